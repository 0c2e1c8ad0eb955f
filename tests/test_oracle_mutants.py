"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (the mistakes live only in a temporary copy; the
oracle itself is untouched)."""
import os
import tempfile

import pytest

import oracle as O
from oracle_pins import ALL_PINS

SRC = open(O._SRC).read()

MUTANTS = {
    "dropped indexer weight": ("s += (int64_t)wI[h] * dot;", "s += dot;"),
    "indexer head/channel transposed": ("qI[((b * Tq + t) * H_I + h) * D_I + c]", "qI[((b * Tq + t) * D_I + c) * H_I + h]"),
    "diagonal left out of the prefix": ("long n = q_offset + t + 1;", "long n = q_offset + t;"),
    "ties go to the higher position": ("return (a->j < b->j) ? -1 : (a->j > b->j);", "return (a->j > b->j) ? -1 : (a->j < b->j);"),
    "score order flipped": ("return (a->s > b->s) ? -1 : 1;", "return (a->s < b->s) ? -1 : 1;"),
    "index set not sorted ascending": ("int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;\n    return (a < b) ? -1 : (a > b);",
                                       "int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;\n    return (a > b) ? -1 : (a < b);"),
    "wrong key/value head": ("int kh = h / G;", "int kh = h % Hkv;"),
    "scale dropped": ("logit[i] = dot * scale;", "logit[i] = dot;"),
    "gate sides swapped": ("oc = gh * oc + (1.0 - gh) * bf16_to_double(lrow[c]);", "oc = (1.0 - gh) * oc + gh * bf16_to_double(lrow[c]);"),
    "gate applied to full heads": ("if (!full && g != NULL && lrow != NULL)", "if (g != NULL && lrow != NULL)"),
    "lse misses the max": ("lse[r * Hq + h] = m + log(den);", "lse[r * Hq + h] = log(den);"),
    "value row from the key cache": ("const uint16_t *vrow = v + ", "const uint16_t *vrow = k + "),
    "full heads skip the diagonal": ("nk = p + 1;\n                for (long j = 0; j < nk; j++)", "nk = p;\n                for (long j = 0; j < nk; j++)"),
    "threshold form from the (K+1)-th position": ("const scored_pos kth = order[K - 1];",
                                                  "const scored_pos kth = order[K];"),
    "threshold form of a whole prefix off by one": ("tr[1] = (int32_t)p;",
                                                    "tr[1] = (int32_t)(p + 1);"),
    "per-head threshold form scored by every head": ("const int scored_head = per_head ? set : -1;",
                                                      "const int scored_head = -1;"),
    "ReLU not applied": ("if (relu && dot < 0) dot = 0;", ";"),
    "ReLU clamps the weighted sum instead of each head": ("if (relu && dot < 0) dot = 0;", "if (relu && dot < 0 && H_I == 1) dot = 0;"),
    "per-head score weighted": ("if (head >= 0) s += dot;", "if (head >= 0) s += (int64_t)wI[h] * dot;"),
    "per-head set scored by every head": ("if (head >= 0 && h != head) continue;", ";"),
    "query head reads the wrong set": ("long set = r * nsets + h / (Hq / nsets);", "long set = r * nsets + h % nsets;"),
    "router sums instead of averaging": ("x[c] = Tk > 0 ? acc / (double)Tk : 0.0;", "x[c] = acc;"),
    "router without its ReLU": ("hid[f] = acc > 0.0 ? acc : 0.0;", "hid[f] = acc;"),
    "router decision flipped": ("route[b * Hq + h] = (uint8_t)(z[1] >= z[0] ? 1 : 0);", "route[b * Hq + h] = (uint8_t)(z[0] >= z[1] ? 1 : 0);"),
    "router ties go full": ("route[b * Hq + h] = (uint8_t)(z[1] >= z[0] ? 1 : 0);", "route[b * Hq + h] = (uint8_t)(z[1] > z[0] ? 1 : 0);"),
    "KDA forgets along value channels": ("for (int c = 0; c < Dv; c++) S[i * Dv + c] *= (double)at[i];",
                                         "for (int c = 0; c < Dv; c++) S[i * Dv + c] *= (double)at[c % Dk];"),
    "KDA forgetting left out": ("for (int c = 0; c < Dv; c++) S[i * Dv + c] *= (double)at[i];", ";"),
    "KDA erase without beta": ("S[i * Dv + c] += bt * bf16_to_double(kt[i]) * (bf16_to_double(vt[c]) - u[c]);",
                               "S[i * Dv + c] += bf16_to_double(kt[i]) * (bt * bf16_to_double(vt[c]) - u[c]);"),
    "KDA adds instead of erasing": ("(bf16_to_double(vt[c]) - u[c])", "(bf16_to_double(vt[c]) + u[c])"),
    "KDA reads out with the key": ("acc += bf16_to_double(qt[i]) * S[i * Dv + c];", "acc += bf16_to_double(kt[i]) * S[i * Dv + c];"),
    "KDA output scale dropped": ("o[row * Dv + c] = scale * acc;", "o[row * Dv + c] = acc;"),
    "KDA initial state transposed": ("(double)state_in[(bh * Dk + i) * Dv + c]", "(double)state_in[(bh * Dv + c) * Dk + i]"),
    "KDA final state not kept": ("state_out[bh * Dk * Dv + e] = S[e];", "state_out[bh * Dk * Dv + e] = 0.0;"),
    "KDA heads mixed up": ("const long row = (b * T + t) * H + h;", "const long row = (b * T + t) * H + (H - 1 - h);"),
    "KDA reads out before the write": (
        "acc += bf16_to_double(qt[i]) * S[i * Dv + c];",
        "acc += bf16_to_double(qt[i]) * (S[i * Dv + c] - bt * bf16_to_double(kt[i]) * (bf16_to_double(vt[c]) - u[c]));"),
    "router reads the first position only": ("for (long j = 0; j < Tk; j++) acc += bf16_to_double(k[(b * Tk + j) * C + c]);", "for (long j = 0; j < 1; j++) acc += bf16_to_double(k[(b * Tk + j) * C + c]) * (double)Tk;"),
}


def _caught(lib):
    for pin in ALL_PINS:
        try:
            pin(lib)
        except Exception:
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name):
    old, new = MUTANTS[name]
    assert SRC.count(old) == 1, f"mutation site not unique: {name}"
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "mutant.c")
        with open(src, "w") as f:
            f.write(SRC.replace(old, new))
        so = O.build(src=src, out=os.path.join(d, "libmutant.so"))
        assert _caught(O.lib(so)), f"no pin catches: {name}"
