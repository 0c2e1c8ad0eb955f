"""Pins that tie the CPU oracle to something other than itself.

Each ``pin_*`` function takes a compiled oracle handle (``oracle.lib()`` or a
deliberately broken copy built by the mutation tests) and raises
AssertionError when the oracle disagrees with:
  * the hand-worked example in ``tests/golden/indexer_tiny.txt``;
  * brute force on tiny inputs (the counting definition of top-K);
  * library routines (numpy int64 einsum, numpy lexsort, torch fp64
    scaled_dot_product_attention with a causal or explicit mask);
  * closed forms and invariants (t=0 gives v_0, V=1 gives 1, softmax sums to
    one, permutation invariance, gate end points and affinity, needles);
  * for the KDA linear branch: the hand-worked tests/golden/kda_tiny.txt, the
    full transition-matrix form, the delta rule's retrieval invariant, basis
    keys (per-row moving averages), orthonormal keys without forgetting
    (causal linear attention) and state chaining.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch

import esa_inputs as E
import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "indexer_tiny.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def _bf16_f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def _small(seed=11, **over):
    cfg = E.small_config(seed=seed, **over)
    return cfg, E.shape_of(cfg), E.make_inputs(cfg)


def _sdpa_masked(inp, shape, allowed, rows):
    """fp64 torch SDPA for the listed flat rows with boolean mask allowed[r, j]."""
    B, Tq, Hq, Hkv, D = shape["B"], shape["Tq"], shape["Hq"], shape["Hkv"], shape["D"]
    G = Hq // Hkv
    q = _bf16_f64(inp["q"]).reshape(B * Tq, Hq, D)[torch.as_tensor(rows)]
    out = torch.empty(len(rows), Hq, D, dtype=torch.float64)
    lse = torch.empty(len(rows), Hq, dtype=torch.float64)
    for i, r in enumerate(rows):
        b = r // Tq
        k = _bf16_f64(inp["k"][b]).repeat_interleave(G, dim=1).transpose(0, 1)  # [Hq, Tk, D]
        v = _bf16_f64(inp["v"][b]).repeat_interleave(G, dim=1).transpose(0, 1)
        m = torch.as_tensor(allowed[i])[None, None, :]
        o = torch.nn.functional.scaled_dot_product_attention(q[i][:, None, :], k, v, attn_mask=m)
        out[i] = o[:, 0, :]
        logits = (q[i][:, None, :] @ k.transpose(-1, -2))[:, 0, :] / math.sqrt(D)
        lse[i] = torch.logsumexp(logits.masked_fill(~m[0], -math.inf), dim=-1)
    return out.numpy(), lse.numpy()


# ---------------------------------------------------------------- indexer
def pin_indexer_golden(L):
    gv = _golden()
    qI = np.array(gv["qI"], dtype=np.int8).reshape(1, 3, 2, 3)
    kI = np.array(gv["kI"], dtype=np.int8).reshape(1, 3, 3)
    w = np.array(gv["w"], dtype=np.int32)
    sh = dict(B=1, Tq=3, Tk=3, q_offset=0, Hq=1, Hkv=1, D=64, H_I=2, D_I=3)
    for t in range(3):
        got = O.indexer_row(qI, kI, w, sh, 0, t, L=L)
        assert got.tolist() == gv[f"scores_t{t}"], (t, got)
    idx1, _ = O.topk(qI, kI, w, sh, 1, L=L)
    assert idx1.reshape(-1).tolist() == gv["top1"], idx1
    idx2, cnt2 = O.topk(qI, kI, w, sh, 2, L=L)
    assert idx2.reshape(-1).tolist() == gv["top2"], idx2
    assert cnt2.tolist() == gv["cnt2"], cnt2


def pin_indexer_numpy(L, seed=3):
    rng = np.random.default_rng(seed)
    for (B, Tq, Tk, qo, HI, DI) in [(2, 5, 9, 4, 3, 16), (1, 1, 40, 39, 1, 64), (3, 7, 7, 0, 4, 8)]:
        qI = rng.integers(-128, 128, (B, Tq, HI, DI), dtype=np.int8)
        kI = rng.integers(-128, 128, (B, Tk, DI), dtype=np.int8)
        w = rng.integers(-3, 5, HI).astype(np.int32)
        sh = dict(B=B, Tq=Tq, Tk=Tk, q_offset=qo, Hq=1, Hkv=1, D=64, H_I=HI, D_I=DI)
        ref = np.einsum("bthc,bjc,h->btj", qI.astype(np.int64), kI.astype(np.int64), w.astype(np.int64))
        for b in range(B):
            for t in range(Tq):
                got = O.indexer_row(qI, kI, w, sh, b, t, L=L)
                assert np.array_equal(got, ref[b, t, :qo + t + 1]), (b, t)


def pin_indexer_onehot(L):
    rng = np.random.default_rng(5)
    kI = rng.integers(-8, 8, (1, 12, 8), dtype=np.int8)
    for h, c, w in [(0, 3, 1), (2, 7, 4), (1, 0, 2)]:
        qI = np.zeros((1, 12, 3, 8), dtype=np.int8)
        qI[0, 11, h, c] = 1
        wv = np.array([1, 2, 4], dtype=np.int32)
        sh = dict(B=1, Tq=12, Tk=12, q_offset=0, Hq=1, Hkv=1, D=64, H_I=3, D_I=8)
        got = O.indexer_row(qI, kI, wv, sh, 0, 11, L=L)
        assert np.array_equal(got, wv[h] * kI[0, :, c].astype(np.int32)), (h, c, w)


def pin_indexer_bound(L):
    cfg, sh, inp = _small(seed=21, Tq=32, Tk=32, H_I=4, D_I=64, weights="1to4")
    bound = int(inp["wI"].abs().sum()) * 64 * 64
    for t in (0, 15, 31):
        s = O.indexer_row(inp["qI"], inp["kI"], inp["wI"], sh, 0, t, L=L)
        assert np.abs(s).max() <= bound


# ---------------------------------------------------------------- top-K
def _topk_bruteforce(s: np.ndarray, K: int):
    """Counting definition: j is kept iff fewer than K positions beat it
    (higher score, or equal score at a lower position)."""
    n = len(s)
    keep = [j for j in range(n) if sum(1 for i in range(n) if s[i] > s[j] or (s[i] == s[j] and i < j)) < K]
    return keep


def pin_topk_bruteforce(L, seed=9):
    rng = np.random.default_rng(seed)
    for trial in range(6):
        B, Tq, Tk, qo = 2, 6, 30, 24
        DI = 4
        qI = rng.integers(-2, 2, (B, Tq, 1, DI), dtype=np.int8)  # small range: many ties
        kI = rng.integers(-2, 2, (B, Tk, DI), dtype=np.int8)
        w = np.ones(1, dtype=np.int32)
        sh = dict(B=B, Tq=Tq, Tk=Tk, q_offset=qo, Hq=1, Hkv=1, D=64, H_I=1, D_I=DI)
        K = [1, 3, 7, 25, 26, 40][trial]
        idx, cnt = O.topk(qI, kI, w, sh, K, L=L)
        for r in range(B * Tq):
            b, t = divmod(r, Tq)
            s = O.indexer_row(qI, kI, w, sh, b, t, L=L)
            keep = _topk_bruteforce(s, K)
            assert cnt[r] == len(keep) == min(K, qo + t + 1)
            assert idx[r, :cnt[r]].tolist() == keep, (trial, r)
            assert (idx[r, cnt[r]:] == -1).all()


def pin_threshold_form(L, seed=23):
    """The threshold form (T, P) of a row's set: the hand-worked rows of the
    golden file, then on tie-heavy rows the set it describes
    ({j : s_j > T or (s_j == T and j <= P)}) equals the brute-force counting
    set, T equals the K-th largest score (numpy sort) and s_P == T; whole
    prefixes give (INT32_MIN, p)."""
    gv = _golden()
    qI = np.array(gv["qI"], dtype=np.int8).reshape(1, 3, 2, 3)
    kI = np.array(gv["kI"], dtype=np.int8).reshape(1, 3, 3)
    w = np.array(gv["w"], dtype=np.int32)
    sh = dict(B=1, Tq=3, Tk=3, q_offset=0, Hq=1, Hkv=1, D=64, H_I=2, D_I=3)
    for K in (1, 2):
        thr = O.threshold(qI, kI, w, sh, K, L=L)
        assert thr.reshape(-1).tolist() == gv[f"thr{K}"], (K, thr)
    rng = np.random.default_rng(seed)
    imin = np.iinfo(np.int32).min
    for trial in range(6):
        B, Tq, Tk, qo, DI = 2, 6, 30, 24, 4
        qI = rng.integers(-2, 2, (B, Tq, 1, DI), dtype=np.int8)  # small range: many ties
        kI = rng.integers(-2, 2, (B, Tk, DI), dtype=np.int8)
        w = np.ones(1, dtype=np.int32)
        sh = dict(B=B, Tq=Tq, Tk=Tk, q_offset=qo, Hq=1, Hkv=1, D=64, H_I=1, D_I=DI)
        K = [1, 2, 5, 24, 25, 31][trial]
        thr = O.threshold(qI, kI, w, sh, K, L=L)
        for r in range(B * Tq):
            b, t = divmod(r, Tq)
            s = O.indexer_row(qI, kI, w, sh, b, t, L=L)
            T, P = int(thr[r, 0]), int(thr[r, 1])
            n = len(s)
            if n <= K:
                assert (T, P) == (imin, n - 1), (trial, r, T, P)
                continue
            assert T == int(np.sort(s)[::-1][K - 1]) and int(s[P]) == T, (trial, r, T, P)
            described = [j for j in range(n) if s[j] > T or (s[j] == T and j <= P)]
            assert described == _topk_bruteforce(s, K), (trial, r)


def pin_threshold_form_per_head(L, seed=29):
    """With per-head sets (and the ReLU), each set's threshold form equals
    the one-set threshold form of the query sliced to that indexer head
    (weight 1)."""
    cfg, sh, inp = _small(seed=seed, Tq=40, Tk=40, H_I=3, D_I=16, top_k=9, weights="1to4")
    for flags in (2, 3):
        shp = dict(sh, flags=flags)
        thr = O.threshold(inp["qI"], inp["kI"], inp["wI"], shp, 9, L=L)
        assert thr.shape == (40, 3, 2)
        for hh in range(3):
            one = dict(sh, H_I=1, flags=flags & 1)
            ref = O.threshold(inp["qI"][:, :, hh:hh + 1].contiguous(), inp["kI"], np.ones(1, np.int32), one, 9, L=L)
            assert np.array_equal(thr[:, hh], ref), (flags, hh)


def pin_topk_lexsort(L, seed=13):
    cfg, sh, inp = _small(seed=seed, Tq=48, Tk=48, H_I=2, D_I=16, top_k=20, weights="1to4")
    K = 20
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
    qI = inp["qI"].numpy().astype(np.int64)
    kI = inp["kI"].numpy().astype(np.int64)
    w = inp["wI"].numpy().astype(np.int64)
    for t in range(48):
        s = np.einsum("hc,jc,h->j", qI[0, t], kI[0, :t + 1], w)
        order = np.lexsort((np.arange(t + 1), -s))  # score desc, then position asc
        ref = np.sort(order[:K])
        assert idx[t, :cnt[t]].tolist() == ref.tolist(), t


def pin_topk_special(L):
    cfg, sh, inp = _small(seed=17, Tq=40, Tk=40, D_I=32)
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 64, L=L)  # K >= every prefix
    for t in range(40):
        assert cnt[t] == t + 1
        assert idx[t, :t + 1].tolist() == list(range(t + 1))
        assert (idx[t, t + 1:] == -1).all()
    kz = torch.zeros_like(inp["kI"])  # all scores equal: the first K positions win
    idx, cnt = O.topk(inp["qI"], kz, inp["wI"], sh, 5, L=L)
    for t in range(40):
        assert idx[t, :cnt[t]].tolist() == list(range(min(5, t + 1)))


def pin_topk_needles(L):
    cfg = E.small_config(B=1, Tq=1, Tk=16384, q_offset=16383, Hq=4, Hkv=1, D=64, H_I=1, D_I=64,
                         top_k=256, needles=64, seed=2005)
    inp = E.make_inputs(cfg)
    sh = E.shape_of(cfg)
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 256, L=L)
    assert set(inp["needles"].tolist()) <= set(idx[0].tolist())


# ---------------------------------------------------------------- attention
def pin_attention_full_is_sdpa(L):
    for over in [dict(Tq=33, Tk=33, Hq=4, Hkv=1, D=64), dict(Tq=20, Tk=20, Hq=8, Hkv=2, D=128),
                 dict(B=2, Tq=5, Tk=29, q_offset=24, Hq=6, Hkv=3, D=64)]:
        cfg, sh, inp = _small(seed=23, **over)
        K = sh["Tk"]
        rows = list(range(sh["B"] * sh["Tq"]))
        idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
        out, lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, L=L)
        allowed = np.array([[j <= sh["q_offset"] + r % sh["Tq"] for j in range(sh["Tk"])] for r in rows])
        ref, ref_lse = _sdpa_masked(inp, sh, allowed, rows)
        assert np.abs(out - ref).max() < 1e-12, np.abs(out - ref).max()
        assert np.abs(lse - ref_lse).max() < 1e-12
        if sh["q_offset"] == 0:  # also the library's own causal flag
            B, Tq, Hq, Hkv, D = sh["B"], sh["Tq"], sh["Hq"], sh["Hkv"], sh["D"]
            G = Hq // Hkv
            q = _bf16_f64(inp["q"]).permute(0, 2, 1, 3)
            k = _bf16_f64(inp["k"]).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
            v = _bf16_f64(inp["v"]).repeat_interleave(G, dim=2).permute(0, 2, 1, 3)
            o = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
            assert np.abs(out - o.permute(0, 2, 1, 3).reshape(B * Tq, Hq, D).numpy()).max() < 1e-12


def pin_attention_sparse_is_masked_sdpa(L):
    cfg, sh, inp = _small(seed=29, Tq=40, Tk=40, Hq=8, Hkv=2, D=64, D_I=16)
    K = 9
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
    out, lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, L=L)
    rows = list(range(40))
    allowed = np.zeros((40, 40), dtype=bool)
    for r in rows:
        allowed[r, idx[r, :cnt[r]]] = True
    ref, ref_lse = _sdpa_masked(inp, sh, allowed, rows)
    assert np.abs(out - ref).max() < 1e-12
    assert np.abs(lse - ref_lse).max() < 1e-12


def pin_attention_closed_forms(L):
    cfg, sh, inp = _small(seed=31, Tq=16, Tk=16, Hq=4, Hkv=2, D=64)
    K = 6
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
    out, lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, L=L)
    v0 = _bf16_f64(inp["v"][0, 0]).numpy()  # [Hkv, D]
    for h in range(4):
        assert np.array_equal(out[0, h], v0[h // 2])  # row 0 attends to key 0 alone
        assert lse[0, h] == _bf16_f64(inp["q"][0, 0, h]).dot(_bf16_f64(inp["k"][0, 0, h // 2])).item() / 8.0
    ones = torch.ones_like(inp["v"])
    o1, _ = O.attention(inp["q"], inp["k"], ones, idx, cnt, sh, K, L=L)
    assert np.abs(o1 - 1.0).max() < 1e-14
    perm = idx.copy()
    rng = np.random.default_rng(0)
    for r in range(16):
        perm[r, :cnt[r]] = rng.permutation(perm[r, :cnt[r]])
    op, lp = O.attention(inp["q"], inp["k"], inp["v"], perm, cnt, sh, K, L=L)
    assert np.abs(op - out).max() < 1e-13 and np.abs(lp - lse).max() < 1e-13
    # softmax over the selected keys sums to one: sum_j exp(logit_j - lse) = 1
    q = _bf16_f64(inp["q"][0])
    k = _bf16_f64(inp["k"][0])
    for r in (3, 9, 15):
        for h in range(4):
            sel = torch.as_tensor(idx[r, :cnt[r]], dtype=torch.long)
            logits = (k[sel, h // 2] @ q[r, h]) / 8.0
            assert abs(torch.exp(logits - lse[r, h]).sum().item() - 1.0) < 1e-13


def pin_empty_set(L):
    """cnt = 0: no key is attended: o = 0, lse = -inf, gated out = (1-g) lin."""
    cfg, sh, inp = _small(seed=43, Tq=8, Tk=8, Hq=2, Hkv=1, D=64)
    K = 4
    idx = np.full((8, K), -1, dtype=np.int32)
    cnt = np.zeros(8, dtype=np.int32)
    o, lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, L=L)
    assert (o == 0).all() and np.isneginf(lse).all()
    og, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"], L=L)
    lin = _bf16_f64(inp["lin"]).reshape(8, 2, 64).numpy()
    g = inp["g"].double().numpy()
    assert np.array_equal(og, (1.0 - g)[None, :, None] * lin)


def pin_gate(L):
    cfg, sh, inp = _small(seed=37, Tq=24, Tk=24, Hq=4, Hkv=1, D=64)
    K = 7
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
    plain, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, L=L)
    lin = _bf16_f64(inp["lin"]).reshape(24, 4, 64).numpy()
    g0, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=torch.zeros(4), lin=inp["lin"], L=L)
    g1, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=torch.ones(4), lin=inp["lin"], L=L)
    assert np.array_equal(g0, lin)  # g = 0 gives the linear branch exactly
    assert np.array_equal(g1, plain)  # g = 1 gives the sparse attention exactly
    gv = torch.tensor([0.25, 0.5, 0.75, 0.125])
    gm, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=gv, lin=inp["lin"], L=L)
    for h in range(4):  # affine in g between the two end points
        ref = g0[:, h] + gv[h].item() * (g1[:, h] - g0[:, h])
        assert np.abs(gm[:, h] - ref).max() < 1e-12


def pin_routing(L):
    cfg, sh, inp = _small(seed=41, B=2, Tq=20, Tk=20, Hq=4, Hkv=4, D=64, routed=True)
    K = 5
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K, L=L)
    rows = list(range(40))
    full = torch.zeros(2, 4, dtype=torch.uint8)
    of, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"], route=full, L=L)
    allowed = np.array([[j <= r % 20 for j in range(20)] for r in rows])
    ref, _ = _sdpa_masked(inp, sh, allowed, rows)
    assert np.abs(of - ref).max() < 1e-12  # full heads: causal attention, no gate
    sparse = torch.ones(2, 4, dtype=torch.uint8)
    osp, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"], route=sparse, L=L)
    ou, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"], L=L)
    assert np.array_equal(osp, ou)
    mixed = torch.tensor([[1, 0, 1, 0], [0, 0, 1, 1]], dtype=torch.uint8)
    om, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"], route=mixed, L=L)
    for b in range(2):
        for h in range(4):
            src = osp if mixed[b, h] else of
            assert np.array_equal(om[b * 20:(b + 1) * 20, h], src[b * 20:(b + 1) * 20, h])


def pin_needles_closed_form(L):
    cfg = E.small_config(B=1, Tq=1, Tk=16384, q_offset=16383, Hq=4, Hkv=1, D=128, H_I=1, D_I=64,
                         top_k=256, needles=64, seed=2005)
    inp = E.make_inputs(cfg)
    sh = E.shape_of(cfg)
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 256, L=L)
    out, _ = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, 256, L=L)
    # head 0's query meets 64 identical needle keys 4*q: their logits sit ~40
    # above the rest, so the output is the plain mean of the needles' values.
    vmean = _bf16_f64(inp["v"][0, torch.as_tensor(inp["needles"]), 0]).mean(0).numpy()
    assert np.abs(out[0, 0] - vmean).max() < 1e-9



# ------------------------------------------------------------------ indexer options: ReLU, per-head sets
def _golden_example():
    gv = _golden()
    qI = np.array(gv["qI"], dtype=np.int8).reshape(1, 3, 2, 3)
    kI = np.array(gv["kI"], dtype=np.int8).reshape(1, 3, 3)
    w = np.array(gv["w"], dtype=np.int32)
    sh = dict(B=1, Tq=3, Tk=3, q_offset=0, Hq=2, Hkv=1, D=64, H_I=2, D_I=3, flags=0)
    return gv, qI, kI, w, sh


def pin_indexer_modes_golden(L):
    """The hand-worked example of tests/golden/indexer_tiny.txt with the ReLU
    per head and with one index set per head."""
    gv, qI, kI, w, sh = _golden_example()
    assert O.indexer_row(qI, kI, w, sh, 0, 2, L=L, relu=True).tolist() == gv["relu_scores_t2"]
    rs = dict(sh, flags=O.RELU)
    assert O.topk(qI, kI, w, rs, 1, L=L)[0].reshape(-1).tolist() == gv["relu_top1"]
    assert O.topk(qI, kI, w, rs, 2, L=L)[0].reshape(-1).tolist() == gv["relu_top2"]
    heads = O.indexer_row(qI, kI, w, sh, 0, 2, L=L, head=0).tolist() + \
        O.indexer_row(qI, kI, w, sh, 0, 2, L=L, head=1).tolist()
    assert heads == gv["head_scores_t2"], heads
    ph = dict(sh, flags=O.PER_HEAD)
    idx, cnt = O.topk(qI, kI, w, ph, 2, L=L)
    assert idx.shape == (3, 2, 2) and cnt.shape == (3, 2)
    assert idx.reshape(-1).tolist() == gv["head_top2"], idx
    assert cnt.reshape(-1).tolist() == gv["head_cnt2"], cnt
    idx, _ = O.topk(qI, kI, w, dict(sh, flags=O.PER_HEAD | O.RELU), 2, L=L)
    assert idx[2].reshape(-1).tolist() == gv["head_relu_top2_t2"], idx[2]


def pin_relu_special_and_numpy(L, seed=19):
    """ReLU indexer: equal to the linear one when every head's dot product is
    >= 0; all scores 0 (so the first K positions) when every one is <= 0;
    and numpy's elementwise maximum of int64 einsum products elsewhere."""
    rng = np.random.default_rng(seed)
    B, Tq, Tk, HI, DI = 1, 6, 30, 3, 16
    sh = dict(B=B, Tq=Tq, Tk=Tk, q_offset=Tk - Tq, Hq=1, Hkv=1, D=64, H_I=HI, D_I=DI, flags=0)
    w = np.array([2, 1, 3], dtype=np.int32)
    qpos = rng.integers(0, 8, (B, Tq, HI, DI), dtype=np.int8)
    kpos = rng.integers(0, 8, (B, Tk, DI), dtype=np.int8)
    kneg = -kpos
    for t in range(Tq):
        assert np.array_equal(O.indexer_row(qpos, kpos, w, sh, 0, t, L=L, relu=True),
                              O.indexer_row(qpos, kpos, w, sh, 0, t, L=L)), t
        assert not O.indexer_row(qpos, kneg, w, sh, 0, t, L=L, relu=True).any(), t
    K = 7
    idx, cnt = O.topk(qpos, kneg, w, dict(sh, flags=O.RELU), K, L=L)
    assert (idx == np.arange(K)[None, :]).all() and (cnt == K).all()
    qI = rng.integers(-128, 128, (2, 5, HI, DI), dtype=np.int8)
    kI = rng.integers(-128, 128, (2, 11, DI), dtype=np.int8)
    sh2 = dict(B=2, Tq=5, Tk=11, q_offset=6, Hq=1, Hkv=1, D=64, H_I=HI, D_I=DI, flags=0)
    dots = np.einsum("bthc,bjc->bthj", qI.astype(np.int64), kI.astype(np.int64))
    ref = np.einsum("bthj,h->btj", np.maximum(dots, 0), w.astype(np.int64))
    for b in range(2):
        for t in range(5):
            assert np.array_equal(O.indexer_row(qI, kI, w, sh2, b, t, L=L, relu=True), ref[b, t, :7 + t]), (b, t)


def pin_per_head_sets_are_sliced_queries(L):
    """One index set per indexer head: head h's set equals the one-set
    selection of the query sliced to head h with weight 1 (and the same with
    the ReLU, which on one head clamps its negative scores to 0)."""
    cfg, sh, inp = _small(seed=47, B=2, Tq=20, Tk=40, q_offset=20, H_I=3, D_I=16, top_k=9, weights="1to4")
    K = 9
    for flags in (O.PER_HEAD, O.PER_HEAD | O.RELU):
        idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], dict(sh, flags=flags), K, L=L)
        for h in range(3):
            q1 = inp["qI"][:, :, h:h + 1, :].contiguous()
            one = dict(sh, H_I=1, flags=flags & O.RELU)
            i1, c1 = O.topk(q1, inp["kI"], np.array([1], dtype=np.int32), one, K, L=L)
            assert np.array_equal(idx[:, h], i1) and np.array_equal(cnt[:, h], c1), (flags, h)


def pin_per_head_attention_uses_its_set(L):
    """With one index set per indexer head, query head h's output equals the
    one-set attention given head h's set (query head h reads set h // (Hq // H_I))."""
    cfg, sh, inp = _small(seed=53, Tq=24, Tk=24, Hq=8, Hkv=2, D=64, H_I=4, D_I=16, top_k=6)
    K = 6
    ph = dict(sh, flags=O.PER_HEAD)
    idx, cnt = O.topk(inp["qI"], inp["kI"], inp["wI"], ph, K, L=L)
    out, lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, ph, K, g=inp["g"], lin=inp["lin"], L=L)
    for s in range(4):
        o1, l1 = O.attention(inp["q"], inp["k"], inp["v"], idx[:, s], cnt[:, s], dict(sh, flags=0), K,
                             g=inp["g"], lin=inp["lin"], L=L)
        for h in range(2 * s, 2 * s + 2):
            assert np.array_equal(out[:, h], o1[:, h]) and np.array_equal(lse[:, h], l1[:, h]), (s, h)


# ------------------------------------------------------------------ attention router
ROUTER_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "router_tiny.txt")


def pin_router_golden(L):
    """The hand-worked router example of tests/golden/router_tiny.txt."""
    gv = {}
    for line in open(ROUTER_GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            key, *rest = line.split()
            gv[key] = [float(x) for x in rest]
    k = torch.tensor(gv["k"], dtype=torch.float32).to(torch.bfloat16).reshape(1, 2, 1, 2)
    sh = dict(B=1, Tk=2, Hkv=1, D=2, Hq=2)
    W1 = np.array(gv["W1"], dtype=np.float32).reshape(2, 2)
    W2 = np.array(gv["W2"], dtype=np.float32).reshape(4, 2)
    route, margin = O.route_heads(k, sh, W1, np.array(gv["b1"], np.float32), W2, np.array(gv["b2"], np.float32), L=L)
    assert route.reshape(-1).tolist() == [int(x) for x in gv["route"]], route
    assert np.allclose(margin.reshape(-1), gv["margin"], atol=0, rtol=0), margin


def _router_case(seed, B=2, Tk=37, Hkv=2, D=16, Hq=4, F=8):
    rng = np.random.default_rng(seed)
    k = torch.from_numpy(rng.standard_normal((B, Tk, Hkv, D)).astype(np.float32) + 0.5).to(torch.bfloat16)
    C = Hkv * D
    W = dict(W1=rng.standard_normal((F, C)).astype(np.float32), b1=rng.standard_normal(F).astype(np.float32),
             W2=rng.standard_normal((2 * Hq, F)).astype(np.float32), b2=rng.standard_normal(2 * Hq).astype(np.float32))
    return k, dict(B=B, Tk=Tk, Hkv=Hkv, D=D, Hq=Hq), W


def pin_router_numpy(L):
    """numpy: mean over positions, matrix products, elementwise maximum."""
    for seed in (1, 2, 3):
        k, sh, W = _router_case(seed)
        route, margin = O.route_heads(k, sh, W["W1"], W["b1"], W["W2"], W["b2"], L=L)
        x = k.to(torch.float64).numpy().reshape(sh["B"], sh["Tk"], -1).mean(axis=1)
        hid = np.maximum(x @ W["W1"].astype(np.float64).T + W["b1"], 0.0)
        z = (hid @ W["W2"].astype(np.float64).T + W["b2"]).reshape(sh["B"], sh["Hq"], 2)
        assert np.allclose(margin, z[..., 1] - z[..., 0], rtol=1e-12, atol=1e-12)
        assert np.array_equal(route, (z[..., 1] >= z[..., 0]).astype(np.uint8))


def pin_router_closed_forms(L):
    """W1 = 0: hid = max(0, b1) whatever the keys; equal full and sparse rows
    tie and go sparse; permuting the cached positions changes nothing."""
    k, sh, W = _router_case(7)
    W0 = dict(W, W1=np.zeros_like(W["W1"]))
    r0, m0 = O.route_heads(k, sh, W0["W1"], W0["b1"], W0["W2"], W0["b2"], L=L)
    hid = np.maximum(W["b1"].astype(np.float64), 0.0)
    z = (W["W2"].astype(np.float64) @ hid + W["b2"]).reshape(sh["Hq"], 2)
    assert np.allclose(m0, np.broadcast_to(z[:, 1] - z[:, 0], m0.shape), rtol=1e-12, atol=1e-12)
    Wt = dict(W)
    Wt["W2"] = np.repeat(W["W2"][0::2], 2, axis=0)
    Wt["b2"] = np.repeat(W["b2"][0::2], 2)
    rt, mt = O.route_heads(k, sh, Wt["W1"], Wt["b1"], Wt["W2"], Wt["b2"], L=L)
    assert (mt == 0).all() and (rt == 1).all()
    perm = torch.from_numpy(np.random.default_rng(8).permutation(sh["Tk"]))
    r1, m1 = O.route_heads(k, sh, W["W1"], W["b1"], W["W2"], W["b2"], L=L)
    r2, m2 = O.route_heads(k[:, perm].contiguous(), sh, W["W1"], W["b1"], W["W2"], W["b2"], L=L)
    assert np.allclose(m1, m2, rtol=1e-12, atol=1e-12) and np.array_equal(r1, r2)

KDA_GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kda_tiny.txt")


def _bf(x) -> torch.Tensor:
    return torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)


def pin_kda_golden(L):
    """The two hand-worked KDA examples of tests/golden/kda_tiny.txt."""
    gv = {}
    for line in open(KDA_GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            key, *rest = line.split()
            gv[key] = [float(x) for x in rest]
    o, st = O.kda(_bf(gv["c1_q"]).reshape(1, 2, 1, 2), _bf(gv["c1_k"]).reshape(1, 2, 1, 2),
                  _bf(gv["c1_v"]).reshape(1, 2, 1, 1), np.float32(gv["c1_alpha"]).reshape(1, 2, 1, 2),
                  np.float32(gv["c1_beta"]).reshape(1, 2, 1), scale=1.0, L=L)
    assert o.reshape(-1).tolist() == gv["c1_o"], o
    assert st.reshape(-1).tolist() == gv["c1_state"], st
    o, st = O.kda(_bf(gv["c2_q"]).reshape(1, 1, 1, 2), _bf(gv["c2_k"]).reshape(1, 1, 1, 2),
                  _bf(gv["c2_v"]).reshape(1, 1, 1, 2), np.float32(gv["c2_alpha"]).reshape(1, 1, 1, 2),
                  np.float32(gv["c2_beta"]).reshape(1, 1, 1), state_in=np.float32(gv["c2_state_in"]).reshape(1, 1, 2, 2),
                  scale=0.5, L=L)
    assert o.reshape(-1).tolist() == gv["c2_o"], o
    assert st.reshape(-1).tolist() == gv["c2_state"], st


def _kda_case(seed, B=2, T=12, H=3, Dk=8, Dv=5, state=True):
    rng = np.random.default_rng(seed)
    q = _bf(rng.standard_normal((B, T, H, Dk)) / math.sqrt(Dk))
    k = rng.standard_normal((B, T, H, Dk))
    k = _bf(k / np.linalg.norm(k, axis=-1, keepdims=True))
    v = _bf(rng.standard_normal((B, T, H, Dv)))
    alpha = rng.uniform(0.5, 1.0, (B, T, H, Dk)).astype(np.float32)
    beta = rng.uniform(0.0, 1.0, (B, T, H)).astype(np.float32)
    s0 = rng.standard_normal((B, H, Dk, Dv)).astype(np.float32) if state else None
    return q, k, v, alpha, beta, s0


def _f64(x):
    return (x.to(torch.float64).numpy() if isinstance(x, torch.Tensor) else np.asarray(x, dtype=np.float64))


def pin_kda_transition_matrices(L):
    """numpy matrix form: S_t = (I - beta_t k_t k_t^T) diag(alpha_t) S_{t-1} +
    beta_t k_t v_t^T, o_t = scale S_t^T q_t, with the transition built as a
    full Dk x Dk matrix per step (Dk != Dv, several heads and sequences)."""
    for seed in (1, 2):
        q, k, v, alpha, beta, s0 = _kda_case(seed)
        o, st = O.kda(q, k, v, alpha, beta, state_in=s0, scale=0.7, L=L)
        qd, kd, vd, ad, bd = (_f64(x) for x in (q, k, v, alpha, beta))
        B, T, H, Dk = qd.shape
        for b in range(B):
            for h in range(H):
                S = _f64(s0[b, h])
                for t in range(T):
                    kk = kd[b, t, h][:, None]
                    A = (np.eye(Dk) - bd[b, t, h] * (kk @ kk.T)) @ np.diag(ad[b, t, h])
                    S = A @ S + bd[b, t, h] * kk @ vd[b, t, h][None, :]
                    assert np.allclose(o[b, t, h], 0.7 * S.T @ qd[b, t, h], rtol=1e-12, atol=1e-12)
                assert np.allclose(st[b, h], S, rtol=1e-12, atol=1e-12)


def pin_kda_retrieval(L):
    """Delta-rule invariant: with beta_t = 1 and a unit key, the state returns
    v_t for k_t right after step t, whatever the forgetting factors and the
    history; so q_t = k_t and scale = 1 give o_t = v_t. The keys are four
    entries of +-1/2 (exactly unit in bf16)."""
    rng = np.random.default_rng(5)
    B, T, H, Dk, Dv = 2, 16, 2, 8, 6
    q, _, v, alpha, beta, s0 = _kda_case(5, B, T, H, Dk, Dv)
    kk = np.zeros((B, T, H, Dk))
    for idx in np.ndindex(B, T, H):
        pos = rng.choice(Dk, 4, replace=False)
        kk[idx][pos] = rng.choice([-0.5, 0.5], 4)
    hit = rng.random((B, T, H)) < 0.5
    beta = np.where(hit, 1.0, beta).astype(np.float32)
    k = _bf(kk)
    qn = torch.where(torch.from_numpy(hit)[..., None], k, q)
    o, _ = O.kda(qn, k, v, alpha, beta, state_in=s0, scale=1.0, L=L)
    assert np.allclose(o[hit], _f64(v)[hit], rtol=0, atol=1e-12), np.abs(o[hit] - _f64(v)[hit]).max()
    assert not np.allclose(o[~hit], _f64(v)[~hit], atol=1e-3)


def pin_kda_basis_keys(L):
    """Keys that are basis vectors e_j make each state row an exponential
    moving average: every row i decays by alpha_t[i]; row j = key(t) becomes
    (1 - beta_t) row + beta_t v_t; o_t = scale sum_i q_t[i] row_i. Keys repeat,
    the initial state is random and Dk != Dv."""
    rng = np.random.default_rng(9)
    B, T, H, Dk, Dv = 2, 14, 2, 6, 4
    q, _, v, alpha, beta, s0 = _kda_case(9, B, T, H, Dk, Dv)
    j = rng.integers(0, Dk, (B, T, H))
    k = torch.nn.functional.one_hot(torch.from_numpy(j), Dk).to(torch.bfloat16)
    o, st = O.kda(q, k, v, alpha, beta, state_in=s0, scale=0.25, L=L)
    qd, vd = _f64(q), _f64(v)
    for b in range(B):
        for h in range(H):
            rows = _f64(s0[b, h]).copy()
            for t in range(T):
                rows *= alpha[b, t, h].astype(np.float64)[:, None]
                jj = j[b, t, h]
                bt = float(beta[b, t, h])
                rows[jj] = (1.0 - bt) * rows[jj] + bt * vd[b, t, h]
                assert np.allclose(o[b, t, h], 0.25 * (qd[b, t, h][:, None] * rows).sum(0), rtol=1e-12, atol=1e-12)
            assert np.allclose(st[b, h], rows, rtol=1e-12, atol=1e-12)


def pin_kda_linear_attention(L):
    """No forgetting (alpha = 1), zero initial state and orthonormal keys (rows
    of a 16 x 16 Hadamard matrix / 4, exact in bf16): nothing stored is ever
    erased, so o_t = scale sum_{j<=t} beta_j (q_t . k_j) v_j — causal linear
    attention (torch einsum under a lower-triangular mask)."""
    rng = np.random.default_rng(13)
    Hd = np.array([[1.0]])
    while Hd.shape[0] < 16:
        Hd = np.block([[Hd, Hd], [Hd, -Hd]])
    B, T, H, Dk, Dv = 2, 16, 2, 16, 7
    q, _, v, _, beta, _ = _kda_case(13, B, T, H, Dk, Dv, state=False)
    kk = np.stack([np.stack([Hd[rng.permutation(16)[:T]] / 4.0 for _ in range(H)], axis=1) for _ in range(B)])
    k = _bf(kk)
    alpha = np.ones((B, T, H, Dk), dtype=np.float32)
    o, _ = O.kda(q, k, v, alpha, beta, scale=0.3, L=L)
    qt, kt, vt = (x.to(torch.float64) for x in (q, k, v))
    att = torch.einsum("bthd,bshd->bhts", qt, kt) * torch.from_numpy(beta.astype(np.float64)).permute(0, 2, 1)[:, :, None, :]
    att = att * torch.tril(torch.ones(T, T, dtype=torch.float64))
    ref = 0.3 * torch.einsum("bhts,bshc->bthc", att, vt)
    assert np.allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


def pin_kda_chunked_form(L):
    """The chunked (matrix) form of the recurrence, chunk by chunk of C steps
    with g_t = prod_{tau <= t} alpha_tau inside the chunk: reads of the
    chunk-start state W = (K*G) S, Z = (Q*G) S; intra-chunk couplings
    A = strictly-lower((K*G)(K/G)^T), B = lower((Q*G)(K/G)^T); writes
    D = (I + diag(beta) A)^{-1} diag(beta) (V - W); outputs scale (Z + B D);
    state g_last * S + ((K/G) * g_last)^T D. Equal to the step-by-step
    recurrence (C = 4, a ragged last chunk, an initial state, Dk != Dv)."""
    q, k, v, alpha, beta, s0 = _kda_case(31, B=2, T=13, H=2, Dk=8, Dv=5)
    o, st = O.kda(q, k, v, alpha, beta, state_in=s0, scale=0.6, L=L)
    qd, kd, vd, ad = (_f64(x) for x in (q, k, v, alpha))
    bd = beta.astype(np.float64)
    B, T, H, _ = qd.shape
    C = 4
    for b in range(B):
        for h in range(H):
            S = s0[b, h].astype(np.float64)
            for c0 in range(0, T, C):
                sl = slice(c0, min(T, c0 + C))
                Kc, Qc, Vc, Ac, bc = kd[b, sl, h], qd[b, sl, h], vd[b, sl, h], ad[b, sl, h], bd[b, sl, h]
                G = np.cumprod(Ac, axis=0)
                Kt, Qt, Ki = Kc * G, Qc * G, Kc / G
                A = np.tril(Kt @ Ki.T, -1)
                Bm = np.tril(Qt @ Ki.T)
                D = np.linalg.solve(np.eye(len(bc)) + bc[:, None] * A, bc[:, None] * (Vc - Kt @ S))
                assert np.allclose(o[b, sl, h], 0.6 * (Qt @ S + Bm @ D), rtol=1e-10, atol=1e-10)
                S = G[-1][:, None] * S + (Ki * G[-1]).T @ D
            assert np.allclose(st[b, h], S, rtol=1e-10, atol=1e-10)


def pin_kda_extreme_gates(L):
    """alpha_t = 0 wipes the state before the write, so
    o_t = scale * beta_t * (q_t . k_t) * v_t whatever came before; beta = 0
    writes nothing, so with alpha = 1 every output reads the initial state:
    o_t = scale * S_0^T q_t."""
    q, k, v, alpha, beta, s0 = _kda_case(21, T=9)
    a0 = alpha.copy()
    a0[:, 4] = 0.0
    o, _ = O.kda(q, k, v, a0, beta, state_in=s0, scale=0.5, L=L)
    qd, kd, vd = _f64(q), _f64(k), _f64(v)
    ref = 0.5 * beta[:, 4].astype(np.float64)[..., None] * (qd[:, 4] * kd[:, 4]).sum(-1)[..., None] * vd[:, 4]
    assert np.allclose(o[:, 4], ref, rtol=1e-12, atol=1e-12)
    o1, st1 = O.kda(q, k, v, np.ones_like(alpha), np.zeros_like(beta), state_in=s0, scale=0.5, L=L)
    ref1 = 0.5 * np.einsum("bhic,bthi->bthc", s0.astype(np.float64), qd)
    assert np.allclose(o1, ref1, rtol=1e-12, atol=1e-12) and np.array_equal(st1, s0.astype(np.float64))


def pin_kda_chaining(L):
    """Running T steps at once equals running the first T1 and then the rest
    from the carried state (chunked prefill, decode); T = 0 hands the initial
    state straight back."""
    q, k, v, alpha, beta, s0 = _kda_case(17, T=20)
    o, st = O.kda(q, k, v, alpha, beta, state_in=s0, L=L)
    o1, st1 = O.kda(q[:, :7], k[:, :7], v[:, :7], alpha[:, :7], beta[:, :7], state_in=s0, L=L)
    o2, st2 = O.kda(q[:, 7:], k[:, 7:], v[:, 7:], alpha[:, 7:], beta[:, 7:], state_in=st1.astype(np.float32), L=L)
    assert np.allclose(o[:, :7], o1, rtol=0, atol=0)
    assert np.allclose(o[:, 7:], o2, rtol=1e-6, atol=1e-6) and np.allclose(st, st2, rtol=1e-6, atol=1e-6)
    _, st0 = O.kda(q[:, :0], k[:, :0], v[:, :0], alpha[:, :0], beta[:, :0], state_in=s0, L=L)
    assert np.array_equal(st0, s0.astype(np.float64))


ALL_PINS = [pin_indexer_golden, pin_indexer_numpy, pin_indexer_onehot, pin_indexer_bound,
            pin_topk_bruteforce, pin_threshold_form, pin_threshold_form_per_head, pin_topk_lexsort, pin_topk_special, pin_topk_needles,
            pin_attention_full_is_sdpa, pin_attention_sparse_is_masked_sdpa, pin_attention_closed_forms,
            pin_empty_set, pin_gate, pin_routing, pin_needles_closed_form,
            pin_indexer_modes_golden, pin_relu_special_and_numpy, pin_per_head_sets_are_sliced_queries,
            pin_per_head_attention_uses_its_set, pin_router_golden, pin_router_numpy, pin_router_closed_forms,
            pin_kda_golden, pin_kda_transition_matrices, pin_kda_retrieval, pin_kda_basis_keys,
            pin_kda_linear_attention, pin_kda_chaining, pin_kda_extreme_gates, pin_kda_chunked_form]
