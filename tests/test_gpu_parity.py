"""CUDA path (through the C ABI) against the CPU oracle, element by element.

Index sets and counts must match bit-exactly; fp32 outputs within 2e-3
max-abs (bf16 inputs, fp32 accumulation). Small cases span several tiles
and ragged tails; the five workloads run at full size, compared on all rows
(decode; index sets of every prefill workload) or on seeded row samples
plus edge rows (prefill outputs)."""
import math
import os

import numpy as np
import pytest
import torch

import esa_inputs as E
import oracle as O
from gpu_helpers import (ATOL, assert_close, assert_idx_equal, assert_thr_equal, esa, gpu_attn, gpu_routed,
                         gpu_threshold, gpu_topk, sample_rows, to_dev)

pytestmark = pytest.mark.gpu


def _case(**over):
    cfg = E.small_config(**over)
    return cfg, E.shape_of(cfg), E.make_inputs(cfg)


# ------------------------------------------------------------------ top-K
TOPK_CASES = [
    # prefill, row-tiled selection: ragged row tiles, t around K, several key tiles
    dict(B=1, Tq=300, Tk=300, top_k=64, D_I=32),
    dict(B=2, Tq=200, Tk=200, top_k=100, D_I=64, H_I=4, weights="1to4"),
    dict(B=1, Tq=130, Tk=130, top_k=1, D_I=16),
    dict(B=1, Tq=300, Tk=300, top_k=200, D_I=64, H_I=2, weights="1to4"),  # thresholds near 0 and below
    dict(B=1, Tq=257, Tk=257, top_k=256, D_I=128, H_I=2, weights="1to4"),
    # chunked prefill: queries at positions q_offset..q_offset+Tq-1
    dict(B=2, Tq=70, Tk=600, q_offset=530, top_k=128, D_I=64),
    # decode, split selection across blocks
    dict(B=1, Tq=1, Tk=5000, q_offset=4999, top_k=2048, D_I=64),
    dict(B=3, Tq=1, Tk=40000, q_offset=39999, top_k=700, D_I=32, H_I=3, weights="1to4"),
    dict(B=8, Tq=1, Tk=1500, q_offset=1499, top_k=2048, D_I=64),   # n <= K: whole prefix
    dict(B=2, Tq=1, Tk=9000, q_offset=8999, top_k=2048, D_I=128),
    dict(B=1, Tq=1, Tk=3000, q_offset=2999, top_k=2999, D_I=16),   # K = n-1
    dict(B=4, Tq=2, Tk=6000, q_offset=5998, top_k=1000, D_I=64),   # two query rows per sequence
]


@pytest.mark.parametrize("over", TOPK_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_topk_small(over):
    cfg, sh, inp = _case(seed=101, **over)
    K = cfg["top_k"]
    gi, gc = gpu_topk(to_dev(inp), sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi, oc)


THR_CASES = [
    dict(B=1, Tq=300, Tk=300, top_k=64, D_I=32),
    dict(B=2, Tq=200, Tk=200, top_k=100, D_I=64, H_I=4, weights="1to4"),
    dict(B=1, Tq=130, Tk=130, top_k=1, D_I=16),
    dict(B=2, Tq=70, Tk=600, q_offset=530, top_k=128, D_I=64),
    dict(B=1, Tq=257, Tk=257, top_k=256, D_I=128, H_I=2, weights="1to4"),  # dp4a kernel (D_I = 128)
]


@pytest.mark.parametrize("over", THR_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_topk_threshold_small(over):
    """The routed call's selection step, (T, P) per row, bit-exact against the
    oracle's threshold form, and the set it describes equal to the idx row
    of esa_topk_select."""
    cfg, sh, inp = _case(seed=111, **over)
    K = cfg["top_k"]
    d = to_dev(inp)
    thr = gpu_threshold(d, sh, K)
    assert_thr_equal(thr, O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, K))
    gi, gc = gpu_topk(d, sh, K)
    for r in range(0, sh["B"] * sh["Tq"], 7):
        b, t = divmod(r, sh["Tq"])
        s = O.indexer_row(inp["qI"], inp["kI"], inp["wI"], sh, b, t)
        T, P = thr[r]
        j = np.arange(len(s))
        described = j[(s > T) | ((s == T) & (j <= P))]
        assert described.tolist() == gi[r, :gc[r]].tolist(), r


def test_topk_threshold_ties():
    """All scores equal, and tie-heavy small-range scores: the last tie taken
    (P) must be exactly the oracle's."""
    cfg, sh, inp = _case(seed=112, B=1, Tq=260, Tk=260, top_k=50, D_I=64)
    inp["kI"] = torch.zeros_like(inp["kI"])
    d = to_dev(inp)
    assert_thr_equal(gpu_threshold(d, sh, 50), O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, 50))
    g = torch.Generator().manual_seed(5)
    inp["qI"] = torch.randint(-1, 2, inp["qI"].shape, dtype=torch.int8, generator=g)
    inp["kI"] = torch.randint(-1, 2, inp["kI"].shape, dtype=torch.int8, generator=g)
    d = to_dev(inp)
    assert_thr_equal(gpu_threshold(d, sh, 50), O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, 50))


@pytest.mark.parametrize("decode", [False, True])
def test_topk_all_equal_scores(decode):
    """Every score equal: the K lowest positions win (worst case for ties)."""
    over = dict(B=2, Tq=1, Tk=20000, q_offset=19999, top_k=2048) if decode else dict(B=1, Tq=200, Tk=200, top_k=50)
    cfg, sh, inp = _case(seed=5, D_I=64, **over)
    inp["kI"] = torch.zeros_like(inp["kI"])
    K = cfg["top_k"]
    gi, gc = gpu_topk(to_dev(inp), sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi, oc)


@pytest.mark.parametrize("decode", [False, True])
def test_topk_wide_scores(decode):
    """Full-range int8 and large, mixed-sign weights: scores near 2^30 take
    the deeper histogram levels, and the indexer heads cannot be collapsed."""
    over = dict(B=2, Tq=1, Tk=30000, q_offset=29999, top_k=1500) if decode else dict(B=1, Tq=160, Tk=160, top_k=40)
    cfg, sh, inp = _case(seed=77, D_I=64, H_I=4, **over)
    g = torch.Generator().manual_seed(3)
    inp["qI"] = torch.randint(-128, 128, inp["qI"].shape, dtype=torch.int8, generator=g)
    inp["kI"] = torch.randint(-128, 128, inp["kI"].shape, dtype=torch.int8, generator=g)
    inp["wI"] = torch.tensor([500, -300, 200, 7], dtype=torch.int32)
    K = cfg["top_k"]
    gi, gc = gpu_topk(to_dev(inp), sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi, oc)


def test_topk_repeated_calls_reuse_workspace():
    """The split selection returns its workspace to zero: back-to-back calls
    with different shapes on one workspace stay exact."""
    m = esa()
    shapes = [dict(B=4, Tq=1, Tk=30000, q_offset=29999, top_k=512), dict(B=1, Tq=1, Tk=90000, q_offset=89999,
                                                                         top_k=2048)]
    cases = [_case(seed=200 + i, D_I=64, **s) for i, s in enumerate(shapes)]
    need = max(m.esa_workspace_size(m.OP_TOPK_SELECT, m.shape_from(c[1]), c[0]["top_k"]) for c in cases)
    ws = m.Workspace(need)
    for rep in range(3):
        for cfg, sh, inp in cases:
            gi, gc = gpu_topk(to_dev(inp), sh, cfg["top_k"], ws=ws)
            oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, cfg["top_k"])
            assert_idx_equal(gi, gc, oi, oc)


# ------------------------------------------------------------------ prefill selection: tensor-core and dp4a kernels
def test_topk_prefill_two_sequences_offset():
    """Two sequences, a ragged 128-row tail and queries deep in the cache:
    the fp16 key copy of each sequence starts at its own padded offset."""
    cfg, sh, inp = _case(seed=404, B=2, Tq=300, Tk=5000, q_offset=4700, top_k=1024, D_I=64, H_I=2,
                         weights="1to4")
    gi, gc = gpu_topk(to_dev(inp), sh, 1024)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 1024)
    assert_idx_equal(gi, gc, oi, oc)


def test_topk_prefill_deep_levels():
    """Full-range int8 vectors and weight 8: the collapsed query still fits
    fp16 exactly, and scores up to ~2^21 take three histogram levels."""
    cfg, sh, inp = _case(seed=405, B=1, Tq=260, Tk=2600, q_offset=2340, top_k=300, D_I=64, H_I=1)
    g = torch.Generator().manual_seed(11)
    inp["qI"] = torch.randint(-128, 128, inp["qI"].shape, dtype=torch.int8, generator=g)
    inp["kI"] = torch.randint(-128, 128, inp["kI"].shape, dtype=torch.int8, generator=g)
    inp["wI"] = torch.tensor([8], dtype=torch.int32)
    gi, gc = gpu_topk(to_dev(inp), sh, 300)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 300)
    assert_idx_equal(gi, gc, oi, oc)


def test_topk_prefill_mixed_tiles():
    """One 128-row query tile whose collapsed indexer query leaves the exact
    fp16 range goes to the dp4a kernel; the other tiles stay on the tensor
    cores. Both halves of the result must match."""
    cfg, sh, inp = _case(seed=406, B=2, Tq=400, Tk=400, top_k=96, D_I=32, H_I=2, weights="1to4")
    inp["qI"] = inp["qI"].clone()
    inp["wI"] = torch.tensor([20, 1], dtype=torch.int32)  # |q_eff| = |20 q_0 + q_1| <= 168 ...
    inp["qI"][1, 130, 0, 5] = 127  # ... except row 130 of sequence 1: 2540 + q_1 > 2048
    gi, gc = gpu_topk(to_dev(inp), sh, 96)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 96)
    assert_idx_equal(gi, gc, oi, oc)


def test_topk_prefill_kernels_agree(monkeypatch):
    """The tensor-core selection and the dp4a kernel (ESA_ROW_SELECT=dp4a)
    give identical index sets on a chunk of 1000 queries over 6000 keys."""
    cfg, sh, inp = _case(seed=407, B=1, Tq=1000, Tk=6000, q_offset=5000, top_k=2048, D_I=64, H_I=4,
                         weights="1to4")
    d = to_dev(inp)
    ti, tc = gpu_topk(d, sh, 2048)
    monkeypatch.setenv("ESA_ROW_SELECT", "dp4a")
    di, dc = gpu_topk(d, sh, 2048)
    monkeypatch.delenv("ESA_ROW_SELECT")
    assert np.array_equal(tc, dc)
    assert np.array_equal(ti, di)
    rows = sample_rows(sh["B"], sh["Tq"], 2048, 64, seed=9)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 2048, rows=rows)
    assert_idx_equal(ti, tc, oi, oc, rows=rows)


# ------------------------------------------------------------------ attention
ATTN_CASES = [
    dict(B=1, Tq=150, Tk=150, Hq=4, Hkv=1, D=64, top_k=40),
    dict(B=2, Tq=90, Tk=90, Hq=16, Hkv=2, D=128, top_k=70, D_I=64, H_I=4, weights="1to4"),
    dict(B=1, Tq=65, Tk=65, Hq=6, Hkv=3, D=64, top_k=200),               # K >= every prefix
    dict(B=2, Tq=1, Tk=9000, q_offset=8999, Hq=32, Hkv=1, D=128, top_k=2048, D_I=64),   # decode, splits
    dict(B=1, Tq=1, Tk=20000, q_offset=19999, Hq=64, Hkv=1, D=128, top_k=2048, D_I=64),  # 64 heads per KV head
    dict(B=3, Tq=1, Tk=4000, q_offset=3999, Hq=8, Hkv=2, D=64, top_k=300, D_I=32),
    dict(B=1, Tq=40, Tk=500, q_offset=460, Hq=48, Hkv=1, D=128, top_k=100, D_I=64),     # chunked, 48 heads
    dict(B=1, Tq=1, Tk=12000, q_offset=11999, Hq=32, Hkv=1, D=128, top_k=4000, D_I=64),  # decode, two stages
    dict(B=8, Tq=1, Tk=3000, q_offset=2999, Hq=64, Hkv=1, D=64, top_k=1024, D_I=32),     # decode, 64-head blocks
]


@pytest.mark.parametrize("over", ATTN_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
@pytest.mark.parametrize("gate", [True, False])
def test_sparse_attn_small(over, gate):
    cfg, sh, inp = _case(seed=303, **over)
    K = cfg["top_k"]
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    ref, ref_lse = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K, g=inp["g"] if gate else None,
                               lin=inp["lin"] if gate else None)
    st, out, lse = gpu_attn(to_dev(inp), sh, K, oi, oc, gate=gate)
    assert st == 0
    assert_close(out, ref)
    assert_close(lse, ref_lse, what="lse")


def test_sparse_attn_edge_counts():
    """cnt = 0 (empty set: out = linear share, lse = -inf), cnt = 1, and an
    index list given in non-ascending order (attention is order-free)."""
    cfg, sh, inp = _case(seed=9, B=1, Tq=1, Tk=3000, q_offset=2999, Hq=32, Hkv=1, D=128, top_k=512, D_I=64)
    K = 512
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    d = to_dev(inp)
    for c in (0, 1, 511):
        idx = oi.copy()
        idx[0, c:] = -1
        cnt = np.array([c], dtype=np.int32)
        idx[0, :c] = idx[0, :c][::-1].copy()
        ref, ref_lse = O.attention(inp["q"], inp["k"], inp["v"], idx, cnt, sh, K, g=inp["g"], lin=inp["lin"])
        st, out, lse = gpu_attn(d, sh, K, idx, cnt)
        assert st == 0
        assert_close(out, ref)
        if c == 0:
            assert np.isneginf(lse).all()
        else:
            assert_close(lse, ref_lse, what="lse")


@pytest.mark.parametrize("decode", [False, True])
def test_sparse_attn_bad_index_sets_status(decode):
    """An index past the causal prefix is reported in the status word (no
    fault); the row is left unwritten and the other rows are exact."""
    over = dict(B=2, Tq=1, Tk=5000, q_offset=4999, Hq=32, D=128, D_I=64, top_k=1024) if decode else \
        dict(B=1, Tq=50, Tk=50, Hq=4, D=64, top_k=16)
    cfg, sh, inp = _case(seed=12, Hkv=1, **over)
    K = cfg["top_k"]
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    bad_row = 1 if decode else 20
    idx = oi.copy()
    idx[bad_row, 0] = (sh["q_offset"] + bad_row % sh["Tq"]) + 1  # one past the prefix
    st, out, _ = gpu_attn(to_dev(inp), sh, K, idx, oc)
    assert st == esa().ERR_BAD_INDEX
    assert np.isnan(out[bad_row]).all()
    ref, _ = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K, g=inp["g"], lin=inp["lin"])
    keep = [r for r in range(len(oc)) if r != bad_row]
    assert_close(out[keep], ref[keep])


def test_gated_mix():
    m = esa()
    cfg, sh, inp = _case(seed=41, B=2, Tq=33, Tk=33, Hq=8, Hkv=2, D=128, top_k=9, routed=True)
    K = 9
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    plain, _ = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K)
    gated, _ = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K, g=inp["g"], lin=inp["lin"])
    attn = torch.as_tensor(plain, dtype=torch.float32).reshape(2, 33, 8, 128).cuda()
    out = torch.empty_like(attn)
    d = to_dev(inp)
    m.esa_gated_mix(attn, d["lin"], d["g"], None, m.shape_from(sh), out)
    assert_close(out.reshape(66, 8, 128).cpu().numpy(), gated)
    # with a head mask: unmasked heads copy attn; also in place (out aliases attn)
    m.esa_gated_mix(attn, d["lin"], d["g"], d["route"], m.shape_from(sh), attn)
    got = attn.reshape(66, 8, 128).cpu().numpy()
    route = inp["route"].numpy()
    for b in range(2):
        for h in range(8):
            src = gated if route[b, h] else plain
            assert_close(got[b * 33:(b + 1) * 33, h], src[b * 33:(b + 1) * 33, h])


# ------------------------------------------------------------------ routed
ROUTED_CASES = [
    dict(B=2, Tq=200, Tk=200, Hq=8, Hkv=8, D=128, top_k=50, D_I=64),
    dict(B=1, Tq=130, Tk=130, Hq=4, Hkv=2, D=64, top_k=16, D_I=32, H_I=2, weights="1to4"),
    dict(B=1, Tq=64, Tk=300, q_offset=236, Hq=6, Hkv=6, D=128, top_k=100, D_I=128),
    dict(B=1, Tq=70, Tk=70, Hq=4, Hkv=1, D=64, top_k=12, D_I=16),
    dict(B=1, Tq=300, Tk=300, Hq=2, Hkv=1, D=128, top_k=64, D_I=64, H_I=4, weights="1to4"),
]


@pytest.mark.parametrize("over", ROUTED_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
@pytest.mark.parametrize("routes", ["drawn", "all_full", "all_sparse"])
def test_routed_small(over, routes):
    cfg, sh, inp = _case(seed=55, routed=True, **over)
    if routes == "all_full":
        inp["route"] = torch.zeros_like(inp["route"])
    elif routes == "all_sparse":
        inp["route"] = torch.ones_like(inp["route"])
    K = cfg["top_k"]
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, K)
    out = gpu_routed(to_dev(inp), sh, K)
    assert_close(out, ref)


def test_routed_equal_scores():
    """All-equal indexer scores: sparse heads keep the K lowest positions."""
    cfg, sh, inp = _case(seed=8, routed=True, B=1, Tq=150, Tk=150, Hq=4, Hkv=4, D=64, top_k=20, D_I=64)
    inp["kI"] = torch.zeros_like(inp["kI"])
    inp["route"] = torch.tensor([[1, 0, 1, 1]], dtype=torch.uint8)
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, 20)
    assert_close(gpu_routed(to_dev(inp), sh, 20), ref)


def test_routed_wide_scores():
    """Full-range int8 indexer vectors with large, mixed-sign weights: the
    collapsed indexer query is not exact in fp16, so the tensor-core kernel
    takes its exact integer mask path; results must still match."""
    cfg, sh, inp = _case(seed=19, routed=True, B=1, Tq=200, Tk=200, Hq=4, Hkv=2, D=128, top_k=30, D_I=64, H_I=4)
    g = torch.Generator().manual_seed(5)
    inp["qI"] = torch.randint(-128, 128, inp["qI"].shape, dtype=torch.int8, generator=g)
    inp["kI"] = torch.randint(-128, 128, inp["kI"].shape, dtype=torch.int8, generator=g)
    inp["wI"] = torch.tensor([500, -300, 200, 7], dtype=torch.int32)
    inp["route"] = torch.tensor([[1, 0, 1, 1]], dtype=torch.uint8)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, 30)
    assert_close(gpu_routed(to_dev(inp), sh, 30), ref)


def test_routed_values_beyond_fp16():
    """A value above the fp16 range in V makes the routed launch take its
    bf16 hi + lo variant for P V (the fp16 one stands down). Only the last
    query row sees that key: the other rows must match within 2e-3, and the
    last row, whose outputs are large, within a relative 5e-5 (bf16 hi + lo
    P keeps ~2^-17; an fp16 P would be off by ~2^-12)."""
    cfg, sh, inp = _case(seed=23, routed=True, B=1, Tq=300, Tk=300, Hq=4, Hkv=2, D=128, top_k=40, D_I=64)
    inp["v"] = inp["v"].clone()
    inp["v"][0, 299, :, 7] = 70000.0  # bf16 70144, > 65504
    inp["route"] = torch.tensor([[1, 0, 1, 0]], dtype=torch.uint8)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, 40)
    got = gpu_routed(to_dev(inp), sh, 40)
    assert_close(got[:-1], ref[:-1])
    err = np.abs(got[-1].astype(np.float64) - ref[-1])
    assert (err <= 5e-5 * np.maximum(1.0, np.abs(ref[-1]))).all(), err.max()


# ------------------------------------------------------------------ indexer options: ReLU, per-head index sets
RELU, PER_HEAD = 1, 2


@pytest.mark.parametrize("flags", [0, RELU, PER_HEAD, RELU | PER_HEAD])
def test_indexer_score_modes(flags):
    """Diagnostic scores: weighted sum (or one head's own score) of the
    int8 dot products, with the ReLU per head when asked; INT32_MIN past the
    causal prefix."""
    m = esa()
    cfg, sh, inp = _case(seed=500 + flags, B=2, Tq=5, Tk=300, q_offset=295, H_I=3, D_I=32, weights="1to4",
                         flags=flags)
    d = to_dev(inp)
    H = sh["H_I"] if flags & PER_HEAD else 1
    B, Tq, Tk = sh["B"], sh["Tq"], sh["Tk"]
    scores = torch.full((B, Tq, H, Tk), 7, dtype=torch.int32, device="cuda")
    shape = m.shape_from(sh)
    ws = m.workspace_for(m.OP_INDEXER_SCORE, shape, 1)
    m.esa_indexer_score(d["qI"], d["kI"], d["wI"], shape, scores, ws)
    assert m.esa_read_status(ws) == m.OK
    got = scores.cpu().numpy()
    for b in range(B):
        for t in range(Tq):
            n = sh["q_offset"] + t + 1
            for h in range(H):
                ref = O.indexer_row(inp["qI"], inp["kI"], inp["wI"], sh, b, t, relu=bool(flags & RELU),
                                    head=h if flags & PER_HEAD else -1)
                assert np.array_equal(got[b, t, h, :n], ref), (b, t, h)
                assert (got[b, t, h, n:] == np.iinfo(np.int32).min).all()


MODE_TOPK_CASES = [
    # decode, split selection: ReLU on one head; per-head sets (4 single-head rows per query)
    dict(B=2, Tq=1, Tk=20000, q_offset=19999, top_k=1024, D_I=64, H_I=1, flags=RELU),
    dict(B=2, Tq=1, Tk=20000, q_offset=19999, top_k=1024, D_I=64, H_I=4, flags=PER_HEAD),
    dict(B=2, Tq=1, Tk=20000, q_offset=19999, top_k=1024, D_I=64, H_I=4, flags=RELU | PER_HEAD),
    # decode, ReLU on several heads: the row kernel
    dict(B=1, Tq=1, Tk=9000, q_offset=8999, top_k=512, D_I=32, H_I=3, weights="1to4", flags=RELU),
    # prefill: tensor-core rows (ReLU on one head, per-head sets), dp4a rows (ReLU on several heads)
    dict(B=1, Tq=300, Tk=300, top_k=64, D_I=64, H_I=1, flags=RELU),
    dict(B=2, Tq=200, Tk=200, top_k=50, D_I=32, H_I=4, weights="1to4", flags=RELU),
    dict(B=1, Tq=150, Tk=700, q_offset=550, top_k=128, D_I=64, H_I=4, flags=PER_HEAD),
    dict(B=1, Tq=150, Tk=700, q_offset=550, top_k=128, D_I=64, H_I=4, flags=RELU | PER_HEAD),
]


@pytest.mark.parametrize("over", MODE_TOPK_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_topk_modes(over):
    cfg, sh, inp = _case(seed=511, **over)
    K = cfg["top_k"]
    gi, gc = gpu_topk(to_dev(inp), sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi.reshape(-1, K), oc.reshape(-1))


def test_topk_relu_weight_sign():
    """ReLU on one head with a negative weight: the scores are w * max(0, q.k)
    (not max(0, w * q.k)), on the tensor cores and in decode."""
    for over in (dict(B=1, Tq=200, Tk=200, top_k=40), dict(B=2, Tq=1, Tk=12000, q_offset=11999, top_k=300)):
        cfg, sh, inp = _case(seed=512, D_I=64, H_I=1, flags=RELU, **over)
        inp["wI"] = torch.tensor([-3], dtype=torch.int32)
        K = cfg["top_k"]
        gi, gc = gpu_topk(to_dev(inp), sh, K)
        oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
        assert_idx_equal(gi, gc, oi.reshape(-1, K), oc.reshape(-1))


PER_HEAD_ATTN_CASES = [
    dict(B=1, Tq=90, Tk=90, Hq=16, Hkv=2, D=128, H_I=16, D_I=32, top_k=30, flags=PER_HEAD),  # a set per query head
    dict(B=1, Tq=90, Tk=90, Hq=16, Hkv=2, D=128, H_I=4, D_I=32, top_k=30, flags=RELU | PER_HEAD),  # 4 heads per set
    dict(B=2, Tq=60, Tk=60, Hq=8, Hkv=4, D=64, H_I=2, D_I=16, top_k=20, flags=PER_HEAD),  # a set spans 2 KV heads
    dict(B=1, Tq=1, Tk=9000, q_offset=8999, Hq=32, Hkv=1, D=128, H_I=4, D_I=64, top_k=2048, flags=PER_HEAD),  # decode
]


@pytest.mark.parametrize("over", PER_HEAD_ATTN_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_attention_per_head_sets(over):
    """Query head h attends to the index set of indexer head h // (Hq // H_I)."""
    cfg, sh, inp = _case(seed=513, **over)
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc, ref, ref_lse = O.gated_sparse_attention(inp, sh, K)
    assert_idx_equal(gi, gc, oi.reshape(-1, K), oc.reshape(-1))
    st, out, lse = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out, ref)
    assert_close(lse, ref_lse, what="lse")


def test_routed_relu():
    """Routed heads with the ReLU indexer: the sparse heads' masks come from
    the clamped per-head scores (dp4a), the thresholds from the row selection."""
    cfg, sh, inp = _case(seed=514, routed=True, B=1, Tq=200, Tk=200, Hq=4, Hkv=2, D=128, top_k=30, D_I=64, H_I=2,
                         weights="1to4", flags=RELU)
    inp["route"] = torch.tensor([[1, 0, 1, 1]], dtype=torch.uint8)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, 30)
    assert_close(gpu_routed(to_dev(inp), sh, 30), ref)


ROUTED_PER_HEAD_CASES = [
    # a set per query head, drawn routes
    dict(B=1, Tq=300, Tk=300, Hq=8, Hkv=2, D=128, H_I=8, D_I=64, top_k=64, flags=PER_HEAD),
    # 2 query heads per set, with the ReLU (one head per set: exact on the tensor cores)
    dict(B=2, Tq=200, Tk=200, Hq=8, Hkv=8, D=128, H_I=4, D_I=32, top_k=40, flags=RELU | PER_HEAD),
    # D = 64, a set spanning two key/value heads, queries deep in a cache
    dict(B=1, Tq=130, Tk=700, q_offset=570, Hq=8, Hkv=4, D=64, H_I=2, D_I=16, top_k=100, flags=PER_HEAD),
]


@pytest.mark.parametrize("routes", ["drawn", "all_sparse"])
@pytest.mark.parametrize("over", ROUTED_PER_HEAD_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_routed_per_head_sets(over, routes):
    """Routed attention with one index set per indexer head: each sparse
    head masks with the set of indexer head h // (Hq // H_I), rebuilt from
    that head's own scores and its threshold form; full heads stay exact
    causal attention."""
    cfg, sh, inp = _case(seed=515, routed=True, **over)
    if routes == "all_sparse":
        inp["route"] = torch.ones_like(inp["route"])
    K = cfg["top_k"]
    d = to_dev(inp)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K)
    assert_close(gpu_routed(d, sh, K), ref)
    thr = gpu_threshold(d, sh, K).reshape(-1, sh["H_I"], 2)
    assert_thr_equal(thr.reshape(-1, 2), O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, K).reshape(-1, 2))


@pytest.mark.parametrize("over", [ROUTED_CASES[1], ROUTED_CASES[2], ROUTED_PER_HEAD_CASES[2]],
                         ids=["gqa-D64", "chunk-in-cache", "per-head-sets"])
def test_routed_with_dp4a_selection(monkeypatch, over):
    """The dp4a row selection (ESA_ROW_SELECT=dp4a; the path of query tiles
    outside the exact fp16 range) writes the same bitmask of selected keys
    that the routed kernel masks sparse heads with: exact outputs, with one
    set per row and with per-head sets."""
    monkeypatch.setenv("ESA_ROW_SELECT", "dp4a")
    cfg, sh, inp = _case(seed=516, routed=True, **over)
    inp["route"] = torch.ones_like(inp["route"])
    inp["route"][..., 0] = 0  # one full head, the rest sparse
    K = cfg["top_k"]
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K)
    assert_close(gpu_routed(to_dev(inp), sh, K), ref)


def test_threshold_per_head_ties():
    """Per-head threshold forms on tie-heavy scores (small int8 range), with
    and without the ReLU."""
    for flags in (PER_HEAD, RELU | PER_HEAD):
        cfg, sh, inp = _case(seed=516, B=1, Tq=260, Tk=260, H_I=3, D_I=64, top_k=50, flags=flags)
        g = torch.Generator().manual_seed(6)
        inp["qI"] = torch.randint(-1, 2, inp["qI"].shape, dtype=torch.int8, generator=g)
        inp["kI"] = torch.randint(-1, 2, inp["kI"].shape, dtype=torch.int8, generator=g)
        d = to_dev(inp)
        assert_thr_equal(gpu_threshold(d, sh, 50), O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, 50).reshape(-1, 2))


# ------------------------------------------------------------------ attention router
def _gpu_route(d_k, sh, W):
    m = esa()
    shape = m.shape_from(sh)
    ws = m.workspace_for(m.OP_ROUTE_HEADS, shape, 1)
    route = torch.full((sh["B"], sh["Hq"]), 7, dtype=torch.uint8, device="cuda")
    margin = torch.full((sh["B"], sh["Hq"]), float("nan"), dtype=torch.float32, device="cuda")
    Wd = {n: t.cuda() for n, t in W.items()}
    m.esa_route_heads(d_k, Wd["W1"], Wd["b1"], Wd["W2"], Wd["b2"], shape, route, margin, ws)
    assert m.esa_read_status(ws) == m.OK
    return route.cpu().numpy(), margin.cpu().numpy()


def _check_route(route, margin, oroute, omargin):
    """Margins within the fp32 error of the sums; route bits equal wherever
    the oracle's margin is outside that band (inside it both bits are valid)."""
    band = 1e-4 * (1.0 + np.abs(omargin))
    assert (np.abs(margin - omargin) <= band).all(), np.abs(margin - omargin).max()
    decided = np.abs(omargin) > band
    assert np.array_equal(route[decided], oroute[decided])
    assert decided.mean() > 0.9


@pytest.mark.parametrize("name", ["small", "routed_prefill"])
def test_route_heads_matches_oracle(name):
    if name == "small":
        cfg, sh, inp = _case(seed=515, routed=True, B=2, Tq=300, Tk=300, Hq=8, Hkv=2, D=64)
        inp["k"] = (inp["k"].float() + 0.4).to(torch.bfloat16)  # a mean key state away from 0
        W = E.router_weights(cfg, hidden=32)
    else:
        cfg, sh, inp = _full("routed_prefill")
        W = E.router_weights(cfg)
    route, margin = _gpu_route(inp["k"].cuda(), sh, W)
    oroute, omargin = O.route_heads(inp["k"], sh, W["W1"], W["b1"], W["W2"], W["b2"])
    _check_route(route, margin, oroute, omargin)
    r2, m2 = _gpu_route(inp["k"].cuda(), sh, W)
    assert np.array_equal(route, r2) and np.array_equal(margin, m2)  # fixed summation order


def test_router_drives_routed_attention():
    """The router's bits are the routed launch's metadata: router -> routed
    attention, compared with the oracle run on the same bits."""
    cfg, sh, inp = _case(seed=516, routed=True, B=2, Tq=160, Tk=160, Hq=8, Hkv=8, D=64, top_k=24, D_I=32)
    W = E.router_weights(cfg, hidden=16)
    d = to_dev(inp)
    route, _ = _gpu_route(d["k"], sh, W)
    d["route"] = torch.from_numpy(route).cuda()
    inp["route"] = torch.from_numpy(route)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, 24)
    assert_close(gpu_routed(d, sh, 24), ref)


# ------------------------------------------------------------------ the five workloads at full size
def _full(name):
    cfg = E.CONFIGS[name]
    return cfg, E.shape_of(cfg), E.make_inputs(cfg)


def test_tiny_prefill_full():
    cfg, sh, inp = _full("tiny_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc, ref, ref_lse = O.gated_sparse_attention(inp, sh, K)
    assert_idx_equal(gi, gc, oi, oc)
    st, out, lse = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out, ref)
    assert_close(lse, ref_lse, what="lse")


@pytest.mark.parametrize("name", ["decode", "million_decode"])
def test_decode_full(name):
    cfg, sh, inp = _full(name)
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc, ref, ref_lse = O.gated_sparse_attention(inp, sh, K)
    assert_idx_equal(gi, gc, oi, oc)
    if inp["needles"] is not None:
        assert set(inp["needles"].tolist()) <= set(gi[0].tolist())
    st, out, lse = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out, ref)
    assert_close(lse, ref_lse, what="lse")


def test_long_prefill_full():
    """Index sets on all 32768 rows; outputs on 1024 seeded rows plus edges."""
    cfg, sh, inp = _full("long_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi, oc)
    assert (gc == np.minimum(K, np.arange(sh["Tq"]) + 1)).all()
    rows = sample_rows(sh["B"], sh["Tq"], K, 1024, seed=1)
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, K, rows=rows)
    st, out, _ = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out[rows], ref)


def test_chunked_prefill_full():
    """A 16384-token chunk at the end of a 131072-token cache (queries at
    positions 114688..131071): index sets on all rows, outputs on 512 seeded
    rows plus the chunk's edge rows."""
    cfg, sh, inp = _full("chunked_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi, oc)
    assert (gc == K).all()
    rows = sample_rows(sh["B"], sh["Tq"], K, 512, seed=3)
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, K, rows=rows)
    st, out, _ = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out[rows], ref)


def test_per_head_prefill_full():
    """One ReLU'd index set per query head (16 sets per query row) at
    S=8192: every set of every row; outputs on 512 seeded rows plus edge
    rows, every head."""
    cfg, sh, inp = _full("per_head_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    gi, gc = gpu_topk(d, sh, K)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    assert_idx_equal(gi, gc, oi.reshape(-1, K), oc.reshape(-1))
    rows = sample_rows(sh["B"], sh["Tq"], K, 512, seed=4)
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, K, rows=rows)
    st, out, _ = gpu_attn(d, sh, K, gi, gc)
    assert st == 0
    assert_close(out[rows], ref)


def test_per_head_prefill_routed_full():
    """The per-head workload (S=8192, a ReLU'd set per query head) through
    the routed launch with every head sparse: the per-head threshold forms on
    every row and set, bit-exact; outputs on 512 seeded rows plus edge rows,
    equal to the gathered path's definition."""
    cfg, sh, inp = _full("per_head_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    d["route"] = torch.ones(sh["B"], sh["Hq"], dtype=torch.uint8, device="cuda")
    thr = gpu_threshold(d, sh, K)
    assert_thr_equal(thr, O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, K).reshape(-1, 2))
    rows = sample_rows(sh["B"], sh["Tq"], K, 512, seed=5)
    out = gpu_routed(d, sh, K)
    _, _, ref, _ = O.gated_sparse_attention(dict(inp, route=None), sh, K, rows=rows)
    assert_close(out[rows], ref)


def test_routed_prefill_full():
    """The routed call's selection, its threshold form (T, P), on all 131072
    rows, bit-exact; outputs of every head on 512 seeded rows per sequence
    plus edge rows."""
    cfg, sh, inp = _full("routed_prefill")
    K = cfg["top_k"]
    d = to_dev(inp)
    thr = gpu_threshold(d, sh, K)
    assert_thr_equal(thr, O.threshold(inp["qI"], inp["kI"], inp["wI"], sh, K))
    rows = sample_rows(sh["B"], sh["Tq"], K, 512, seed=2)
    out = gpu_routed(d, sh, K)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K, rows=rows)
    assert_close(out[rows], ref)


# ------------------------------------------------------------------ bounded waits
def test_wait_timeout_reports_status(monkeypatch):
    """A barrier made unreachable (extra arrivals nobody provides) runs out
    after its short limit: the call returns, the status word says TIMEOUT,
    and the context stays usable (a parity check follows on a fresh
    workspace)."""
    m = esa()
    cfg, sh, inp = _case(seed=31, B=2, Tq=1, Tk=20000, q_offset=19999, top_k=512, D_I=64)
    d = to_dev(inp)
    shape = m.shape_from(sh)
    ws = m.workspace_for(m.OP_TOPK_SELECT, shape, 512)
    idx = torch.empty(2, 1, 512, dtype=torch.int32, device="cuda")
    cnt = torch.empty(2, 1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("ESA_DEBUG_EXTRA_ARRIVALS", "1")
    monkeypatch.setenv("ESA_WAIT_LIMIT_NS", "20000000")
    m.esa_topk_select(d["qI"], d["kI"], d["wI"], shape, 512, idx, cnt, ws)
    assert m.esa_read_status(ws) == m.ERR_TIMEOUT
    monkeypatch.delenv("ESA_DEBUG_EXTRA_ARRIVALS")
    monkeypatch.delenv("ESA_WAIT_LIMIT_NS")
    m.esa_workspace_init(ws)
    gi, gc = gpu_topk(d, sh, 512, ws=ws)
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, 512)
    assert_idx_equal(gi, gc, oi, oc)


def test_decode_attention_wait_timeout_reports_status(monkeypatch):
    """The decode attention's blocks of one row meet at a bounded counter
    barrier; made unreachable it runs out: the call returns, the status word
    says TIMEOUT, the rows stay unwritten, and after re-initialising the
    workspace the same call is exact."""
    m = esa()
    cfg, sh, inp = _case(seed=33, B=2, Tq=1, Tk=9000, q_offset=8999, Hq=32, Hkv=1, D=128, top_k=2048, D_I=64)
    K = 2048
    oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
    d = to_dev(inp)
    ws = m.workspace_for(m.OP_SPARSE_ATTN, m.shape_from(sh), K)
    monkeypatch.setenv("ESA_DEBUG_EXTRA_ARRIVALS", "1")
    monkeypatch.setenv("ESA_WAIT_LIMIT_NS", "20000000")
    st, out, _ = gpu_attn(d, sh, K, oi, oc, ws=ws)
    assert st == m.ERR_TIMEOUT
    assert np.isnan(out).all()
    monkeypatch.delenv("ESA_DEBUG_EXTRA_ARRIVALS")
    monkeypatch.delenv("ESA_WAIT_LIMIT_NS")
    m.esa_workspace_init(ws)
    st, out, lse = gpu_attn(d, sh, K, oi, oc, ws=ws)
    assert st == 0
    ref, ref_lse = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K, g=inp["g"], lin=inp["lin"])
    assert_close(out, ref)
    assert_close(lse, ref_lse, what="lse")


def test_decode_attention_repeated_calls():
    """The barrier's counters are cleared by each call: many calls on one
    workspace (two shapes alternating, sized for the larger) stay exact."""
    m = esa()
    cases = []
    for seed, over in ((34, dict(B=2, Tq=1, Tk=9000, q_offset=8999, Hq=32, Hkv=1, D=128, top_k=2048, D_I=64)),
                       (35, dict(B=1, Tq=1, Tk=20000, q_offset=19999, Hq=64, Hkv=1, D=128, top_k=1024, D_I=64))):
        cfg, sh, inp = _case(seed=seed, **over)
        K = cfg["top_k"]
        oi, oc = O.topk(inp["qI"], inp["kI"], inp["wI"], sh, K)
        ref, ref_lse = O.attention(inp["q"], inp["k"], inp["v"], oi, oc, sh, K, g=inp["g"], lin=inp["lin"])
        cases.append((sh, K, to_dev(inp), oi, oc, ref))
    n = max(m.esa_workspace_size(m.OP_SPARSE_ATTN, m.shape_from(sh), K) for sh, K, *_ in cases)
    ws = m.Workspace(n)
    for it in range(6):
        sh, K, d, oi, oc, ref = cases[it % 2]
        st, out, _ = gpu_attn(d, sh, K, oi, oc, ws=ws, want_lse=False)
        assert st == 0
        assert_close(out, ref)


# ------------------------------------------------------------------ cache append
@pytest.mark.parametrize("Tq", [1, 5])
def test_cache_append_writes_exactly_the_new_rows(Tq):
    """The new positions' rows land at q_offset..q_offset+Tq-1 of each
    sequence, bit for bit; every other cache byte is unchanged; a skipped
    cache (both pointers NULL) is untouched."""
    m = esa()
    B, Tk, Hkv, D, DI = 3, 40, 2, 128, 64
    q_offset = Tk - Tq
    sh = dict(B=B, Tq=Tq, Tk=Tk, q_offset=q_offset, Hq=4, Hkv=Hkv, D=D, H_I=1, D_I=DI)
    g = torch.Generator().manual_seed(5)
    k = torch.randn(B, Tk, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Tk, Hkv, D, generator=g).to(torch.bfloat16)
    kI = torch.randint(-128, 128, (B, Tk, DI), generator=g, dtype=torch.int8)
    kn = torch.randn(B, Tq, Hkv, D, generator=g).to(torch.bfloat16)
    vn = torch.randn(B, Tq, Hkv, D, generator=g).to(torch.bfloat16)
    kIn = torch.randint(-128, 128, (B, Tq, DI), generator=g, dtype=torch.int8)
    dk, dv, dkI = k.cuda(), v.cuda(), kI.cuda()
    m.esa_cache_append(kn.cuda(), vn.cuda(), kIn.cuda(), dk, dv, dkI, m.shape_from(sh))
    ek, ev, ekI = k.clone(), v.clone(), kI.clone()
    ek[:, q_offset:] = kn
    ev[:, q_offset:] = vn
    ekI[:, q_offset:] = kIn
    assert torch.equal(dk.cpu().view(torch.int16), ek.view(torch.int16))
    assert torch.equal(dv.cpu().view(torch.int16), ev.view(torch.int16))
    assert torch.equal(dkI.cpu(), ekI)
    dk2 = k.cuda()
    m.esa_cache_append(None, None, kIn.cuda(), None, None, dkI, m.shape_from(sh))
    assert torch.equal(dk2.cpu().view(torch.int16), k.view(torch.int16))
