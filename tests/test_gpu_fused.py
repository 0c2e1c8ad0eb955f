"""esa_gated_sparse_attn — the whole path in one call — against the CPU
oracle, through the C ABI, on both of its implementations: the selection
and gathered-attention kernels back to back (the default), and, with
ESA_DECODE_PATH=fused, the single cooperative launch for decode-like shapes
(selection, attention over each block's own selected keys, the row's
partials merged in the same launch, gate mix). Index sets bit-exact; fp32
outputs and lse within 2e-3 max-abs."""
import math

import numpy as np
import pytest
import torch

import esa_inputs as E
import oracle as O
from gpu_helpers import assert_close, assert_idx_equal, esa, gpu_attn, gpu_topk, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["two-launch", "fused"], autouse=True)
def decode_path(request, monkeypatch):
    if request.param == "fused":
        monkeypatch.setenv("ESA_DECODE_PATH", "fused")
    else:
        monkeypatch.delenv("ESA_DECODE_PATH", raising=False)
    return request.param


def _case(**over):
    cfg = E.small_config(**over)
    return cfg, E.shape_of(cfg), E.make_inputs(cfg)


def gpu_gated(d, sh, K, want_idx=True, gate=True, want_lse=True, ws=None):
    m = esa()
    shape = m.shape_from(sh)
    ws = ws or m.workspace_for(m.OP_GATED_SPARSE_ATTN, shape, K)
    B, Tq, Hq, D = sh["B"], sh["Tq"], sh["Hq"], sh["D"]
    sets = (sh["H_I"],) if sh.get("flags", 0) & 2 else ()
    out = torch.full((B, Tq, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, Tq, Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    idx = torch.full((B, Tq, *sets, K), -7, dtype=torch.int32, device="cuda") if want_idx else None
    cnt = torch.full((B, Tq, *sets), -7, dtype=torch.int32, device="cuda") if want_idx else None
    m.esa_gated_sparse_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], shape, K, 1.0 / math.sqrt(D),
                            d["g"] if gate else None, d["lin"] if gate else None, out, lse, idx, cnt, ws)
    st = m.esa_read_status(ws)
    assert st == m.OK, m.status_string(st)
    res = {"out": out.reshape(B * Tq, Hq, D).cpu().numpy()}
    if want_lse:
        res["lse"] = lse.reshape(B * Tq, Hq).cpu().numpy()
    if want_idx:
        res["idx"] = idx.reshape(-1, K).cpu().numpy()
        res["cnt"] = cnt.reshape(-1).cpu().numpy()
    return res


def check_against_oracle(inp, sh, K, res, gate=True):
    oi, oc, ref, ref_lse = O.gated_sparse_attention(inp, sh, K, gate=gate)
    if "idx" in res:
        assert_idx_equal(res["idx"], res["cnt"], oi.reshape(-1, K), oc.reshape(-1))
    assert_close(res["out"], ref)
    if "lse" in res:
        assert_close(res["lse"], ref_lse, what="lse")


FUSED_CASES = [
    # the decode workload's head layout on one row (2 m-tiles of 16 heads)
    dict(B=1, Tq=1, Tk=5000, q_offset=4999, Hq=32, Hkv=1, D=128, D_I=64, top_k=2048),
    # whole prefixes (n <= K): every key of every span
    dict(B=8, Tq=1, Tk=1500, q_offset=1499, Hq=32, Hkv=1, D=128, D_I=64, top_k=2048),
    # GQA, D = 64, three weighted indexer heads
    dict(B=3, Tq=1, Tk=40000, q_offset=39999, Hq=16, Hkv=2, D=64, H_I=3, D_I=32, top_k=700, weights="1to4"),
    # 64 heads over one key/value head (4 m-tiles), D_I = 128
    dict(B=2, Tq=1, Tk=9000, q_offset=8999, Hq=64, Hkv=1, D=128, D_I=128, top_k=2048),
    # 8 heads per key/value head (half-empty m-tiles), two query rows per sequence
    dict(B=4, Tq=2, Tk=6000, q_offset=5998, Hq=8, Hkv=1, D=128, D_I=64, top_k=1000),
    dict(B=2, Tq=1, Tk=20000, q_offset=19999, Hq=32, Hkv=4, D=128, D_I=16, top_k=512),
    # K = n - 1, and K = 1
    dict(B=1, Tq=1, Tk=3000, q_offset=2999, Hq=16, Hkv=1, D=64, D_I=16, top_k=2999),
    dict(B=2, Tq=1, Tk=7000, q_offset=6999, Hq=16, Hkv=1, D=128, D_I=64, top_k=1),
    # the ReLU indexer (one head)
    dict(B=2, Tq=1, Tk=30000, q_offset=29999, Hq=32, Hkv=1, D=128, D_I=64, top_k=2048, flags=1),
]


@pytest.mark.parametrize("over", FUSED_CASES, ids=lambda o: "-".join(f"{k}{v}" for k, v in o.items()))
def test_fused_decode_small(over):
    cfg, sh, inp = _case(seed=303, **over)
    K = cfg["top_k"]
    m = esa()
    # these shapes take the single launch: its workspace is the fused plan's
    assert m.esa_workspace_size(m.OP_GATED_SPARSE_ATTN, m.shape_from(sh), K) > 0
    res = gpu_gated(to_dev(inp), sh, K)
    check_against_oracle(inp, sh, K, res)


def test_fused_without_index_output_or_gate():
    """idx/cnt not requested (the index list never leaves the chip), and no
    gate: the same outputs as with them, the plain attention without it."""
    cfg, sh, inp = _case(seed=304, B=4, Tq=1, Tk=50000, q_offset=49999, Hq=32, Hkv=1, D=128, D_I=64, top_k=2048)
    d = to_dev(inp)
    a = gpu_gated(d, sh, 2048)
    b = gpu_gated(d, sh, 2048, want_idx=False)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
    c = gpu_gated(d, sh, 2048, want_idx=False, gate=False, want_lse=False)
    check_against_oracle(inp, sh, 2048, c, gate=False)


def test_fused_matches_the_two_calls():
    """Same index sets as esa_topk_select and outputs within the tolerance of
    esa_sparse_attn's on the same inputs."""
    cfg, sh, inp = _case(seed=305, B=8, Tq=1, Tk=60000, q_offset=59999, Hq=32, Hkv=1, D=128, D_I=64, top_k=2048)
    d = to_dev(inp)
    res = gpu_gated(d, sh, 2048)
    gi, gc = gpu_topk(d, sh, 2048)
    assert np.array_equal(res["idx"], gi) and np.array_equal(res["cnt"], gc)
    st, out, lse = gpu_attn(d, sh, 2048, gi, gc)
    assert st == 0
    assert np.abs(res["out"] - out).max() <= 2e-3 and np.abs(res["lse"] - lse).max() <= 2e-3


@pytest.mark.parametrize("decode", [False, True])
def test_fused_ties_and_wide_scores(decode):
    """All-equal indexer scores (the lowest positions win), then full-range
    int8 with large mixed-sign weights (the deeper histogram levels)."""
    cfg, sh, inp = _case(seed=306, B=2, Tq=1, Tk=30000, q_offset=29999, Hq=32, Hkv=1, D=128, D_I=64, H_I=4,
                         top_k=1500)
    if decode:
        g = torch.Generator().manual_seed(3)
        inp["qI"] = torch.randint(-128, 128, inp["qI"].shape, dtype=torch.int8, generator=g)
        inp["kI"] = torch.randint(-128, 128, inp["kI"].shape, dtype=torch.int8, generator=g)
        inp["wI"] = torch.tensor([500, -300, 200, 7], dtype=torch.int32)
    else:
        inp["kI"] = torch.zeros_like(inp["kI"])
    res = gpu_gated(to_dev(inp), sh, 1500)
    check_against_oracle(inp, sh, 1500, res)


@pytest.mark.parametrize("over", [
    dict(B=1, Tq=300, Tk=300, Hq=4, Hkv=1, D=64, D_I=32, top_k=64),                  # prefill rows
    dict(B=2, Tq=70, Tk=600, q_offset=530, Hq=8, Hkv=2, D=128, D_I=64, top_k=128),   # chunked prefill
    dict(B=2, Tq=1, Tk=20000, q_offset=19999, Hq=8, Hkv=2, D=64, H_I=4, D_I=64, top_k=512, flags=3),  # per-head sets
], ids=["prefill", "chunked", "per-head-sets"])
def test_fused_call_on_shapes_that_take_two_launches(over):
    cfg, sh, inp = _case(seed=307, **over)
    K = cfg["top_k"]
    res = gpu_gated(to_dev(inp), sh, K)
    check_against_oracle(inp, sh, K, res)
    res = gpu_gated(to_dev(inp), sh, K, want_idx=False)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K)
    assert_close(res["out"], ref)


@pytest.mark.parametrize("over", [
    dict(B=1, Tq=300, Tk=300, Hq=4, Hkv=1, D=64, D_I=32, top_k=64),                  # prefill rows
    dict(B=2, Tq=70, Tk=600, q_offset=530, Hq=8, Hkv=2, D=128, D_I=64, top_k=128),   # chunked prefill
    dict(B=1, Tq=200, Tk=200, Hq=8, Hkv=2, D=128, H_I=4, D_I=64, top_k=40, flags=3),  # per-head sets, ReLU
], ids=["prefill", "chunked", "per-head-sets"])
def test_gated_call_on_the_routed_path(over):
    """Prefill shapes whose causal prefixes hold few times the selected keys,
    called without lse, take the routed kernel with every head sparse (the
    selection's bitmask masks dense tiles): the same index sets and outputs
    within tolerance, with and without the index outputs."""
    cfg, sh, inp = _case(seed=308, **over)
    K = cfg["top_k"]
    res = gpu_gated(to_dev(inp), sh, K, want_lse=False)
    check_against_oracle(inp, sh, K, res)
    res = gpu_gated(to_dev(inp), sh, K, want_idx=False, want_lse=False)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K)
    assert_close(res["out"], ref)
    res = gpu_gated(to_dev(inp), sh, K, want_idx=False, want_lse=False, gate=False)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K, gate=False)
    assert_close(res["out"], ref)


def test_small_prefill_default_rule(monkeypatch):
    """The library's own choice for a small prefill (no ESA_ROW_SELECT): the
    dp4a row selection for 1024 queries over 1024 keys (8 row tiles of 128),
    with its bitmask feeding the routed kernel in the one call: exact index
    sets, and outputs within tolerance, with and without the index outputs."""
    monkeypatch.delenv("ESA_ROW_SELECT", raising=False)
    cfg, sh, inp = _case(seed=612, B=1, Tq=1024, Tk=1024, q_offset=0, Hq=4, Hkv=1, D=64, top_k=128, D_I=32)
    K = cfg["top_k"]
    res = gpu_gated(to_dev(inp), sh, K, want_lse=False)
    check_against_oracle(inp, sh, K, res)
    res = gpu_gated(to_dev(inp), sh, K, want_idx=False, want_lse=False)
    _, _, ref, _ = O.gated_sparse_attention(inp, sh, K)
    assert_close(res["out"], ref)


def test_fused_workspace_reuse_across_shapes():
    """Back-to-back calls on one workspace, alternating shapes: the control
    state each call leaves behind is what the next one needs."""
    m = esa()
    shapes = [dict(B=4, Tq=1, Tk=30000, q_offset=29999, top_k=512), dict(B=1, Tq=1, Tk=90000, q_offset=89999,
                                                                         top_k=2048)]
    cases = [_case(seed=310 + i, Hq=32, Hkv=1, D=128, D_I=64, **s) for i, s in enumerate(shapes)]
    need = max(m.esa_workspace_size(m.OP_GATED_SPARSE_ATTN, m.shape_from(c[1]), c[0]["top_k"]) for c in cases)
    ws = m.Workspace(need)
    for rep in range(3):
        for cfg, sh, inp in cases:
            res = gpu_gated(to_dev(inp), sh, cfg["top_k"], ws=ws)
            check_against_oracle(inp, sh, cfg["top_k"], res)


@pytest.mark.parametrize("name", ["decode", "million_decode"])
def test_fused_full(name):
    """The two decode workloads at full size, every row and head."""
    cfg = E.CONFIGS[name]
    sh, inp = E.shape_of(cfg), E.make_inputs(cfg)
    K = cfg["top_k"]
    res = gpu_gated(to_dev(inp), sh, K)
    check_against_oracle(inp, sh, K, res)
    if inp["needles"] is not None:
        assert set(inp["needles"].tolist()) <= set(res["idx"][0].tolist())


def test_fused_wait_timeout_reports_status(monkeypatch):
    """A row barrier made unreachable runs out after its short limit: the
    call returns, the status word says TIMEOUT, and a fresh workspace then
    gives exact results."""
    m = esa()
    cfg, sh, inp = _case(seed=320, B=2, Tq=1, Tk=20000, q_offset=19999, Hq=32, Hkv=1, D=128, D_I=64, top_k=512)
    d = to_dev(inp)
    shape = m.shape_from(sh)
    ws = m.workspace_for(m.OP_GATED_SPARSE_ATTN, shape, 512)
    out = torch.empty(2, 1, 32, 128, dtype=torch.float32, device="cuda")
    monkeypatch.setenv("ESA_DEBUG_EXTRA_ARRIVALS", "1")
    monkeypatch.setenv("ESA_WAIT_LIMIT_NS", "20000000")
    m.esa_gated_sparse_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], shape, 512, 1.0 / math.sqrt(128),
                            d["g"], d["lin"], out, None, None, None, ws)
    assert m.esa_read_status(ws) == m.ERR_TIMEOUT
    monkeypatch.delenv("ESA_DEBUG_EXTRA_ARRIVALS")
    monkeypatch.delenv("ESA_WAIT_LIMIT_NS")
    m.esa_workspace_init(ws)
    res = gpu_gated(d, sh, 512, ws=ws)
    check_against_oracle(inp, sh, 512, res)
