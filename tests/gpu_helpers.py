"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import esa_inputs as E
import oracle as O

ATOL = 2e-3  # max-abs error allowed on fp32 outputs (bf16 inputs, fp32 accumulation)


def esa():
    import long_context_sparse_20_b300 as m
    return m


def to_dev(inp: dict) -> dict:
    return {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def _sets(sh: dict) -> tuple:
    """() with one index set per query row, (H_I,) with per-head sets."""
    return (sh["H_I"],) if sh.get("flags", 0) & 2 else ()


def gpu_topk(d: dict, sh: dict, K: int, ws=None):
    m = esa()
    shape = m.shape_from(sh)
    ws = ws or m.workspace_for(m.OP_TOPK_SELECT, shape, K)
    sets = _sets(sh)  # per-head index sets: [B, Tq, H_I, K]
    idx = torch.full((sh["B"], sh["Tq"], *sets, K), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((sh["B"], sh["Tq"], *sets), -7, dtype=torch.int32, device="cuda")
    m.esa_topk_select(d["qI"], d["kI"], d["wI"], shape, K, idx, cnt, ws)
    st = m.esa_read_status(ws)
    assert st == m.OK, m.status_string(st)
    return idx.reshape(-1, K).cpu().numpy(), cnt.reshape(-1).cpu().numpy()


def gpu_threshold(d: dict, sh: dict, K: int, ws=None):
    """The threshold form (T, P) of every row's set, int32 [rows, 2], from the
    routed call's selection step (esa_topk_threshold)."""
    m = esa()
    shape = m.shape_from(sh)
    ws = ws or m.workspace_for(m.OP_TOPK_THRESHOLD, shape, K)
    sets = _sets(sh)  # per-head index sets: [B, Tq, H_I, 2]
    thr = torch.full((sh["B"], sh["Tq"], *sets, 2), -7, dtype=torch.int32, device="cuda")
    m.esa_topk_threshold(d["qI"], d["kI"], d["wI"], shape, K, thr, ws)
    st = m.esa_read_status(ws)
    assert st == m.OK, m.status_string(st)
    return thr.reshape(-1, 2).cpu().numpy()


def assert_thr_equal(got, ref):
    bad = np.nonzero((got != ref).any(axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} rows differ; first row {bad[0] if len(bad) else None}: " \
                          f"{got[bad[0]] if len(bad) else None} vs {ref[bad[0]] if len(bad) else None}"


def gpu_attn(d: dict, sh: dict, K: int, idx, cnt, gate=True, want_lse=True, ws=None, scale=None):
    m = esa()
    shape = m.shape_from(sh)
    ws = ws or m.workspace_for(m.OP_SPARSE_ATTN, shape, K)
    B, Tq, Hq, D = sh["B"], sh["Tq"], sh["Hq"], sh["D"]
    out = torch.full((B, Tq, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((B, Tq, Hq), float("nan"), dtype=torch.float32, device="cuda") if want_lse else None
    sets = _sets(sh)
    idx_d = torch.as_tensor(np.asarray(idx, dtype=np.int32)).reshape(B, Tq, *sets, K).cuda()
    cnt_d = torch.as_tensor(np.asarray(cnt, dtype=np.int32)).reshape(B, Tq, *sets).cuda()
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    m.esa_sparse_attn(d["q"], d["k"], d["v"], idx_d, cnt_d, shape, K, scale, d["g"] if gate else None,
                      d["lin"] if gate else None, out, lse, ws)
    st = m.esa_read_status(ws)
    return st, out.reshape(B * Tq, Hq, D).cpu().numpy(), (lse.reshape(B * Tq, Hq).cpu().numpy() if want_lse else None)


def gpu_routed(d: dict, sh: dict, K: int, gate=True):
    m = esa()
    shape = m.shape_from(sh)
    ws = m.workspace_for(m.OP_ROUTED_ATTN, shape, K)
    B, Tq, Hq, D = sh["B"], sh["Tq"], sh["Hq"], sh["D"]
    out = torch.full((B, Tq, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    m.esa_routed_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], d["route"], shape, K, 1.0 / math.sqrt(D),
                      d["g"] if gate else None, d["lin"] if gate else None, out, ws)
    st = m.esa_read_status(ws)
    assert st == m.OK, m.status_string(st)
    return out.reshape(B * Tq, Hq, D).cpu().numpy()


def sample_rows(B: int, Tq: int, K: int, n: int, seed: int = 0) -> np.ndarray:
    """A seeded uniform sample of n flat rows per sequence plus the edge rows
    of every sequence (0, 1, K-2, K-1, K, Tq-1)."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(B):
        rows |= set((b * Tq + rng.choice(Tq, size=min(n, Tq), replace=False)).tolist())
    for b in range(B):
        for t in (0, 1, K - 2, K - 1, K, Tq - 1):
            if 0 <= t < Tq:
                rows.add(b * Tq + t)
    return np.array(sorted(rows), dtype=np.int64)


def assert_idx_equal(gi, gc, oi, oc, rows=None):
    if rows is not None:
        gi, gc = gi[rows], gc[rows]
    bad = np.nonzero((gc != oc) | (gi != oi).any(axis=1))[0]
    assert len(bad) == 0, f"{len(bad)} rows differ; first row {bad[0] if len(bad) else None}"


def assert_close(got, ref, atol=ATOL, what="out"):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    assert err.max() <= atol, f"{what}: max abs err {err.max():.3e} > {atol}"
