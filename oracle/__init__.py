"""CPU oracle for gated fine-grained sparse attention — TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The product path (the C-ABI library and
its Python binding) never calls it and shares no code with it.

The arithmetic lives in ``esa_oracle.c`` (plain C, int64 / fp64, OpenMP over
query rows); this file only compiles it with gcc and marshals numpy/torch
arrays. What each function computes, and which passage of the pages it
follows, is stated in the C source. Every function is pinned by the CPU tests
(brute force, closed forms, invariants, numpy/torch library routines); no
function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "esa_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "libesa_oracle.so")
_lib = None

c_long = ctypes.c_long
c_int = ctypes.c_int
vp = ctypes.c_void_p


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle with gcc (-O2, OpenMP). Returns the .so path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.oracle_indexer_row.restype = c_long
    lib.oracle_indexer_row.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_int, c_int, c_long, c_long, vp]
    lib.oracle_indexer_row_mode.restype = c_long
    lib.oracle_indexer_row_mode.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_int, c_int, c_long, c_long,
                                            c_int, c_int, vp]
    lib.oracle_topk_rows_mode.restype = c_int
    lib.oracle_topk_rows_mode.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_int, c_int, c_int, c_int, vp,
                                          c_long, vp, vp, c_int]
    lib.oracle_attention_rows_sets.restype = c_int
    lib.oracle_attention_rows_sets.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_long, c_long, c_long, c_long, c_int,
                                               c_int, c_int, ctypes.c_double, vp, vp, vp, vp, c_long, vp, vp, c_int]
    lib.oracle_topk_rows.restype = c_int
    lib.oracle_topk_rows.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_int, c_int, c_int, vp, c_long,
                                     vp, vp, c_int]
    lib.oracle_attention_rows.restype = c_int
    lib.oracle_attention_rows.argtypes = [vp, vp, vp, vp, vp, c_int, c_long, c_long, c_long, c_long, c_int, c_int,
                                          c_int, ctypes.c_double, vp, vp, vp, vp, c_long, vp, vp, c_int]
    lib.oracle_route_heads.restype = c_int
    lib.oracle_route_heads.argtypes = [vp, c_long, c_long, c_int, c_int, c_int, c_int, vp, vp, vp, vp, vp, vp]
    lib.oracle_kda.restype = c_int
    lib.oracle_kda.argtypes = [vp, vp, vp, vp, vp, vp, c_long, c_long, c_int, c_int, c_int, ctypes.c_double, vp, vp,
                               c_int]
    lib.oracle_threshold_rows.restype = c_int
    lib.oracle_threshold_rows.argtypes = [vp, vp, vp, c_long, c_long, c_long, c_long, c_int, c_int, c_int, c_int, vp,
                                          c_long, vp, c_int]
    return lib


def lib(path: str | None = None):
    """The compiled oracle (built on first use when missing or stale)."""
    global _lib
    if path is not None:
        return _bind(path)
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
            build()
        _lib = _bind(_LIB_PATH)
    return _lib


def threads() -> int:
    return int(os.environ.get("ESA_ORACLE_THREADS", os.cpu_count() or 1))


def _np(x, dtype):
    """numpy array of ``dtype``; bf16 tensors become their uint16 bit patterns."""
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            x = x.view(torch.int16)
        x = x.numpy()
    a = np.ascontiguousarray(x)
    if dtype == np.uint16 and a.dtype in (np.int16, np.uint16):
        return a.view(np.uint16)
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(vp) if a is not None else None


def _rows(B, Tq, rows):
    if rows is None:
        return np.arange(B * Tq, dtype=np.int64)
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


# shape["flags"] bits (the same values as the C ABI's)
RELU = 1       # ReLU on each indexer head's dot product before the weighted sum
PER_HEAD = 2   # one index set per indexer head, scored by that head alone


def indexer_row(qI, kI, wI, shape: dict, b: int, t: int, L=None, relu: bool = False, head: int = -1) -> np.ndarray:
    """int32 scores of row (b,t) against keys 0..q_offset+t: the weighted sum
    over indexer heads (head < 0) or one head's own unweighted score."""
    L = L or lib()
    qa, ka, wa = _np(qI, np.int8), _np(kI, np.int8), _np(wI, np.int32)
    n = shape["q_offset"] + t + 1
    out = np.empty(n, dtype=np.int32)
    r = L.oracle_indexer_row_mode(_ptr(qa), _ptr(ka), _ptr(wa), shape["B"], shape["Tq"], shape["Tk"],
                                  shape["q_offset"], shape["H_I"], shape["D_I"], b, t, int(relu), head, _ptr(out))
    if r != n:
        raise ValueError(f"oracle_indexer_row failed ({r}): score outside int32 or row beyond Tk")
    return out


def topk(qI, kI, wI, shape: dict, K: int, rows=None, L=None):
    """(idx, cnt) int32 for the listed flat rows: [n_rows,K] and [n_rows], or
    with per-head sets (shape flags) [n_rows,H_I,K] and [n_rows,H_I]."""
    L = L or lib()
    qa, ka, wa = _np(qI, np.int8), _np(kI, np.int8), _np(wI, np.int32)
    rr = _rows(shape["B"], shape["Tq"], rows)
    flags = int(shape.get("flags", 0))
    sets = (shape["H_I"],) if flags & PER_HEAD else ()
    idx = np.empty((len(rr), *sets, K), dtype=np.int32)
    cnt = np.empty((len(rr), *sets), dtype=np.int32)
    rc = L.oracle_topk_rows_mode(_ptr(qa), _ptr(ka), _ptr(wa), shape["B"], shape["Tq"], shape["Tk"],
                                 shape["q_offset"], shape["H_I"], shape["D_I"], K, flags, _ptr(rr), len(rr), _ptr(idx),
                                 _ptr(cnt), threads())
    if rc != 0:
        raise ValueError("oracle_topk_rows: a score does not fit in int32")
    return idx, cnt


def attention(q, k, v, idx, cnt, shape: dict, K: int, scale: float | None = None, g=None, lin=None, route=None,
              rows=None, L=None):
    """(out [n_rows,Hq,D] fp64, lse [n_rows,Hq] fp64) for the listed rows.

    idx/cnt are given per listed row (as returned by :func:`topk`); with
    per-head sets (shape flags) query head h reads set h // (Hq // H_I)."""
    L = L or lib()
    B, Tq, Hq, D = shape["B"], shape["Tq"], shape["Hq"], shape["D"]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    qa, ka, va = _np(q, np.uint16), _np(k, np.uint16), _np(v, np.uint16)
    rr = _rows(B, Tq, rows)
    nsets = shape["H_I"] if int(shape.get("flags", 0)) & PER_HEAD else 1
    ia = np.ascontiguousarray(np.asarray(idx, dtype=np.int32).reshape(len(rr) * nsets, K))
    ca = np.ascontiguousarray(np.asarray(cnt, dtype=np.int32).reshape(len(rr) * nsets))
    ga = _np(g, np.float32) if g is not None else None
    la = _np(lin, np.uint16) if lin is not None else None
    ra = _np(route, np.uint8) if route is not None else None
    out = np.empty((len(rr), Hq, D), dtype=np.float64)
    lse = np.empty((len(rr), Hq), dtype=np.float64)
    rc = L.oracle_attention_rows_sets(_ptr(qa), _ptr(ka), _ptr(va), _ptr(ia), _ptr(ca), K, nsets, B, Tq, shape["Tk"],
                                      shape["q_offset"], Hq, shape["Hkv"], D, float(scale), _ptr(ga), _ptr(la),
                                      _ptr(ra), _ptr(rr), len(rr), _ptr(out), _ptr(lse), threads())
    if rc != 0:
        raise ValueError("oracle_attention_rows: an index lies outside the causal prefix")
    return out, lse


def gated_sparse_attention(inp: dict, shape: dict, K: int, rows=None, gate=True, L=None):
    """The whole path for the listed rows: indexer -> top-K -> attention over the
    selected keys (or all keys for heads routed full) -> gate mix.

    Returns (idx, cnt, out, lse)."""
    L = L or lib()
    idx, cnt = topk(inp["qI"], inp["kI"], inp["wI"], shape, K, rows=rows, L=L)
    out, lse = attention(inp["q"], inp["k"], inp["v"], idx, cnt, shape, K,
                         g=inp["g"] if gate else None, lin=inp["lin"] if gate else None,
                         route=inp.get("route"), rows=rows, L=L)
    return idx, cnt, out, lse


def route_heads(k, shape: dict, W1, b1, W2, b2, L=None):
    """(route uint8 [B, Hq], margin fp64 [B, Hq]) of the attention router:
    mean key state over the cache -> ReLU(W1 x + b1) -> W2 h + b2, sparse iff
    the sparse logit >= the full one; margin = sparse - full logit."""
    L = L or lib()
    B, Hq = shape["B"], shape["Hq"]
    ka = _np(k, np.uint16)
    w1, bb1, w2, bb2 = (_np(a, np.float32) for a in (W1, b1, W2, b2))
    F = w1.shape[0]
    route = np.empty((B, Hq), dtype=np.uint8)
    margin = np.empty((B, Hq), dtype=np.float64)
    L.oracle_route_heads(_ptr(ka), B, shape["Tk"], shape["Hkv"], shape["D"], Hq, F, _ptr(w1), _ptr(bb1), _ptr(w2),
                         _ptr(bb2), _ptr(route), _ptr(margin))
    return route, margin


def kda(q, k, v, alpha, beta, state_in=None, scale: float | None = None, L=None):
    """(o fp64 [B, T, H, Dv], final state fp64 [B, H, Dk, Dv]) of the KDA
    linear-attention branch: per (sequence, head) the state forgets with
    alpha_t per key channel, then takes v_t under key k_t with strength beta_t
    (delta rule), and o_t = scale * S_t^T q_t. q, k bf16 [B, T, H, Dk]; v bf16
    [B, T, H, Dv]; alpha fp32 [B, T, H, Dk]; beta fp32 [B, T, H]; state_in
    fp32 [B, H, Dk, Dv] or None (zero). scale defaults to 1/sqrt(Dk)."""
    L = L or lib()
    qa, ka, va = _np(q, np.uint16), _np(k, np.uint16), _np(v, np.uint16)
    B, T, H, Dk = qa.shape
    Dv = va.shape[-1]
    aa, ba = _np(alpha, np.float32), _np(beta, np.float32)
    assert ka.shape == qa.shape and va.shape == (B, T, H, Dv) and aa.shape == qa.shape and ba.shape == (B, T, H)
    sa = _np(state_in, np.float32)
    assert sa is None or sa.shape == (B, H, Dk, Dv)
    o = np.empty((B, T, H, Dv), dtype=np.float64)
    st = np.empty((B, H, Dk, Dv), dtype=np.float64)
    sc = 1.0 / math.sqrt(Dk) if scale is None else float(scale)
    L.oracle_kda(_ptr(qa), _ptr(ka), _ptr(va), _ptr(aa), _ptr(ba), _ptr(sa), B, T, H, Dk, Dv, sc, _ptr(o), _ptr(st),
                 threads())
    return o, st


def threshold(qI, kI, wI, shape: dict, K: int, rows=None, L=None) -> np.ndarray:
    """int32 [n_rows, 2] threshold form (T, P) of each listed row's index set
    ([n_rows, H_I, 2] with per-head sets): key j <= p is selected iff
    s_j > T, or s_j == T and j <= P; T = INT32_MIN and P = p when the prefix
    holds at most K keys."""
    L = L or lib()
    qa, ka, wa = _np(qI, np.int8), _np(kI, np.int8), _np(wI, np.int32)
    rr = _rows(shape["B"], shape["Tq"], rows)
    flags = int(shape.get("flags", 0))
    sets = (shape["H_I"],) if flags & PER_HEAD else ()
    thr = np.empty((len(rr), *sets, 2), dtype=np.int32)
    rc = L.oracle_threshold_rows(_ptr(qa), _ptr(ka), _ptr(wa), shape["B"], shape["Tq"], shape["Tk"],
                                 shape["q_offset"], shape["H_I"], shape["D_I"], K, flags, _ptr(rr), len(rr), _ptr(thr),
                                 threads())
    if rc != 0:
        raise ValueError("oracle_threshold_rows: a score does not fit in int32")
    return thr
