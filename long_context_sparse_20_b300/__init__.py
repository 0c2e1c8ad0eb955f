"""Python binding of libesa.so — gated fine-grained sparse attention on B300.

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Functions carry the names of the C entry points (see
``include/esa.h``) and take torch CUDA tensors (device memory) plus an
optional stream; they raise :class:`EsaError` when a call returns a non-zero
status. There is no CPU fallback: importing this package without the built
library raises ImportError.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libesa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with `python long_context_sparse_20_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_BAD_INDEX, ERR_WORKSPACE, ERR_INTERNAL = range(8)
(OP_INDEXER_SCORE, OP_TOPK_SELECT, OP_SPARSE_ATTN, OP_GATED_MIX, OP_ROUTED_ATTN, OP_ROUTE_HEADS, OP_TOPK_THRESHOLD,
 OP_GATED_SPARSE_ATTN) = range(8)
INDEXER_RELU, PER_HEAD_SETS = 1, 2  # esa_shape.flags


class esa_shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("Tq", ctypes.c_int64), ("Tk", ctypes.c_int64), ("q_offset", ctypes.c_int64),
                ("Hq", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("D", ctypes.c_int32), ("H_I", ctypes.c_int32),
                ("D_I", ctypes.c_int32), ("flags", ctypes.c_int32)]


class EsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_sp = ctypes.POINTER(esa_shape)
_SIGS = {
    "esa_workspace_size": (_sz, [ctypes.c_int, _sp, ctypes.c_int]),
    "esa_workspace_init": (_i32, [_vp, _sz, _vp]),
    "esa_indexer_score": (_i32, [_vp, _vp, _vp, _sp, _vp, _vp, _sz, _vp]),
    "esa_topk_select": (_i32, [_vp, _vp, _vp, _sp, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]),
    "esa_sparse_attn": (_i32, [_vp, _vp, _vp, _vp, _vp, _sp, ctypes.c_int, ctypes.c_float, _vp, _vp, _vp, _vp, _vp,
                               _sz, _vp]),
    "esa_gated_mix": (_i32, [_vp, _vp, _vp, _vp, _sp, _vp, _vp]),
    "esa_gated_sparse_attn": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _sp, ctypes.c_int, ctypes.c_float, _vp, _vp, _vp,
                                     _vp, _vp, _vp, _vp, _sz, _vp]),
    "esa_routed_attn": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _sp, ctypes.c_int, ctypes.c_float, _vp, _vp, _vp,
                               _vp, _sz, _vp]),
    "esa_topk_threshold": (_i32, [_vp, _vp, _vp, _sp, ctypes.c_int, _vp, _vp, _sz, _vp]),
    "esa_topk_select_noalloc": (_i32, [_vp, _vp, _vp, _sp, ctypes.c_int, _vp, _vp, _vp, _vp]),
    "esa_route_heads": (_i32, [_vp, _vp, _vp, _vp, _vp, _sp, ctypes.c_int, _vp, _vp, _vp, _sz, _vp]),
    "esa_kda": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64, _i32, _i32, _i32, ctypes.c_float,
                       _vp, _vp, _vp, _vp, _sz, _vp]),
    "esa_kda_workspace_size": (_sz, [ctypes.c_int64, ctypes.c_int64, _i32, _i32, _i32]),
    "esa_read_status": (_i32, [_vp, _vp, ctypes.POINTER(_i32)]),
    "esa_status_string": (ctypes.c_char_p, [_i32]),
    "esa_binary_version": (ctypes.c_int, []),
    "esa_cache_append": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _sp, _vp]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.restype, _f.argtypes = _res, _args


def exported_symbols():
    return sorted(_SIGS)


def status_string(st: int) -> str:
    return _lib.esa_status_string(st).decode()


def make_shape(B, Tq, Tk, q_offset, Hq=1, Hkv=1, D=64, H_I=1, D_I=64, flags=0) -> esa_shape:
    return esa_shape(B, Tq, Tk, q_offset, Hq, Hkv, D, H_I, D_I, flags)


def shape_from(d: dict) -> esa_shape:
    return make_shape(*(d[k] for k in ("B", "Tq", "Tk", "q_offset", "Hq", "Hkv", "D", "H_I", "D_I")),
                      flags=int(d.get("flags", 0)))


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, ref: torch.Tensor):
    if stream is None:
        stream = torch.cuda.current_stream(ref.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(st: int, where: str):
    if st != OK:
        raise EsaError(st, where)


class Workspace:
    """A zero-initialised device workspace (torch-allocated uint8 buffer)."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = max(256, int(nbytes))
        self.buf = torch.zeros(self.nbytes, dtype=torch.uint8, device=device)

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    def fits(self, nbytes: int) -> bool:
        return nbytes <= self.nbytes


def esa_workspace_size(op: int, shape: esa_shape, top_k: int = 1) -> int:
    return int(_lib.esa_workspace_size(op, ctypes.byref(shape), top_k))


def esa_workspace_init(ws: Workspace, stream=None):
    _check(_lib.esa_workspace_init(ws.ptr, ws.nbytes, _stream(stream, ws.buf)), "esa_workspace_init")


def workspace_for(op: int, shape: esa_shape, top_k: int = 1, device="cuda") -> Workspace:
    n = esa_workspace_size(op, shape, top_k)
    if n == 0:
        raise EsaError(ERR_INVALID, "esa_workspace_size")
    return Workspace(n, device)


def esa_indexer_score(qI, kI, wI, shape: esa_shape, scores, ws: Workspace, stream=None):
    _check(_lib.esa_indexer_score(_p(qI), _p(kI), _p(wI), ctypes.byref(shape), _p(scores), ws.ptr, ws.nbytes,
                                  _stream(stream, qI)), "esa_indexer_score")


def esa_topk_select(qI, kI, wI, shape: esa_shape, top_k: int, idx, cnt, ws: Workspace, stream=None):
    _check(_lib.esa_topk_select(_p(qI), _p(kI), _p(wI), ctypes.byref(shape), top_k, _p(idx), _p(cnt), ws.ptr,
                                ws.nbytes, _stream(stream, qI)), "esa_topk_select")


def esa_topk_threshold(qI, kI, wI, shape: esa_shape, top_k: int, thr, ws: Workspace, stream=None):
    """thr int32 [B, Tq, 2]: the threshold form (T, P) of every row's Top-K set."""
    _check(_lib.esa_topk_threshold(_p(qI), _p(kI), _p(wI), ctypes.byref(shape), top_k, _p(thr), ws.ptr, ws.nbytes,
                                   _stream(stream, qI)), "esa_topk_threshold")


def esa_topk_select_noalloc(qI, kI, wI, shape: esa_shape, top_k: int, idx, cnt, dev_status=None, stream=None):
    """esa_topk_select without a workspace: for callers that may not allocate
    device memory (the library's own fixed scratch array is used)."""
    _check(_lib.esa_topk_select_noalloc(_p(qI), _p(kI), _p(wI), ctypes.byref(shape), top_k, _p(idx), _p(cnt),
                                        _p(dev_status), _stream(stream, qI)), "esa_topk_select_noalloc")


def _bits(t):
    """bf16 tensors travel as their 16-bit patterns."""
    if t is None:
        return None
    assert t.dtype == torch.bfloat16, t.dtype
    return t


def esa_sparse_attn(q, k, v, idx, cnt, shape: esa_shape, top_k: int, scale: float, g, lin, out, lse,
                    ws: Workspace, stream=None):
    _check(_lib.esa_sparse_attn(_p(_bits(q)), _p(_bits(k)), _p(_bits(v)), _p(idx), _p(cnt), ctypes.byref(shape),
                                top_k, float(scale), _p(g), _p(_bits(lin)), _p(out), _p(lse), ws.ptr, ws.nbytes,
                                _stream(stream, q)), "esa_sparse_attn")


def esa_gated_sparse_attn(q, k, v, qI, kI, wI, shape: esa_shape, top_k: int, scale: float, g, lin, out, lse=None,
                          idx=None, cnt=None, ws: Workspace = None, stream=None):
    """The whole path (indexer, top-K, gathered attention, gate mix) in one
    call; one launch for decode-like shapes. idx/cnt optional outputs."""
    _check(_lib.esa_gated_sparse_attn(_p(_bits(q)), _p(_bits(k)), _p(_bits(v)), _p(qI), _p(kI), _p(wI),
                                      ctypes.byref(shape), top_k, float(scale), _p(g), _p(_bits(lin)), _p(out), _p(lse),
                                      _p(idx), _p(cnt), ws.ptr, ws.nbytes, _stream(stream, q)), "esa_gated_sparse_attn")


def esa_gated_mix(attn, lin, g, head_mask, shape: esa_shape, out, stream=None):
    _check(_lib.esa_gated_mix(_p(attn), _p(_bits(lin)), _p(g), _p(head_mask), ctypes.byref(shape), _p(out),
                              _stream(stream, attn)), "esa_gated_mix")


def esa_cache_append(k_new, v_new, kI_new, k, v, kI, shape: esa_shape, stream=None):
    ref = next(t for t in (k, v, kI) if t is not None)
    _check(_lib.esa_cache_append(_p(_bits(k_new)), _p(_bits(v_new)), _p(kI_new), _p(_bits(k)), _p(_bits(v)), _p(kI),
                                 ctypes.byref(shape), _stream(stream, ref)), "esa_cache_append")


def esa_routed_attn(q, k, v, qI, kI, wI, route, shape: esa_shape, top_k: int, scale: float, g, lin, out,
                    ws: Workspace, stream=None):
    _check(_lib.esa_routed_attn(_p(_bits(q)), _p(_bits(k)), _p(_bits(v)), _p(qI), _p(kI), _p(wI), _p(route),
                                ctypes.byref(shape), top_k, float(scale), _p(g), _p(_bits(lin)), _p(out), ws.ptr,
                                ws.nbytes, _stream(stream, q)), "esa_routed_attn")


def esa_route_heads(k, W1, b1, W2, b2, shape: esa_shape, route, margin, ws: Workspace, stream=None):
    hidden = int(W1.shape[0])
    _check(_lib.esa_route_heads(_p(_bits(k)), _p(W1), _p(b1), _p(W2), _p(b2), ctypes.byref(shape), hidden, _p(route),
                                _p(margin), ws.ptr, ws.nbytes, _stream(stream, k)), "esa_route_heads")


def esa_kda_workspace_size(B: int, T: int, H: int, Dk: int, Dv: int) -> int:
    """Bytes of workspace the chunked form of esa_kda needs (0: none)."""
    return int(_lib.esa_kda_workspace_size(B, T, H, Dk, Dv))


def esa_kda(q, k, v, alpha, beta, state_in=None, o=None, lin=None, state_out=None, scale: float | None = None,
            ws=None, chunked: bool = True, stream=None):
    """The KDA linear-attention branch: q, k bf16 [B, T, H, Dk]; v bf16
    [B, T, H, Dv]; alpha fp32 [B, T, H, Dk]; beta fp32 [B, T, H]; state_in /
    state_out fp32 [B, H, Dk, Dv] (may be the same tensor); o fp32 and lin
    bf16 [B, T, H, Dv]. scale defaults to 1/sqrt(Dk). chunked: the chunked
    form, in ``ws`` (a uint8 device tensor of esa_kda_workspace_size bytes;
    allocated here when None); otherwise the steps one by one."""
    B, T, H, Dk = (int(x) for x in q.shape)
    Dv = int(v.shape[-1])
    for t, want in ((k, q.shape), (alpha, q.shape), (v, (B, T, H, Dv)), (beta, (B, T, H))):
        assert tuple(t.shape) == tuple(want), (tuple(t.shape), tuple(want))
        assert t.is_contiguous()
    for t in (state_in, state_out, o, lin):
        assert t is None or t.is_contiguous()
    for t in (alpha, beta, state_in, state_out, o):
        assert t is None or t.dtype == torch.float32, t.dtype
    sc = Dk ** -0.5 if scale is None else float(scale)
    wp, wn = None, 0
    if chunked:
        need = esa_kda_workspace_size(B, T, H, Dk, Dv)
        if need:
            if ws is None:
                ws = torch.empty(need + 256, dtype=torch.uint8, device=q.device)
            off = (-ws.data_ptr()) % 256
            wp, wn = ctypes.c_void_p(ws.data_ptr() + off), ws.numel() - off
    _check(_lib.esa_kda(_p(_bits(q)), _p(_bits(k)), _p(_bits(v)), _p(alpha), _p(beta), _p(state_in), B, T, H, Dk, Dv,
                        sc, _p(o), _p(_bits(lin)), _p(state_out), wp, wn, _stream(stream, q)), "esa_kda")


def esa_read_status(ws: Workspace, stream=None) -> int:
    st = _i32(0)
    _check(_lib.esa_read_status(ws.ptr, _stream(stream, ws.buf), ctypes.byref(st)), "esa_read_status")
    return int(st.value)
