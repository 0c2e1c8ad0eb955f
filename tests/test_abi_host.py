"""The C-ABI library without a GPU: it loads, exports every symbol that
include/*.h declares, and rejects bad arguments on the host before any
launch (no CUDA call is made by these checks)."""
import ctypes
import glob
import os
import re

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names |= set(re.findall(r"ESA_API\s+[\w\s\*]*?\b(esa_\w+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_five_calls():
    d = _declared()
    for name in ["esa_indexer_score", "esa_topk_select", "esa_sparse_attn", "esa_gated_mix", "esa_routed_attn",
                 "esa_workspace_size", "esa_read_status"]:
        assert name in d


def test_library_exports_every_declared_symbol():
    import long_context_sparse_20_b300 as esa
    lib = ctypes.CDLL(esa.LIB_PATH)
    for name in _declared():
        assert hasattr(lib, name), name
    assert set(_declared()) <= set(esa.exported_symbols())


def test_library_is_built_for_sm_103a_only():
    """The build compiles every kernel for sm_103a and nothing else; without
    a GPU the runtime cannot load the kernels and the query says so."""
    import long_context_sparse_20_b300 as esa
    from long_context_sparse_20_b300 import build
    gencode = [build.ARCH[i + 1] for i, a in enumerate(build.ARCH) if a == "-gencode"]
    assert gencode == ["arch=compute_103a,code=sm_103a"]
    if not torch.cuda.is_available():
        assert esa._lib.esa_binary_version() == -1


@pytest.mark.gpu
def test_kernels_load_as_sm_103():
    import long_context_sparse_20_b300 as esa
    assert esa._lib.esa_binary_version() == 103


def _shape(esa, **kw):
    d = dict(B=1, Tq=4, Tk=4, q_offset=0, Hq=4, Hkv=1, D=64, H_I=1, D_I=32)
    d.update(kw)
    return esa.shape_from(d)


def test_cache_append_validation():
    import long_context_sparse_20_b300 as esa
    L = esa._lib
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    s = _shape(esa, Tq=1, Tk=8, q_offset=7)
    # a cache without its new rows, and nothing to write
    assert L.esa_cache_append(None, fake, fake, fake, fake, fake, ctypes.byref(s), None) == esa.ERR_INVALID
    assert L.esa_cache_append(None, None, None, None, None, None, ctypes.byref(s), None) == esa.ERR_INVALID
    # misaligned pointer
    odd = ctypes.c_void_p(0x1008)
    assert L.esa_cache_append(fake, fake, fake, fake, fake, odd, ctypes.byref(s), None) == esa.ERR_INVALID
    # positions past the cache
    bad = _shape(esa, Tq=2, Tk=8, q_offset=7)
    assert L.esa_cache_append(fake, fake, fake, fake, fake, fake, ctypes.byref(bad), None) == esa.ERR_INVALID
    # nothing to do: B * Tq = 0 launches nothing
    empty = _shape(esa, B=0, Tq=1, Tk=8, q_offset=7)
    assert L.esa_cache_append(fake, fake, fake, fake, fake, fake, ctypes.byref(empty), None) == esa.OK


def test_host_validation_rejects_before_launch():
    import long_context_sparse_20_b300 as esa
    L = esa._lib
    fake = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    s = _shape(esa)
    # null pointers
    assert L.esa_topk_select(None, fake, fake, ctypes.byref(s), 4, fake, fake, fake, 1 << 20, None) == esa.ERR_INVALID
    # top_k out of range
    assert L.esa_topk_select(fake, fake, fake, ctypes.byref(s), 0, fake, fake, fake, 1 << 20, None) == esa.ERR_INVALID
    # q_offset + Tq > Tk
    bad = _shape(esa, Tq=5)
    assert L.esa_topk_select(fake, fake, fake, ctypes.byref(bad), 4, fake, fake, fake, 1 << 20, None) == esa.ERR_INVALID
    # Hq not a multiple of Hkv; unsupported D; unsupported D_I / H_I
    for kw, code in [(dict(Hq=6, Hkv=4), esa.ERR_INVALID), (dict(D=96), esa.ERR_UNSUPPORTED)]:
        sh = _shape(esa, **kw)
        assert L.esa_sparse_attn(fake, fake, fake, fake, fake, ctypes.byref(sh), 4, 0.125, None, None, fake, None,
                                 fake, 1 << 20, None) == code
    for kw in [dict(D_I=48), dict(H_I=17), dict(H_I=0)]:
        sh = _shape(esa, **kw)
        assert L.esa_topk_select(fake, fake, fake, ctypes.byref(sh), 4, fake, fake, fake, 1 << 20, None) == \
            esa.ERR_UNSUPPORTED
    # gate without lin (both or neither)
    assert L.esa_sparse_attn(fake, fake, fake, fake, fake, ctypes.byref(s), 4, 0.125, fake, None, fake, None, fake,
                             1 << 20, None) == esa.ERR_INVALID
    # non-positive scale
    assert L.esa_sparse_attn(fake, fake, fake, fake, fake, ctypes.byref(s), 4, 0.0, None, None, fake, None, fake,
                             1 << 20, None) == esa.ERR_INVALID
    # misaligned tensor
    odd = ctypes.c_void_p(0x1008)
    assert L.esa_gated_mix(odd, fake, fake, None, ctypes.byref(s), fake, None) == esa.ERR_INVALID
    # routed attention: head dim outside {64, 128}
    sh = _shape(esa, D=96)
    assert L.esa_routed_attn(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(sh), 4, 0.125, None, None, fake,
                             fake, 1 << 20, None) == esa.ERR_UNSUPPORTED
    # workspace: null or misaligned
    assert L.esa_indexer_score(fake, fake, fake, ctypes.byref(s), fake, None, 1 << 20, None) == esa.ERR_WORKSPACE
    assert L.esa_indexer_score(fake, fake, fake, ctypes.byref(s), fake, ctypes.c_void_p(0x1010), 1 << 20, None) == \
        esa.ERR_WORKSPACE


def test_host_validation_of_indexer_flags():
    """Unknown flag bits are invalid; per-head sets need Hq % H_I == 0 and, for
    attention, heads per set and heads per key/value head dividing one
    another. All of it is decided before any launch."""
    import long_context_sparse_20_b300 as esa
    L = esa._lib
    fake = ctypes.c_void_p(0x1000)
    sh = _shape(esa, flags=4)
    assert L.esa_topk_select(fake, fake, fake, ctypes.byref(sh), 4, fake, fake, fake, 1 << 20, None) == esa.ERR_INVALID
    for kw, code in [(dict(Hq=6, Hkv=1, H_I=4), esa.ERR_INVALID),            # 6 % 4
                     (dict(Hq=12, Hkv=3, H_I=2), esa.ERR_UNSUPPORTED)]:      # 6 heads per set, 4 per KV head
        sh = _shape(esa, flags=esa.PER_HEAD_SETS, **kw)
        assert L.esa_sparse_attn(fake, fake, fake, fake, fake, ctypes.byref(sh), 4, 0.125, None, None, fake, None,
                                 fake, 1 << 20, None) == code, kw
    sh = _shape(esa, flags=esa.PER_HEAD_SETS, Hq=6, Hkv=6, H_I=4)
    assert L.esa_routed_attn(fake, fake, fake, fake, fake, fake, fake, ctypes.byref(sh), 4, 0.125, None, None, fake,
                             fake, 1 << 20, None) == esa.ERR_INVALID  # 6 % 4


def test_workspace_size_rejects_bad_shapes():
    import long_context_sparse_20_b300 as esa
    assert esa.esa_workspace_size(esa.OP_TOPK_SELECT, _shape(esa, Tq=9), 4) == 0
    assert esa.esa_workspace_size(99, _shape(esa), 4) == 0
    assert esa.esa_workspace_size(esa.OP_SPARSE_ATTN, _shape(esa), 0) == 0


def test_status_strings():
    import long_context_sparse_20_b300 as esa
    assert esa.status_string(esa.ERR_TIMEOUT) == "device wait timed out"
    assert esa.status_string(esa.OK) == "ok"
    assert esa.status_string(123) == "unknown status"


def test_host_validation_of_kda():
    import long_context_sparse_20_b300 as esa
    L = esa._lib
    f = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails (or returns) first
    mis = ctypes.c_void_p(0x1008)

    def call(q=f, k=f, v=f, a=f, b=f, s_in=None, B=1, T=4, H=2, Dk=128, Dv=128, o=f, lin=None, s_out=None, ws=None,
             ws_bytes=0):
        return L.esa_kda(q, k, v, a, b, s_in, B, T, H, Dk, Dv, 0.1, o, lin, s_out, ws, ws_bytes, None)

    assert call(Dk=96) == esa.ERR_UNSUPPORTED
    assert call(Dv=24) == esa.ERR_UNSUPPORTED and call(Dv=1024) == esa.ERR_UNSUPPORTED
    assert call(H=0) == esa.ERR_INVALID and call(T=-1) == esa.ERR_INVALID
    assert call(B=70000) == esa.ERR_UNSUPPORTED
    assert call(q=None) == esa.ERR_INVALID and call(b=None) == esa.ERR_INVALID
    assert call(k=mis) == esa.ERR_INVALID and call(o=mis) == esa.ERR_INVALID and call(s_out=mis) == esa.ERR_INVALID
    assert call(lin=ctypes.c_void_p(0x1004)) == esa.ERR_INVALID
    # nothing to do: no launch
    assert call(B=0) == esa.OK
    assert call(q=None, k=None, v=None, a=None, b=None, T=0) == esa.OK
    # the chunked form's workspace: too small or misaligned
    need = esa.esa_kda_workspace_size(1, 100, 2, 128, 128)
    assert need > 0
    assert call(T=100, ws=ctypes.c_void_p(0x100000), ws_bytes=need - 1) == esa.ERR_WORKSPACE
    assert call(T=100, ws=ctypes.c_void_p(0x100010), ws_bytes=need) == esa.ERR_WORKSPACE


def test_kda_workspace_size():
    """A 256-byte status word, then one record per (sequence, head, chunk of
    16 steps) of fp32 words: two 16 x Dk matrices with rows padded to Dk + 4,
    one with rows padded to Dk + 8, g_last (Dk), a flag (padded to four) and
    two 16 x Dv matrices (the records 256-byte aligned as a whole); at most
    256 chunks at a time, plus the carried state (256-byte aligned) and a
    second set of records beyond that. None for T <= 4 or unsupported
    shapes."""
    import long_context_sparse_20_b300 as esa
    rec = lambda Dk, Dv: 4 * (2 * 16 * (Dk + 4) + 16 * (Dk + 8) + Dk + 4 + 2 * 16 * Dv)
    a256 = lambda n: (n + 255) // 256 * 256
    assert esa.esa_kda_workspace_size(2, 100, 3, 128, 64) == 256 + a256(2 * 3 * 7 * rec(128, 64))
    assert esa.esa_kda_workspace_size(1, 4096, 2, 64, 128) == 256 + a256(2 * 256 * rec(64, 128))
    carry = 1 * 16 * 128 * 128 * 4
    # more than 256 chunks: two record buffers (one filled while the other is read)
    assert esa.esa_kda_workspace_size(1, 32768, 16, 128, 128) == 256 + carry + 2 * a256(16 * 256 * rec(128, 128))
    assert esa.esa_kda_workspace_size(1, 4, 2, 128, 128) == 0
    assert esa.esa_kda_workspace_size(1, 100, 2, 96, 128) == 0
