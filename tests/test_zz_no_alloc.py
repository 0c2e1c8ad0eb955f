"""esa_topk_select_noalloc: top-K selection for callers that cannot allocate.

Code that runs inside a runtime owning every device allocation (a caching
allocator, a serving engine's reserved pool) may not call cudaMalloc, so it
cannot give esa_topk_select() a workspace. The no-allocation entry point
keeps that scratch in a fixed array inside the library. These tests call it
through the C ABI and compare its index sets with esa_topk_select()'s on the
same inputs, bit for bit (integer results), on two calls in a row — the
shared array must be left ready for the next call. This file is collected
last so that a run stopping at the first failure has run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import esa_inputs as E

pytestmark = pytest.mark.gpu

CASES = [
    # decode: the split selection, whose scratch holds barrier counters,
    # level histograms and per-block published counts
    dict(B=8, Tq=1, Tk=131072, q_offset=131071, Hq=32, Hkv=1, D=128, H_I=1, D_I=64, top_k=2048),
    dict(B=2, Tq=1, Tk=30000, q_offset=29999, Hq=8, Hkv=1, D=64, H_I=3, D_I=32, top_k=700, weights="1to4"),
    # per-head index sets with the ReLU indexer: 2 x 4 single-head selection
    # rows, one weight of 1 from the library's own constant
    dict(B=2, Tq=1, Tk=30000, q_offset=29999, Hq=8, Hkv=1, D=64, H_I=4, D_I=64, top_k=512, flags=3),
    # prefill: the row-tiled selection (only the status word in scratch)
    dict(B=1, Tq=300, Tk=300, Hq=4, Hkv=1, D=64, H_I=1, D_I=64, top_k=64),
]


@pytest.mark.parametrize("over", CASES, ids=["decode-8x131072", "decode-2x30000", "decode-per-head-relu",
                                             "prefill-300"])
def test_noalloc_matches_workspace_call(over):
    import long_context_sparse_20_b300 as esa
    cfg = E.small_config(seed=909, **over)
    sh = E.shape_of(cfg)
    K = cfg["top_k"]
    inp = E.make_inputs(cfg)
    qI, kI, wI = inp["qI"].cuda(), inp["kI"].cuda(), inp["wI"].cuda()
    shape = esa.shape_from(sh)
    B, Tq = sh["B"], sh["Tq"]
    sets = (sh["H_I"],) if sh["flags"] & esa.PER_HEAD_SETS else ()  # per-head sets: [B, Tq, H_I, K]

    ws = esa.workspace_for(esa.OP_TOPK_SELECT, shape, K)
    ref_idx = torch.empty(B, Tq, *sets, K, dtype=torch.int32, device="cuda")
    ref_cnt = torch.empty(B, Tq, *sets, dtype=torch.int32, device="cuda")
    esa.esa_topk_select(qI, kI, wI, shape, K, ref_idx, ref_cnt, ws)
    assert esa.esa_read_status(ws) == esa.OK

    lib = esa._lib
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        idx = torch.full((B, Tq, *sets, K), -7, dtype=torch.int32, device="cuda")
        cnt = torch.full((B, Tq, *sets), -7, dtype=torch.int32, device="cuda")
        status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        rc = lib.esa_topk_select_noalloc(ctypes.c_void_p(qI.data_ptr()), ctypes.c_void_p(kI.data_ptr()),
                                         ctypes.c_void_p(wI.data_ptr()), ctypes.byref(shape), K,
                                         ctypes.c_void_p(idx.data_ptr()), ctypes.c_void_p(cnt.data_ptr()),
                                         ctypes.c_void_p(status.data_ptr()), stream)
        assert rc == esa.OK, esa.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == esa.OK, (call, int(status.item()))
        assert torch.equal(cnt, ref_cnt), call
        assert torch.equal(idx, ref_idx), (call, int((idx != ref_idx).any(dim=-1).sum()))


def test_noalloc_rejects_shapes_beyond_its_scratch():
    """A decode batch of 64 rows: the split selection's scratch (per-block
    publications plus per-row control state) exceeds the fixed array, so the
    call returns ESA_ERR_UNSUPPORTED and writes nothing. The tensors are real
    and sized for the shape, so that even a call that went ahead would only
    touch valid memory."""
    import long_context_sparse_20_b300 as esa
    K = 512
    sh = dict(B=64, Tq=1, Tk=20000, q_offset=19999, Hq=8, Hkv=1, D=64, H_I=1, D_I=64)
    shape = esa.shape_from(sh)
    # the entry point's own rule: the split plan (one block per SM, at least
    # two blocks per row, spans of at most 16384 keys) whose workspace is
    # larger than the fixed scratch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = sh["B"] * sh["Tq"]
    split = rows <= sms // 2 and -(-(sh["q_offset"] + 1) // (sms // rows)) <= 16384
    need = esa.esa_workspace_size(esa.OP_TOPK_SELECT, shape, K)
    if not (split and need > (8 << 20)):
        pytest.skip("on this device the shape's selection fits the fixed scratch")
    qI = torch.zeros(sh["B"], 1, 1, sh["D_I"], dtype=torch.int8, device="cuda")
    kI = torch.zeros(sh["B"], sh["Tk"], sh["D_I"], dtype=torch.int8, device="cuda")
    wI = torch.ones(1, dtype=torch.int32, device="cuda")
    idx = torch.full((sh["B"], 1, K), -7, dtype=torch.int32, device="cuda")
    cnt = torch.full((sh["B"], 1), -7, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = esa._lib.esa_topk_select_noalloc(p(qI), p(kI), p(wI), ctypes.byref(shape), K, p(idx), p(cnt), None, stream)
    assert rc == esa.ERR_UNSUPPORTED, esa.status_string(rc)
    torch.cuda.synchronize()
    assert (idx == -7).all() and (cnt == -7).all()
