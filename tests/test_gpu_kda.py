"""KDA linear-attention branch: the CUDA path (through the C ABI) against the
CPU oracle on the same seeded inputs.

Tolerance. The kernel keeps the state in fp32 and sums in a fixed order; the
oracle is fp64. The recurrence contracts (forgetting factors <= 1, unit keys,
write strengths in [0, 1]), so rounding errors do not grow with T: an fp32
emulation of the same steps on the workload's inputs stays within 4e-7 of
max|o| over 4000 steps. The tests allow REL = 1e-4 of the largest reference
magnitude (o, and the state separately), 250 times that; the bf16 `lin`
output may differ from o by one bf16 rounding (2^-8 relative) beyond it."""
import numpy as np
import pytest
import torch

import esa_inputs as E
import oracle as O
from gpu_helpers import assert_close, assert_idx_equal, esa, gpu_attn, gpu_topk, to_dev

pytestmark = pytest.mark.gpu

REL = 1e-4


def _inputs(B, T, H, Dk, Dv, seed, state):
    return E.kda_inputs(B, T, H, Dk, Dv, seed, state=state)


def _gpu(x: dict, state_in=None, inplace=False, lin=True, o=True, chunked=True, ws=None):
    m = esa()
    B, T, H, Dk = (int(s) for s in x["q"].shape)
    Dv = int(x["v"].shape[-1])
    d = {k: v.cuda() for k, v in x.items() if k != "state"}
    out = torch.full((B, T, H, Dv), float("nan"), dtype=torch.float32, device="cuda") if o else None
    lo = torch.zeros((B, T, H, Dv), dtype=torch.bfloat16, device="cuda") if lin else None
    si = state_in.cuda() if state_in is not None else None
    so = si if inplace else torch.full((B, H, Dk, Dv), float("nan"), dtype=torch.float32, device="cuda")
    m.esa_kda(d["q"], d["k"], d["v"], d["alpha"], d["beta"], state_in=si, o=out, lin=lo, state_out=so,
              chunked=chunked, ws=ws)
    torch.cuda.synchronize()
    return (out.cpu() if o else None), (lo.cpu() if lin else None), so.cpu()


# both forms of the recurrence: chunks of 16 steps (a workspace given), and
# the steps one by one
FORMS = pytest.mark.parametrize("chunked", [True, False], ids=["chunked", "stepwise"])


def _check(o, lin, so, ro, rs):
    tol = REL * float(np.abs(ro).max())
    assert torch.isfinite(o).all()
    err = np.abs(o.double().numpy() - ro)
    assert err.max() <= tol, f"o: max err {err.max():.3e} > {tol:.3e}"
    if lin is not None:
        lerr = np.abs(lin.double().numpy() - ro) - np.abs(ro) * 2.0 ** -8
        assert lerr.max() <= 1.01 * tol, f"lin: {lerr.max():.3e}"
        assert torch.equal(lin, o.to(torch.bfloat16)), "lin is not o rounded to bf16"
    stol = REL * max(float(np.abs(rs).max()), 1e-30)
    serr = np.abs(so.double().numpy() - rs)
    assert serr.max() <= stol, f"state: max err {serr.max():.3e} > {stol:.3e}"


KDA_CASES = [
    dict(B=1, T=1, H=2, Dk=128, Dv=128, state=True),   # one decode step
    dict(B=2, T=4, H=2, Dk=64, Dv=128, state=True),    # few steps (the streaming kernel)
    dict(B=2, T=37, H=3, Dk=64, Dv=64, state=False),   # one ragged chunk
    dict(B=1, T=5, H=1, Dk=128, Dv=48, state=True),    # three column blocks
    dict(B=1, T=100, H=2, Dk=128, Dv=64, state=True),  # several chunks, ragged tail
    dict(B=1, T=257, H=2, Dk=128, Dv=128, state=False),
    dict(B=3, T=70, H=1, Dk=64, Dv=16, state=True),    # one column block
    # at Dk = 128 a grid that fits on the SMs at one block each holds one
    # column per lane, larger ones two: this one launches 1024 blocks
    dict(B=4, T=41, H=32, Dk=128, Dv=128, state=True),
]


@FORMS
@pytest.mark.parametrize("c", KDA_CASES, ids=lambda c: "-".join(f"{k}{v}" for k, v in c.items()))
def test_kda_small(c, chunked):
    x = _inputs(c["B"], c["T"], c["H"], c["Dk"], c["Dv"], 300 + c["T"], c["state"])
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x.get("state"))
    o, lin, so = _gpu(x, state_in=x.get("state"), chunked=chunked)
    _check(o, lin, so, ro, rs)


@pytest.mark.parametrize("inplace", [False, True])
def test_kda_chunked_over_segments(inplace):
    """More than 256 chunks (4096 steps) in one call: the chunked form runs
    in segments and carries the state between them; a ragged last chunk;
    the final state written over the initial one when asked."""
    x = _inputs(2, 4500, 2, 64, 48, 77, True)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"].clone(), inplace=inplace)
    _check(o, lin, so, ro, rs)


@FORMS
def test_kda_state_carried_across_calls(chunked):
    """Chunked prefill: 100 steps in one call, or 64 then 36 with the state
    updated in place, give the same bits (the state is carried in fp32 and
    the split falls on a boundary of both forms' step groups, 32 staged
    steps and 16-step chunks, so every step is computed alike); a split at
    45 (steps grouped differently) matches the oracle; both match the
    oracle."""
    x = _inputs(2, 100, 2, 128, 128, 71, True)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"], chunked=chunked)
    _check(o, lin, so, ro, rs)
    for cut, exact in ((64, True), (45, False)):
        st = x["state"].clone().cuda()
        parts = []
        for a, b in ((0, cut), (cut, 100)):
            xs = {k: (v[:, a:b].contiguous() if k != "state" else v) for k, v in x.items()}
            po, _, _ = _gpu(xs, state_in=st, inplace=True, lin=False, chunked=chunked)
            parts.append(po)
        oc = torch.cat(parts, dim=1)
        if exact:
            assert torch.equal(oc, o)
            assert torch.equal(st.cpu(), so)
        else:
            _check(oc, None, st.cpu(), ro, rs)


@FORMS
def test_kda_empty_and_state_only(chunked):
    """T = 0 hands the initial state back; no outputs requested still
    advances the state."""
    x = _inputs(1, 6, 2, 64, 64, 72, True)
    m = esa()
    si = x["state"].cuda()
    so = torch.full_like(si, float("nan"))
    e = {k: v[:, :0].contiguous().cuda() for k, v in x.items() if k != "state"}
    m.esa_kda(e["q"], e["k"], e["v"], e["alpha"], e["beta"], state_in=si, state_out=so)
    torch.cuda.synchronize()
    assert torch.equal(so, si)
    _, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    _, _, so2 = _gpu(x, state_in=x["state"], lin=False, o=False, chunked=chunked)
    assert np.abs(so2.double().numpy() - rs).max() <= REL * np.abs(rs).max()
    # zero initial state when none is given
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    o, lin, so = _gpu(x, chunked=chunked)
    _check(o, lin, so, ro, rs)


@FORMS
@pytest.mark.parametrize("T", [3, 70])
def test_kda_extreme_gates(T, chunked):
    """Gates at their ends on every kernel (a few steps and many, both
    forms): alpha = 0 (the state is wiped), alpha = 1 (nothing forgotten),
    beta = 0 (no write) and beta = 1 (full replacement) mixed over steps,
    heads and channels. In the chunked form nearly every chunk then holds a
    zero forgetting factor and runs step by step."""
    x = _inputs(2, T, 3, 128, 64, 90 + T, True)
    rng = np.random.default_rng(T)
    a = x["alpha"].numpy().copy()
    pick = rng.random(a.shape)
    a[pick < 0.1] = 0.0
    a[pick > 0.8] = 1.0
    x["alpha"] = torch.from_numpy(a)
    bt = x["beta"].numpy().copy()
    pb = rng.random(bt.shape)
    bt[pb < 0.2] = 0.0
    bt[pb > 0.8] = 1.0
    x["beta"] = torch.from_numpy(bt)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"], chunked=chunked)
    _check(o, lin, so, ro, rs)


def test_kda_chunked_few_flagged_chunks():
    """Forgetting factors of 0 or near it in a few places: chunks whose
    cumulative factor falls below 2^-60 run step by step, the others as
    matrix products (one with factors down to 2^-35), and the state passes
    between the two kinds of chunk."""
    x = _inputs(1, 200, 2, 128, 32, 78, True)
    a = x["alpha"].numpy().copy()
    a[0, 37, 0, 5] = 0.0        # chunk 2, head 0: flagged
    a[0, 38:56, 1, 70] = 0.09   # head 1: 0.09^10 ~ 2^-35 in chunk 2, 0.09^8 in chunk 3: products
    a[0, 100:116, 0, 9] = 0.01  # head 0: 0.01^12 ~ 2^-80 in chunk 6 (flagged), 0.01^4 in chunk 7
    a[0, 150, :, :] = 0.0       # chunk 9, every channel of both heads: flagged
    x["alpha"] = torch.from_numpy(a)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"])
    _check(o, lin, so, ro, rs)


def test_kda_chunked_in_a_cuda_graph():
    """A call of several segments (their preps on a side stream beside the
    scans, joined by events) captured in a CUDA graph and replayed gives the
    bits of the same call made directly."""
    m = esa()
    x = _inputs(1, 8300, 2, 128, 32, 80, True)
    d = {k: v.cuda() for k, v in x.items()}
    B, T, H, Dk, Dv = 1, 8300, 2, 128, 32
    ws = torch.empty(m.esa_kda_workspace_size(B, T, H, Dk, Dv) + 256, dtype=torch.uint8, device="cuda")
    outs = []
    for graph in (False, True):
        o = torch.full((B, T, H, Dv), float("nan"), device="cuda")
        so = torch.full((B, H, Dk, Dv), float("nan"), device="cuda")

        def call():
            m.esa_kda(d["q"], d["k"], d["v"], d["alpha"], d["beta"], state_in=d["state"], o=o, state_out=so, ws=ws)

        if graph:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=s):
                    call()
            torch.cuda.current_stream().wait_stream(s)
            g.replay()
        else:
            call()
        torch.cuda.synchronize()
        outs.append((o.cpu(), so.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    _check(outs[1][0], None, outs[1][1], ro, rs)


def test_kda_chunked_wait_timeout_reports_status(monkeypatch):
    """The scan's compute warps wait, bounded, for each chunk's record. With
    the copy warp held after the first chunk the wait runs out: the call
    returns, the workspace's status word says TIMEOUT, the first chunk's
    outputs are written and the later steps and the final state are not;
    the next call clears the status and is exact."""
    import ctypes
    m = esa()
    B, T, H, Dk, Dv = 1, 100, 2, 64, 32
    x = _inputs(B, T, H, Dk, Dv, 79, True)
    ws = torch.zeros(m.esa_kda_workspace_size(B, T, H, Dk, Dv) + 256, dtype=torch.uint8, device="cuda")
    wptr = ctypes.c_void_p(ws.data_ptr() + (-ws.data_ptr()) % 256)

    def status():
        v = ctypes.c_int32(0)
        assert m._lib.esa_read_status(wptr, ctypes.c_void_p(torch.cuda.current_stream().cuda_stream),
                                      ctypes.byref(v)) == m.OK
        return v.value

    monkeypatch.setenv("ESA_DEBUG_EXTRA_ARRIVALS", "1")
    monkeypatch.setenv("ESA_WAIT_LIMIT_NS", "20000000")
    o, _, so = _gpu(x, state_in=x["state"], ws=ws)
    assert status() == m.ERR_TIMEOUT
    assert torch.isfinite(o[:, :16]).all() and torch.isnan(o[:, 16:]).all() and torch.isnan(so).all()
    monkeypatch.delenv("ESA_DEBUG_EXTRA_ARRIVALS")
    monkeypatch.delenv("ESA_WAIT_LIMIT_NS")
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"], ws=ws)
    assert status() == m.OK
    _check(o, lin, so, ro, rs)


def test_kda_decode_full():
    """The decode workload's shape (8 sequences, 32 heads, 128 x 128 state per
    head, one step), every output and the whole state."""
    x = _inputs(8, 1, 32, 128, 128, 2002, True)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"])
    o, lin, so = _gpu(x, state_in=x["state"])
    _check(o, lin, so, ro, rs)


@FORMS
def test_kda_long_prefill_sampled_heads(chunked):
    """The long-prefill shape (32768 steps, 16 heads, 128 x 128 state): the
    GPU runs every head; the oracle recomputes two heads in full (every step,
    every output and the final state)."""
    x = _inputs(1, 32768, 16, 128, 128, 2003, False)
    o, lin, so = _gpu(x, chunked=chunked)
    heads = [0, 11]
    xs = {k: v[:, :, heads].contiguous() for k, v in x.items()}
    ro, rs = O.kda(xs["q"], xs["k"], xs["v"], xs["alpha"], xs["beta"])
    _check(o[:, :, heads].contiguous(), lin[:, :, heads].contiguous(), so[:, heads].contiguous(), ro, rs)
    assert torch.isfinite(o).all() and torch.isfinite(so).all()


def test_kda_feeds_the_gate_mix():
    """The linear branch's bf16 output is the gate mix's lin: KDA -> sparse
    attention with the gate on the GPU, against the oracle's KDA output
    rounded to bf16 -> the oracle's gated attention."""
    cfg = E.small_config(seed=73, B=1, Tq=96, Tk=96, Hq=4, Hkv=1, D=64, top_k=24)
    sh = E.shape_of(cfg)
    inp = E.make_inputs(cfg)
    x = _inputs(1, 96, 4, 64, 64, 74, False)
    ro, _ = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"])
    inp["lin"] = torch.from_numpy(ro.astype(np.float32)).to(torch.bfloat16)
    oi, oc, ref, _ = O.gated_sparse_attention(inp, sh, 24)
    d = to_dev(inp)
    _, lin, _ = _gpu(x, o=False)
    d["lin"] = lin.cuda()
    gi, gc = gpu_topk(d, sh, 24)
    assert_idx_equal(gi, gc, oi, oc)
    st, out, _ = gpu_attn(d, sh, 24, gi, gc)
    assert st == 0
    assert_close(out, ref)
