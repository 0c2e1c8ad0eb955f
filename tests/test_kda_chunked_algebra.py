"""The chunked KDA kernels' algebra, on the CPU in fp64, against the oracle:
the rearrangement the scan uses (D = U - Wk S, O = scale (Qp S + Up),
S' = g_last * S + Kl^T D, with M solved by the same row-update forward
substitution), and the error bound of the three-product tf32 split that the
scan's tensor-core products use. No GPU: these check the method the CUDA
kernels implement, not the kernels."""
import numpy as np
import pytest
import torch

import esa_inputs as E
import oracle as O

C = 16


def _f64(t):
    return t.to(torch.float64).numpy()


def _chunked(q, k, v, alpha, beta, s0, scale):
    """The prep and scan of the chunked form, written out per (sequence,
    head) and chunk of C steps (steps past the end: k = q = 0, alpha = 1,
    beta = 0, v = 0)."""
    B, T, H, Dk = q.shape
    Dv = v.shape[-1]
    o = np.zeros((B, T, H, Dv))
    st = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = s0[b, h].copy()
            for t0 in range(0, T, C):
                n = min(C, T - t0)
                K = np.zeros((C, Dk)); Q = np.zeros((C, Dk)); A = np.ones((C, Dk)); V = np.zeros((C, Dv))
                be = np.zeros(C)
                K[:n], Q[:n], A[:n] = k[b, t0:t0 + n, h], q[b, t0:t0 + n, h], alpha[b, t0:t0 + n, h]
                V[:n], be[:n] = v[b, t0:t0 + n, h], beta[b, t0:t0 + n, h]
                G = np.cumprod(A, axis=0)
                Kt, Qt, Ki = K * G, Q * G, K / G
                gl = G[-1]
                Kl = Ki * gl
                Am = np.tril(Kt @ Ki.T, -1)
                Bm = np.tril(Qt @ Ki.T)
                # forward substitution, each new entry added into the rows below
                M = np.zeros((C, C))
                for j in range(C):
                    acc = np.zeros(C)
                    for i in range(C):
                        m = be[i] * ((1.0 if i == j else 0.0) - acc[i])
                        M[i, j] = m
                        acc[i + 1:] += Am[i + 1:, i] * m
                Wk, U = M @ Kt, M @ V
                Qp, Up = Qt - Bm @ Wk, Bm @ U
                D = U - Wk @ S
                o[b, t0:t0 + n, h] = (scale * (Qp @ S + Up))[:n]
                S = gl[:, None] * S + Kl.T @ D
            st[b, h] = S
    return o, st


@pytest.mark.parametrize("shape", [(1, 53, 2, 32, 16), (2, 16, 1, 64, 48), (1, 5, 3, 16, 8)],
                         ids=["ragged", "one-chunk", "short"])
def test_chunked_rearrangement_equals_the_recurrence(shape):
    B, T, H, Dk, Dv = shape
    x = E.kda_inputs(B, T, H, Dk, Dv, 91 + T, state=True)
    ro, rs = O.kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=x["state"], scale=0.4)
    o, st = _chunked(_f64(x["q"]), _f64(x["k"]), _f64(x["v"]), _f64(x["alpha"]), _f64(x["beta"]),
                     _f64(x["state"]), 0.4)
    assert np.allclose(o, ro, rtol=1e-10, atol=1e-12)
    assert np.allclose(st, rs, rtol=1e-10, atol=1e-12)


def _tf32_split(x: np.ndarray):
    """The scan's split: hi = x with the low 13 bits of its fp32 pattern
    cleared, lo = the same of the exact remainder x - hi."""
    x = x.astype(np.float32)
    hi = (x.view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    lo = ((x - hi).astype(np.float32).view(np.uint32) & np.uint32(0xFFFFE000)).view(np.float32)
    return hi.astype(np.float64), lo.astype(np.float64)


def test_three_tf32_products_bound():
    """hi and lo keep 11 significant bits each and the remainder x - hi has
    at most 13, so |x - hi - lo| < 2^-21 |x|; hi*hi + hi*lo + lo*hi (each
    term exact, as the tensor cores form it) is within 2^-19 |a b| of the
    product, the dropped lo*lo term (up to 2^-20 |a b|) the largest part."""
    rng = np.random.default_rng(5)
    a = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    b = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 30, 200000))).astype(np.float32)
    ah, al = _tf32_split(a)
    bh, bl = _tf32_split(b)
    a64, b64 = a.astype(np.float64), b.astype(np.float64)
    assert np.all(np.abs(a64 - ah - al) < 2.0 ** -21 * np.abs(a64))
    approx = ah * bh + ah * bl + al * bh
    assert np.all(np.abs(approx - a64 * b64) < 2.0 ** -19 * np.abs(a64 * b64))
    # one tf32 product alone is off by up to ~2^-10: why the split is needed
    assert np.max(np.abs(ah * bh - a64 * b64) / np.abs(a64 * b64)) > 2.0 ** -12
