"""Seeded synthetic inputs for gated fine-grained sparse attention.

This module is shared by the CPU oracle's tests, the GPU parity tests and the
benchmark. It holds none of the method's arithmetic (no indexer scoring, no
selection, no softmax, no gate mix): it only draws counter-based random
numbers and shapes them like the workloads of the pages.

Generator (its definition, so that anyone can re-derive every value):

* SplitMix64 finaliser ``mix(z)``: ``z ^= z>>30; z *= 0xBF58476D1CE4E5B9;
  z ^= z>>27; z *= 0x94D049BB133111EB; z ^= z>>31`` (all mod 2**64).
* A stream key is ``key(seed, tid) = mix(seed*GAMMA + tid)`` with
  ``GAMMA = 0x9E3779B97F4A7C15``; tensor ``tid`` draws word ``i`` as
  ``mix(key + (i+1)*GAMMA)``.
* int8 uniform on {-8..7}: ``(u >> 60) - 8`` (exact).
* integer weights on {1..4}: ``(u >> 62) + 1``.
* Bernoulli(3/4) "sparse" routing bit: ``(u >> 62) != 0``.
* N(0,1): element ``i`` uses words ``2i`` and ``2i+1`` as ``u1, u2 =
  ((w >> 11) + 0.5) * 2**-53`` and Box-Muller ``sqrt(-2 ln u1) cos(2 pi u2)``
  in fp64, rounded to fp32 (RNE) and then to bf16 (RNE).
* gate value: ``fp32(1 / (1 + exp(-z)))`` with ``z`` N(0,1) in fp64; the gate
  reaches the method already squashed into (0,1).
* needles: distinct positions ``w mod (L-1)`` taken in counter order.
* KDA linear branch: q and k are N(0,1) vectors (fp64) scaled to unit length,
  then rounded to fp32 and bf16; v bf16 N(0,1); forgetting factors
  ``0.9 + 0.1 * (w >> 11) * 2**-53`` in fp64, rounded to fp32; write
  strengths ``fp32(1 / (1 + exp(-z)))``; initial state ``fp32(0.1 * z)``.
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_GAMMA_U = np.uint64(GAMMA)

# Tensor ids: every tensor of a workload draws from its own stream.
TID = dict(qI=1, kI=2, wI=3, q=4, k=5, v=6, g=7, lin=8, route=9, needles=10, router=11,
           kda_q=12, kda_k=13, kda_v=14, kda_alpha=15, kda_beta=16, kda_state=17)

_CHUNK = 1 << 22
_THREADS = max(1, min(16, os.cpu_count() or 1))


def _mix_py(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> int:
    return _mix_py((seed * GAMMA + tid) & MASK64)


def words(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    """Words ``start .. start+n-1`` of stream (seed, tid) as uint64."""
    key = np.uint64(stream_key(seed, tid))
    ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix_np(ctr * _GAMMA_U + key)


def _chunked(n: int, fn, out: np.ndarray) -> np.ndarray:
    """Fill ``out`` (flat, length n) by calling fn(start, count) on chunks."""
    starts = list(range(0, n, _CHUNK))

    def run(s):
        c = min(_CHUNK, n - s)
        out[s:s + c] = fn(s, c)

    if len(starts) <= 1:
        for s in starts:
            run(s)
    else:
        with ThreadPoolExecutor(_THREADS) as ex:
            list(ex.map(run, starts))
    return out


def _f32_to_bf16_bits(x32: np.ndarray) -> np.ndarray:
    b = x32.view(np.uint32).astype(np.uint64)
    r = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def _normal_f64(seed: int, tid: int, start: int, n: int) -> np.ndarray:
    w = words(seed, tid, 2 * start, 2 * n)
    u = ((w >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)
    u1, u2 = u[0::2], u[1::2]
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


_HERE = os.path.dirname(os.path.abspath(__file__))
_GEN_SRC = os.path.join(_HERE, "gen.c")
_GEN_SO = os.path.join(_HERE, "_build", "libesa_gen.so")
_gen = None


def _genlib():
    """The C version of the same generator (bulk tensors), built on first use."""
    global _gen
    if _gen is None:
        if not os.path.exists(_GEN_SO) or os.path.getmtime(_GEN_SO) < os.path.getmtime(_GEN_SRC):
            os.makedirs(os.path.dirname(_GEN_SO), exist_ok=True)
            subprocess.run(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", _GEN_SO, _GEN_SRC, "-lm"], check=True)
        _gen = ctypes.CDLL(_GEN_SO)
        for f in (_gen.gen_normal_bf16, _gen.gen_int8_uniform):
            f.restype = None
            f.argtypes = [ctypes.c_uint64, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p]
    return _gen


def normal_bf16_bits(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    _genlib().gen_normal_bf16(stream_key(seed, tid), 0, n, out.ctypes.data_as(ctypes.c_void_p))
    return out


def int8_uniform(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int8)
    _genlib().gen_int8_uniform(stream_key(seed, tid), 0, n, out.ctypes.data_as(ctypes.c_void_p))
    return out


def normal_bf16_bits_np(seed: int, tid: int, n: int) -> np.ndarray:
    """numpy restatement of :func:`normal_bf16_bits` (checks the C loop)."""
    out = np.empty(n, dtype=np.uint16)
    return _chunked(n, lambda s, c: _f32_to_bf16_bits(_normal_f64(seed, tid, s, c).astype(np.float32)), out)


def int8_uniform_np(seed: int, tid: int, n: int) -> np.ndarray:
    out = np.empty(n, dtype=np.int8)
    return _chunked(n, lambda s, c: ((words(seed, tid, s, c) >> np.uint64(60)).astype(np.int16) - 8).astype(np.int8), out)


def bf16_tensor(bits: np.ndarray, shape) -> torch.Tensor:
    return torch.from_numpy(bits.view(np.int16).reshape(shape)).view(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """uint16 bit patterns of a CPU bf16 tensor."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------
# Workloads. Shapes follow the five configurations the method is measured on:
# a tiny prefill, a 131K-cache batched decode, a 32K GQA prefill with four
# weighted indexer heads, a 64K per-head routed (elastic) prefill and a
# 1M-token decode with planted needles.
# --------------------------------------------------------------------------
CONFIGS = {
    "tiny_prefill": dict(B=1, Tq=1024, Tk=1024, q_offset=0, Hq=4, Hkv=1, D=64, H_I=1, D_I=32,
                         top_k=128, weights="ones", routed=False, needles=0, seed=2001),
    "decode": dict(B=8, Tq=1, Tk=131072, q_offset=131071, Hq=32, Hkv=1, D=128, H_I=1, D_I=64,
                   top_k=2048, weights="ones", routed=False, needles=0, seed=2002),
    "long_prefill": dict(B=1, Tq=32768, Tk=32768, q_offset=0, Hq=16, Hkv=2, D=128, H_I=4, D_I=64,
                         top_k=2048, weights="1to4", routed=False, needles=0, seed=2003),
    "routed_prefill": dict(B=2, Tq=65536, Tk=65536, q_offset=0, Hq=32, Hkv=32, D=128, H_I=1, D_I=64,
                           top_k=2048, weights="ones", routed=True, needles=0, seed=2004),
    # chunked prefill against an existing cache: the last 16384 tokens of a
    # 131072-token context, with the long_prefill head and indexer layout
    "chunked_prefill": dict(B=1, Tq=16384, Tk=131072, q_offset=114688, Hq=16, Hkv=2, D=128, H_I=4, D_I=64,
                            top_k=2048, weights="1to4", routed=False, needles=0, seed=2006),
    "million_decode": dict(B=1, Tq=1, Tk=1048576, q_offset=1048575, Hq=64, Hkv=1, D=128, H_I=1, D_I=64,
                           top_k=2048, weights="ones", routed=False, needles=64, seed=2005),
    # one index set per query head (the per-head [batch, heads, top_k] shape),
    # each scored by its own ReLU'd int8 dot products: flags 1 | 2
    "per_head_prefill": dict(B=1, Tq=8192, Tk=8192, q_offset=0, Hq=16, Hkv=2, D=128, H_I=16, D_I=64,
                             top_k=2048, weights="ones", routed=False, needles=0, seed=2007, flags=3),
}


def shape_of(cfg: dict) -> dict:
    sh = {k: cfg[k] for k in ("B", "Tq", "Tk", "q_offset", "Hq", "Hkv", "D", "H_I", "D_I")}
    sh["flags"] = int(cfg.get("flags", 0))  # indexer options: 1 = ReLU per head, 2 = per-head index sets
    return sh


def needle_positions(seed: int, L: int, count: int) -> np.ndarray:
    """``count`` distinct positions in [0, L-1), in draw order."""
    got, seen, start = [], set(), 0
    while len(got) < count:
        w = words(seed, TID["needles"], start, 4 * count)
        start += 4 * count
        for x in (w % np.uint64(L - 1)).tolist():
            if x not in seen:
                seen.add(x)
                got.append(x)
                if len(got) == count:
                    break
    return np.array(got, dtype=np.int64)


def make_inputs(cfg: dict, seed: int | None = None, p_sparse_bits: bool = True) -> dict:
    """All input tensors of one workload on the CPU (torch), from one seed.

    Layouts: qI int8 [B,Tq,H_I,D_I]; kI int8 [B,Tk,D_I]; wI int32 [H_I];
    q bf16 [B,Tq,Hq,D]; k, v bf16 [B,Tk,Hkv,D]; g fp32 [Hq];
    lin bf16 [B,Tq,Hq,D]; route uint8 [B,Hq] (1 = sparse) or None.
    """
    c = dict(cfg)
    seed = c["seed"] if seed is None else seed
    B, Tq, Tk, Hq, Hkv, D, HI, DI = (c[k] for k in ("B", "Tq", "Tk", "Hq", "Hkv", "D", "H_I", "D_I"))
    out = {}
    out["qI"] = torch.from_numpy(int8_uniform(seed, TID["qI"], B * Tq * HI * DI).reshape(B, Tq, HI, DI))
    kI = int8_uniform(seed, TID["kI"], B * Tk * DI).reshape(B, Tk, DI)
    if c.get("weights", "ones") == "1to4":
        w = ((words(seed, TID["wI"], 0, HI) >> np.uint64(62)).astype(np.int64) + 1).astype(np.int32)
    else:
        w = np.ones(HI, dtype=np.int32)
    out["wI"] = torch.from_numpy(w)
    q = normal_bf16_bits(seed, TID["q"], B * Tq * Hq * D).reshape(B, Tq, Hq, D)
    k = normal_bf16_bits(seed, TID["k"], B * Tk * Hkv * D).reshape(B, Tk, Hkv, D)
    out["v"] = bf16_tensor(normal_bf16_bits(seed, TID["v"], B * Tk * Hkv * D), (B, Tk, Hkv, D))
    z = _normal_f64(seed, TID["g"], 0, Hq)
    out["g"] = torch.from_numpy((1.0 / (1.0 + np.exp(-z))).astype(np.float32))
    out["lin"] = bf16_tensor(normal_bf16_bits(seed, TID["lin"], B * Tq * Hq * D), (B, Tq, Hq, D))
    if c.get("routed"):
        bits = (words(seed, TID["route"], 0, B * Hq) >> np.uint64(62)) != 0
        out["route"] = torch.from_numpy(bits.astype(np.uint8).reshape(B, Hq))
    else:
        out["route"] = None
    npos = None
    if c.get("needles", 0):
        # Needle keys: K row = 4x the first query head's vector (exact in bf16),
        # indexer key = the indexer query of head 0. Values keep their draw.
        npos = needle_positions(seed, Tk, c["needles"])
        qI0 = out["qI"].numpy()
        for b in range(B):
            qv = q[b, 0, 0, :].astype(np.uint32) << np.uint32(16)
            four_q = (qv.view(np.float32) * np.float32(4.0))
            for p in npos:
                k[b, p, :, :] = _f32_to_bf16_bits(four_q)[None, :]
                kI[b, p, :] = qI0[b, 0, 0, :]
    out["q"] = bf16_tensor(q.reshape(-1), (B, Tq, Hq, D))
    out["k"] = bf16_tensor(k.reshape(-1), (B, Tk, Hkv, D))
    out["kI"] = torch.from_numpy(kI)
    out["needles"] = npos
    return out


def router_weights(cfg: dict, hidden: int = 64, seed: int | None = None) -> dict:
    """Seeded weights of the 2-layer attention router (no trained weights
    exist): W1 fp32 [hidden, Hkv*D] ~ N(0, 1/(Hkv*D)), b1 [hidden] ~ N(0, 1/4),
    W2 fp32 [2*Hq, hidden] ~ N(0, 1/hidden), b2 [2*Hq] ~ N(0, 1/4), from one
    SplitMix64 N(0,1) stream (fp64, rounded to fp32) in that order."""
    seed = cfg["seed"] if seed is None else seed
    C, Hq = cfg["Hkv"] * cfg["D"], cfg["Hq"]
    sizes = [hidden * C, hidden, 2 * Hq * hidden, 2 * Hq]
    z = _normal_f64(seed, TID["router"], 0, sum(sizes))
    out, o = {}, 0
    for name, n, sd, shp in (("W1", sizes[0], C ** -0.5, (hidden, C)), ("b1", sizes[1], 0.5, (hidden,)),
                             ("W2", sizes[2], hidden ** -0.5, (2 * Hq, hidden)), ("b2", sizes[3], 0.5, (2 * Hq,))):
        out[name] = torch.from_numpy((z[o:o + n] * sd).astype(np.float32).reshape(shp))
        o += n
    return out


def kda_inputs(B: int, T: int, H: int, Dk: int, Dv: int, seed: int, state: bool = False) -> dict:
    """Seeded inputs of the KDA linear-attention branch (CPU tensors), shaped
    like the model's: q, k bf16 [B, T, H, Dk] are N(0,1) vectors scaled to
    unit length in fp64, then rounded to fp32 and bf16 (the model normalises
    its queries and keys); v bf16 [B, T, H, Dv] ~ N(0,1); alpha fp32
    [B, T, H, Dk] uniform in [0.9, 1) as 0.9 + 0.1 * (w >> 11) * 2**-53;
    beta fp32 [B, T, H] = 1 / (1 + exp(-z)), z ~ N(0,1); with ``state`` also
    an initial state fp32 [B, H, Dk, Dv] ~ 0.1 N(0,1)."""
    n = B * T * H * Dk

    def unit(tid):
        z = _chunked(n, lambda s, c: _normal_f64(seed, TID[tid], s, c), np.empty(n, dtype=np.float64))
        z = z.reshape(B, T, H, Dk)
        z /= np.linalg.norm(z, axis=-1, keepdims=True)
        return torch.from_numpy(z.astype(np.float32)).to(torch.bfloat16)

    def uniform(s, c):
        return 0.9 + 0.1 * (words(seed, TID["kda_alpha"], s, c) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53

    out = dict(q=unit("kda_q"), k=unit("kda_k"),
               v=bf16_tensor(normal_bf16_bits(seed, TID["kda_v"], B * T * H * Dv), (B, T, H, Dv)))
    alpha = _chunked(n, uniform, np.empty(n, dtype=np.float64))
    out["alpha"] = torch.from_numpy(alpha.astype(np.float32).reshape(B, T, H, Dk))
    zb = _normal_f64(seed, TID["kda_beta"], 0, B * T * H)
    out["beta"] = torch.from_numpy((1.0 / (1.0 + np.exp(-zb))).astype(np.float32).reshape(B, T, H))
    if state:
        zs = _normal_f64(seed, TID["kda_state"], 0, B * H * Dk * Dv)
        out["state"] = torch.from_numpy((0.1 * zs).astype(np.float32).reshape(B, H, Dk, Dv))
    return out


def small_config(**over) -> dict:
    """A small workload for parity tests: defaults overridden by keywords."""
    base = dict(B=1, Tq=64, Tk=64, q_offset=0, Hq=4, Hkv=1, D=64, H_I=1, D_I=32, top_k=16,
                weights="ones", routed=False, needles=0, seed=7)
    base.update(over)
    return base
