"""Benchmark of the gated fine-grained sparse attention hot path on B300.

One step = one decode pass of the whole path for every sequence of the batch:
indexer scores over the full 131,072-key cache, exact top-2048 selection,
gathered sparse attention with the gate mix fused. Workload: 8 sequences, 1
new token each, 32 query heads sharing 1 KV head, head dim 128, indexer
1 head x 64 (int8), synthetic seeded inputs. Multi-GPU runs are replicas
(each rank its own batch, no collective on the data path): scaling "weak",
value = tokens of all ranks / max time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl esa|reference]

Rank 0 also times every other workload (the 1M-token decode, the tiny,
long, chunked, per-head and routed prefills, the attention router and the
KDA linear branch), each next to the oracle on the host cores. The stdout
JSON line is compact: its "configs" map holds one short entry per workload
(time, rate, roofline fraction, oracle rate); the full per-workload detail
goes to stderr as a second JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "sparse-attn prefill tok/s + decode µs/step @1 B300; % HBM/tensor roofline"
NSETS = 4  # rotating input sets: their kI caches together exceed the 126 MB L2


def _load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d.get("bf16_tflops"), "measured"
    return 6400.0, 1800.0, "fallback"


def max_over_ranks(values, world: int, device) -> list:
    """Per-rank timings reduced to their maximum over all ranks (the whole
    job ends when its slowest rank does); the identity on one rank."""
    if world <= 1:
        return list(values)
    import torch.distributed as dist
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job throughput: every rank's units over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while a region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def _traffic_for(kernel: str, src_files: list[str]):
    """dram bytes per launch recorded from an ncu capture, if the kernel source
    is unchanged since (the capture stores a hash of its sources)."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel)
    if not d:
        return None
    h = hashlib.sha256()
    for f in src_files:
        h.update(open(os.path.join(ROOT, f), "rb").read())
    return d["bytes_per_launch"] if d.get("src_sha256") == h.hexdigest() else None


SELECT_SRC = ["long_context_sparse_20_b300/csrc/k_select_split.cu", "long_context_sparse_20_b300/csrc/esa_device.cuh"]
FUSED_SRC = SELECT_SRC
ATTN_SRC = ["long_context_sparse_20_b300/csrc/k_sparse_attn.cu", "long_context_sparse_20_b300/csrc/esa_device.cuh"]


def decode_bytes(sh: dict, K: int):
    """Algorithmic HBM bytes of one decode step, per kernel: the selection
    streams every indexer key once and writes the index list; the attention
    reads the index list, gathers one K and one V row per selected key and
    KV head, and reads q and lin and writes the fp32 output."""
    B, L, Hq, Hkv, D, HI, DI = (sh[k] for k in ("B", "Tk", "Hq", "Hkv", "D", "H_I", "D_I"))
    sel = B * L * DI + B * HI * DI + B * K * 4 + B * 4            # kI stream, qI, idx + cnt written
    k_sel = min(K, L)
    attn = B * k_sel * Hkv * D * 2 * 2 + B * k_sel * 4 + B * 4      # gathered K and V rows, idx + cnt read
    attn += B * Hq * D * 2 * 2 + B * Hq * D * 4 + Hq * 4            # q, lin in; out (fp32) out; g
    return sel, attn


def fused_step_bytes(sh: dict, K: int) -> int:
    """Algorithmic HBM bytes of one fused decode step: every indexer key
    streamed once, the indexer queries, one K and one V row per selected key
    and KV head, q and lin read, the fp32 output written, the gate. The index
    list, the scores and the attention partials stay on chip (the partials
    pass through L2 once)."""
    B, L, Hq, Hkv, D, HI, DI = (sh[k] for k in ("B", "Tk", "Hq", "Hkv", "D", "H_I", "D_I"))
    k_sel = min(K, L)
    return (B * L * DI + B * HI * DI + B * k_sel * Hkv * D * 2 * 2 + B * Hq * D * (2 + 2 + 4) + Hq * 4)


def run_cpu_baseline(cfg: dict, inp: dict, seconds: float = 10.0):
    """The oracle, as it stands, on whole decode steps (all rows of the batch),
    repeated for about `seconds`; returns tok/s, threads, sample text."""
    sys.path.insert(0, ROOT)
    import esa_inputs as E
    import oracle as O
    sh = E.shape_of(cfg)
    K = cfg["top_k"]
    O.lib()
    reps, t0 = 0, time.perf_counter()
    while True:
        O.gated_sparse_attention(inp, sh, K)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    rows = sh["B"] * sh["Tq"]
    threads = min(O.threads(), rows)
    return rows * reps / el, threads, f"{reps} full decode steps ({rows} rows each), {el:.1f} s"


def run_cpu_baseline_1thread(cfg: dict, inp: dict, seconds: float = 5.0):
    """The same on one host thread: decode steps row by row, for about `seconds`."""
    sys.path.insert(0, ROOT)
    import esa_inputs as E
    import oracle as O
    sh = E.shape_of(cfg)
    K = cfg["top_k"]
    old = os.environ.get("ESA_ORACLE_THREADS")
    os.environ["ESA_ORACLE_THREADS"] = "1"
    try:
        rows, n, t0 = sh["B"] * sh["Tq"], 0, time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            O.gated_sparse_attention(inp, sh, K, rows=[n % rows])
            n += 1
        el = time.perf_counter() - t0
    finally:
        if old is None:
            del os.environ["ESA_ORACLE_THREADS"]
        else:
            os.environ["ESA_ORACLE_THREADS"] = old
    return n / el, f"{n} decode rows one at a time, {el:.1f} s"


def oracle_row_sample(host: dict, sh: dict, K: int, n_rows: int = 16, seed: int = 0) -> dict:
    """The oracle, as it stands, on a seeded uniform sample of a prefill
    workload's query rows (all host threads), extrapolated to the whole
    forward: est = rows / n_sample * t_sample (unbiased: a row's cost depends
    only on its position, drawn uniformly)."""
    sys.path.insert(0, ROOT)
    import oracle as O
    O.lib()
    total = sh["B"] * sh["Tq"]
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(total, size=min(n_rows, total), replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    O.gated_sparse_attention(host, sh, K, rows=rows)
    el = time.perf_counter() - t0
    est = el * total / len(rows)
    whole = len(rows) == total
    return {"tok_per_s": total / est, "unit": "tok/s", "cores": min(O.threads(), len(rows)),
            "kind": "oracle" if whole else "oracle, extrapolated",
            "sample": f"all {total} rows, {el:.2f} s" if whole else f"{len(rows)} seeded uniform rows of {total}, {el:.2f} s"}


def decode_label(name: str, sh: dict, K: int) -> str:
    """The workload string of a decode configuration, the same in both arms."""
    return (f"{name}: B={sh['B']} x 1 new token, cache {sh['Tk']}, Hq={sh['Hq']}, Hkv={sh['Hkv']}, D={sh['D']}, "
            f"indexer {sh['H_I']}x{sh['D_I']} int8, top_k={K}")


def run_config(name: str, sh: dict, K: int, world: int) -> dict:
    """The JSON line's "config" object, identical in both arms."""
    return {"workload": decode_label(name, sh, K), "global_batch": sh["B"] * world, "seq_len": sh["Tk"],
            "parallelism": f"replicas x{world}"}


def reference_arm(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    sys.path.insert(0, ROOT)
    import esa_inputs as E
    cfg = E.CONFIGS[args.workload]
    inp = E.make_inputs(cfg)
    import oracle as O
    sh = E.shape_of(cfg)
    K = cfg["top_k"]
    O.lib()
    rows = sh["B"] * sh["Tq"]
    # each step: one query row of the workload, in turn (a bounded sample)
    for i in range(args.warmup):
        O.gated_sparse_attention(inp, sh, K, rows=[i % rows])
    t0 = time.perf_counter()
    for i in range(args.steps):
        O.gated_sparse_attention(inp, sh, K, rows=[i % rows])
    el = time.perf_counter() - t0
    val = args.steps / el
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": run_config(args.workload, sh, K, 1),
            "cpu_baseline": {"value": val, "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": f"{args.steps} steps of one query row each (rows taken in turn)"},
            "e2e": {"value": val, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def prefill_section(dev, esa, E, reps: int = 2, seq: int = 0,
                    names=("tiny_prefill", "long_prefill", "chunked_prefill", "per_head_prefill", "routed_prefill"),
                    oracle_rows: int = 0) -> dict:
    """The prefill workloads, one forward each (after one untimed warm-up),
    timed with CUDA events on the launching stream. Inputs exceed the 126 MB
    L2 except for the tiny prefill's (a few MB: launch-bound at any rate). Algorithmic flops count what the method
    computes: causal pairs for full heads, selected pairs (min(K, p+1) per
    row) for sparse heads, 4*D flops per pair (Q.K and P.V)."""
    _, tf_peak, kind = _load_peaks()
    res = {}
    st = torch.cuda.current_stream(dev)

    def timed(fn):
        fn()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    for name in names:
        cfg = dict(E.CONFIGS[name])
        if seq:  # a shorter sequence (profiling of small cases)
            cfg["Tk"] = cfg["Tk"] * seq // cfg["Tq"]
            cfg["q_offset"] = cfg["Tk"] - seq
            cfg["Tq"] = seq
        sh = E.shape_of(cfg)
        K = cfg["top_k"]
        host = E.make_inputs(cfg)
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        shape = esa.shape_from(sh)
        B, S, Hq, D = sh["B"], sh["Tq"], sh["Hq"], sh["D"]
        scale = 1.0 / math.sqrt(D)
        out = torch.empty(B, S, Hq, D, dtype=torch.float32, device=dev)
        n = np.arange(sh["q_offset"] + 1, sh["q_offset"] + S + 1, dtype=np.float64)  # prefix lengths
        sel_pairs = float(np.minimum(n, K).sum())  # per (sequence, head)
        causal_pairs = float(n.sum())
        opts = {0: "", 1: " ReLU", 2: " per-head sets", 3: " ReLU, per-head sets"}[sh["flags"]]
        entry = {"workload": f"{name}: B={B} S={S} (queries at {sh['q_offset']}..{sh['q_offset'] + S - 1} of a "
                             f"{sh['Tk']}-key cache) Hq={Hq} Hkv={sh['Hkv']} D={D} indexer {sh['H_I']}x{sh['D_I']}"
                             f"{opts} top_k={K}"}
        if cfg.get("routed"):
            ws = esa.workspace_for(esa.OP_ROUTED_ATTN, shape, K, dev)
            ms = timed(lambda: esa.esa_routed_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], d["route"], shape,
                                                   K, scale, d["g"], d["lin"], out, ws, st))
            assert esa.esa_read_status(ws, st) == 0
            nfull = int((host["route"] == 0).sum())
            nsparse = B * Hq - nfull
            flops = 4.0 * D * (nfull * causal_pairs + nsparse * sel_pairs)
            entry.update({"full_heads": nfull, "sparse_heads": nsparse, "kernels_ms": {"routed_attn": ms}})
            # the attention router on the same keys (seeded weights, hidden 64):
            # bound by one read of k
            W = {n: t.to(dev) for n, t in E.router_weights(cfg).items()}
            wsr = esa.workspace_for(esa.OP_ROUTE_HEADS, shape, 1, dev)
            rt = torch.empty(B, Hq, dtype=torch.uint8, device=dev)
            ms_r = timed(lambda: esa.esa_route_heads(d["k"], W["W1"], W["b1"], W["W2"], W["b2"], shape, rt, None, wsr,
                                                     st))
            assert esa.esa_read_status(wsr, st) == 0
            rbytes = B * sh["Tk"] * sh["Hkv"] * D * 2 + sum(t.numel() * 4 for t in W.values()) + B * Hq
            hbm_peak = _load_peaks()[0]
            entry["router"] = {"ms": ms_r, "algorithmic_bytes": rbytes, "GB_per_s": rbytes / (ms_r / 1e3) / 1e9,
                               "frac_of_hbm": rbytes / (ms_r / 1e3) / 1e9 / hbm_peak, "peak_kind": kind,
                               "sparse_heads_routed": int(rt.sum().item())}
        else:
            wsel = esa.workspace_for(esa.OP_TOPK_SELECT, shape, K, dev)
            watt = esa.workspace_for(esa.OP_SPARSE_ATTN, shape, K, dev)
            sets = (sh["H_I"],) if sh["flags"] & esa.PER_HEAD_SETS else ()  # per-head index sets
            idx = torch.empty(B, S, *sets, K, dtype=torch.int32, device=dev)
            cnt = torch.empty(B, S, *sets, dtype=torch.int32, device=dev)
            ms_sel = timed(lambda: esa.esa_topk_select(d["qI"], d["kI"], d["wI"], shape, K, idx, cnt, wsel, st))
            ms_att = timed(lambda: esa.esa_sparse_attn(d["q"], d["k"], d["v"], idx, cnt, shape, K, scale, d["g"],
                                                       d["lin"], out, None, watt, st))
            assert esa.esa_read_status(wsel, st) == 0 and esa.esa_read_status(watt, st) == 0
            ms = ms_sel + ms_att
            flops = 4.0 * D * B * Hq * sel_pairs
            entry["kernels_ms"] = {"topk_select": ms_sel, "sparse_attn": ms_att}
            # the same outputs through the one-call API (no lse, no index
            # outputs): prefill shapes whose prefixes hold few times the
            # selected keys take the routed kernel with every head sparse
            del idx, cnt, wsel, watt
            torch.cuda.empty_cache()
            wsg = esa.workspace_for(esa.OP_GATED_SPARSE_ATTN, shape, K, dev)
            ms_g = timed(lambda: esa.esa_gated_sparse_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], shape, K,
                                                           scale, d["g"], d["lin"], out, None, None, None, wsg, st))
            assert esa.esa_read_status(wsg, st) == 0
            entry["kernels_ms"]["gated_one_call"] = ms_g
            entry["path"] = "esa_topk_select + esa_sparse_attn"
            if ms_g < ms:
                entry["path"] = "esa_gated_sparse_attn (one call)"
                ms = ms_g
            del wsg
        entry.update({"ms": ms, "tok_per_s": B * S / (ms / 1e3), "algorithmic_tflops": flops / (ms / 1e3) / 1e12,
                      "tensor_peak_tflops": tf_peak, "frac_of_bf16_peak": flops / (ms / 1e3) / 1e12 / tf_peak,
                      "peak_kind": kind})
        if oracle_rows:
            entry["cpu_baseline"] = oracle_row_sample(host, sh, K, n_rows=min(oracle_rows, B * S) if B * S > 4096
                                                      else B * S)
        res[name] = entry
        del d, host, out
        torch.cuda.empty_cache()
    return res


def kda_section(dev, esa, E, reps: int = 3, T: int = 32768, oracle: bool = False) -> dict:
    """The KDA linear branch (the gate mix's lin input) at the decode shape
    (8 sequences x 32 heads, one step, 128 x 128 fp32 state per head updated
    in place) and the long-prefill shape (1 x T steps x 16 heads, zero initial
    state), timed with CUDA events on the launching stream.

    decode: bound by HBM — each step reads and writes the whole state; 16
    state buffers rotate (256 MiB > the 126 MB L2); the 16 launches are one
    CUDA graph, replayed (the per-launch host cost would otherwise hide the
    ~5 us kernel). Algorithmic bytes: state read + write, the step's q, k, v,
    alpha, beta, and o (fp32) + lin (bf16).
    prefill: bound by the fp32 pipes — 7 flops per state element per step
    (forget 1, read 2, write 2, output 2); peak = 148 SMs x 128 fp32 lanes x
    2 flops x the maximum SM clock.
    With `oracle`, the oracle as it stands is timed beside each: whole decode
    steps repeated for ~2 s; the prefill on one head in full, extrapolated to
    every head over the host threads (heads are independent)."""
    peak_gbs, _, kind = _load_peaks()
    sm_mhz = 2032.0
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        sm_mhz = float(json.load(open(p)).get("sm_max_mhz", sm_mhz))
    alu_peak = 148 * 128 * 2 * sm_mhz * 1e6 / 1e12  # TFLOP/s
    st = torch.cuda.current_stream(dev)
    res = {}

    if oracle:
        sys.path.insert(0, ROOT)
        import oracle as O
        O.lib()
    B, H, D, NB = 8, 32, 128, 16
    xh = E.kda_inputs(B, 1, H, D, D, 2002, state=True)
    x = {k: v.to(dev) for k, v in xh.items()}
    states = [x["state"].clone() for _ in range(NB)]
    o = torch.empty(B, 1, H, D, dtype=torch.float32, device=dev)
    lin = torch.empty(B, 1, H, D, dtype=torch.bfloat16, device=dev)

    def launch(i):
        esa.esa_kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], state_in=states[i], o=o, lin=lin,
                    state_out=states[i])

    for i in range(NB):
        launch(i)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(NB):
            launch(i)
    g.replay()
    torch.cuda.synchronize()
    best = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(10):
            g.replay()
        e1.record(st)
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (10 * NB)
        best = us if best is None else min(best, us)
    nbytes = 2 * B * H * D * D * 4 + B * H * (2 * D * 2 + D * 2 + D * 4 + 4) + B * H * D * (4 + 2)
    res["decode"] = {"workload": f"KDA decode: B={B} x 1 step, H={H}, Dk=Dv={D}, state in place",
                     "us": best, "algorithmic_bytes": nbytes, "GB_per_s": nbytes / (best / 1e6) / 1e9,
                     "frac_of_hbm": nbytes / (best / 1e6) / 1e9 / peak_gbs, "peak_gbs": peak_gbs, "peak_kind": kind,
                     "l2": f"{NB} state buffers in rotation ({NB * B * H * D * D * 4 / 2**20:.0f} MiB > 126 MB L2)",
                     "timing": "CUDA graph of 16 launches, replayed 10 times; best of 3"}
    if oracle:
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 2.0:
            O.kda(xh["q"], xh["k"], xh["v"], xh["alpha"], xh["beta"], state_in=xh["state"])
            n += 1
        el = time.perf_counter() - t0
        res["decode"]["cpu_baseline"] = {"us": el / n * 1e6, "tok_per_s": B * n / el, "cores": min(O.threads(), B * H),
                                         "kind": "oracle", "sample": f"{n} whole decode steps, {el:.1f} s"}
    del x, states, o, lin, g
    torch.cuda.empty_cache()

    B, H = 1, 16
    xh = E.kda_inputs(B, T, H, D, D, 2003)
    x = {k: v.to(dev) for k, v in xh.items()}
    o = torch.empty(B, T, H, D, dtype=torch.float32, device=dev)
    lin = torch.empty(B, T, H, D, dtype=torch.bfloat16, device=dev)
    so = torch.empty(B, H, D, D, dtype=torch.float32, device=dev)
    ws = torch.empty(esa.esa_kda_workspace_size(B, T, H, D, D) + 256, dtype=torch.uint8, device=dev)

    def timed(chunked):
        def run():
            esa.esa_kda(x["q"], x["k"], x["v"], x["alpha"], x["beta"], o=o, lin=lin, state_out=so, ws=ws,
                        chunked=chunked)

        run()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            run()
            e1.record(st)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1)
            best = ms if best is None else min(best, ms)
        return best

    step_ms = timed(False)
    best = timed(True)
    flops = 7.0 * B * H * T * D * D
    res["long_prefill"] = {"workload": f"KDA prefill: B={B} x {T} steps, H={H}, Dk=Dv={D}, zero initial state",
                           "form": "chunked (16-step chunks: prep + scan kernels)",
                           "ms": best, "tok_per_s": B * T / (best / 1e3), "algorithmic_flops": flops,
                           "achieved_tflops": flops / (best / 1e3) / 1e12, "bound": "alu",
                           "alu_peak_tflops": alu_peak, "frac_of_alu": flops / (best / 1e3) / 1e12 / alu_peak,
                           "alu_peak_from": f"148 SMs x 128 fp32 lanes x 2 flops x {sm_mhz:.0f} MHz",
                           "stepwise_ms": step_ms, "workspace_bytes": int(ws.numel() - 256)}
    # the chunked form's tensor-core work: per step and head, X = [Wk; Qp] S
    # (2 Dk Dv MACs) and the state update (Dk Dv MACs), each fp32 product as
    # three tf32 products; against the tf32 peak scaled from the measured bf16
    # peak by the nominal ratio (1.1 / 2.25 PFLOP/s dense)
    _, bf16_peak, bkind = _load_peaks()
    tf32_peak = bf16_peak * 1.1 / 2.25
    tflops = 3 * 2 * 3.0 * B * H * T * D * D
    res["long_prefill"]["tensor_view"] = {
        "executed_tf32_flops": tflops, "achieved_tflops": tflops / (best / 1e3) / 1e12,
        "tf32_peak_tflops": tf32_peak, "peak_from": f"{bkind} bf16 {bf16_peak:.0f} TFLOP/s x 1.1/2.25",
        "frac": tflops / (best / 1e3) / 1e12 / tf32_peak}
    if oracle:
        one = {k: v[:, :, :1].contiguous() for k, v in xh.items()}
        t0 = time.perf_counter()
        O.kda(one["q"], one["k"], one["v"], one["alpha"], one["beta"])
        el = time.perf_counter() - t0
        cores = min(O.threads(), B * H)
        est = el * B * H / cores
        res["long_prefill"]["cpu_baseline"] = {"ms": est * 1e3, "tok_per_s": B * T / est, "cores": cores,
                                               "kind": "oracle, extrapolated",
                                               "sample": f"one head of {B * H}, {T} steps, {el:.1f} s"}
    del x, o, lin, so, ws
    torch.cuda.empty_cache()
    return res


def decode_section(dev, esa, E, name: str, args, world: int, e2e: bool) -> dict:
    """Time decode steps of workload `name` (inputs resident in HBM).

    NSETS rotating copies of the whole decode state (their kI caches exceed
    the 126 MB L2). The K = args.steps timed steps are captured once into a
    CUDA graph (host launch overhead would otherwise starve the GPU),
    replayed once untimed, then `args.repeats` times timed, each replay
    bracketed by a barrier and a synchronize with CUDA events on the
    launching stream; the step time is the median replay over K (the max
    over ranks of each replay first). The timed graph holds kernels only: an
    event between the kernels of a step would cut the programmatic
    (early-launch) edge between them; a second graph of the same steps with
    an event around each kernel gives the per-kernel durations (the
    roofline's launch time). With `e2e`, the same steps also run end to end
    through host buffers."""
    cfg = dict(E.CONFIGS[name])
    assert cfg["Tq"] == 1, "the step benchmark runs decode workloads"
    sh = E.shape_of(cfg)
    K = cfg["top_k"]
    B, L, Hq, Hkv, D, HI, DI = (sh[k] for k in ("B", "Tk", "Hq", "Hkv", "D", "H_I", "D_I"))
    rank = _dist()[1]
    host = E.make_inputs(cfg, seed=cfg["seed"] + 1000 * rank)
    shape = esa.shape_from(sh)
    scale = 1.0 / math.sqrt(D)

    # the decode step: esa_topk_select + esa_sparse_attn (two public calls,
    # each kernel timed apart for the roofline), or the one-call
    # esa_gated_sparse_attn (--gated; a single launch with ESA_DECODE_PATH=fused)
    fused = args.gated or os.environ.get("ESA_DECODE_PATH") == "fused"
    sets = []
    for _ in range(args.sets):
        d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in host.items()}
        d["out"] = torch.empty(B, 1, Hq, D, dtype=torch.float32, device=dev)
        if fused:
            d["ws"] = esa.workspace_for(esa.OP_GATED_SPARSE_ATTN, shape, K, dev)
        else:
            d["idx"] = torch.empty(B, 1, K, dtype=torch.int32, device=dev)
            d["cnt"] = torch.empty(B, 1, dtype=torch.int32, device=dev)
            d["ws_sel"] = esa.workspace_for(esa.OP_TOPK_SELECT, shape, K, dev)
            d["ws_att"] = esa.workspace_for(esa.OP_SPARSE_ATTN, shape, K, dev)
        sets.append(d)
    single = fused and os.environ.get("ESA_DECODE_PATH") == "fused"  # one cooperative launch per step
    launches_per_step = 1 if single else 2

    def step(d, ev=None):
        st = torch.cuda.current_stream(dev)
        if ev:
            ev[0].record(st)
        if fused:  # the whole path in one call
            esa.esa_gated_sparse_attn(d["q"], d["k"], d["v"], d["qI"], d["kI"], d["wI"], shape, K, scale, d["g"],
                                      d["lin"], d["out"], None, None, None, d["ws"], st)
            if ev:
                ev[1].record(st)
                ev[2].record(st)
            return
        esa.esa_topk_select(d["qI"], d["kI"], d["wI"], shape, K, d["idx"], d["cnt"], d["ws_sel"], st)
        if ev:
            ev[1].record(st)
        esa.esa_sparse_attn(d["q"], d["k"], d["v"], d["idx"], d["cnt"], shape, K, scale, d["g"], d["lin"], d["out"],
                            None, d["ws_att"], st)
        if ev:
            ev[2].record(st)

    def check_status():
        for d in sets:
            for w in ((d["ws"],) if fused else (d["ws_sel"], d["ws_att"])):
                assert esa.esa_read_status(w) == 0

    for i in range(max(3, args.warmup)):
        step(sets[i % len(sets)])
    torch.cuda.synchronize()
    check_status()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)] for _ in range(args.steps)]
    timing = f"median of {args.repeats} timed replays of a {args.steps}-step CUDA graph"

    def capture(with_events):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(args.steps):
                step(sets[i % len(sets)], evs[i] if with_events else None)
        gr.replay()
        torch.cuda.synchronize()
        return gr.replay

    try:
        run = capture(False)
        run_breakdown = capture(True)
    except Exception as exc:  # capture unsupported: time eager launches
        timing = f"median of {args.repeats} timed runs of {args.steps} eager steps ({type(exc).__name__})"
        torch.cuda.synchronize()

        def run():
            for i in range(args.steps):
                step(sets[i % len(sets)])

        def run_breakdown():
            for i in range(args.steps):
                step(sets[i % len(sets)], evs[i])
    replays = []
    with Clocks(torch.cuda.current_device()) as clk:
        for _ in range(args.repeats):
            barrier()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record()
            run()
            t1.record()
            barrier()
            replays.append(t0.elapsed_time(t1))
    clocks = clk.summary()
    replays = max_over_ranks(replays, world, dev)
    ms_step = statistics.median(replays) / args.steps
    # per-kernel times: the event-bracketed graph replayed five times, each
    # kernel's mean over the steps of a replay, the median over the replays
    sel_r, att_r = [], []
    for _ in range(5):
        run_breakdown()
        torch.cuda.synchronize()
        sel_r.append(statistics.mean(e[0].elapsed_time(e[1]) for e in evs))
        att_r.append(statistics.mean(e[1].elapsed_time(e[2]) for e in evs))
    sel_avg, att_avg = statistics.median(sel_r), statistics.median(att_r)
    check_status()

    peak_gbs, _, peak_kind = _load_peaks()
    if fused:
        # the single launch keeps the index list on chip; two launches
        # write it and read it back
        step_bytes = fused_step_bytes(sh, K) if single else sum(decode_bytes(sh, K))
        sel_bytes, att_bytes = step_bytes, 0
        dom_name = "decode_step (single launch)" if single else "esa_gated_sparse_attn (select + attention)"
        dom_ms, dom_bytes = sel_avg, step_bytes
        traffic = _traffic_for("decode_step", FUSED_SRC)
        kernels = {"decode_step": sel_avg * 1e3}
    else:
        sel_bytes, att_bytes = decode_bytes(sh, K)
        dom_is_sel = sel_avg >= att_avg
        dom_name = "split_select" if dom_is_sel else "sparse_attn"
        dom_ms, dom_bytes = (sel_avg, sel_bytes) if dom_is_sel else (att_avg, att_bytes)
        traffic = _traffic_for(dom_name, SELECT_SRC if dom_is_sel else ATTN_SRC)
        kernels = {"split_select": sel_avg * 1e3, "sparse_attn": att_avg * 1e3}
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    res = {
        "name": name, "sh": sh, "K": K, "host": host, "cfg": cfg, "ms_per_step": ms_step,
        "replay_ms": replays, "timing": timing, "clocks": clocks, "launches_per_step": launches_per_step,
        "l2": f"{args.sets} rotating input sets (kI caches {args.sets * B * L * DI / 2**20:.0f} MiB"
              f"{' > 126 MB L2' if args.sets * B * L * DI > 126e6 else ', within L2'})",
        "roofline": {"bound": "hbm", "kernel": dom_name,
                     "achieved": achieved, "peak": peak_gbs, "unit": "GB/s", "frac": achieved / peak_gbs,
                     "peak_kind": peak_kind, "traffic": traffic, "algorithmic_bytes": dom_bytes,
                     "avg_launch_us": dom_ms * 1e3},
        "kernels_us": kernels,
        "kernel_replays_us": {"first": [round(x * 1e3, 2) for x in sel_r], "second": [round(x * 1e3, 2) for x in att_r]},
        "step_roofline": {"achieved": (sel_bytes + att_bytes) / (ms_step / 1e3) / 1e9, "peak": peak_gbs,
                          "frac": (sel_bytes + att_bytes) / (ms_step / 1e3) / 1e9 / peak_gbs,
                          "algorithmic_bytes": sel_bytes + att_bytes},
    }
    if not e2e:
        del sets
        torch.cuda.empty_cache()
        return res

    # ---- end to end through host buffers: per step copy the new token's
    # inputs in (q, qI, lin, and its K/V/kI rows, written into the caches at
    # position L-1) and the output back. The inputs travel as ONE copy from a
    # pinned staging buffer into a device staging buffer whose typed views
    # are the step's q, qI and lin; esa_cache_append (one launch) places the
    # new cache rows. Each input set's whole step (copy in, cache append, the
    # library calls, copy out) is captured once into a CUDA graph and
    # replayed per step. A decode step's inputs depend on the previous step's
    # output, so the steps are serialised on one stream.
    parts = [host["q"], host["qI"], host["lin"], host["k"][:, L - 1:L], host["v"][:, L - 1:L], host["kI"][:, L - 1:L]]
    parts = [t.contiguous() for t in parts]
    nbytes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in nbytes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    h_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
    for t, o, n in zip(parts, offs, nbytes):
        h_in[o:o + n].copy_(t.view(-1).view(torch.uint8))
    h_out = torch.empty(B, 1, Hq, D, dtype=torch.float32).pin_memory()
    h2d = sum(nbytes)
    d2h = h_out.numel() * 4

    def make_e2e(d):
        d_in = torch.empty(offs[-1], dtype=torch.uint8, device=dev)
        v = [d_in[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, nbytes)]
        dd = dict(d, q=v[0], qI=v[1], lin=v[2])

        def e2e_step():
            d_in.copy_(h_in, non_blocking=True)
            esa.esa_cache_append(v[3], v[4], v[5], d["k"], d["v"], d["kI"], shape)
            step(dd)
            h_out.copy_(d["out"], non_blocking=True)
        return e2e_step

    e2e_steps = [make_e2e(d) for d in sets]
    e2e_timing = "cuda-graph per step"
    try:
        e2e_run = []
        for fn in e2e_steps:
            fn()
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                fn()
            g.replay()
            torch.cuda.synchronize()
            e2e_run.append(g.replay)
    except Exception as exc:  # capture unsupported: eager steps
        e2e_timing = f"eager ({type(exc).__name__})"
        torch.cuda.synchronize()
        e2e_run = e2e_steps
    for i in range(3):
        e2e_run[i % len(e2e_run)]()
    e2e_reps = []
    for _ in range(args.repeats):
        barrier()
        a0 = time.perf_counter()
        for i in range(args.steps):
            e2e_run[i % len(e2e_run)]()
        torch.cuda.synchronize()
        e2e_reps.append((time.perf_counter() - a0) * 1e3)
        barrier()
    check_status()
    e2e_reps = max_over_ranks(e2e_reps, world, dev)
    e2e_ms = statistics.median(e2e_reps) / args.steps
    res["e2e"] = {"value": job_rate(B, world, e2e_ms), "unit": "tok/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                  "timing": f"{e2e_timing}, median of {args.repeats} runs of {args.steps} steps (host clock)"}
    del sets, e2e_run, e2e_steps
    torch.cuda.empty_cache()
    return res


def _r(x, n=4):
    """A number rounded to n significant digits (keeps the JSON line short)."""
    if x is None or not isinstance(x, (int, float)) or x == 0 or not math.isfinite(x):
        return x
    return float(f"{x:.{n}g}")


def summarise(dec: dict, mdec: dict | None, prefill: dict | None, kda: dict | None, cpu: dict | None,
              mcpu: dict | None) -> dict:
    """One short entry per workload: time, rate, roofline fraction, oracle rate."""
    out = {}
    if prefill and "tiny_prefill" in prefill:
        p = prefill["tiny_prefill"]
        out["1_tiny_prefill"] = {"ms": _r(p["ms"]), "tok_s": _r(p["tok_per_s"]), "bound": "latency",
                                 "cpu_tok_s": _r((p.get("cpu_baseline") or {}).get("tok_per_s"))}
    for key, d, c in (("2_decode", dec, cpu), ("5_million_decode", mdec, mcpu)):
        if d:
            out[key] = {"us": _r(d["ms_per_step"] * 1e3), "tok_s": _r(d["sh"]["B"] / d["ms_per_step"] * 1e3),
                        "hbm_frac": _r(d["step_roofline"]["frac"], 3),
                        "top_kernel_frac": _r(d["roofline"]["frac"], 3),
                        "cpu_tok_s": _r((c or {}).get("value"))}
    for key, name in (("3_long_prefill", "long_prefill"), ("4_routed_prefill", "routed_prefill"),
                      ("chunked_prefill", "chunked_prefill"), ("per_head_prefill", "per_head_prefill")):
        if prefill and name in prefill:
            p = prefill[name]
            e = {"ms": _r(p["ms"]), "tok_s": _r(p["tok_per_s"]), "bf16_frac": _r(p["frac_of_bf16_peak"], 3)}
            e.update({k: _r(v) for k, v in p["kernels_ms"].items()})
            if "path" in p:
                e["path"] = "one call" if p["path"].startswith("esa_gated") else "two calls"
            e["cpu_tok_s"] = _r((p.get("cpu_baseline") or {}).get("tok_per_s"))
            out[key] = e
            if "router" in p:
                out["router"] = {"ms": _r(p["router"]["ms"]), "hbm_frac": _r(p["router"]["frac_of_hbm"], 3)}
    if kda:
        if "decode" in kda:
            k = kda["decode"]
            out["kda_decode"] = {"us": _r(k["us"]), "hbm_frac": _r(k["frac_of_hbm"], 3),
                                 "cpu_tok_s": _r((k.get("cpu_baseline") or {}).get("tok_per_s"))}
        if "long_prefill" in kda:
            k = kda["long_prefill"]
            out["kda_prefill"] = {"ms": _r(k["ms"]), "alu_frac": _r(k["frac_of_alu"], 3),
                                  "tf32_frac": _r((k.get("tensor_view") or {}).get("frac"), 3),
                                  "stepwise_ms": _r(k.get("stepwise_ms")),
                                  "cpu_tok_s": _r((k.get("cpu_baseline") or {}).get("tok_per_s"))}
    return out


def esa_arm(args):
    world, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.kda_only:  # profiling aid: the KDA linear branch alone
        sys.path.insert(0, ROOT)
        import esa_inputs as E
        import long_context_sparse_20_b300 as esa
        if rank == 0:
            print(json.dumps({"linear_branch": kda_section(dev, esa, E, T=args.kda_steps)}), flush=True)
        return
    if args.prefill_only:  # profiling aid: the prefill workloads alone
        sys.path.insert(0, ROOT)
        import esa_inputs as E
        import long_context_sparse_20_b300 as esa
        if rank == 0:
            print(json.dumps({"prefill": prefill_section(dev, esa, E, seq=args.prefill_seq,
                                                         names=args.prefill_names.split(","))}), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    sys.path.insert(0, ROOT)
    import esa_inputs as E
    import long_context_sparse_20_b300 as esa

    dec = decode_section(dev, esa, E, args.workload, args, world, e2e=True)
    sh, K, B = dec["sh"], dec["K"], dec["sh"]["B"]
    ms_step = dec["ms_per_step"]
    value = job_rate(B, world, ms_step)

    mdec = prefill = kda = cpu = mcpu = None
    other = "million_decode" if args.workload != "million_decode" else "decode"
    if rank == 0 and not args.no_extra_decode:
        mdec = decode_section(dev, esa, E, other, args, 1, e2e=False)
    if rank == 0 and not args.no_prefill:
        prefill = prefill_section(dev, esa, E, seq=args.prefill_seq,
                                  oracle_rows=0 if args.no_cpu_baseline else args.oracle_rows)
    if rank == 0 and not args.no_kda:
        kda = kda_section(dev, esa, E, T=args.kda_steps, oracle=not args.no_cpu_baseline)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            v, cores, sample = run_cpu_baseline(dec["cfg"], dec["host"], seconds=args.cpu_seconds)
            v1, sample1 = run_cpu_baseline_1thread(dec["cfg"], dec["host"], seconds=args.cpu_seconds / 2)
            cpu = {"value": v, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample,
                   "one_thread": {"value": v1, "unit": "tok/s", "cores": 1, "sample": sample1}}
            if mdec:
                v, cores, sample = run_cpu_baseline(mdec["cfg"], mdec["host"], seconds=args.cpu_seconds / 2)
                mcpu = {"value": v, "unit": "tok/s", "cores": cores, "kind": "oracle", "sample": sample}
        configs = summarise(dec if args.workload == "decode" else mdec, mdec if args.workload == "decode" else dec,
                            prefill, kda, cpu if args.workload == "decode" else mcpu,
                            mcpu if args.workload == "decode" else cpu)
        roof = {k: (_r(v) if isinstance(v, float) else v) for k, v in dec["roofline"].items()}
        line = {
            "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "us_per_step": _r(ms_step * 1e3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": run_config(args.workload, sh, K, world),
            "timing": f"{dec['timing']}; {dec['l2']}",
            "roofline": roof,
            "step_roofline_frac": _r(dec["step_roofline"]["frac"], 3),
            "gpu_launches": dec["launches_per_step"] * args.steps,
            "e2e": {k: (_r(v) if isinstance(v, float) else v) for k, v in dec["e2e"].items() if k != "timing"},
            "clocks": dec["clocks"],
            "cpu_baseline": ({k: (_r(v) if isinstance(v, float) else v) for k, v in cpu.items() if k != "one_thread"}
                             if cpu else None),
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
        detail = {"decode": {k: v for k, v in dec.items() if k not in ("host", "cfg")},
                  "other_decode": {k: v for k, v in mdec.items() if k not in ("host", "cfg")} if mdec else None,
                  "cpu_baseline": cpu, "other_cpu_baseline": mcpu, "prefill": prefill, "linear_branch": kda}
        print(json.dumps({"detail": detail}, default=str), file=sys.stderr, flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--repeats", type=int, default=7, help="timed replays of the K-step graph (median taken)")
    ap.add_argument("--impl", default="esa", choices=["esa", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sets", type=int, default=NSETS, help="rotating input sets (small profiling cases use 1)")
    ap.add_argument("--no-prefill", action="store_true", help="skip the prefill workloads' timings")
    ap.add_argument("--prefill-only", action="store_true", help="time the prefill workloads only (profiling)")
    ap.add_argument("--prefill-seq", type=int, default=0, help="override the prefill sequence length (profiling)")
    ap.add_argument("--prefill-names", default="tiny_prefill,long_prefill,chunked_prefill,per_head_prefill,routed_prefill",
                    help="comma-separated prefill workloads for --prefill-only (profiling)")
    ap.add_argument("--no-kda", action="store_true", help="skip the KDA linear branch's timings")
    ap.add_argument("--no-extra-decode", action="store_true", help="skip the second decode workload")
    ap.add_argument("--gated", action="store_true",
                    help="decode step as the one-call esa_gated_sparse_attn instead of esa_topk_select + "
                         "esa_sparse_attn")
    ap.add_argument("--oracle-rows", type=int, default=64,
                    help="query rows per prefill workload on which the oracle is timed (extrapolated)")
    ap.add_argument("--kda-only", action="store_true", help="time the KDA linear branch alone (profiling)")
    ap.add_argument("--kda-steps", type=int, default=32768, help="KDA prefill steps (profiling of small cases)")
    args = ap.parse_args()
    if args.impl == "reference":
        reference_arm(args)
    else:
        esa_arm(args)


if __name__ == "__main__":
    main()
