"""The benchmark's CPU-side baselines on a tiny workload (no GPU): the
oracle timed on a seeded row sample and extrapolated, and the one-thread
decode figure — they run, report what they sampled, and give positive
rates."""
import os
import sys

import esa_inputs as E

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_oracle_row_sample_extrapolates():
    cfg = E.small_config(seed=5, B=2, Tq=96, Tk=96, Hq=4, Hkv=1, D=64, top_k=24)
    r = bench.oracle_row_sample(E.make_inputs(cfg), E.shape_of(cfg), cfg["top_k"], n_rows=8)
    assert r["tok_per_s"] > 0 and r["kind"] == "oracle, extrapolated" and r["cores"] >= 1
    assert r["sample"].startswith("8 seeded uniform rows of 192")


def test_one_thread_decode_figure_restores_the_thread_setting():
    cfg = E.small_config(seed=6, B=2, Tq=1, Tk=300, q_offset=299, Hq=4, Hkv=1, D=64, top_k=32)
    before = os.environ.get("ESA_ORACLE_THREADS")
    v, sample = bench.run_cpu_baseline_1thread(cfg, E.make_inputs(cfg), seconds=0.2)
    assert v > 0 and "decode rows one at a time" in sample
    assert os.environ.get("ESA_ORACLE_THREADS") == before


def test_summary_line_is_compact_and_covers_every_config():
    """The JSON line's per-workload map stays short enough for a log tail to
    hold the whole line, and names the five configurations."""
    import json
    sh = dict(B=8, Tk=131072)
    dec = {"ms_per_step": 0.02, "sh": sh, "step_roofline": {"frac": 0.6}, "roofline": {"frac": 0.7}}
    mdec = {"ms_per_step": 0.02, "sh": dict(B=1, Tk=1 << 20), "step_roofline": {"frac": 0.5},
            "roofline": {"frac": 0.6}}
    pre = {n: {"ms": 1.234567, "tok_per_s": 123456.789, "frac_of_bf16_peak": 0.0123456,
               "kernels_ms": {"topk_select": 1.0, "sparse_attn": 2.0}, "cpu_baseline": {"tok_per_s": 600.123}}
           for n in ("tiny_prefill", "long_prefill", "chunked_prefill", "per_head_prefill", "routed_prefill")}
    pre["routed_prefill"]["router"] = {"ms": 0.19, "frac_of_hbm": 0.87}
    kda = {"decode": {"us": 8.9, "frac_of_hbm": 0.59, "cpu_baseline": {"tok_per_s": 2700.0}},
           "long_prefill": {"ms": 5.5, "frac_of_alu": 0.14, "cpu_baseline": {"tok_per_s": 21000.0}}}
    s = bench.summarise(dec, mdec, pre, kda, {"value": 43.0}, {"value": 3.3})
    for key in ("1_tiny_prefill", "2_decode", "3_long_prefill", "4_routed_prefill", "5_million_decode"):
        assert key in s
    assert len(json.dumps(s)) < 1600


def test_both_arms_print_the_same_config():
    sh = E.shape_of(E.CONFIGS["decode"])
    c = bench.run_config("decode", sh, 2048, 1)
    assert c["workload"] == bench.decode_label("decode", sh, 2048)
    assert c["workload"].startswith("decode: B=8 x 1 new token, cache 131072")
