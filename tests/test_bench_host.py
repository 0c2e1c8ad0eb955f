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
