"""The seeded input generator: the C loops agree with the numpy restatement,
values have the stated ranges, and the workloads have the stated shapes."""
import numpy as np

import esa_inputs as E


def test_c_generator_matches_numpy():
    for seed, tid, n in [(1, 4, 10001), (2005, 2, 4097), (7, 9, 3)]:
        a = E.normal_bf16_bits(seed, tid, n)
        b = E.normal_bf16_bits_np(seed, tid, n)
        # libm and numpy may differ in the last ulp of log/cos; after rounding to
        # bf16 a disagreement is a one-ulp step at most, and must be rare
        diff = np.abs(a.astype(np.int32) - b.astype(np.int32))
        assert diff.max() <= 1 and (diff > 0).mean() < 1e-3
        assert np.array_equal(E.int8_uniform(seed, tid, n), E.int8_uniform_np(seed, tid, n))


def test_value_ranges_and_shapes():
    cfg = E.CONFIGS["tiny_prefill"]
    inp = E.make_inputs(cfg)
    assert tuple(inp["qI"].shape) == (1, 1024, 1, 32) and tuple(inp["kI"].shape) == (1, 1024, 32)
    assert int(inp["qI"].min()) >= -8 and int(inp["qI"].max()) <= 7
    assert tuple(inp["q"].shape) == (1, 1024, 4, 64) and tuple(inp["k"].shape) == (1, 1024, 1, 64)
    x = inp["q"].float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1) < 0.02
    assert ((inp["g"] > 0) & (inp["g"] < 1)).all()
    cfg3 = E.small_config(H_I=4, weights="1to4", routed=True, B=3, Hq=8, Hkv=8)
    inp3 = E.make_inputs(cfg3)
    assert set(inp3["wI"].tolist()) <= {1, 2, 3, 4}
    assert set(inp3["route"].flatten().tolist()) <= {0, 1}
