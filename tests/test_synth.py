"""The synthetic workloads have the shapes, formats and load structure they claim."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle


def test_skew_workload_load_structure():
    inp = moe_synth.make_inputs("skew", router_only=True)
    _, ids, _ = oracle.route(oracle.x_values(inp), inp.w_router, inp.bias, inp.cfg.k)
    counts = np.bincount(ids.reshape(-1), minlength=128)
    assert abs(counts.max() / counts.mean() - 8.0) < 0.25
    assert (counts == 0).sum() >= 4


def test_decode_workload_routing_spread():
    inp = moe_synth.make_inputs("decode", router_only=True)
    _, ids, _ = oracle.route(oracle.x_values(inp), inp.w_router, inp.bias, inp.cfg.k)
    assert len(np.unique(ids)) > 110           # nearly every expert is active at T=64


def test_seed_determinism_and_independence():
    a = moe_synth.make_custom(8, 64, 8, 2, 32, 32, "bf16", "e4m3", seed=3)
    b = moe_synth.make_custom(8, 64, 8, 2, 32, 32, "bf16", "e4m3", seed=3)
    c = moe_synth.make_custom(8, 64, 8, 2, 32, 32, "bf16", "e4m3", seed=4)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.w13, b.w13)
    assert not np.array_equal(a.x, c.x)


@pytest.mark.parametrize("w_dtype", ["f32", "e4m3", "nvfp4"])
def test_stored_shapes(w_dtype):
    inp = moe_synth.make_custom(4, 64, 8, 2, 32, 48, "bf16", w_dtype)
    E, d, f, fs = 8, 64, 32, 48
    if w_dtype == "nvfp4":
        assert inp.w13.shape == (E, 2 * f, d // 2) and inp.w13_scale.shape == (E, 2 * f, d // 16)
        assert inp.w2.shape == (E, d, f // 2) and inp.w2_gscale.shape == (E,)
        assert inp.s13.shape == (1, 2 * fs, d // 2) and inp.s2_scale.shape == (1, d, fs // 16)
    else:
        assert inp.w13.shape == (E, 2 * f, d) and inp.w2.shape == (E, d, f)
        assert inp.s13.shape == (1, 2 * fs, d) and inp.s2.shape == (1, d, fs)
    assert inp.x.dtype == np.uint16 and inp.x.shape == (4, d)


def test_weight_distribution_scale():
    inp = moe_synth.make_custom(4, 1024, 4, 2, 256, 256, "bf16", "e4m3")
    W13, _ = oracle.expert_weights(inp, 0)
    assert abs(W13.std() * np.sqrt(1024) - 1.0) < 0.02
    x = oracle.x_values(inp)
    assert abs(x.std() - 1.0) < 0.05
    # x really is bf16-representable
    assert np.array_equal(torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy(), x)
