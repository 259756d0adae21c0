"""Host-side checks of the seeded input generator and the accuracy gate."""
import numpy as np
import pytest
import torch

from transformer_encoder_layer_gb300.gate import gate
from transformer_encoder_layer_gb300.inputs import (
    SHAPES, from_storage, make_inputs, round_to_dtype, tiny_shape, to_storage)


def test_bf16_rounding_matches_torch_for_fp32_values():
    rng = np.random.default_rng(0)
    a = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ours = round_to_dtype(a.astype(np.float64), "bf16")
    ref = torch.tensor(a).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_bf16_rounding_is_single_step_from_fp64():
    # 1 + 2^-8 + 2^-30 lies just above the bf16 midpoint between 1 and 1+2^-7:
    # direct RNE rounds up; rounding through fp32 first would keep the
    # midpoint... and tie to even (down).  Our conversion must round up.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -30
    assert round_to_dtype(np.array([v]), "bf16")[0] == 1.0 + 2.0 ** -7


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_storage_roundtrip(dtype):
    rng = np.random.default_rng(1)
    a = round_to_dtype(rng.standard_normal(1000) * 3, dtype)
    assert np.array_equal(from_storage(to_storage(a, dtype), dtype), a)


def test_inputs_are_seeded_and_prefix_consistent():
    s = SHAPES["short_d128_L64_B4096"].with_(batch=64)
    a = make_inputs(s, seed=0, input_scale=10.0)
    b = make_inputs(s, seed=0, input_scale=10.0)
    c = make_inputs(s, seed=0, input_scale=10.0, batch=8)
    assert np.array_equal(a.x, b.x) and np.array_equal(a.valid_len, b.valid_len)
    assert np.array_equal(c.x, a.x[:8]) and np.array_equal(c.valid_len, a.valid_len[:8])
    for pa, pc in zip(a.layers, c.layers):
        for k in pa:
            assert np.array_equal(pa[k], pc[k])
    assert a.valid_len.min() >= 32 and a.valid_len.max() <= 64


def test_weight_statistics():
    s = tiny_shape(d_model=256, d_ff=1024, n_heads=4, n_layers=1, batch=1, seq_len=1)
    p = make_inputs(s, seed=2).layers[0]
    assert abs(p["w_qkv"].std() - 1 / 16) < 2e-3
    assert abs(p["w_2"].std() - 1 / 32) < 1e-3
    assert abs(p["b_1"].std() - 0.02) < 2e-3
    assert abs(p["ln1_g"].mean() - 1.0) < 0.03


def test_gate_semantics():
    ref = np.array([1.0, 0.0, 100.0, -0.05])
    ok, util, _ = gate(ref + np.array([0.019, 0.0019, 1.9, 0.0019]), ref)
    assert ok and util < 1
    ok, util, idx = gate(ref + np.array([0.0, 0.0021, 0.0, 0.0]), ref)
    assert not ok and idx == (1,)
    ok, _, _ = gate(np.array([np.nan, 0, 0, 0]), np.zeros(4))
    assert not ok
