"""The CPU rounding-emulation probe that sets the tensor-core paths'
precision plan, pinned here so that its conclusions are reproducible:

* plain 16-bit activation operands fail the gate (fp16 at input scale 10 and
  above, bf16 everywhere);
* a (hi, lo) pair for every activation operand passes with a wide margin;
* with fp16, dropping the lo part of P (the Pl.Vh product) and of the FFN
  hidden (FFN2 on h_hi) still passes: the megakernel's fp16 plan; P alone is
  the layered fp16 attention's plan;
* with bf16 the same removal fails, so bf16 keeps every lo part.

The measured GPU envelopes agree with the probe's all-split prediction
(0.024 on the d128 workload, 0.19-0.26 on the d1024 one).
"""
import numpy as np
import pytest

import oracle
import precision_probe as pp
from transformer_encoder_layer_gb300.gate import gate
from transformer_encoder_layer_gb300.inputs import SHAPES, make_inputs

FP16_MEGA = pp.Plan(p_lo=False, h_lo=False)


def _envelopes(shape, nseq, scale, plans, seed=0):
    inp = make_inputs(shape, seed=seed, input_scale=scale, batch=nseq)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, shape.n_heads, check=False)
    out = {}
    for name, plan in plans.items():
        got = pp.forward(inp.x, inp.valid_len, inp.layers, shape.n_heads, shape.dtype, plan)
        out[name] = gate(got, ref)[1]
    return out


def test_probe_without_roundings_is_the_oracle():
    """With no operand rounded (fp32 I/O plan on fp32 inputs, splits exact to
    fp32 resolution) the probe agrees with the oracle to fp32 rounding."""
    s = SHAPES["tiny_d32_L32"]
    inp = make_inputs(s, seed=1)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, s.n_heads)
    got = pp.forward(inp.x, inp.valid_len, inp.layers, s.n_heads, "f32", pp.ALL_SPLIT)
    assert np.max(np.abs(got - ref)) < 1e-4


@pytest.mark.parametrize("scale", [1e-3, 1.0, 10.0, 1e3])
def test_fp16_d128_plans(scale):
    s = SHAPES["short_d128_L64_B4096"]
    e = _envelopes(s, 8, scale, {"split": pp.ALL_SPLIT, "mega": FP16_MEGA, "plain": pp.PLAIN})
    assert e["split"] < 0.1, e
    assert e["mega"] < 0.8, e
    if scale >= 10.0:
        assert e["plain"] > 1.0, e


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_fp16_long_sequence_layer_without_pl(scale):
    """The 100k-token workload's layer (fp16, head_dim 16) on 2 sequences of
    1000 tokens: P without its lo part (the layered fp16 attention's plan)
    stays far inside the gate."""
    s = SHAPES["long_d64_L100k_B8"].with_(seq_len=1000, vl_lo=900, vl_hi=1000)
    e = _envelopes(s, 2, scale, {"split": pp.ALL_SPLIT, "p_hi": pp.Plan(p_lo=False)})
    assert e["p_hi"] < 0.6, e


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_bf16_d1024_needs_every_lo_part(scale):
    s = SHAPES["wide_d1024_L1024_B32"].with_(seq_len=128, vl_lo=64, vl_hi=128)
    e = _envelopes(s, 1, scale, {"split": pp.ALL_SPLIT, "p_hi": pp.Plan(p_lo=False),
                                 "plain": pp.PLAIN})
    assert e["split"] < 0.5, e
    assert e["plain"] > 1.0, e
    assert e["p_hi"] > 0.5, e
