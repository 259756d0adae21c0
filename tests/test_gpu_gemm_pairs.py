"""The layered path's GEMMs on CTA pairs (tcgen05 cta_group::2, one MMA
instruction over a 256-row block shared by two CTAs) against the fp64
oracle, and against the one-CTA GEMMs, on every epilogue (head-major QKV,
GELU, LayerNorm over one and several N tiles) with ragged row counts."""
import numpy as np
import pytest

import oracle
from transformer_encoder_layer_gb300.gate import gate
from transformer_encoder_layer_gb300.inputs import SHAPES, make_inputs, tiny_shape, to_storage

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    binding.load()


def _run(inp, pairs):
    from transformer_encoder_layer_gb300 import binding
    from transformer_encoder_layer_gb300.inputs import from_storage
    s = inp.shape
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    try:
        enc.set_path("layered")
        enc.set_gemm_pairs(pairs)
        st = to_storage(inp.x, s.dtype)
        x = (torch.from_numpy(st.view(np.int16)).view(torch.bfloat16) if s.dtype == "bf16"
             else torch.from_numpy(st)).cuda()
        vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
        o = enc.forward(x, vl).cpu()
        if s.dtype == "bf16":
            return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16")
        return from_storage(o.numpy(), s.dtype)
    finally:
        enc.close()


@pytest.mark.parametrize("dtype,d,H,dff,L,batch", [
    ("bf16", 256, 4, 1024, 100, 3),    # 300 rows: a ragged second pair block
    ("f16", 384, 6, 768, 130, 4),      # N tile 192 (96 weight rows per CTA), LN over two tiles
    ("bf16", 1024, 16, 4096, 256, 2),  # the d1024 layer, LN rows over four N tiles
    ("f16", 64, 4, 256, 600, 2),       # the 100k-token workload's layer (head_dim 16)
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_pair_gemms_pass_the_gate(dtype, d, H, dff, L, batch, scale):
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d, n_heads=H,
                   d_ff=dff, n_layers=2)
    inp = make_inputs(s, seed=13, input_scale=scale)
    got = _run(inp, True)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, H, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"envelope {util:.3f} at {idx}"
    one = _run(inp, False)
    ulp = 2.0 ** (-8 if dtype == "bf16" else -11) * np.abs(one)
    assert np.all(np.abs(got - one) <= np.maximum(2 * ulp, 1e-3))


def test_pairs_on_the_d1024_workload_sample():
    s = SHAPES["wide_d1024_L1024_B32"]
    inp = make_inputs(s, seed=1, batch=2)
    got = _run(inp, True)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, s.n_heads, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"envelope {util:.3f} at {idx}"
