"""Split-K attention (key range cut into chunks whose partial softmax states
are merged; "KernelForge", section "What's next") against the fp64 oracle.

Batch-1 long sequences are the shapes the split exists for: without it the
few (head, query tile) items of the last causal rows leave most SMs idle.
Forced chunk sizes on ragged shapes reach chunks that hold no visible key
(valid_len far below L), single-tile chunks, and the merge of the near-tie
screen's second-best scores at input scale 1e3.
"""
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


def _device_x(inp):
    st = to_storage(inp.x, inp.shape.dtype)
    if inp.shape.dtype == "bf16":
        return torch.from_numpy(st.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(st).cuda()


def _to_f64(t, dtype):
    from transformer_encoder_layer_gb300.inputs import from_storage
    o = t.cpu()
    if dtype == "bf16":
        return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16")
    return from_storage(o.numpy(), dtype)


def _run(inp, split):
    from transformer_encoder_layer_gb300 import binding
    s = inp.shape
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    try:
        enc.set_path("layered")
        enc.set_attention_split(split)
        kc = enc.attention_split(s.batch, s.seq_len)
        x = _device_x(inp)
        vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
        out = enc.forward(x, vl)
        return _to_f64(out, s.dtype), kc
    finally:
        enc.close()


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_batch1_long_sequence_splits_automatically(scale):
    """The 100k-token workload's layers on one sequence of 8192 tokens: the
    plan splits on its own, and the output passes the gate."""
    s = SHAPES["long_d64_L100k_B8"].with_(batch=1, seq_len=8192, vl_lo=7400, vl_hi=8192)
    inp = make_inputs(s, seed=3, input_scale=scale)
    got, kc = _run(inp, -1)
    assert kc > 0
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, s.n_heads, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"scale {scale}: envelope {util:.3f} at {idx}"


@pytest.mark.parametrize("dtype,d,H,L,vl_lo,vl_hi,batch", [
    ("bf16", 256, 4, 4096, 3000, 4096, 1),   # head_dim 64
    ("f16", 128, 4, 3000, 2000, 3000, 1),    # head_dim 32, ragged last query tile
])
def test_batch1_other_head_widths(dtype, d, H, L, vl_lo, vl_hi, batch):
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=vl_lo, vl_hi=vl_hi, d_model=d,
                   n_heads=H, d_ff=2 * d, n_layers=1)
    inp = make_inputs(s, seed=4, input_scale=1.0)
    got, kc = _run(inp, -1)
    assert kc > 0
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, H, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"envelope {util:.3f} at {idx}"
    # against the unsplit kernel: the same function summed in another order,
    # so the outputs differ at most by the I/O rounding of a value next to a
    # rounding boundary (one unit in the last place)
    base, kc0 = _run(inp, 0)
    assert kc0 == 0
    ulp = 2.0 ** (-8 if dtype == "bf16" else -11) * np.abs(base)
    assert np.all(np.abs(got - base) <= np.maximum(2 * ulp, 1e-3))


@pytest.mark.parametrize("kc", [1, 2, 3, 5])
@pytest.mark.parametrize("dtype,d,H", [("f16", 64, 4), ("bf16", 64, 2), ("f16", 128, 4)])
@pytest.mark.parametrize("scale", [1.0, 1e3])
def test_forced_chunks_on_ragged_shapes(kc, dtype, d, H, scale):
    """Forced chunk sizes, valid lengths from 1 to L: chunks past the valid
    keys arrive empty, padded rows merge over [0, valid_len)."""
    s = tiny_shape(dtype=dtype, batch=3, seq_len=700, vl_lo=1, vl_hi=700, d_model=d, n_heads=H,
                   d_ff=2 * d, n_layers=2)
    inp = make_inputs(s, seed=kc, input_scale=scale)
    inp.valid_len[0] = 1  # only key 0 visible: every later chunk of the sequence is empty
    got, k = _run(inp, kc)
    assert k == kc
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, H, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"kc {kc} scale {scale}: envelope {util:.3f} at {idx}"


def test_split_forward_captures_in_a_cuda_graph():
    """The counter reset and the split kernel record into a CUDA graph; two
    replays give the eager bits (the counters start from zero each time)."""
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype="f16", batch=1, seq_len=1500, vl_lo=1200, vl_hi=1500, d_model=64,
                   n_heads=4, d_ff=256, n_layers=2)
    inp = make_inputs(s, seed=9)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    enc.set_path("layered")
    enc.set_attention_split(2)
    x = _device_x(inp)
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    ws = torch.empty(enc.workspace_size(1, s.seq_len), dtype=torch.uint8, device="cuda")
    ref = enc.forward(x, vl, workspace=ws)
    out = torch.empty_like(x)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        enc.forward(x, vl, out=out, workspace=ws, stream=side, check=False)
    for _ in range(2):
        out.view(torch.uint8).fill_(0xFF)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    assert enc.get_status() == 0
    enc.close()


def test_split_setting_is_checked():
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["long_d64_L100k_B8"]
    inp = make_inputs(s.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1))
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    for bad in (-2, 4097):
        with pytest.raises(binding.TLError):
            enc.set_attention_split(bad)
    # the full 100k-token workload has items enough: no split, no extra workspace
    assert enc.attention_split(8, 100000) == 0
    enc.set_attention_split(0)
    assert enc.attention_split(1, 8192) == 0
    enc.set_attention_split(-1)
    assert enc.attention_split(1, 8192) > 0
    enc.close()
