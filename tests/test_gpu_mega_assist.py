"""Assisting CTAs for the sequence-resident megakernel: for batches whose
tiles fill at most half the SMs, each 128-row tile runs on a cluster of two
CTAs (the resident one and a helper that takes half the heads and half the
FFN chunks).  Gated against the fp64 oracle over input scales, and against
the unassisted megakernel."""
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


def _run(inp, assist):
    from transformer_encoder_layer_gb300 import binding
    from transformer_encoder_layer_gb300.inputs import from_storage
    s = inp.shape
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    try:
        enc.set_path("mega")
        enc.set_mega_assist(assist)
        used = enc.mega_assisted(s.batch, s.seq_len)
        st = to_storage(inp.x, s.dtype)
        x = (torch.from_numpy(st.view(np.int16)).view(torch.bfloat16) if s.dtype == "bf16"
             else torch.from_numpy(st)).cuda()
        vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
        o = enc.forward(x, vl).cpu()
        if s.dtype == "bf16":
            return from_storage(o.view(torch.int16).numpy().view(np.uint16), "bf16"), used
        return from_storage(o.numpy(), s.dtype), used
    finally:
        enc.close()


@pytest.mark.parametrize("dtype,dff,n_layers,batch", [
    ("f16", 512, 4, 8),      # the d128 workload's layer, 4 tiles
    ("f16", 512, 4, 1),      # one sequence: half a tile
    ("bf16", 512, 2, 13),    # ragged last tile
    ("f16", 384, 3, 6),      # three FFN chunks: two on the resident CTA, one on the helper
    ("f16", 256, 1, 3),      # two chunks, one layer
    ("f16", 512, 2, 152),    # 76 tiles: every SM busy
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_assisted_megakernel_passes_the_gate(dtype, dff, n_layers, batch, scale):
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=64, vl_lo=1, vl_hi=64, d_model=128,
                   n_heads=4, d_ff=dff, n_layers=n_layers)
    inp = make_inputs(s, seed=17, input_scale=scale)
    got, used = _run(inp, 1)
    assert used
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 4, check=False)
    ok, util, idx = gate(got, ref)
    assert ok, f"envelope {util:.3f} at {idx}"
    plain, used0 = _run(inp, 0)
    assert not used0
    ulp = 2.0 ** (-8 if dtype == "bf16" else -11) * np.abs(plain)
    assert np.all(np.abs(got - plain) <= np.maximum(2 * ulp, 1e-3))


def test_assist_is_chosen_by_batch_size():
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["short_d128_L64_B4096"]
    inp = make_inputs(s.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1))
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert not enc.mega_assisted(8, 64)                   # automatic: off
    enc.set_mega_assist(1)
    assert enc.mega_assisted(2 * (sms // 2), 64)          # sms/2 tiles: assisted
    assert not enc.mega_assisted(2 * (sms // 2) + 2, 64)  # one more tile: not
    assert not enc.mega_assisted(4096, 64)
    enc.set_mega_assist(0)
    assert not enc.mega_assisted(8, 64)
    with pytest.raises(binding.TLError):
        enc.set_mega_assist(2)
    enc.close()


def test_assisted_status_and_graph_capture():
    """A bad valid_len is reported from the assisted kernel; the forward
    records into a CUDA graph and replays bit for bit."""
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype="f16", batch=4, seq_len=64, vl_lo=64, vl_hi=64, d_model=128, n_heads=4,
                   d_ff=512, n_layers=2)
    inp = make_inputs(s, seed=5)
    enc = binding.Encoder(inp.layers, 128, 4, 512, "f16")
    enc.set_mega_assist(1)
    assert enc.mega_assisted(4, 64)
    x = torch.from_numpy(to_storage(inp.x, "f16")).cuda()
    bad = torch.tensor([0, 65, 64, 10], dtype=torch.int32, device="cuda")
    out = enc.forward(x, bad, check=False)
    assert enc.get_status() == 6
    ref = enc.forward(x, torch.tensor([1, 64, 64, 10], dtype=torch.int32, device="cuda"))
    assert torch.equal(out, ref)
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    eager = enc.forward(x, vl).clone()
    o2 = torch.empty_like(x)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        enc.forward(x, vl, out=o2, stream=side, check=False)
    for _ in range(2):
        o2.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(o2, eager)
    assert enc.get_status() == 0
    enc.close()
