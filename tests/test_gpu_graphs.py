"""Graph mode: the layered path's launches recorded once per (shape,
buffers) into a CUDA graph and replayed ("KernelForge", section "What we
built": a forward captured in a CUDA graph).  Replays give the eager
forward's bits, follow new contents of the same buffers, and a new buffer
set is recorded afresh."""
import numpy as np
import pytest

from transformer_encoder_layer_gb300.inputs import make_inputs, tiny_shape, to_storage

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    binding.load()


def _x(inp):
    st = to_storage(inp.x, inp.shape.dtype)
    if inp.shape.dtype == "bf16":
        return torch.from_numpy(st.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(st).cuda()


@pytest.mark.parametrize("dtype,d,H,L,batch,split", [
    ("bf16", 256, 4, 300, 3, -1),
    ("f16", 64, 4, 1500, 1, 2),      # split-K attention: counter memsets in the graph
    ("bf16", 512, 8, 96, 4, -1),     # LayerNorm apply pass (rows wider than one N tile)
])
def test_graph_replays_match_eager(dtype, d, H, L, batch, split):
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d, n_heads=H,
                   d_ff=2 * d, n_layers=2)
    a = make_inputs(s, seed=21)
    b = make_inputs(s, seed=22)
    enc = binding.Encoder(a.layers, d, H, 2 * d, dtype)
    enc.set_path("layered")
    enc.set_attention_split(split)
    ws = torch.empty(enc.workspace_size(batch, L), dtype=torch.uint8, device="cuda")
    xa, xb = _x(a), _x(b)
    vla = torch.from_numpy(a.valid_len.astype(np.int32)).cuda()
    vlb = torch.from_numpy(b.valid_len.astype(np.int32)).cuda()
    ref_a = enc.forward(xa, vla, workspace=ws).clone()
    ref_b = enc.forward(xb, vlb, workspace=ws).clone()
    enc.set_graphs(True)
    x = xa.clone()
    vl = vla.clone()
    out = torch.empty_like(x)
    for i in range(3):
        out.view(torch.uint8).fill_(0xFF)
        enc.forward(x, vl, out=out, workspace=ws)
        assert torch.equal(out.view(torch.uint8), ref_a.view(torch.uint8)), f"call {i}"
    assert enc.graph_stats() == (1, 2)
    # new contents of the same buffers: the replay reads them
    x.copy_(xb)
    vl.copy_(vlb)
    enc.forward(x, vl, out=out, workspace=ws)
    assert torch.equal(out.view(torch.uint8), ref_b.view(torch.uint8))
    assert enc.graph_stats() == (1, 3)
    # a new output buffer: recorded afresh
    out2 = torch.empty_like(x)
    enc.forward(x, vl, out=out2, workspace=ws)
    enc.forward(x, vl, out=out2, workspace=ws)
    assert torch.equal(out2.view(torch.uint8), ref_b.view(torch.uint8))
    assert enc.graph_stats() == (2, 4)
    enc.set_graphs(False)
    enc.forward(x, vl, out=out, workspace=ws)
    assert enc.graph_stats() == (2, 4)
    assert enc.get_status() == 0
    enc.close()


def test_graph_mode_leaves_other_paths_alone():
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype="f16", batch=4, seq_len=64, vl_lo=1, vl_hi=64, d_model=128, n_heads=4,
                   d_ff=512, n_layers=2)
    inp = make_inputs(s, seed=3)
    enc = binding.Encoder(inp.layers, 128, 4, 512, "f16")
    assert enc.plan(4, 64) == "mega"
    enc.set_graphs(True)
    x = _x(inp)
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    o1 = enc.forward(x, vl).clone()
    o2 = enc.forward(x, vl)
    assert torch.equal(o1, o2)
    assert enc.graph_stats() == (0, 0)
    enc.close()
