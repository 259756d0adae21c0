"""The allocation-free forward (tl_encoder_forward_static) agrees with the
ordinary forward.

Collected last on purpose (file name), so a run that stops at the first
failure has run every other test first.  Calls the entry point through the C
ABI (ctypes) twice in a row on the same handle: the static scratch array
keeps the first call's contents, and the second call must not depend on
them.  Must pass alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest

from transformer_encoder_layer_gb300.gate import gate
from transformer_encoder_layer_gb300.inputs import SHAPES, make_inputs, tiny_shape, to_storage

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _tensor(a, dtype):
    st = to_storage(a, dtype)
    if dtype == "bf16":
        return torch.from_numpy(st.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(st).cuda()


def _as_f64(t):
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("shape,path,batch", [
    # layered path: its workspace lives in the static array
    (SHAPES["short_d128_L64_B4096"].with_(batch=8), "layered", None),
    # CUDA-core path (fp32 I/O) with the batch-1 workload
    (SHAPES["batch1_d256_L512"], "auto", None),
    (tiny_shape(dtype="bf16", batch=3, seq_len=130, vl_lo=1, vl_hi=130, d_model=64,
                n_heads=4, d_ff=256), "auto", None),
])
def test_static_scratch_forward_matches_forward(shape, path, batch):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    lib = binding.load()
    enc = binding.Encoder(make_inputs(shape, seed=0).layers, shape.d_model, shape.n_heads,
                          shape.d_ff, shape.dtype)
    try:
        if path != "auto":
            enc.set_path(path)
        B, L = shape.batch, shape.seq_len
        need = enc.workspace_size(B, L)
        assert 0 < need <= (32 << 20)
        outs = []
        for seed in (1, 2):  # two calls in a row, different inputs
            inp = make_inputs(shape, seed=seed, input_scale=10.0 if seed == 2 else 1.0)
            x = _tensor(inp.x, shape.dtype)
            vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
            ref = enc.forward(x, vl)  # the ordinary entry point, caller workspace
            out = torch.empty_like(x)
            stream = torch.cuda.current_stream()
            rc = lib.tl_encoder_forward_static(enc.handle, ctypes.c_void_p(x.data_ptr()), B, L,
                                               ctypes.c_void_p(vl.data_ptr()),
                                               ctypes.c_void_p(out.data_ptr()),
                                               ctypes.c_void_p(int(stream.cuda_stream)))
            assert rc == 0, binding.STATUS.get(rc, rc)
            assert lib.tl_encoder_get_status(enc.handle, ctypes.c_void_p(int(stream.cuda_stream))) == 0
            ok, util, idx = gate(_as_f64(out), _as_f64(ref))
            assert ok, f"call with seed {seed}: envelope {util:.3f} at {idx}"
            outs.append(_as_f64(out))
        assert not np.array_equal(outs[0], outs[1])
    finally:
        enc.close()


def test_static_scratch_rejects_oversized_shapes():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    lib = binding.load()
    s = SHAPES["short_d128_L64_B4096"]
    enc = binding.Encoder(make_inputs(s.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1)).layers,
                          s.d_model, s.n_heads, s.d_ff, s.dtype)
    try:
        enc.set_path("layered")
        B, L = 4096, 64
        assert enc.workspace_size(B, L) > (32 << 20)
        x = torch.zeros((B, L, 128), dtype=torch.float16, device="cuda")
        vl = torch.full((B,), L, dtype=torch.int32, device="cuda")
        out = torch.empty_like(x)
        rc = lib.tl_encoder_forward_static(enc.handle, ctypes.c_void_p(x.data_ptr()), B, L,
                                           ctypes.c_void_p(vl.data_ptr()),
                                           ctypes.c_void_p(out.data_ptr()), None)
        assert rc == 5  # TL_ERR_WORKSPACE_TOO_SMALL, nothing launched
    finally:
        enc.close()
