"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Every comparison is element by element under the pages' gate
(|err| <= 0.002 OR |err| <= 0.02 |ref|, NaN/Inf fail), on seeded inputs, over
seeds and the input-scale sweep 1e-3 .. 1e3.  Sizes the oracle finishes in
seconds are checked in full; full-size workloads are checked on sampled
sequences (sequences are independent) or, for the 100k-token workload, layer
by layer on 4096 sampled query rows of every sequence, and as a whole stack
on a causal prefix (rows < P depend only on tokens < P when P <= valid_len).
"""
import numpy as np
import pytest

import oracle
from transformer_encoder_layer_gb300.gate import gate
from transformer_encoder_layer_gb300.inputs import (
    INPUT_SCALES, SHAPES, make_inputs, tiny_shape, to_storage, from_storage)

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    binding.load()


def _paths_for(shape):
    from transformer_encoder_layer_gb300 import binding
    enc = binding.Encoder(make_inputs(shape.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1)).layers,
                          shape.d_model, shape.n_heads, shape.d_ff, shape.dtype)
    out = []
    for p in ("simt", "layered", "mega", "dag"):
        enc.set_path(p)
        try:
            enc.plan(shape.batch, shape.seq_len)
            out.append(p)
        except binding.TLError:
            pass
    enc.close()
    return out


def _run(inp, path="auto"):
    from transformer_encoder_layer_gb300 import binding
    return binding.run_forward(inp, path=path)


def _check(inp, path="auto", rows=None):
    got = _run(inp, path)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, inp.shape.n_heads)
    if rows is not None:
        got, ref = got[:, rows], ref[:, rows]
    ok, util, idx = gate(got, ref)
    assert ok, f"{inp.shape.name} scale={inp.input_scale} seed={inp.seed} path={path}: " \
               f"envelope {util:.3f} at {idx}: gpu={got[idx]} ref={ref[idx]}"
    return util


# ----------------------------------------------------------- small, in full
@pytest.mark.parametrize("scale", INPUT_SCALES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tiny_d32_full(seed, scale):
    s = SHAPES["tiny_d32_L32"]
    for p in _paths_for(s):
        _check(make_inputs(s, seed=seed, input_scale=scale), p)


@pytest.mark.parametrize("scale", INPUT_SCALES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_batch1_d256_full(seed, scale):
    s = SHAPES["batch1_d256_L512"]
    for p in _paths_for(s):
        _check(make_inputs(s, seed=seed, input_scale=scale), p)


@pytest.mark.parametrize("scale", INPUT_SCALES)
@pytest.mark.parametrize("seed", [0, 1, 2])
def test_short_d128_subsample(seed, scale):
    s = SHAPES["short_d128_L64_B4096"]
    for p in _paths_for(s.with_(batch=32)):
        _check(make_inputs(s, seed=seed, input_scale=scale, batch=32), p)


@pytest.mark.parametrize("scale", INPUT_SCALES)
def test_wide_d1024_subsample(scale):
    s = SHAPES["wide_d1024_L1024_B32"]
    for p in _paths_for(s.with_(batch=2)):
        _check(make_inputs(s, seed=0, input_scale=scale, batch=2), p)


@pytest.mark.parametrize("dtype,d,H,dff,L,batch", [
    ("bf16", 512, 8, 1024, 37, 3),    # 111 rows: one ragged 128-row block
    ("f16", 384, 6, 768, 50, 5),      # 192-wide N tiles, two per row
    ("bf16", 768, 12, 1536, 130, 2),  # three 256-wide N tiles per row
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_layered_rows_over_several_n_tiles(dtype, d, H, dff, L, batch, scale):
    """LayerNorm GEMMs whose rows span several N tiles (the scratch-row
    epilogue), with ragged row blocks."""
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=dff, n_layers=2)
    _check(make_inputs(s, seed=4, input_scale=scale), "layered")


@pytest.mark.parametrize("dtype,d,H,L,batch", [
    ("f16", 64, 8, 40, 3),     # head_dim 8: four heads per 32-column chunk
    ("bf16", 64, 16, 33, 2),   # head_dim 4
    ("f16", 64, 32, 17, 2),    # head_dim 2
    ("bf16", 128, 4, 70, 2),   # head_dim 32: one chunk per head
])
@pytest.mark.parametrize("scale", [1.0, 1e3])
def test_layered_qkv_head_widths(dtype, d, H, L, batch, scale):
    """The head-major QKV epilogue for every head width it handles."""
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=2 * d, n_layers=2)
    _check(make_inputs(s, seed=6, input_scale=scale), "layered")


@pytest.mark.parametrize("scale", INPUT_SCALES)
def test_long_d64_reduced_length(scale):
    # Same layer as the 100k-token workload, 3000 tokens (ragged tail) so the
    # whole output is checked, valid_len spanning the same 90-100% range.
    s = SHAPES["long_d64_L100k_B8"].with_(batch=2, seq_len=3000, vl_lo=2700, vl_hi=3000)
    for p in _paths_for(s):
        _check(make_inputs(s, seed=0, input_scale=scale), p)


# ----------------------------------------------------- full size, sampled
def _sampled_sequences(shape_name, n_sample, scale=1.0, seed=0):
    s = SHAPES[shape_name]
    inp = make_inputs(s, seed=seed, input_scale=scale)
    got = _run(inp)
    idx = np.sort(np.random.default_rng(123).choice(s.batch, size=n_sample, replace=False))
    ref = oracle.encoder_forward(inp.x[idx], inp.valid_len[idx], inp.layers, s.n_heads)
    ok, util, where = gate(got[idx], ref)
    assert ok, f"{shape_name}: envelope {util:.3f} at {where}"
    # Row 0 of every sequence has a closed form (it sees only itself).
    r0 = oracle.first_row_closed_form(inp.x[:, 0], inp.layers)
    ok0, util0, where0 = gate(got[:, 0], r0)
    assert ok0, f"{shape_name} row 0: envelope {util0:.3f} at {where0}"
    return max(util, util0)


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_short_d128_full_size_sampled(scale):
    _sampled_sequences("short_d128_L64_B4096", 48, scale=scale)


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_wide_d1024_full_size_sampled(scale):
    _sampled_sequences("wide_d1024_L1024_B32", 4, scale=scale)


@pytest.fixture(scope="module")
def oracle_pool():
    import oracle_workers
    pool = oracle_workers.make_pool()
    yield pool
    pool.close()
    pool.join()


def _gate_rows(L, vl, n, rng):
    """n increasing query positions of a sequence: a seeded uniform sample
    that always holds rows 0, 1, vl-2, vl-1, vl (when vl < L) and L-1."""
    must = {0, 1, vl - 2, vl - 1, L - 1} | ({vl} if vl < L else set())
    rest = np.setdiff1d(np.arange(L), np.array(sorted(must)))
    extra = rng.choice(rest, size=n - len(must), replace=False)
    return np.sort(np.concatenate([np.array(sorted(must)), extra]))


@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
@pytest.mark.parametrize("layer", [0, 1])
def test_long_d64_full_length_sampled_rows(layer, scale, oracle_pool):
    """Each layer of the 100k-token workload at full size (8 sequences of
    100,000 tokens) as a one-layer encoder on the seeded input: every element
    of 4096 seeded query rows per sequence against the oracle, which
    evaluates just those rows (keys and values from all 100,000 positions).
    The sample reaches the longest key ranges, the padding boundary and the
    padded rows past it."""
    import dataclasses
    s = SHAPES["long_d64_L100k_B8"]
    inp = make_inputs(s, seed=0, input_scale=scale)
    p = inp.layers[layer]
    one = dataclasses.replace(inp, shape=s.with_(n_layers=1), layers=[p])
    got = _run(one)
    assert got.shape == (s.batch, s.seq_len, s.d_model)
    rng = np.random.default_rng(1000 + 10 * layer + INPUT_SCALES.index(scale))
    rows = [_gate_rows(s.seq_len, int(inp.valid_len[b]), 4096, rng) for b in range(s.batch)]
    jobs = [(inp.x[b:b + 1], inp.valid_len[b:b + 1], p, s.n_heads, rows[b][None])
            for b in range(s.batch)]
    import oracle_workers
    refs = oracle_pool.map(oracle_workers.layer_rows, jobs)
    worst = 0.0
    for b in range(s.batch):
        ok, util, where = gate(got[b, rows[b]], refs[b][0])
        assert ok, f"layer {layer} scale {scale} sequence {b}: envelope {util:.3f} at " \
                   f"row {rows[b][where[0]]} col {where[1]}"
        worst = max(worst, util)
    assert np.all(np.isfinite(got))


def test_long_d64_full_size_prefix_and_first_row():
    s = SHAPES["long_d64_L100k_B8"]
    inp = make_inputs(s, seed=0)
    got = _run(inp)
    P = 2048  # every valid_len >= 90000 > P, so rows < P see only tokens < P
    ref = oracle.encoder_forward(inp.x[:, :P], inp.valid_len * 0 + P, inp.layers, s.n_heads)
    ok, util, where = gate(got[:, :P], ref)
    assert ok, f"prefix: envelope {util:.3f} at {where}"
    r0 = oracle.first_row_closed_form(inp.x[:, 0], inp.layers)
    ok0, util0, where0 = gate(got[:, 0], r0)
    assert ok0
    assert np.all(np.isfinite(got))


# ------------------------------------------------------------- edge cases
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("L,vl_lo,vl_hi", [(1, 1, 1), (37, 1, 37), (129, 1, 3), (130, 129, 130)])
def test_edge_lengths(dtype, L, vl_lo, vl_hi):
    s = tiny_shape(dtype=dtype, batch=3, seq_len=L, vl_lo=vl_lo, vl_hi=vl_hi,
                   d_model=64, n_heads=4, d_ff=256)
    for p in _paths_for(s):
        _check(make_inputs(s, seed=5, input_scale=1.0), p)


@pytest.mark.parametrize("dh", [16, 32, 64, 128])
def test_head_dims(dh):
    s = tiny_shape(dtype="f16", batch=2, seq_len=70, vl_lo=5, vl_hi=70,
                   d_model=dh * 2, n_heads=2, d_ff=4 * dh * 2)
    for p in _paths_for(s):
        _check(make_inputs(s, seed=6, input_scale=1.0), p)


# ------------------------------------------------------- GPU invariances
def test_causal_and_padding_invariance_bitwise():
    s = SHAPES["short_d128_L64_B4096"].with_(batch=8)
    inp = make_inputs(s, seed=1)
    base = _run(inp)
    x2 = inp.x.copy()
    t = 20
    x2[:, t + 1:] = -x2[:, t + 1:]
    inp2 = make_inputs(s, seed=1)
    inp2.x = x2
    out = _run(inp2)
    assert np.array_equal(out[:, :t + 1], base[:, :t + 1])
    # A padded position p changes only row p.
    b = 0
    vl = int(inp.valid_len[b])
    if vl < s.seq_len:
        x3 = inp.x.copy()
        x3[b, s.seq_len - 1] = -x3[b, s.seq_len - 1]
        inp3 = make_inputs(s, seed=1)
        inp3.x = x3
        out3 = _run(inp3)
        changed = np.any(out3 != base, axis=-1)
        assert changed[b, s.seq_len - 1] and changed.sum() == 1


@pytest.mark.parametrize("shape_name,batch", [("short_d128_L64_B4096", 9), ("wide_d1024_L1024_B32", 3),
                                              ("batch1_d256_L512", 1), ("tiny_d32_L32", 4)])
def test_layer_by_layer(shape_name, batch):
    """Each layer alone: a one-layer encoder built from layer k's weights,
    fed the oracle's layer k-1 output rounded to the I/O dtype, against the
    oracle's one-layer result on that same input."""
    import dataclasses
    from transformer_encoder_layer_gb300.inputs import round_to_dtype
    s = SHAPES[shape_name]
    L = min(s.seq_len, 256)
    s = s.with_(seq_len=L, vl_lo=min(s.vl_lo, L), vl_hi=L)
    inp = make_inputs(s, seed=3, batch=batch)
    h = inp.x
    for k, p in enumerate(inp.layers):
        one = dataclasses.replace(inp, shape=inp.shape.with_(n_layers=1), x=h, layers=[p])
        got = _run(one)
        ref = oracle.encoder_forward(h, inp.valid_len, [p], s.n_heads)
        ok, util, idx = gate(got, ref)
        assert ok, f"{shape_name} layer {k}: envelope {util:.3f} at {idx}"
        h = round_to_dtype(ref, s.dtype)


@pytest.mark.parametrize("shape_name", ["short_d128_L64_B4096", "wide_d1024_L1024_B32"])
def test_batch_permutation_permutes_outputs(shape_name):
    """Sequences are independent: permuting the batch permutes the output rows
    bit for bit."""
    s = SHAPES[shape_name]
    batch = 6 if shape_name.startswith("short") else 3
    inp = make_inputs(s, seed=5, batch=batch)
    base = _run(inp)
    perm = np.random.default_rng(7).permutation(batch)
    inp2 = make_inputs(s, seed=5, batch=batch)
    inp2.x = inp.x[perm].copy()
    inp2.valid_len = inp.valid_len[perm].copy()
    out = _run(inp2)
    assert np.array_equal(out, base[perm])


def test_argument_errors_with_a_handle():
    """Host-side checks on a live handle return a status before any launch."""
    import ctypes
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype="f16", batch=2, seq_len=40, vl_lo=1, vl_hi=40, d_model=64, n_heads=4,
                   d_ff=256)
    inp = make_inputs(s, seed=0)
    enc = binding.Encoder(inp.layers, 64, 4, 256, "f16")
    enc.set_path("layered")
    lib, h = enc.lib, enc.handle
    x = torch.from_numpy(to_storage(inp.x, "f16")).cuda()
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    out = torch.empty_like(x)
    need = enc.workspace_size(2, 40)
    assert need > 0
    ws = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    fwd = lambda xp, B, op, wsp, nb: lib.tl_encoder_forward(h, xp, B, 40, vl.data_ptr(), op, wsp, nb, None)
    assert fwd(x.data_ptr(), 2, out.data_ptr(), ws.data_ptr(), need - 1) == 5      # workspace too small
    assert fwd(x.data_ptr(), 2, x.data_ptr(), ws.data_ptr(), need) == 1           # out overlaps x
    assert fwd(x.data_ptr() + 2, 2, out.data_ptr(), ws.data_ptr(), need) == 1     # x not 16-byte aligned
    assert fwd(x.data_ptr(), 2, out.data_ptr(), ws.data_ptr() + 16, need) == 1    # workspace misaligned
    assert fwd(x.data_ptr(), 0, out.data_ptr(), ws.data_ptr(), need) == 1         # B = 0
    assert fwd(x.data_ptr(), 2, out.data_ptr(), ws.data_ptr(), need) == 0
    assert lib.tl_encoder_set_path(h, 99) == 1
    # more tokens than the kernels' int row counts allow: refused, nothing allocated
    with pytest.raises(binding.TLError):
        enc.plan(1 << 20, 1 << 11)
    with pytest.raises(binding.TLError):
        enc.workspace_size(1 << 20, 1 << 11)
    # a forced path that is not built for the shape: the megakernel needs d = 128
    enc.set_path("mega")
    with pytest.raises(binding.TLError):
        enc.plan(2, 40)
    assert fwd(x.data_ptr(), 2, out.data_ptr(), ws.data_ptr(), need) == 2
    enc.set_path("auto")
    # host-buffer forward: workspace below the reported size
    hn = enc.host_workspace_size(2, 40)
    xh, vh = x.cpu().pin_memory(), vl.cpu().pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    hws = torch.empty(hn, dtype=torch.uint8, device="cuda")
    assert lib.tl_encoder_forward_host(h, xh.data_ptr(), 2, 40, vh.data_ptr(), oh.data_ptr(),
                                       hws.data_ptr(), hn - 1, None) == 5
    assert lib.tl_encoder_forward_host(h, xh.data_ptr(), 2, 40, vh.data_ptr(), oh.data_ptr(),
                                       hws.data_ptr(), hn, None) == 0
    torch.cuda.synchronize()
    assert enc.get_status() == 0
    enc.close()


@pytest.mark.parametrize("path,dtype,d,H,dff,L", [
    ("simt", "f16", 32, 2, 128, 16),
    ("layered", "f16", 64, 4, 256, 16),     # tcgen05 attention, head_dim 16
    ("layered", "bf16", 128, 2, 256, 40),   # tcgen05 attention, head_dim 64
    ("mega", "f16", 128, 4, 512, 64),       # tensor-core megakernel
    ("mega", "f32", 32, 2, 128, 32),        # CUDA-core megakernel
    ("dag", "f32", 64, 2, 256, 40),         # task graph
])
def test_bad_valid_len_is_reported_and_clamped(path, dtype, d, H, dff, L):
    """Every path clamps a valid_len outside [1, L] and reports it through
    the status word; the result equals a run with the clamped lengths."""
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype=dtype, batch=2, seq_len=L, vl_lo=L, vl_hi=L, d_model=d, n_heads=H,
                   d_ff=dff)
    inp = make_inputs(s, seed=0)
    enc = binding.Encoder(inp.layers, d, H, dff, dtype)
    enc.set_path(path)
    assert enc.plan(2, L) == path
    st = to_storage(inp.x, dtype)
    x = (torch.from_numpy(st.view(np.int16)).view(torch.bfloat16) if dtype == "bf16"
         else torch.from_numpy(st)).cuda()
    vl = torch.tensor([0, L + 1], dtype=torch.int32, device="cuda")
    out = enc.forward(x, vl, check=False)
    assert enc.get_status() == 6  # TL_ERR_BAD_VALID_LEN
    assert enc.get_status() == 0  # cleared by the read
    # Clamped to [1, L]: equal to running with valid_len = [1, L].
    ref = enc.forward(x, torch.tensor([1, L], dtype=torch.int32, device="cuda"))
    assert torch.equal(out.view(torch.uint8) if dtype == "bf16" else out,
                       ref.view(torch.uint8) if dtype == "bf16" else ref)
    assert enc.get_status() == 0
    enc.close()


def test_forward_host_matches_device_forward():
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["short_d128_L64_B4096"].with_(batch=16)
    inp = make_inputs(s, seed=2)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    xh = torch.from_numpy(to_storage(inp.x, "f16")).pin_memory()
    vh = torch.from_numpy(inp.valid_len.astype(np.int32)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    enc.forward_host(xh, vh, oh)
    od = enc.forward(xh.cuda(), vh.cuda()).cpu()
    assert torch.equal(oh, od)
    enc.close()


@pytest.mark.parametrize("path,dtype,d,H,dff,L,batch", [
    ("mega", "f16", 128, 4, 512, 64, 37),
    ("mega", "f32", 32, 2, 128, 32, 9),
    ("layered", "bf16", 128, 2, 256, 96, 7),
    ("dag", "f32", 64, 2, 256, 40, 5),
    ("simt", "f32", 64, 4, 128, 33, 6),
])
@pytest.mark.parametrize("chunks", [0, 1, 2, 3, 64])
@pytest.mark.parametrize("pinned", [True, False])
def test_forward_host_slices_are_bit_identical(path, dtype, d, H, dff, L, batch, chunks, pinned):
    """The host-buffer forward cut into batch slices on two streams gives the
    device forward's bits, pinned or pageable, with a ragged last slice."""
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=dff, n_layers=2)
    inp = make_inputs(s, seed=11)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    enc.set_path(path)
    assert enc.plan(batch, L) == path
    enc.set_host_chunks(chunks)
    xh = torch.from_numpy(to_storage(inp.x, dtype))
    vh = torch.from_numpy(inp.valid_len.astype(np.int32))
    oh = torch.empty_like(xh)
    oh.view(torch.uint8).fill_(0xFF)  # NaN in every dtype: each element must be written
    if pinned:
        xh, vh, oh = xh.pin_memory(), vh.pin_memory(), oh.pin_memory()
    enc.forward_host(xh, vh, oh)
    od = enc.forward(xh.cuda(), vh.cuda()).cpu()
    assert torch.equal(oh.view(torch.uint8), od.view(torch.uint8))
    assert enc.get_status() == 0
    enc.close()


@pytest.mark.parametrize("path,dtype,d,H,dff,L,batch", [
    ("mega", "f16", 128, 4, 512, 64, 6),
    ("mega", "f32", 32, 2, 128, 32, 4),
    ("layered", "bf16", 512, 8, 1024, 70, 2),   # d > 256: GEMM + LayerNorm apply pass
    ("layered", "f16", 64, 4, 256, 200, 2),     # head_dim 16 attention
    ("dag", "f32", 64, 2, 256, 40, 2),          # counter memset + one launch
    ("simt", "f32", 64, 4, 128, 33, 3),
])
def test_forward_captures_in_a_cuda_graph(path, dtype, d, H, dff, L, batch):
    """forward() neither allocates nor synchronises, so it records into a CUDA
    graph as it is; the replay gives the eager forward's bits."""
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=dff, n_layers=2)
    inp = make_inputs(s, seed=12)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    enc.set_path(path)
    assert enc.plan(batch, L) == path
    x = torch.from_numpy(to_storage(inp.x, dtype)).cuda()
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    ws = torch.empty(max(enc.workspace_size(batch, L), 256), dtype=torch.uint8, device="cuda")
    ref = enc.forward(x, vl, workspace=ws)  # eager, also sets the kernels' attributes
    out = torch.empty_like(x)
    side = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side, capture_error_mode="thread_local"):
        enc.forward(x, vl, out=out, workspace=ws, stream=side, check=False)
    out.view(torch.uint8).fill_(0xFF)
    torch.cuda.synchronize()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), ref.view(torch.uint8))
    assert enc.get_status() == 0
    enc.close()


def test_forward_host_automatic_slices_with_ramp():
    """A batch large enough for the automatic plan to pipeline (4+ slices of
    8 MiB, with quarter slices at both ends) still gives the device forward's
    bits."""
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["short_d128_L64_B4096"].with_(batch=2048)
    inp = make_inputs(s, seed=8)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    xh = torch.from_numpy(to_storage(inp.x, "f16")).pin_memory()
    vh = torch.from_numpy(inp.valid_len.astype(np.int32)).pin_memory()
    oh = torch.empty_like(xh).pin_memory()
    oh.view(torch.uint8).fill_(0xFF)
    enc.forward_host(xh, vh, oh)
    od = enc.forward(xh.cuda(), vh.cuda()).cpu()
    assert torch.equal(oh.view(torch.uint8), od.view(torch.uint8))
    enc.close()


def test_host_chunks_setting_is_checked():
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["short_d128_L64_B4096"].with_(batch=4)
    inp = make_inputs(s, seed=2)
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    for bad in (-1, 65):
        with pytest.raises(RuntimeError):
            enc.set_host_chunks(bad)
    enc.set_host_chunks(1)
    one = enc.host_workspace_size(4, 64)
    enc.set_host_chunks(4)
    assert enc.host_workspace_size(4, 64) >= one
    enc.close()


# ------------------------------------------------- sequence-resident path
@pytest.mark.parametrize("dtype,L,dff,n_layers,batch", [
    ("f16", 64, 512, 4, 37),     # the d128 workload's layer, ragged last tile
    ("bf16", 64, 512, 2, 6),
    ("f16", 64, 256, 2, 9),
    ("f16", 64, 128, 1, 3),      # d_ff = d
    ("bf16", 64, 384, 3, 2),
    ("bf16", 64, 512, 2, 5),
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_mega_shapes(dtype, L, dff, n_layers, batch, scale):
    from transformer_encoder_layer_gb300 import binding
    s = tiny_shape(dtype=dtype, batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=128,
                   n_heads=4, d_ff=dff, n_layers=n_layers)
    inp = make_inputs(s, seed=3, input_scale=scale)
    assert "mega" in _paths_for(s)
    _check(inp, "mega")


def test_mega_matches_layered_closely():
    # Two tensor-core paths over the same function: the layered path keeps
    # every (hi, lo) operand, the fp16 megakernel rounds P and the FFN hidden
    # to one 16-bit value; both pass the gate against the oracle, and they
    # are within twice the gate's absolute bound of each other.
    s = SHAPES["short_d128_L64_B4096"].with_(batch=64)
    inp = make_inputs(s, seed=4)
    a = _run(inp, "mega")
    b = _run(inp, "layered")
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, s.n_heads)
    assert gate(a, ref)[0] and gate(b, ref)[0]
    assert np.max(np.abs(a - b)) < 4e-3


# ------------------------------------------------------ task-graph path
@pytest.mark.parametrize("d,H,dff,n_layers,batch,L,vl_lo", [
    (256, 8, 1024, 2, 1, 512, 384),   # the batch-1 d256 workload's layer
    (32, 2, 128, 2, 4, 32, 16),       # the d32 workload: two sequences per row block
    (64, 1, 256, 3, 3, 100, 1),       # head_dim 64, ragged row blocks
    (80, 5, 320, 2, 2, 70, 5),        # ragged column tiles and K chunks
    (1024, 16, 512, 1, 1, 96, 60),    # split-K out-projection (4 chunks)
    (128, 8, 512, 8, 2, 33, 1),       # eight layers
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_dag_shapes(d, H, dff, n_layers, batch, L, vl_lo, scale):
    s = tiny_shape(dtype="f32", batch=batch, seq_len=L, vl_lo=vl_lo, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=dff, n_layers=n_layers)
    assert "dag" in _paths_for(s)
    _check(make_inputs(s, seed=7, input_scale=scale), "dag")


def test_auto_dispatch_for_fp32():
    from transformer_encoder_layer_gb300 import binding
    for name, want in (("batch1_d256_L512", "dag"), ("tiny_d32_L32", "mega")):
        s = SHAPES[name]
        inp = make_inputs(s.with_(batch=1, seq_len=1, vl_lo=1, vl_hi=1))
        enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
        assert enc.plan(s.batch, s.seq_len) == want
        assert enc.plan(64, 1024) == "simt"  # 65536 tokens of long sequences: layer by layer
        enc.close()


# ------------------------------------- sequence-resident path, CUDA cores
@pytest.mark.parametrize("d,H,dff,n_layers,batch,L", [
    (32, 2, 128, 2, 4, 32),     # the d32 workload's layer
    (64, 2, 256, 2, 3, 64),     # head_dim 32, the largest supported sizes
    (64, 4, 256, 3, 5, 17),     # head_dim 16, ragged length
    (32, 1, 64, 1, 2, 1),       # one token
    (48, 3, 192, 2, 3, 40),     # head_dim 16, d not a power of two
])
@pytest.mark.parametrize("scale", [1e-3, 1.0, 1e3])
def test_mega_simt_shapes(d, H, dff, n_layers, batch, L, scale):
    s = tiny_shape(dtype="f32", batch=batch, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                   n_heads=H, d_ff=dff, n_layers=n_layers)
    assert "mega" in _paths_for(s)
    _check(make_inputs(s, seed=8, input_scale=scale), "mega")


def test_mega_simt_matches_dag_and_simt():
    s = SHAPES["tiny_d32_L32"]
    inp = make_inputs(s, seed=12)
    a = _run(inp, "mega")
    assert np.array_equal(a, _run(inp, "mega"))  # deterministic
    for other in ("dag", "simt"):
        assert np.max(np.abs(a - _run(inp, other))) < 1e-4


def test_dag_deterministic_and_matches_simt():
    s = SHAPES["batch1_d256_L512"]
    inp = make_inputs(s, seed=11)
    a = _run(inp, "dag")
    b = _run(inp, "dag")
    assert np.array_equal(a, b)  # no atomics in the arithmetic
    c = _run(inp, "simt")
    assert np.max(np.abs(a - c)) < 1e-3


def test_dag_stalled_dependency_times_out(monkeypatch):
    # The first task waits on a counter target no task reaches: the bounded
    # wait gives up, every CTA drains the queue, and the status word reports
    # the timeout.  The context stays usable for the next forward.
    from transformer_encoder_layer_gb300 import binding
    s = SHAPES["batch1_d256_L512"]
    inp = make_inputs(s, seed=0)
    x = torch.from_numpy(to_storage(inp.x, "f32")).cuda()
    vl = torch.from_numpy(inp.valid_len.astype(np.int32)).cuda()
    monkeypatch.setenv("TL_DAG_INJECT_STALL", "1")
    enc = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    monkeypatch.delenv("TL_DAG_INJECT_STALL")
    assert enc.plan(1, s.seq_len) == "dag"
    enc.forward(x, vl, check=False)
    torch.cuda.synchronize()
    assert enc.get_status() == 7  # TL_ERR_DEVICE_TIMEOUT
    enc.close()
    good = binding.Encoder(inp.layers, s.d_model, s.n_heads, s.d_ff, s.dtype)
    out = good.forward(x, vl)
    ref = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, s.n_heads)
    ok, util, where = gate(out.cpu().numpy().astype(np.float64), ref)
    assert ok, f"after timeout: envelope {util:.3f} at {where}"
    good.close()
