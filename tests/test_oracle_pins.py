"""Pins for the fp64 oracle: checks against things other than itself.

Each test fixes the oracle to something the pages or the mathematics fix:
an independent library implementation of the same layer (PyTorch's
``TransformerEncoderLayer`` in float64), closed forms, invariants of the
causal and padding masks, LayerNorm's moments, and a scalar brute force.  The
set is chosen so that a dropped term, a wrong sign or index, or a transposed
operand anywhere in the oracle fails at least one of them (see
``test_planted_mistakes_are_caught``).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import encoder_fp64 as ofp
from transformer_encoder_layer_gb300.inputs import make_inputs, tiny_shape

SCALES = (1e-3, 1.0, 1e3)


def _inputs(seed=0, scale=1.0, **kw):
    return make_inputs(tiny_shape(**kw), seed=seed, input_scale=scale)


# ---------------------------------------------------------------- K8 library
def torch_stack(inp):
    """The same stack through torch.nn.TransformerEncoderLayer (float64, CPU),
    post-LN, exact GELU, no dropout, causal src_mask + key-padding mask."""
    s = inp.shape
    x = torch.tensor(inp.x, dtype=torch.float64)
    L = s.seq_len
    causal = torch.triu(torch.ones(L, L, dtype=torch.bool), diagonal=1)
    kpm = torch.arange(L)[None, :] >= torch.tensor(inp.valid_len)[:, None]
    for p in inp.layers:
        layer = torch.nn.TransformerEncoderLayer(
            d_model=s.d_model, nhead=s.n_heads, dim_feedforward=s.d_ff, dropout=0.0,
            activation="gelu", batch_first=True, norm_first=False, dtype=torch.float64)
        with torch.no_grad():
            T = lambda a: torch.tensor(a, dtype=torch.float64)  # noqa: E731
            layer.self_attn.in_proj_weight.copy_(T(p["w_qkv"]))
            layer.self_attn.in_proj_bias.copy_(T(p["b_qkv"]))
            layer.self_attn.out_proj.weight.copy_(T(p["w_o"]))
            layer.self_attn.out_proj.bias.copy_(T(p["b_o"]))
            layer.norm1.weight.copy_(T(p["ln1_g"]))
            layer.norm1.bias.copy_(T(p["ln1_b"]))
            layer.linear1.weight.copy_(T(p["w_1"]))
            layer.linear1.bias.copy_(T(p["b_1"]))
            layer.linear2.weight.copy_(T(p["w_2"]))
            layer.linear2.bias.copy_(T(p["b_2"]))
            layer.norm2.weight.copy_(T(p["ln2_g"]))
            layer.norm2.bias.copy_(T(p["ln2_b"]))
        layer.train()  # dropout is 0; training mode keeps PyTorch off its fused fast path
        with torch.no_grad():
            x = layer(x, src_mask=causal, src_key_padding_mask=kpm)
    return x.numpy()


@pytest.mark.parametrize("scale", SCALES)
@pytest.mark.parametrize("seed", [0, 1])
def test_k8_matches_torch_transformer_encoder_layer(seed, scale):
    inp = _inputs(seed=seed, scale=scale, batch=3, seq_len=11, d_model=16, n_heads=4,
                  d_ff=64, n_layers=2, vl_lo=1, vl_hi=11)
    ref = torch_stack(inp)
    got = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, inp.shape.n_heads)
    # Every row, padded rows included: PyTorch's combined mask gives padded
    # query rows the keys [0, valid_len), the same reading as the oracle.
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-9)


# ------------------------------------------------------------ K7 brute force
def brute_force_stack(inp):
    """Scalar loops over every index, math.erf/math.exp, no numpy algebra."""
    s = inp.shape
    B, L, d, H = s.batch, s.seq_len, s.d_model, s.n_heads
    dh = d // H
    X = [[[float(inp.x[b, i, c]) for c in range(d)] for i in range(L)] for b in range(B)]

    def linear(row, W, bias):
        return [sum(W[o][c] * row[c] for c in range(len(row))) + bias[o] for o in range(len(W))]

    def ln(row, g, be):
        n = len(row)
        mu = sum(row) / n
        var = sum((r - mu) ** 2 for r in row) / n
        return [(row[c] - mu) / math.sqrt(var + 1e-5) * g[c] + be[c] for c in range(n)]

    for p in inp.layers:
        P = {k: v.tolist() for k, v in p.items()}
        new = []
        for b in range(B):
            vl = int(inp.valid_len[b])
            qkv = [linear(X[b][i], P["w_qkv"], P["b_qkv"]) for i in range(L)]
            seq_out = []
            for i in range(L):
                ctx = []
                for h in range(H):
                    qi = qkv[i][h * dh:(h + 1) * dh]
                    keys = [j for j in range(L) if j <= i and j < vl]
                    sc = []
                    for j in keys:
                        kj = qkv[j][d + h * dh:d + (h + 1) * dh]
                        sc.append(sum(qi[t] * kj[t] for t in range(dh)) / math.sqrt(dh))
                    mx = max(sc)
                    ex = [math.exp(z - mx) for z in sc]
                    tot = sum(ex)
                    for t in range(dh):
                        ctx.append(sum(ex[n] / tot * qkv[keys[n]][2 * d + h * dh + t]
                                       for n in range(len(keys))))
                a = linear(ctx, P["w_o"], P["b_o"])
                y = ln([X[b][i][c] + a[c] for c in range(d)], P["ln1_g"], P["ln1_b"])
                u = linear(y, P["w_1"], P["b_1"])
                f = [0.5 * z * (1 + math.erf(z / math.sqrt(2))) for z in u]
                g = linear(f, P["w_2"], P["b_2"])
                seq_out.append(ln([y[c] + g[c] for c in range(d)], P["ln2_g"], P["ln2_b"]))
            new.append(seq_out)
        X = new
    return np.array(X)


@pytest.mark.parametrize("scale", SCALES)
def test_k7_brute_force_tiny(scale):
    inp = _inputs(seed=3, scale=scale, batch=3, seq_len=7, d_model=8, n_heads=2,
                  d_ff=16, n_layers=2, vl_lo=1, vl_hi=7)
    got = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2)
    ref = brute_force_stack(inp)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-11)


def test_k7_brute_force_random_shapes():
    """K7 over randomly drawn tiny shapes: batch, length, heads, widths,
    layer count, valid lengths (including 1 and L), seed and input scale."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")

    @hyp.settings(max_examples=30, deadline=None, derandomize=True)
    @hyp.given(batch=st.integers(1, 3), seq_len=st.integers(1, 8), heads=st.sampled_from([1, 2, 4]),
               dh=st.sampled_from([1, 2, 3]), d_ff=st.sampled_from([4, 8, 12]),
               n_layers=st.integers(1, 2), seed=st.integers(0, 1000),
               scale=st.sampled_from(list(SCALES)), vl_lo=st.integers(1, 8))
    def check(batch, seq_len, heads, dh, d_ff, n_layers, seed, scale, vl_lo):
        vl_lo = min(vl_lo, seq_len)
        inp = _inputs(seed=seed, scale=scale, batch=batch, seq_len=seq_len, d_model=heads * dh,
                      n_heads=heads, d_ff=d_ff, n_layers=n_layers, vl_lo=vl_lo, vl_hi=seq_len)
        got = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, heads)
        np.testing.assert_allclose(got, brute_force_stack(inp), rtol=1e-10, atol=1e-10)

    check()


# -------------------------------------------------------- K2 / K3 invariances
@pytest.mark.parametrize("scale", SCALES)
def test_k2_causal_invariance(scale):
    inp = _inputs(seed=4, scale=scale, batch=2, seq_len=12, vl_lo=12, vl_hi=12)
    base = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2)
    rng = np.random.default_rng(9)
    for t in (0, 5, 10):
        x2 = inp.x.copy()
        x2[:, t + 1:] += rng.standard_normal(x2[:, t + 1:].shape) * scale
        out = oracle.encoder_forward(x2, inp.valid_len, inp.layers, 2)
        assert np.array_equal(out[:, :t + 1], base[:, :t + 1])
        assert not np.allclose(out[:, t + 1:], base[:, t + 1:])


@pytest.mark.parametrize("scale", SCALES)
def test_k3_padding_invariance(scale):
    inp = _inputs(seed=5, scale=scale, batch=3, seq_len=12, vl_lo=3, vl_hi=9)
    base = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2)
    rng = np.random.default_rng(1)
    for b in range(3):
        vl = int(inp.valid_len[b])
        for p in range(vl, 12):
            x2 = inp.x.copy()
            x2[b, p] += rng.standard_normal(x2.shape[-1]) * scale
            out = oracle.encoder_forward(x2, inp.valid_len, inp.layers, 2)
            changed = np.any(out != base, axis=-1)
            expect = np.zeros_like(changed)
            expect[b, p] = True
            assert np.array_equal(changed, expect), (b, p)


# ---------------------------------------------------------- K4 closed form
@pytest.mark.parametrize("scale", SCALES)
def test_k4_first_row_closed_form(scale):
    inp = _inputs(seed=6, scale=scale, batch=3, seq_len=10, vl_lo=1, vl_hi=10)
    out = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2)
    ref = oracle.first_row_closed_form(inp.x[:, 0], inp.layers)
    np.testing.assert_allclose(out[:, 0], ref, rtol=0, atol=1e-12)


def test_k4_length_one_sequence():
    inp = _inputs(seed=7, batch=4, seq_len=1, vl_lo=1, vl_hi=1)
    out = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2)
    ref = oracle.first_row_closed_form(inp.x[:, 0], inp.layers)
    np.testing.assert_allclose(out[:, 0], ref, rtol=0, atol=1e-12)


# ------------------------------------------------------------- K5 LayerNorm
@pytest.mark.parametrize("scale", [1e-4, 1e-2, 1.0, 1e3])
def test_k5_layernorm_moments(scale):
    rng = np.random.default_rng(2)
    r = rng.standard_normal((50, 64)) * scale + rng.standard_normal((50, 1)) * scale
    y = oracle.layer_norm(r, np.ones(64), np.zeros(64))
    var = r.var(axis=-1)
    np.testing.assert_allclose(y.mean(axis=-1), 0, atol=1e-12)
    np.testing.assert_allclose(y.var(axis=-1), var / (var + 1e-5), rtol=1e-12)
    g, b = rng.standard_normal(64), rng.standard_normal(64)
    y2 = oracle.layer_norm(r, g, b)
    np.testing.assert_allclose(y2, y * g + b, rtol=1e-12, atol=1e-12)


def test_k5_gelu_special_values():
    # gelu(0) = 0; gelu(u) -> u for large u, -> 0 for very negative u;
    # gelu(u) - gelu(-u) = u (erf is odd).
    u = np.linspace(-8, 8, 161)
    g = oracle.gelu_erf(u)
    assert oracle.gelu_erf(np.array([0.0]))[0] == 0.0
    np.testing.assert_allclose(g - oracle.gelu_erf(-u), u, atol=1e-14)
    assert abs(oracle.gelu_erf(np.array([30.0]))[0] - 30.0) < 1e-12
    assert abs(oracle.gelu_erf(np.array([-30.0]))[0]) < 1e-12
    # gelu(1) = 0.5 (1 + erf(1/sqrt 2)) = Phi(1) = 0.8413447460685429...
    assert abs(oracle.gelu_erf(np.array([1.0]))[0] - 0.8413447460685429) < 1e-15


# -------------------------------------------------- K6 uniform attention
def test_k6_uniform_attention_prefix_means():
    inp = _inputs(seed=8, batch=3, seq_len=10, vl_lo=2, vl_hi=10)
    p = dict(inp.layers[0])
    d = inp.shape.d_model
    p["w_qkv"] = p["w_qkv"].copy()
    p["b_qkv"] = p["b_qkv"].copy()
    p["w_qkv"][:d] = 0.0
    p["b_qkv"][:d] = 0.0
    q, k, v = oracle.qkv_projection(inp.x, p["w_qkv"], p["b_qkv"], 2)
    assert np.all(q == 0)
    ctx = oracle.masked_attention(q, k, v, inp.valid_len)
    vm = oracle.merge_heads(v)
    for b in range(3):
        vl = int(inp.valid_len[b])
        for i in range(10):
            n = min(i + 1, vl)
            np.testing.assert_allclose(ctx[b, i], vm[b, :n].mean(axis=0), atol=1e-14)


# ------------------------------------------------ K1 rows sum to one
@pytest.mark.parametrize("scale", SCALES)
def test_k1_rows_sum_to_one(scale):
    inp = _inputs(seed=10, scale=scale, batch=2, seq_len=16, vl_lo=4, vl_hi=16)
    q, k, v = oracle.qkv_projection(inp.x, inp.layers[0]["w_qkv"], inp.layers[0]["b_qkv"], 2)
    # With v = 1 everywhere the output is sum_j p_j = 1 exactly up to rounding.
    ones = np.ones_like(v)
    ctx = oracle.masked_attention(q, k, ones, inp.valid_len, check=True)
    np.testing.assert_allclose(ctx, 1.0, atol=1e-12)


# ---------------------------------------------------- K9 head permutation
def test_k9_head_permutation():
    inp = _inputs(seed=11, batch=2, seq_len=8, d_model=16, n_heads=4, d_ff=32, vl_lo=3, vl_hi=8)
    d, H = 16, 4
    dh = d // H
    perm = [2, 0, 3, 1]
    cols = np.concatenate([np.arange(h * dh, (h + 1) * dh) for h in perm])
    layers = []
    for p in inp.layers:
        p2 = dict(p)
        rows = np.concatenate([cols, d + cols, 2 * d + cols])
        p2["w_qkv"] = p["w_qkv"][rows]
        p2["b_qkv"] = p["b_qkv"][rows]
        p2["w_o"] = p["w_o"][:, cols]
        layers.append(p2)
    a = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, H)
    b = oracle.encoder_forward(inp.x, inp.valid_len, layers, H)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_row_blocking_does_not_change_rows():
    inp = _inputs(seed=12, batch=2, seq_len=40, vl_lo=10, vl_hi=40)
    a = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2, row_block=7)
    b = oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 2, row_block=256)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", range(12))
def test_row_selection_matches_full_result(seed):
    """Evaluating only some query rows (the sampled gate of the 100k-token
    workload) gives those rows of the full evaluation.  The two runs group
    the same sums differently (BLAS picks its kernels by the number of rows),
    so they agree to rounding, 1e-13 of the output's scale, not bit for bit;
    a wrong row, key range or residual row would be off by O(1)."""
    rng = np.random.default_rng(100 + seed)
    B, L = int(rng.integers(1, 4)), int(rng.integers(2, 60))
    H = int(rng.choice([1, 2, 4]))
    d = H * int(rng.choice([1, 2, 4, 8]))
    scale = float(rng.choice(SCALES))
    inp = _inputs(seed=seed, scale=scale, batch=B, seq_len=L, vl_lo=1, vl_hi=L, d_model=d,
                  n_heads=H, d_ff=2 * d, n_layers=1)
    rb = int(rng.integers(1, 16))
    full = oracle.encoder_layer(inp.x, inp.valid_len, inp.layers[0], H, row_block=rb)
    n = int(rng.integers(min(L, 5), L + 1))  # rows per sequence
    rows = []
    for b in range(B):
        vl = int(inp.valid_len[b])
        # always the first and last rows and those around the padding boundary
        pick = {0, L - 1, max(vl - 2, 0), vl - 1, min(vl, L - 1)}
        for r in rng.permutation(L):
            if len(pick) >= n:
                break
            pick.add(int(r))
        rows.append(sorted(pick)[:n] if len(pick) > n else sorted(pick))
    rows = np.array(rows)
    sel = oracle.encoder_layer(inp.x, inp.valid_len, inp.layers[0], H, row_block=rb, rows=rows)
    ref = full[np.arange(B)[:, None], rows]
    assert sel.shape == (B, n, d)
    np.testing.assert_allclose(sel, ref, rtol=0, atol=1e-13 * np.max(np.abs(ref)))
    # every row: the selection of all positions is the full evaluation itself
    allr = np.broadcast_to(np.arange(L), (B, L))
    assert np.array_equal(
        oracle.encoder_layer(inp.x, inp.valid_len, inp.layers[0], H, row_block=rb, rows=allr), full)


def test_planted_mistakes_are_caught(monkeypatch):
    """Plant plausible mistakes in the oracle (on the CPU) and check that the
    library pin K8 rejects each of them."""
    inp = _inputs(seed=13, batch=3, seq_len=9, d_model=16, n_heads=4, d_ff=32,
                  vl_lo=3, vl_hi=7)
    ref = torch_stack(inp)

    def run():
        return oracle.encoder_forward(inp.x, inp.valid_len, inp.layers, 4)

    np.testing.assert_allclose(run(), ref, atol=1e-9)
    planted = {
        "no_sqrt_scale": lambda q, k, v, vl, **kw: orig_attn(q * math.sqrt(q.shape[-1]), k, v, vl, **kw),
        "k_v_swapped": lambda q, k, v, vl, **kw: orig_attn(q, v, k, vl, **kw),
    }
    orig_attn = ofp.masked_attention
    for name, fn in planted.items():
        monkeypatch.setattr(ofp, "masked_attention", fn)
        assert not np.allclose(run(), ref, atol=1e-6), name
        monkeypatch.setattr(ofp, "masked_attention", orig_attn)
    orig_allowed = ofp.allowed_keys
    for name, fn in {"no_causal": lambda i, vl: np.full(np.shape(i), vl),
                     "no_padding": lambda i, vl: np.asarray(i) + 1,
                     "off_by_one": lambda i, vl: np.minimum(np.asarray(i), vl) + (np.asarray(i) == 0)}.items():
        monkeypatch.setattr(ofp, "allowed_keys", fn)
        assert not np.allclose(run(), ref, atol=1e-6), name
        monkeypatch.setattr(ofp, "allowed_keys", orig_allowed)
    orig_ln = ofp.layer_norm
    monkeypatch.setattr(ofp, "layer_norm", lambda r, g, b, eps=1e-5: orig_ln(r, g, b, eps=1e-3))
    assert not np.allclose(run(), ref, atol=1e-6)
    monkeypatch.setattr(ofp, "layer_norm", orig_ln)
    monkeypatch.setattr(ofp, "gelu_erf", lambda u: 0.5 * u * (1 + np.tanh(0.7978845608 * (u + 0.044715 * u ** 3))))
    assert not np.allclose(run(), ref, atol=1e-6)
