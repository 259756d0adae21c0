"""fp64 CPU oracle for the forward pass of a masked post-LN encoder stack.

TEST INFRASTRUCTURE.  This module exists to check the CUDA path.  Only the
test suite, the smoke check and the CPU-baseline leg of the benchmark may
import it; the library never does, and it imports nothing from the library.

It is the plain definition of what the pages' kernels compute, written out in
float64 with numpy (matrix products and ``scipy.special.erf`` are the only
library primitives).  The layer, as the three pages describe the task
("Hyper-optimized megakernel-hybrid transformer inference", "KernelForge",
"Implement a GPU Kernel for a Transformer Layer"):

* fused QKV projection ("KernelForge", section "What we built"; the
  megakernel page, section "Hybrid", for the head-major split);
* multi-head attention under a causal mask combined with a right-padding key
  mask ("KernelForge", sections "What we built" and "Why it matters");
* output projection, residual add, LayerNorm ("KernelForge", "What we built":
  fused add + LayerNorm; the megakernel page, "Challenges", for PyTorch's
  LayerNorm as the convention);
* FFN with exact-erf GELU ("KernelForge", "How the LLM is used": a polynomial
  erf failed a tolerance measured against exact erf);
* second residual add and LayerNorm.  Post-LN order, no dropout.

Readings taken where the pages are silent: attention scale 1/sqrt(dh); LayerNorm eps 1e-5 with the biased variance and an
affine gamma/beta; every linear has a bias; W_qkv rows are Q, K, V blocks in
that order and head h owns rows h*dh .. (h+1)*dh-1 of each block; key j is
visible to query i iff j <= i and j < valid_len (so padded query rows attend to
[0, valid_len) and are part of the output); masked keys are excluded, not
added as a large negative number.

Arrays are float64.  Shapes: x [B, L, d]; valid_len int [B]; one dict per
layer with w_qkv [3d, d], b_qkv [3d], w_o [d, d], b_o [d], ln1_g/ln1_b [d],
w_1 [d_ff, d], b_1 [d_ff], w_2 [d, d_ff], b_2 [d], ln2_g/ln2_b [d]
(PyTorch's [out, in] weight layout).
"""
from __future__ import annotations

import math
from typing import Dict, List, Sequence

import numpy as np
from scipy.special import erf

LN_EPS = 1e-5


def split_heads(t: np.ndarray, n_heads: int) -> np.ndarray:
    """[B, L, d] -> [B, H, L, dh]: head h is columns h*dh .. (h+1)*dh-1."""
    B, L, d = t.shape
    dh = d // n_heads
    return t.reshape(B, L, n_heads, dh).transpose(0, 2, 1, 3)


def merge_heads(t: np.ndarray) -> np.ndarray:
    """[B, H, L, dh] -> [B, L, H*dh], heads concatenated in order."""
    B, H, L, dh = t.shape
    return t.transpose(0, 2, 1, 3).reshape(B, L, H * dh)


def qkv_projection(x: np.ndarray, w_qkv: np.ndarray, b_qkv: np.ndarray,
                   n_heads: int):
    """One fused projection qkv = x W_qkv^T + b_qkv, split into Q, K, V and
    then into heads (head-major [B, H, L, dh] each)."""
    d = x.shape[-1]
    qkv = x @ w_qkv.T + b_qkv
    q, k, v = qkv[..., :d], qkv[..., d:2 * d], qkv[..., 2 * d:]
    return split_heads(q, n_heads), split_heads(k, n_heads), split_heads(v, n_heads)


def allowed_keys(i, valid_len):
    """Number of keys visible to query row i (an int or an index array):
    keys j with j <= i (causal) and j < valid_len (right padding), i.e. the
    prefix [0, min(i + 1, valid_len))."""
    return np.minimum(np.asarray(i) + 1, valid_len)


def masked_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray,
                     valid_len: Sequence[int], row_block: int = 256,
                     check: bool = True, rows: np.ndarray | None = None) -> np.ndarray:
    """Causal + key-padding multi-head attention.  k, v [B, H, L, dh];
    q [B, H, R, dh] holds the query rows at positions ``rows[b]`` ([B, R],
    increasing; default: every position, R = L).  Returns the context
    [B, R, H*dh].

    Each query row i takes an exact two-pass softmax over the keys the mask
    leaves visible, j < min(i + 1, valid_len).  Rows are independent; they are
    evaluated in blocks of the positions [r0, r0 + row_block), which only
    bounds memory for 100k-token sequences.  A block's score matrix spans the
    keys its last position may see; entries of keys hidden from a row are
    set to -inf before the max, so their exponentials are exactly 0.  A
    subset of rows is evaluated in the same blocks as the full set, so every
    selected row goes through the same operations as in the full result."""
    B, H, R, dh = q.shape
    L = k.shape[2]
    if rows is None:
        rows = np.broadcast_to(np.arange(L), (B, L))
    rows = np.asarray(rows)
    assert rows.shape == (B, R)
    out = np.empty_like(q)
    scale = 1.0 / math.sqrt(dh)
    for b in range(B):
        vl = int(valid_len[b])
        assert 1 <= vl <= L
        pos = rows[b]
        assert np.all(np.diff(pos) > 0) and pos[0] >= 0 and pos[-1] < L
        for r0 in range(0, L, row_block):
            r1 = min(L, r0 + row_block)
            sel = np.nonzero((pos >= r0) & (pos < r1))[0]  # entries of q in this block
            if sel.size == 0:
                continue
            n_keys = allowed_keys(pos[sel], vl)        # visible prefix per row
            kmax = int(allowed_keys(r1 - 1, vl))       # the block's widest prefix
            hidden = np.arange(kmax)[None, :] >= n_keys[:, None]
            for h in range(H):
                s = (q[b, h, sel] @ k[b, h, :kmax].T) * scale
                s[hidden] = -np.inf
                m = s.max(axis=1, keepdims=True)
                e = np.exp(s - m)
                den = e.sum(axis=1, keepdims=True)
                p = e / den
                if check:
                    assert np.all(np.abs(p.sum(axis=1) - 1.0) < 1e-12)
                out[b, h, sel] = p @ v[b, h, :kmax]
    return merge_heads(out)


def layer_norm(r: np.ndarray, gamma: np.ndarray, beta: np.ndarray,
               eps: float = LN_EPS) -> np.ndarray:
    """LayerNorm over the last axis: two-pass mean and biased variance,
    (r - mean) / sqrt(var + eps) * gamma + beta."""
    mu = r.mean(axis=-1, keepdims=True)
    dev = r - mu
    var = (dev * dev).mean(axis=-1, keepdims=True)
    return dev / np.sqrt(var + eps) * gamma + beta


def gelu_erf(u: np.ndarray) -> np.ndarray:
    """Exact GELU: 0.5 u (1 + erf(u / sqrt(2)))."""
    return 0.5 * u * (1.0 + erf(u / math.sqrt(2.0)))


def encoder_layer(x: np.ndarray, valid_len: Sequence[int], p: Dict[str, np.ndarray],
                  n_heads: int, row_block: int = 256, check: bool = True,
                  rows: np.ndarray | None = None) -> np.ndarray:
    """One post-LN encoder layer, no dropout:
        y  = LN1(x + MHA(x) W_o^T + b_o)
        x' = LN2(y + gelu(y W_1^T + b_1) W_2^T + b_2).
    With ``rows`` ([B, R] increasing positions per sequence) only those
    query rows are evaluated and [B, R, d] is returned; the keys and values
    still come from every position."""
    q, k, v = qkv_projection(x, p["w_qkv"], p["b_qkv"], n_heads)
    xr = x
    if rows is not None:
        rows = np.asarray(rows)
        bi = np.arange(x.shape[0])[:, None]
        q = q[bi[:, :, None], np.arange(n_heads)[None, :, None], rows[:, None, :]]
        xr = x[bi, rows]
    ctx = masked_attention(q, k, v, valid_len, row_block=row_block, check=check, rows=rows)
    a = ctx @ p["w_o"].T + p["b_o"]
    y = layer_norm(xr + a, p["ln1_g"], p["ln1_b"])
    f = gelu_erf(y @ p["w_1"].T + p["b_1"])
    g = f @ p["w_2"].T + p["b_2"]
    return layer_norm(y + g, p["ln2_g"], p["ln2_b"])


def encoder_forward(x: np.ndarray, valid_len: Sequence[int],
                    layers: List[Dict[str, np.ndarray]], n_heads: int,
                    row_block: int = 256, check: bool = True) -> np.ndarray:
    """The whole stack: the layers applied in order.  Returns fp64 [B, L, d]."""
    h = np.asarray(x, dtype=np.float64)
    for p in layers:
        h = encoder_layer(h, valid_len, p, n_heads, row_block=row_block, check=check)
    return h


def first_row_closed_form(x0: np.ndarray, layers: List[Dict[str, np.ndarray]]
                          ) -> np.ndarray:
    """Row 0 of any sequence sees only key 0, whose softmax weight is exactly
    1, so its attention output is the V projection of that token whatever the
    heads.  The stack's row 0 is then a per-token chain:
        v  = W_v x + b_v
        y  = LN1(x + W_o v + b_o)
        x' = LN2(y + W_2 gelu(W_1 y + b_1) + b_2).
    x0 [d] (or [N, d] for N independent first rows)."""
    h = np.asarray(x0, dtype=np.float64)
    for p in layers:
        d = h.shape[-1]
        v = h @ p["w_qkv"][2 * d:].T + p["b_qkv"][2 * d:]
        y = layer_norm(h + v @ p["w_o"].T + p["b_o"], p["ln1_g"], p["ln1_b"])
        f = gelu_erf(y @ p["w_1"].T + p["b_1"])
        h = layer_norm(y + f @ p["w_2"].T + p["b_2"], p["ln2_g"], p["ln2_b"])
    return h
