"""CPU rounding-emulation probe of the 16-bit tensor-core paths' precision
plan (test infrastructure; it is neither the oracle nor the CUDA path).

The probe evaluates the encoder stack in float64 but rounds, at the stages a
plan names, exactly where the 16-bit tensor-core kernels round: activation
operands of every product to the I/O dtype, either alone ("hi") or as a
(hi, lo) pair whose lo = rn(v - hi) carries the rest; products and
accumulators to fp32; the softmax probabilities and LayerNorm outputs to
fp32.  Weights enter unrounded: they are exact in the I/O dtype.  Comparing
its output with the oracle under the pages' gate predicts a plan's envelope
utilisation before a kernel is changed ("KernelForge", section "What we
learned": the error budget decides the precision of every stage).

The layer-1 near-tie correction of the kernels is modelled: a row whose
emulated top-two score gap is below 12 + 2E logits with E above 2e-3 (E =
2^-19 |q| max|k| / sqrt(dh)) takes its probabilities in fp64, as the kernels'
fix-up recomputes them.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
from scipy.special import erf

from transformer_encoder_layer_gb300.inputs import round_to_dtype


@dataclasses.dataclass(frozen=True)
class Plan:
    """Which activation operands keep their lo part (True) or are rounded to
    the I/O dtype alone (False)."""
    x_lo: bool = True      # layer input of layers >= 2 (QKV A operand and residual)
    qk_lo: bool = True     # S = Qh Kh + Qh Kl + Ql Kh
    v_lo: bool = True      # P V uses Vh + Vl
    p_lo: bool = True      # P V uses Ph + Pl (the Pl Vh product)
    ctx_lo: bool = True    # out-projection A operand
    y_lo: bool = True      # FFN1 A operand (LN1 output)
    h_lo: bool = True      # FFN2 A operand (GELU output)


ALL_SPLIT = Plan()
PLAIN = Plan(False, False, False, False, False, False, False)


def f32(a):
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def split(a, dtype, keep_lo):
    """(hi, lo) of fp32 values a in dtype; lo = 0 when the plan drops it."""
    hi = round_to_dtype(a, dtype)
    if not keep_lo:
        return hi, np.zeros_like(hi)
    return hi, round_to_dtype(a - hi, dtype)


def _ln(r, g, b):
    mu = r.mean(axis=-1, keepdims=True)
    dv = r - mu
    var = (dv * dv).mean(axis=-1, keepdims=True)
    return f32(dv / np.sqrt(var + 1e-5) * g + b)


def _gelu(u):
    return 0.5 * u * (1.0 + erf(u / math.sqrt(2.0)))


def _attention(xin_exact, q, k, v, valid_len, H, dtype, plan, fix_ties):
    """q, k, v: fp32 [B, L, d] projections.  Returns fp32 ctx [B, L, d]."""
    B, L, d = q.shape
    dh = d // H
    qh, ql = split(q, dtype, plan.qk_lo)
    kh, kl = split(k, dtype, plan.qk_lo)
    vh, vl_ = split(v, dtype, plan.v_lo)
    ctx = np.empty_like(q)
    scale = 1.0 / math.sqrt(dh)
    for b in range(B):
        n = int(valid_len[b])
        rows = np.arange(L)
        vis = np.minimum(rows + 1, n)
        hidden = np.arange(L)[None, :] >= vis[:, None]
        for h in range(H):
            c = slice(h * dh, (h + 1) * dh)
            s = f32(qh[b, :, c] @ kh[b, :, c].T + qh[b, :, c] @ kl[b, :, c].T +
                    ql[b, :, c] @ kh[b, :, c].T)
            s = np.where(hidden, -np.inf, s)
            m = s.max(axis=1, keepdims=True)
            p = f32(np.exp(f32(s * scale) - f32(m * scale)))
            if fix_ties:
                # the near-tie screen of the kernels, on the emulated scores
                qn = np.linalg.norm(q[b, :, c], axis=1)
                kmax = np.max(np.linalg.norm(k[b, :n, c], axis=1))
                err = 2.0 ** -19 * qn * kmax / math.sqrt(dh)
                srt = np.sort(np.where(hidden, -np.inf, s), axis=1)
                gap = (srt[:, -1] - srt[:, -2]) * scale
                flag = (err > 2e-3) & (gap < 12 + 2 * err) & (vis >= 2)
                if np.any(flag):
                    se = (q[b][flag][:, c] @ k[b, :, c].T) * scale
                    se = np.where(hidden[flag], -np.inf, se)
                    pe = np.exp(se - se.max(axis=1, keepdims=True))
                    p[flag] = pe
            ph, pl = split(p, dtype, plan.p_lo)
            o = f32(ph @ vh[b, :, c] + ph @ vl_[b, :, c] + pl @ vh[b, :, c])
            lsum = f32(p.sum(axis=1, keepdims=True))
            ctx[b, :, c] = f32(o / lsum)
    return ctx


def forward(x, valid_len, layers, n_heads, dtype, plan=ALL_SPLIT, fix_ties=True):
    """The stack with the plan's roundings.  x: dtype-rounded inputs [B, L, d]
    (fp64 values); returns the output rounded to dtype."""
    h = np.asarray(x, dtype=np.float64)
    for li, p in enumerate(layers):
        d = h.shape[-1]
        if li == 0:
            ah, al = h, np.zeros_like(h)          # the exact 16-bit input
        else:
            ah, al = split(h, dtype, plan.x_lo)
        res = ah + al                             # residual as the kernels read it
        qkv = f32(ah @ p["w_qkv"].T + al @ p["w_qkv"].T + p["b_qkv"])
        q, k, v = qkv[..., :d], qkv[..., d:2 * d], qkv[..., 2 * d:]
        ctx = _attention(h, q, k, v, valid_len, n_heads, dtype, plan, fix_ties and li == 0)
        ch, cl = split(ctx, dtype, plan.ctx_lo)
        a = f32(ch @ p["w_o"].T + cl @ p["w_o"].T)
        y = _ln(f32(a + p["b_o"] + res), p["ln1_g"], p["ln1_b"])
        yh, yl = split(y, dtype, plan.y_lo)
        u = f32(yh @ p["w_1"].T + yl @ p["w_1"].T + p["b_1"])
        g = f32(_gelu(u))
        gh, gl = split(g, dtype, plan.h_lo)
        z = f32(gh @ p["w_2"].T + gl @ p["w_2"].T)
        h = _ln(f32(z + p["b_2"] + (yh + yl)), p["ln2_g"], p["ln2_b"])
    return round_to_dtype(h, dtype)
