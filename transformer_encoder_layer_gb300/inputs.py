"""Seeded synthetic inputs for the masked post-LN encoder stack.

This module is the only code shared by the CUDA path's tests/bench and the
fp64 oracle: it draws random numbers and rounds them to the I/O dtype, and
holds none of the encoder's arithmetic.

Workload shapes follow the five synthetic stand-ins for the organiser's
fourteen shapes ("KernelForge", section "Why it matters": 2-4 layers,
d_model 32-1024, batch 1 to 10,000, causal plus padding masks, a 100,000-token
history).  Draw order, fixed so both sides see the same bytes:

1. ``valid_len = integers(lo, hi + 1, size=B)`` (inclusive range);
2. ``x = standard_normal((B, L, d))`` then ``x * input_scale`` in fp64,
   rounded to the dtype (every scale reuses the same draw);
3. per layer, in order: W_qkv, b_qkv, W_o, b_o, ln1_g, ln1_b, W_1, b_1,
   W_2, b_2, ln2_g, ln2_b.  Weights ~ N(0, 1/fan_in) (variance), biases
   ~ N(0, 0.02^2), gamma = 1 + 0.1 N(0,1), beta ~ 0.1 N(0,1).

All parameters are stored in the I/O dtype; the fp64 copies handed to the
oracle are the dtype-rounded values, so weight rounding is not an error source.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List

import numpy as np

DTYPES = ("f32", "f16", "bf16")
PARAM_NAMES = ("w_qkv", "b_qkv", "w_o", "b_o", "ln1_g", "ln1_b",
               "w_1", "b_1", "w_2", "b_2", "ln2_g", "ln2_b")


@dataclasses.dataclass(frozen=True)
class EncoderShape:
    name: str
    n_layers: int
    d_model: int
    n_heads: int
    d_ff: int
    batch: int
    seq_len: int
    dtype: str
    vl_lo: int
    vl_hi: int

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads

    @property
    def tokens(self) -> int:
        return self.batch * self.seq_len

    def with_(self, **kw) -> "EncoderShape":
        return dataclasses.replace(self, **kw)


# The five workloads, named by what they are.
SHAPES: Dict[str, EncoderShape] = {
    "tiny_d32_L32": EncoderShape("tiny_d32_L32", 2, 32, 2, 128, 4, 32, "f32", 16, 32),
    "short_d128_L64_B4096": EncoderShape("short_d128_L64_B4096", 4, 128, 4, 512, 4096, 64, "f16", 32, 64),
    "batch1_d256_L512": EncoderShape("batch1_d256_L512", 2, 256, 8, 1024, 1, 512, "f32", 384, 512),
    "wide_d1024_L1024_B32": EncoderShape("wide_d1024_L1024_B32", 2, 1024, 16, 4096, 32, 1024, "bf16", 512, 1024),
    "long_d64_L100k_B8": EncoderShape("long_d64_L100k_B8", 2, 64, 4, 256, 8, 100000, "f16", 90000, 100000),
}

INPUT_SCALES = (1e-3, 1e-1, 1.0, 1e1, 1e3)


def round_to_dtype(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 values to ``dtype`` (round-to-nearest-even, in one step from
    fp64, no double rounding) and return them as exact fp64 values."""
    a = np.asarray(a, dtype=np.float64)
    if dtype == "f32":
        return a.astype(np.float32).astype(np.float64)
    if dtype == "f16":
        return a.astype(np.float16).astype(np.float64)
    if dtype == "bf16":
        # bf16 keeps 8 significant bits; frexp gives m in [0.5, 1).
        m, e = np.frexp(a)
        return np.ldexp(np.rint(m * 256.0), e - 8)
    raise ValueError(f"unknown dtype {dtype!r}")


def _layer_params(rng: np.random.Generator, d: int, d_ff: int) -> Dict[str, np.ndarray]:
    p = {}
    p["w_qkv"] = rng.standard_normal((3 * d, d)) / np.sqrt(d)
    p["b_qkv"] = rng.standard_normal(3 * d) * 0.02
    p["w_o"] = rng.standard_normal((d, d)) / np.sqrt(d)
    p["b_o"] = rng.standard_normal(d) * 0.02
    p["ln1_g"] = 1.0 + 0.1 * rng.standard_normal(d)
    p["ln1_b"] = 0.1 * rng.standard_normal(d)
    p["w_1"] = rng.standard_normal((d_ff, d)) / np.sqrt(d)
    p["b_1"] = rng.standard_normal(d_ff) * 0.02
    p["w_2"] = rng.standard_normal((d, d_ff)) / np.sqrt(d_ff)
    p["b_2"] = rng.standard_normal(d) * 0.02
    p["ln2_g"] = 1.0 + 0.1 * rng.standard_normal(d)
    p["ln2_b"] = 0.1 * rng.standard_normal(d)
    return p


@dataclasses.dataclass
class EncoderInputs:
    shape: EncoderShape
    input_scale: float
    seed: int
    valid_len: np.ndarray            # int32 [B]
    x: np.ndarray                    # fp64 [B, L, d], dtype-rounded values
    layers: List[Dict[str, np.ndarray]]  # fp64, dtype-rounded values


def make_inputs(shape: EncoderShape, seed: int = 0, input_scale: float = 1.0,
                batch: int | None = None) -> EncoderInputs:
    """Draw one seeded input set.  ``batch`` (<= shape.batch) keeps only the
    first sequences of the same draw, so a subsample is bit-identical to the
    corresponding rows of the full workload."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B, L, d = shape.batch, shape.seq_len, shape.d_model
    vl = rng.integers(shape.vl_lo, shape.vl_hi + 1, size=B).astype(np.int32)
    if batch is not None and batch < B:
        # x is drawn row-major over (B, L, d); the first `batch` sequences are
        # a prefix of the stream, so draw them, then skip the rest.
        x = rng.standard_normal((batch, L, d))
        rng.standard_normal((B - batch) * L * d)
        vl = vl[:batch]
    else:
        x = rng.standard_normal((B, L, d))
    x = round_to_dtype(x * input_scale, shape.dtype)
    layers = []
    for _ in range(shape.n_layers):
        p = _layer_params(rng, d, shape.d_ff)
        layers.append({k: round_to_dtype(v, shape.dtype) for k, v in p.items()})
    return EncoderInputs(shape if batch is None else shape.with_(batch=len(vl)),
                         input_scale, seed, vl, x, layers)


def to_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 values already representable in ``dtype`` -> a numpy array of the
    dtype's storage (bf16 as uint16 bit patterns)."""
    if dtype == "f32":
        return np.ascontiguousarray(a, dtype=np.float32)
    if dtype == "f16":
        return np.ascontiguousarray(a, dtype=np.float16)
    if dtype == "bf16":
        f = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
        return np.ascontiguousarray((f >> 16).astype(np.uint16))
    raise ValueError(dtype)


def from_storage(a: np.ndarray, dtype: str) -> np.ndarray:
    """Inverse of :func:`to_storage`: storage array -> fp64 values."""
    if dtype in ("f32", "f16"):
        return np.asarray(a).astype(np.float64)
    if dtype == "bf16":
        u = np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16
        return u.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def tiny_shape(**kw) -> EncoderShape:
    """A small shape for quick tests; keyword overrides."""
    base = dict(name="tiny", n_layers=2, d_model=32, n_heads=2, d_ff=128,
                batch=3, seq_len=9, dtype="f32", vl_lo=1, vl_hi=9)
    base.update(kw)
    return EncoderShape(**base)

