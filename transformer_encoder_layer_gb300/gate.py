"""The pages' per-element accuracy gate and its envelope utilisation.

Comparison logic only (no encoder arithmetic).  The gate is "atol <= 0.002 OR
rtol <= 0.02" on every element ("Hyper-optimized megakernel-hybrid transformer
inference", section "Headline results"; "KernelForge", section "Inspiration").
"""
from __future__ import annotations

from typing import Tuple

import numpy as np

ATOL = 2e-3
RTOL = 2e-2

def gate(gpu: np.ndarray, ref: np.ndarray, atol: float = ATOL, rtol: float = RTOL
         ) -> Tuple[bool, float, tuple]:
    """Per-element gate: pass iff |e| <= atol OR |e| <= rtol*|ref| (NaN/Inf
    fail).  Returns (passed, envelope utilisation, worst index).  The
    envelope utilisation is max over elements of min(|e|/atol, |e|/(rtol|ref|));
    it is <= 1 iff every element passes ("KernelForge", section "What we
    built": the gate collapsed to one number)."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    e = np.abs(gpu - ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        util = np.minimum(e / atol, e / (rtol * np.abs(ref)))
    util = np.where(np.isfinite(gpu), util, np.inf)
    if util.size == 0:
        return True, 0.0, ()
    idx = np.unravel_index(int(np.argmax(util)), util.shape)
    u = float(util[idx])
    return bool(u <= 1.0), u, tuple(int(i) for i in idx)
