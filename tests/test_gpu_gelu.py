"""The branch-free GELU (erf from Abramowitz & Stegun 7.1.28) against the
erff form and against fp64 exact GELU, on a dense grid."""
import numpy as np
import pytest
from scipy.special import erf

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_gelu_forms_agree():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_encoder_layer_gb300 import binding, build
    build.build()
    lib = binding.load()
    x = torch.linspace(-30.0, 30.0, 2_000_001, dtype=torch.float32, device="cuda")
    x = torch.cat([x, torch.tensor([0.0, -0.0, 1e-30, -1e-30, 1e30, -1e30], device="cuda")])
    ye, yf = torch.empty_like(x), torch.empty_like(x)
    assert lib.tl_eval_gelu(x.data_ptr(), ye.data_ptr(), yf.data_ptr(), x.numel(), None) == 0
    torch.cuda.synchronize()
    xd = x.cpu().numpy().astype(np.float64)
    exact = 0.5 * xd * (1.0 + erf(xd / np.sqrt(2.0)))
    fast, slow = yf.cpu().numpy().astype(np.float64), ye.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(fast))
    # Bound: 0.5 |x| (3e-7 [the formula's erf error] + 2.5e-6 r [fp32: Horner
    # error ~2 ulp amplified 16x by the power, 4 squarings, the reciprocal],
    # r = (...)^-16 <= 1) + 2e-7 |gelu| for the last operations.
    bound = 0.5 * np.abs(xd) * (3e-7 + 2.5e-6) + 2e-7 * np.abs(exact) + 1e-37
    err = np.abs(fast - exact)
    worst = int(np.argmax(err - bound))
    assert np.all(err <= bound), (xd[worst], fast[worst], exact[worst], err[worst], bound[worst])
    assert np.max(np.abs(fast - slow)) < 2e-5
