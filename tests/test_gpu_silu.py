"""The kernels' SiLU forms, element by element, over the range the conv outputs can take.

The tree kernel's x conv evaluates SiLU on the FMA pipe: v / (1 + 2^t), t = -v·log2(e),
2^t by Cody-Waite reduction and a degree-6 Taylor series, 1 / d by three Newton-Raphson
steps; its stated relative error is about 4e-6.  Here it is checked, through the C ABI
(ssm_selftest_silu), against CUDA's expf-based form and against fp64 on the host:
every finite bf16 value with |v| <= 87, a dense grid over [-87, 87] and normal draws.
Beyond |v| = 87 (2^t clamped) the result must stay within 1e-30 of v·sigmoid(v)."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from speculative_decoding_mamba2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need CUDA"


def _inputs():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    allbf = bits.view(np.float32)
    allbf = allbf[np.isfinite(allbf)]
    g = np.random.default_rng(5)
    return np.concatenate([allbf, np.linspace(-87.0, 87.0, 1 << 22, dtype=np.float32),
                           g.normal(0.0, 3.0, 1 << 20).astype(np.float32),
                           np.array([0.0, -0.0, 1e-30, -1e-30, 87.0, -87.0, 88.0, -88.0, 100.0, -100.0], np.float32)])


def _rel(got, ref):
    return np.abs(got - ref) / np.abs(ref)


def test_silu_forms_against_fp64_and_expf():
    from speculative_decoding_mamba2_gb300 import ssm_selftest_silu
    v = _inputs()
    out = ssm_selftest_silu(torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    poly, fast, ref32 = (o.astype(np.float64) for o in out.cpu().numpy())
    v64 = v.astype(np.float64)
    with np.errstate(over="ignore"):
        exact = v64 / (1.0 + np.exp(-v64))
    inside = (np.abs(v64) <= 87.0) & (np.abs(exact) > 1e-30)
    # the FMA-pipe form: relative error below 4e-6 against fp64 and against CUDA's expf form
    assert _rel(poly[inside], exact[inside]).max() <= 4e-6
    assert _rel(poly[inside], ref32[inside]).max() <= 5e-6
    # CUDA's expf form itself (rounded divide): a few ulp
    assert _rel(ref32[inside], exact[inside]).max() <= 1e-6
    # the special-function form on the conv outputs' range (|v| <= 20)
    conv = inside & (np.abs(v64) <= 20.0)
    assert _rel(fast[conv], exact[conv]).max() <= 4e-6
    # outside: v (large positive) or a value within 1e-30 of the tiny exact result
    outside = ~inside
    assert np.all(np.abs(poly[outside] - exact[outside]) <= 1e-30 + 4e-6 * np.abs(exact[outside]))
    assert np.all(np.isfinite(poly)) and np.all(np.isfinite(fast))
