"""The FMA-pipe exp2 on the GPU (dit_attn_check_exp2), against float64 2^x and
against the MUFU ex2.approx instruction it stands in for.

Bounds (relative): the degree-2 evaluation 1.75e-3, degree 3 9e-5 (the
polynomial's minimax error plus the rounding of the clamped argument, derived
in exp2_poly.py and pinned on the CPU by test_exp2_poly.py); ex2.approx.ftz
adds at most 2^-22 relative of its own.  The device results must also equal
the CPU model of the same fp32 operations except where a fused rounding ties.
"""
import numpy as np
import pytest

from test_exp2_poly import BOUND, exp2_model

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dit():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import diffusion_transformer_joint_causal_b300 as lib
    from diffusion_transformer_joint_causal_b300 import build
    build.build()
    lib.create()
    yield lib
    assert lib.get_device_error() == 0


def _inputs():
    rng = np.random.default_rng(2)
    x = np.concatenate([np.linspace(-125, 127, 1 << 20), rng.uniform(-125, 127, 1 << 18),
                        np.arange(-125, 128) + 0.5, np.arange(-125, 128) - 0.5,
                        np.arange(-125, 128).astype(float)])
    x = x.astype(np.float32)
    return x[(x >= -125) & (x <= 127)]


@pytest.mark.parametrize("deg", [2, 3])
def test_exp2_fma_against_float64_and_mufu(dit, deg):
    import torch
    x = _inputs()
    y_fma, y_mufu = dit.check_exp2(torch.from_numpy(x).cuda(), deg)
    torch.cuda.synchronize()
    y_fma = y_fma.cpu().numpy().astype(np.float64)
    y_mufu = y_mufu.cpu().numpy().astype(np.float64)
    exact = np.exp2(x.astype(np.float64))
    rel = np.abs(y_fma / exact - 1)
    assert float(rel.max()) <= BOUND[deg], float(rel.max())
    ok = x > -126                                   # ex2.approx.ftz flushes below 2^-126
    rel_mufu = np.abs(y_fma[ok] / y_mufu[ok] - 1)
    assert float(rel_mufu.max()) <= BOUND[deg] + 2.0 ** -22
    model = exp2_model(x, deg).astype(np.float64)
    assert np.count_nonzero(model != y_fma) <= 1e-4 * x.size


@pytest.mark.parametrize("deg", [2, 3])
def test_exp2_fma_clamps(dit, deg):
    import torch
    x = np.array([-126.0, -300.0, -1e30, -np.inf, 128.0, 300.0, 1e30, np.inf], np.float32)
    y_fma, _ = dit.check_exp2(torch.from_numpy(x).cuda(), deg)
    torch.cuda.synchronize()
    y = y_fma.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(y[:4] / 2.0 ** -125 - 1) <= BOUND[deg])
    assert np.all(np.abs(y[4:] / 2.0 ** 127 - 1) <= BOUND[deg])
