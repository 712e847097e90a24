"""The FMA-pipe polynomial the forward kernel uses for part of its softplus
evaluations: log2(1 + u) for u = 2^-|z| in [0, 1], evaluated as
u (c1 + u (c2 + ... + u c6)) in fp32 Horner arithmetic, with max(z, 0) added
in the last step.  Checked here against the exact function (numpy float64):
the stated largest error, exactness at u = 0 (a masked column, z = -inf,
must give exactly 0), and the resulting softplus error in log2 units over
the z range the kernel sees.  The coefficients are read from the CUDA
header, so the test follows any change to them."""

import pathlib
import re

import numpy as np

HEADER = pathlib.Path(__file__).resolve().parents[1] / "lssar_attn_fwd_gb300" / "csrc" / "softplus_poly.cuh"


def coefficients():
    """c1..c6 in the order the header's Horner steps use them (innermost first)."""
    text = HEADER.read_text()
    body = text[text.index("sp2x2_poly"):]
    body = body[:body.index("}\n")]
    # each __ffma2_rn(..., make_float2(c, c)) carries one coefficient; the
    # first call carries two (the leading product's factor and addend)
    nums = [float(x) for x in re.findall(r"make_float2\(\s*(-?[0-9.]+(?:e-?[0-9]+)?)f\s*,", body)]
    assert len(nums) == 6, nums
    c6, c5, c4, c3, c2, c1 = nums
    return [c1, c2, c3, c4, c5, c6]


def poly_f32(u):
    c1, c2, c3, c4, c5, c6 = (np.float32(c) for c in coefficients())
    u = u.astype(np.float32)
    h = (u * c6 + c5).astype(np.float32)
    h = (h * u + c4).astype(np.float32)
    h = (h * u + c3).astype(np.float32)
    h = (h * u + c2).astype(np.float32)
    h = (h * u + c1).astype(np.float32)
    return (h * u).astype(np.float32)


def test_error_bound_on_unit_interval():
    u = np.linspace(0.0, 1.0, 1_000_001)
    err = np.abs(poly_f32(u).astype(np.float64) - np.log2(1.0 + u))
    assert err.max() <= 2.3e-6, err.max()


def test_masked_column_gives_exact_zero():
    assert poly_f32(np.array([0.0]))[0] == 0.0


def test_softplus_error_over_score_range():
    # z = log2(e) ln(d) ln(i) cos: |z| < 117 for every shape the C ABI accepts
    z = np.linspace(-117.0, 117.0, 400_001)
    u = np.exp2(-np.abs(z))
    sp_poly = np.maximum(z, 0.0) + poly_f32(u).astype(np.float64)
    sp_exact = np.logaddexp2(0.0, z)
    assert np.abs(sp_poly - sp_exact).max() <= 2.5e-6


def test_polynomial_is_monotone():
    # the kernel's ReLU threshold compares softplus values: a polynomial that
    # rose and fell could reorder nearby scores
    u = np.linspace(0.0, 1.0, 100_001)
    assert np.all(np.diff(poly_f32(u).astype(np.float64)) >= -1e-7)


def test_coefficients_are_reproduced_by_the_fitting_script():
    # the committed fit (Lawson minimax, constant term 0), rounded to fp32,
    # gives exactly the header's coefficients
    import importlib.util
    path = HEADER.parent / "fit_softplus_poly.py"
    spec = importlib.util.spec_from_file_location("fit_softplus_poly", path)
    fit = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(fit)
    c = fit.fit(6)
    assert [np.float32(x) for x in c] == [np.float32(x) for x in coefficients()]
    assert fit.max_error_f32(c) < 2.3e-6
