"""The software exp2 (csrc/exp2_poly.cuh) on the CPU: its coefficients are the
ones the committed fitting script produces, and the method -- Cody and
Waite's range reduction, the degree-3 polynomial, n added to the exponent
field -- restated in numpy float32 stays within the stated relative error
of 1.01e-4 against float64 exp2 over the clamped range [-125, 64], with
integers exact.  The CUDA evaluation itself is checked on the GPU
(tests/test_exp2_poly_gpu.py)."""
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "exact_io_aware_14_gb300", "csrc")
sys.path.insert(0, CSRC)
import fit_exp2_poly as fit  # noqa: E402

BOUND = 1.02e-4


def _header_coefficients():
    text = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    found = dict(re.findall(r"const float (c\d) = __uint_as_float\(0x([0-9a-f]{8})u\)", text))
    return [int(found["c%d" % k], 16) for k in (1, 2, 3)]


def test_header_holds_the_fitted_coefficients():
    fitted = [int(np.array(c, dtype=np.float32).view(np.uint32)) for c in fit.coefficients()]
    assert _header_coefficients() == fitted


def test_polynomial_error_on_the_reduced_range():
    c32 = [np.uint32(h).view(np.float32) for h in _header_coefficients()]
    assert fit.rel_error_f32(c32) <= BOUND
    # far better than a Taylor polynomial of the same degree: the fit is not a slip
    taylor = [np.float32(np.log(2.0) ** k / np.prod(np.arange(1, k + 1))) for k in (1, 2, 3)]
    assert fit.rel_error_f32(taylor) > 5 * BOUND


def _method_f32(x):
    """The device steps in float32: clamp, round via 1.5*2^23, polynomial,
    exponent add."""
    c1, c2, c3 = (np.uint32(h).view(np.float32) for h in _header_coefficients())
    x = np.fmin(np.fmax(np.asarray(x, dtype=np.float32), np.float32(-125)), np.float32(64))  # C fmaxf: NaN loses
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)
    f = (x - (t - magic)).astype(np.float32)
    p = fit.eval_f32([c1, c2, c3], f).astype(np.float32)
    ex = (t.view(np.uint32).astype(np.uint64) << np.uint64(23)) & np.uint64(0xFFFFFFFF)
    return (p.view(np.uint32).astype(np.uint64) + ex).astype(np.uint32).view(np.float32)


def test_method_error_over_the_clamped_range():
    x = np.concatenate([np.linspace(-125.0, 64.0, 400001), np.linspace(-1.0, 1.0, 20001)]).astype(np.float32)
    y = _method_f32(x).astype(np.float64)
    ref = np.exp2(x.astype(np.float64))
    assert np.max(np.abs(y / ref - 1.0)) <= BOUND
    ints = np.arange(-125, 65, dtype=np.float32)
    assert np.array_equal(_method_f32(ints), np.exp2(ints.astype(np.float64)).astype(np.float32))


@pytest.mark.parametrize("x,expect", [(-200.0, 2.0 ** -125), (-np.inf, 2.0 ** -125), (100.0, 2.0 ** 64),
                                      (np.nan, 2.0 ** -125), (0.0, 1.0)])
def test_method_clamps(x, expect):
    assert _method_f32(np.array([x]))[0] == np.float32(expect)
