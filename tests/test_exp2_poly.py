"""The FMA-pipe exponential of the forward kernel (csrc/exp2_poly.cuh), checked on
the CPU: the coefficients are the ones the Remez fit in csrc/exp2_poly_fit.py
produces, and a float32 emulation of the device evaluation (Cody-Waite split,
Horner steps rounded to float32, 2^n from the exponent field) stays within the
fit's bound of 2^x everywhere the softmax uses it.  Also the build's spill
check."""

import math
import os
import re
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "online_softmax_14_b300", "csrc")


def header_coefficients():
    text = open(os.path.join(CSRC, "exp2_poly.cuh")).read()
    out = {}
    for k in range(4):
        m = re.search(rf"kExp2C{k} = (0x[0-9a-fA-F.p+-]+)f;", text)
        out[k] = float.fromhex(m.group(1))
    return [out[k] for k in range(4)]


def fit():
    sys.path.insert(0, CSRC)
    try:
        import exp2_poly_fit
    finally:
        sys.path.remove(CSRC)
    return exp2_poly_fit.remez_exp2()


def test_header_holds_the_fitted_coefficients():
    c, err = fit()
    assert err < 7.6e-5  # the levelled relative error of the degree-3 fit
    for got, want in zip(header_coefficients(), c):
        assert got == float(np.float32(want))


def _f32(x):
    return np.asarray(x, dtype=np.float64).astype(np.float32)


def exp2_fma2_emulated(x):
    """The device steps in float32 (fma emulated exactly in float64, then rounded)."""
    c0, c1, c2, c3 = (np.float64(v) for v in header_coefficients())
    x = np.maximum(_f32(x), np.float32(-127.0))
    magic = np.float32(12582912.0)
    t = (x + magic).astype(np.float32)             # round(x) in the low mantissa bits
    n = (t - magic).astype(np.float32)
    f = (x - n).astype(np.float32)
    fd = f.astype(np.float64)
    p = _f32(c3 * fd + c2)
    p = _f32(p.astype(np.float64) * fd + c1)
    p = _f32(p.astype(np.float64) * fd + c0)
    e = ((t.view(np.uint32).astype(np.uint64) + 127) << 23) & 0xFFFFFFFF
    scale = e.astype(np.uint32).view(np.float32)
    return (p * scale).astype(np.float32)


def test_emulated_device_evaluation_meets_the_bound():
    # the softmax feeds x = s - m_ref <= 8 (the lazy rescale's threshold), and
    # anything below -126 only adds terms under 2^-126 to a row sum of at least 1
    x = np.concatenate([np.linspace(-126.0, 8.0, 2_000_001), np.arange(-126, 9) + 0.5,
                        np.arange(-126, 9).astype(np.float64)])
    x = _f32(x).astype(np.float64)
    got = exp2_fma2_emulated(x).astype(np.float64)
    rel = np.abs(got / np.exp2(x) - 1.0)
    assert rel.max() < 1.0e-4, rel.max()


def test_clamped_inputs_give_exact_zero():
    x = np.array([-127.0, -127.2, -200.0, -1e30, -np.inf], dtype=np.float32)
    assert np.all(exp2_fma2_emulated(x) == 0.0)


def test_integer_inputs_are_exact_powers_of_two():
    n = np.arange(-126, 9)
    got = exp2_fma2_emulated(n.astype(np.float32)).astype(np.float64)
    # p(0) = c0, so 2^n comes out as c0 * 2^n: within the fit's bound of exact
    assert np.all(np.abs(got / np.exp2(n) - 1.0) < 7.6e-5)


def test_build_spill_check_flags_any_spilling_kernel():
    from online_softmax_14_b300.build import spilling_kernels

    log = ("ptxas info    : Compiling entry function 'kA' for 'sm_103a'\n"
           "    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n"
           "ptxas info    : Compiling entry function 'kB' for 'sm_103a'\n"
           "    8 bytes stack frame, 4 bytes spill stores, 4 bytes spill loads\n"
           "ptxas info    : Compiling entry function 'kC' for 'sm_103a'\n"
           "    0 bytes stack frame, 0 bytes spill stores, 12 bytes spill loads\n")
    bad = spilling_kernels(log)
    assert len(bad) == 2 and bad[0].startswith("kB") and bad[1].startswith("kC")
