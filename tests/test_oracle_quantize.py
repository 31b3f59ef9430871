"""Pins for the oracle's Q8 activation quantization (C3) and RMSNorm producer (C4).

Pinned by closed forms, exact scaling/sign invariants, the rounding-error bound and an
exact-rational brute force -- never by re-running the oracle's own formula.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quantized_q8_activation_quantize_gb300 import inputs


def test_closed_form_unit_block():
    x = np.zeros((1, 32), np.float32)
    x[0, 0] = 127.0
    q, d, S = oracle.quantize_q8(x)
    assert d[0, 0] == 1.0 and q[0, 0] == 127 and (q[0, 1:] == 0).all() and S[0, 0] == 127


def test_ties_round_half_away_from_zero():
    # amax 127 -> d = 1, id = 1: the products are the inputs themselves
    x = np.zeros((1, 32), np.float32)
    vals = [127.0, 0.5, -0.5, 2.5, -2.5, 1.5, -1.5, 126.5, -126.5, 0.49999997]
    x[0, :len(vals)] = vals
    q, d, S = oracle.quantize_q8(x)
    assert d[0, 0] == 1.0
    assert q[0, :len(vals)].tolist() == [127, 1, -1, 3, -3, 2, -2, 127, -127, 0]
    assert S[0, 0] == sum([127, 1, -1, 3, -3, 2, -2, 127, -127, 0])


def test_zero_block():
    x = np.zeros((2, 64), np.float32)
    x[1, 32:] = 1.0
    q, d, S = oracle.quantize_q8(x)
    assert d[0].tolist() == [0.0, 0.0] and d[1, 0] == 0.0 and (q[0] == 0).all() and S[1, 0] == 0
    assert d[1, 1] == np.float32(1.0) / np.float32(127.0) and (q[1, 32:] == 127).all() and S[1, 1] == 127 * 32


def test_power_of_two_scaling_is_exact():
    x = inputs.activations(np.random.default_rng(7), 4, 256)
    q0, d0, S0 = oracle.quantize_q8(x)
    for k in (-20, -3, 1, 5, 20):
        q, d, S = oracle.quantize_q8(np.ldexp(x, k).astype(np.float32))
        assert np.array_equal(q, q0) and np.array_equal(S, S0)
        assert np.array_equal(d, np.ldexp(d0, k).astype(np.float32))


def test_sign_symmetry():
    x = inputs.activations(np.random.default_rng(8), 4, 256)
    q0, d0, S0 = oracle.quantize_q8(x)
    q, d, S = oracle.quantize_q8(-x)
    assert np.array_equal(q, -q0) and np.array_equal(d, d0) and np.array_equal(S, -S0)


def test_rounding_error_bound_and_range():
    r = np.random.default_rng(9)
    x = inputs.activations(r, 16, 512) * r.uniform(0.01, 100, size=(16, 1)).astype(np.float32)
    x[3, :32] = 0.0
    q, d, S = oracle.quantize_q8(x)
    assert q.min() >= -127 and q.max() <= 127
    dd = np.repeat(d.astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - dd * q)
    # |x - d q| <= d/2 up to the two f32 roundings of d and 1/d (a few ulp of 127)
    assert (err <= dd * (0.5 + 1e-5)).all()
    # the largest element of every non-zero block maps to +-127
    xb = np.abs(x.reshape(16, -1, 32))
    qb = np.abs(q.reshape(16, -1, 32)).astype(int)
    arg = xb.argmax(axis=2)
    top = np.take_along_axis(qb, arg[..., None], 2)[..., 0]
    assert ((top == 127) | (xb.max(axis=2) == 0)).all()
    assert np.array_equal(S, q.reshape(16, -1, 32).astype(np.int32).sum(axis=2))


def test_rmsnorm_constant_row_closed_form():
    for c in (0.5, 1.0, 3.0, 1e-3):
        x = np.full((1, 256), c, np.float32)
        y = oracle.rmsnorm(x, np.ones(256, np.float32), 1e-6)
        exact = float(np.float32(c)) / np.sqrt(float(np.float32(c)) ** 2 + float(np.float32(1e-6)))
        assert np.allclose(y, exact, rtol=3e-7, atol=0)


def test_rmsnorm_exact_rational_brute_force():
    # tiny K: the exact mean of squares as a Fraction, then 1/sqrt to double precision
    r = np.random.default_rng(10)
    x = inputs.activations(r, 3, 64)
    w = inputs.rms_weight(r, 64)
    eps = np.float32(1e-6)
    y = oracle.rmsnorm(x, w, eps)
    for m in range(3):
        ms = sum(Fraction(float(v)) ** 2 for v in x[m]) / 64 + Fraction(float(eps))
        rr = np.float32(1.0 / np.sqrt(float(ms)))          # ms is held exactly, rounded once
        ref = (x[m] * rr).astype(np.float32) * w
        # equal unless the exact and the f64-accumulated mean straddle an f32 rounding boundary
        assert np.array_equal(y[m], ref.astype(np.float32))


def test_rmsnorm_scale_invariance_and_weight_linearity():
    r = np.random.default_rng(11)
    x = inputs.activations(r, 4, 512)
    w = inputs.rms_weight(r, 512)
    y0 = oracle.rmsnorm(x, w, 0.0)
    for k in (-6, 3):
        assert np.array_equal(oracle.rmsnorm(np.ldexp(x, k).astype(np.float32), w, 0.0), y0)
    assert np.array_equal(oracle.rmsnorm(x, 2 * w, 1e-6), 2 * oracle.rmsnorm(x, w, 1e-6))


def test_quantize_with_rms_is_quantize_of_rmsnorm():
    r = np.random.default_rng(12)
    x = inputs.activations(r, 5, 256)
    w = inputs.rms_weight(r, 256)
    a = oracle.quantize_q8(x, w, 1e-6)
    b = oracle.quantize_q8(oracle.rmsnorm(x, w, 1e-6))
    for u, v in zip(a, b):
        assert np.array_equal(u, v)
