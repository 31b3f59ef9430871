"""Pins of the oracle's SwiGLU producer (C8): y = silu(g) * u, silu(g) = g / (1 + exp(-g)),
with exp written out in f32 (reduction by ln2, Taylor series of exp(r)).  Checked against
the mathematics, not against itself: libm's exp, f64 silu, closed forms and identities."""
import math

import numpy as np
import pytest

import oracle

F32_EPS = 2.0 ** -23


def test_exp_f32_against_libm_over_its_range():
    xs = np.concatenate([np.linspace(-86.0, 88.0, 20001), np.linspace(-1.0, 1.0, 4001),
                         np.array([0.0, 0.5 * math.log(2.0), -0.5 * math.log(2.0), math.log(2.0), 1.0, -1.0])])
    worst = 0.0
    for x in xs.astype(np.float32):
        got = oracle.exp_f32(float(x))
        ref = math.exp(float(x))                      # exp of the f32 input, in f64
        worst = max(worst, abs(got - ref) / ref)
    assert worst < 4 * F32_EPS, worst                # a few f32 ulps: reduction + Taylor tail + rounding


def test_exp_f32_exact_points_and_clamps():
    assert oracle.exp_f32(0.0) == 1.0
    # near x = k ln2 the reduction leaves r ~ 0: the result is 2^k times exp of the f32 input's offset
    for k in range(-120, 120, 7):
        x = float(np.float32(k * math.log(2.0)))
        assert abs(oracle.exp_f32(x) / math.exp(x) - 1.0) < 4 * F32_EPS
    # exp(x) exp(-x) = 1
    for x in np.linspace(-80.0, 80.0, 321).astype(np.float32):
        assert abs(oracle.exp_f32(float(x)) * oracle.exp_f32(float(-x)) - 1.0) < 8 * F32_EPS
    # the clamps keep the result a finite normal number
    assert np.isfinite(oracle.exp_f32(1000.0)) and oracle.exp_f32(1000.0) == oracle.exp_f32(88.0)
    assert oracle.exp_f32(-1000.0) == oracle.exp_f32(-86.0) > 0.0


def _silu64(g):
    g = g.astype(np.float64)
    return g / (1.0 + np.exp(-g))


def test_swiglu_matches_f64_definition():
    r = np.random.default_rng(5)
    g = (r.standard_normal((16, 512)) * 6).astype(np.float32)
    u = (r.standard_normal((16, 512)) * 3).astype(np.float32)
    y = oracle.swiglu(g, u).astype(np.float64)
    ref = _silu64(g) * u.astype(np.float64)
    scale = np.maximum(np.abs(ref), 1e-30)
    assert np.max(np.abs(y - ref) / scale) < 8 * F32_EPS


def test_silu_closed_forms_and_identities():
    ones = np.ones((1, 6), np.float32)
    g = np.array([[0.0, 100.0, 87.0, -100.0, 30.0, -30.0]], np.float32)
    y = oracle.swiglu(g, ones)[0]
    assert y[0] == 0.0                                # silu(0) = 0
    assert y[1] == 100.0 and y[2] == 87.0             # silu(g) = g in f32 for large g
    assert 0.0 >= y[3] > -1e-35                        # silu(-100) ~ -3.7e-42: ~0
    assert y[4] == 30.0                               # 1 + e^-30 rounds to 1
    assert abs(y[5] - (-30.0 * math.exp(-30.0))) < 1e-17
    # silu(x) - silu(-x) = x  (to f32 rounding)
    x = np.random.default_rng(6).uniform(-20, 20, (1, 4096)).astype(np.float32)
    d = oracle.swiglu(x, np.ones_like(x)).astype(np.float64) - oracle.swiglu(-x, np.ones_like(x)).astype(np.float64)
    assert np.max(np.abs(d - x.astype(np.float64)) / np.maximum(np.abs(x), 1.0)) < 8 * F32_EPS


def test_swiglu_is_linear_in_up_and_zero_up_gives_zero_plane():
    r = np.random.default_rng(7)
    g = r.standard_normal((4, 256)).astype(np.float32)
    u = r.standard_normal((4, 256)).astype(np.float32)
    y1 = oracle.swiglu(g, u)
    y2 = oracle.swiglu(g, 2 * u)                      # doubling u doubles y exactly (power of two)
    assert np.array_equal(y2, 2 * y1)
    q, d, S = oracle.quantize_swiglu_q8(g, np.zeros_like(u))
    assert not q.any() and not d.any() and not S.any()
    # doubling u leaves the codes and sums unchanged and doubles d (amax and d scale exactly)
    qa, da, Sa = oracle.quantize_swiglu_q8(g, u)
    qb, db, Sb = oracle.quantize_swiglu_q8(g, 2 * u)
    assert np.array_equal(qa, qb) and np.array_equal(Sa, Sb) and np.array_equal(db, 2 * da)


def test_quantize_swiglu_is_quantize_of_swiglu():
    r = np.random.default_rng(8)
    g = (r.standard_normal((3, 768)) * 4).astype(np.float32)
    u = r.standard_normal((3, 768)).astype(np.float32)
    for a, b in zip(oracle.quantize_swiglu_q8(g, u), oracle.quantize_q8(oracle.swiglu(g, u))):
        assert np.array_equal(a, b)


def _negate_d(w):
    """Q4_K bytes with d and dmin negated (fp16 sign bits): the matmul output changes sign exactly."""
    w = w.copy()
    w[..., 1] ^= 0x80
    w[..., 3] ^= 0x80
    return w


def test_gate_up_swiglu_operand_roles_and_closed_form():
    # y(G) - y(-G) = (silu(G) - silu(-G)) U = G U, so the planes of w_gate and of -w_gate differ,
    # after dequantization, by G U within the two quantization steps; swapping the roles of gate
    # and up, or dropping the f32 rounding's input, breaks it.  The plane also matches the f64
    # closed form silu(G) U within its quantization step.
    from quantized_q8_activation_quantize_gb300 import inputs
    r = np.random.default_rng(31)
    M, K, F = 4, 512, 256
    wg = inputs.q4k_weights(r, F, K)
    wu = inputs.q4k_weights(r, F, K)
    plane = oracle.quantize_q8(inputs.activations(r, M, K))
    G = oracle.matmul(wg, "q4k", plane)
    U = oracle.matmul(wu, "q4k", plane)
    assert np.array_equal(oracle.matmul(_negate_d(wg), "q4k", plane), -G)

    def deq(p):
        q, d, _ = p
        return q.reshape(M, -1, 32).astype(np.float64) * d[..., None].astype(np.float64), d

    yp, dp = deq(oracle.gate_up_swiglu_q8(wg, wu, "q4k", plane))
    yn, dn = deq(oracle.gate_up_swiglu_q8(_negate_d(wg), wu, "q4k", plane))
    GU = (G * U).reshape(M, -1, 32)
    step = (dp + dn)[..., None].astype(np.float64)
    assert np.all(np.abs((yp - yn) - GU) <= 0.5 * step * (1 + 1e-6) + 1e-6 * np.abs(GU))
    silu = G / (1 + np.exp(-G))
    ref = (silu * U).reshape(M, -1, 32)
    assert np.all(np.abs(yp - ref) <= 0.5 * dp[..., None] * (1 + 1e-6) + 1e-5 * np.abs(ref).max())
