"""Pins for the oracle's integer block dots (C5, C7) and float-scaled matmul (C6).

* Brute force: f64 dequantize(W) times the f64 dequantized Q8 plane must agree with the
  oracle's block-integer path to ~1e-12 (same sums, different order), for Q4_K, Q5_K and Q6_K.
* Against the unquantized f32 activations the error must stay within the Q8 error bound
  sum_k |W[n,k]| * d_a / 2 (catches a wrong activation-scale index).
* Exact invariants: zero weights, d/dmin doubling, token permutation, activation-scale doubling.
* C7: closed-form extremes (int32 headroom) and exact recomputation of I from decoded ints.
"""
import numpy as np
import pytest

import oracle
from quantized_q8_activation_quantize_gb300 import inputs


def _case(fmt, m, n, k, seed, scale_range=(-64, 63)):
    r = np.random.default_rng(seed)
    if fmt == "q4k":
        w = inputs.q4k_weights(r, n, k)
    elif fmt == "q5k":
        w = inputs.q5k_weights(r, n, k)
    else:
        w = inputs.q6k_weights(r, n, k, scale_range=scale_range)
    x = inputs.activations(r, m, k)
    return w, x


def _dequant_plane(q, d):
    return q.astype(np.float64) * np.repeat(d.astype(np.float64), 32, axis=1)


@pytest.mark.parametrize("fmt,m,n,k", [("q4k", 8, 16, 256), ("q4k", 5, 9, 512), ("q5k", 8, 16, 256),
                                       ("q5k", 4, 11, 512), ("q6k", 8, 16, 256), ("q6k", 3, 7, 512)])
def test_brute_force_dequantized_matmul(fmt, m, n, k):
    w, x = _case(fmt, m, n, k, seed=100 + m + n)
    plane = oracle.quantize_q8(x)
    y = oracle.matmul(w, fmt, plane)
    ref = _dequant_plane(plane[0], plane[1]) @ oracle.dequantize(w, fmt).T
    scale = np.linalg.norm(ref, axis=1, keepdims=True)
    assert np.abs(y - ref).max() <= 1e-12 * scale.max()


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
def test_q8_error_bound_against_unquantized_activations(fmt):
    w, x = _case(fmt, 6, 12, 512, seed=5)
    q, d, S = oracle.quantize_q8(x)
    y = oracle.matmul(w, fmt, (q, d, S))
    W = oracle.dequantize(w, fmt)
    exact = x.astype(np.float64) @ W.T
    bound = (np.abs(W)[None, :, :] * np.repeat(d.astype(np.float64), 32, axis=1)[:, None, :] / 2).sum(-1)
    assert (np.abs(y - exact) <= bound * (1 + 1e-6) + 1e-12).all()
    # and the bound is not vacuous: the error is far below |y|
    assert np.abs(y - exact).max() < 0.05 * np.abs(exact).max()


def test_q4k_zero_weights_give_zero():
    w, x = _case("q4k", 4, 6, 512, seed=6)
    plane = oracle.quantize_q8(x)
    z = w.copy()
    z[..., 0:4] = 0                                   # d = dmin = 0
    assert (oracle.matmul(z, "q4k", plane) == 0).all()
    z = w.copy()
    z[..., 16:] = 0                                   # all quants 0 ...
    z[..., 4:16] = 0                                  # ... and all scales/mins 0
    assert (oracle.matmul(z, "q4k", plane) == 0).all()
    z = w.copy()
    z[..., 16:] = 0                                   # quants 0 with non-zero scales ...
    z[..., 8:12] = 0                                  # ... and the min fields cleared:
    z[..., 12:16] &= 0x0F                             # m0..3 and the min nibbles of m4..7
    _, _, sc, mn, _ = oracle.q4k_fields(z[0, 0])
    assert (mn == 0).all() and (sc > 0).any()
    assert (oracle.matmul(z, "q4k", plane) == 0).all()


def test_q6k_zero_weights_give_zero():
    w, x = _case("q6k", 4, 6, 512, seed=7)
    plane = oracle.quantize_q8(x)
    z = w.copy()
    z[..., 0:128] = 0                                 # low bits 0
    z[..., 128:192] = 0xAA                            # high bit pairs 2 -> q = 32 - 32 = 0
    assert (oracle.matmul(z, "q6k", plane) == 0).all()
    z = w.copy()
    z[..., 208:210] = 0                               # d = 0
    assert (oracle.matmul(z, "q6k", plane) == 0).all()


def _set_half(w, off, value):
    w[..., off:off + 2] = np.array([value], dtype="<f2").view(np.uint8)


def test_q4k_d_and_dmin_are_linear():
    w, x = _case("q4k", 4, 8, 512, seed=8)
    plane = oracle.quantize_q8(x)
    # dmin = 0: doubling d (exact in fp16) doubles Y exactly
    a = w.copy()
    _set_half(a, 2, 0.0)
    b = a.copy()
    b[..., 0:2] = (a[..., 0:2].copy().view("<f2") * 2).view(np.uint8)
    assert np.array_equal(oracle.matmul(b, "q4k", plane), 2 * oracle.matmul(a, "q4k", plane))
    # d = 0: doubling dmin doubles Y exactly
    a = w.copy()
    _set_half(a, 0, 0.0)
    b = a.copy()
    b[..., 2:4] = (a[..., 2:4].copy().view("<f2") * 2).view(np.uint8)
    ya = oracle.matmul(a, "q4k", plane)
    assert np.array_equal(oracle.matmul(b, "q4k", plane), 2 * ya) and np.abs(ya).max() > 0


def test_q6k_d_is_linear():
    w, x = _case("q6k", 4, 8, 512, seed=9)
    plane = oracle.quantize_q8(x)
    b = w.copy()
    b[..., 208:210] = (w[..., 208:210].copy().view("<f2") * 2).view(np.uint8)
    assert np.array_equal(oracle.matmul(b, "q6k", plane), 2 * oracle.matmul(w, "q6k", plane))


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
def test_token_permutation_and_index_lists(fmt):
    w, x = _case(fmt, 7, 10, 512, seed=10)
    plane = oracle.quantize_q8(x)
    y = oracle.matmul(w, fmt, plane)
    perm = np.random.default_rng(1).permutation(7)
    yp = oracle.matmul(w, fmt, oracle.quantize_q8(x[perm]))
    assert np.array_equal(yp, y[perm])
    ms, ns = np.array([6, 0, 3]), np.array([9, 2])
    assert np.array_equal(oracle.matmul(w, fmt, plane, ms, ns), y[np.ix_(ms, ns)])
    assert np.array_equal(oracle.matmul(w, fmt, plane, threads=3), y)


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
def test_activation_scale_doubling(fmt):
    w, x = _case(fmt, 3, 5, 256, seed=11)
    q, d, S = oracle.quantize_q8(x)
    assert np.array_equal(oracle.matmul(w, fmt, (q, 2 * d, S)), 2 * oracle.matmul(w, fmt, (q, d, S)))


def test_q4k_blockdot_extremes():
    b = np.zeros((1, 1, 144), np.uint8)
    b[..., 16:] = 0xFF                                # q = 15 everywhere
    b[..., 4:16] = 0xFF                               # every 6-bit field = 63
    qa = np.full((1, 256), 127, np.int8)
    I, D = oracle.blockdots(b, "q4k", qa)
    assert (D == 15 * 127 * 32).all() and (I == 63 * 15 * 127 * 32).all()


def test_q6k_blockdot_extremes():
    b = np.zeros((1, 1, 210), np.uint8)               # q = -32 everywhere
    b[..., 192:208] = 0x80                            # sc = -128
    qa = np.full((1, 256), -127, np.int8)
    I, D = oracle.blockdots(b, "q6k", qa)
    assert (D == 32 * 127 * 16).all() and (I == -128 * 32 * 127 * 16 * 2).all()
    assert I.min() > np.iinfo(np.int32).min
    b[..., 0:128] = 0xFF
    b[..., 128:192] = 0xFF                            # q = 31 everywhere
    b[..., 192:208] = 127
    I, D = oracle.blockdots(b, "q6k", np.full((1, 256), 127, np.int8))
    assert (I == 127 * 31 * 127 * 16 * 2).all()


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
def test_blockdots_recomputed_from_decoded_integers(fmt):
    w, x = _case(fmt, 3, 4, 512, seed=12, scale_range=(-128, 127))
    q, d, S = oracle.quantize_q8(x)
    I, D = oracle.blockdots(w, fmt, q)
    for n in range(4):
        for sb in range(2):
            if fmt in ("q4k", "q5k"):
                _, _, sc, _, qw = (oracle.q4k_fields if fmt == "q4k" else oracle.q5k_fields)(w[n, sb])
                scb = sc
            else:
                _, sc, qw = oracle.q6k_fields(w[n, sb])
            for m in range(3):
                a = q[m, 256 * sb:256 * sb + 256].astype(np.int64)
                for j in range(8):
                    seg = slice(32 * j, 32 * j + 32)
                    if fmt in ("q4k", "q5k"):
                        ref = scb[j] * int((qw[seg] * a[seg]).sum())
                    else:
                        lo, hi = slice(32 * j, 32 * j + 16), slice(32 * j + 16, 32 * j + 32)
                        ref = sc[2 * j] * int((qw[lo] * a[lo]).sum()) + sc[2 * j + 1] * int((qw[hi] * a[hi]).sum())
                    assert I[m, n, 8 * sb + j] == ref


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
def test_matmul_is_scaled_sum_of_blockdots(fmt):
    # ties C6 to C7: Y = sum_b d_w * da * I (minus the Q4_K min term)
    w, x = _case(fmt, 3, 5, 512, seed=13)
    q, d, S = oracle.quantize_q8(x)
    I, _ = oracle.blockdots(w, fmt, q)
    y = oracle.matmul(w, fmt, (q, d, S))
    for n in range(5):
        for m in range(3):
            acc = 0.0
            for sb in range(2):
                if fmt in ("q4k", "q5k"):
                    dw, dmw, _, mn, _ = (oracle.q4k_fields if fmt == "q4k" else oracle.q5k_fields)(w[n, sb])
                else:
                    dw, _, _ = oracle.q6k_fields(w[n, sb])
                for j in range(8):
                    b = 8 * sb + j
                    acc += dw * float(d[m, b]) * I[m, n, b]
                    if fmt in ("q4k", "q5k"):
                        acc -= dmw * mn[j] * float(d[m, b]) * S[m, b]
            assert abs(acc - y[m, n]) <= 1e-12 * max(1.0, abs(y[m, n]))


def test_q5k_blockdot_extremes():
    b = np.zeros((1, 1, 176), np.uint8)
    b[..., 16:] = 0xFF                                # qh and qs all ones: q = 31 everywhere
    b[..., 4:16] = 0xFF                               # every 6-bit field = 63
    qa = np.full((1, 256), 127, np.int8)
    I, D = oracle.blockdots(b, "q5k", qa)
    assert (D == 31 * 127 * 32).all() and (I == 63 * 31 * 127 * 32).all()
    assert 63 * 31 * 127 * 32 < 2 ** 24                # exact in f32 as well


def test_q5k_d_and_dmin_are_linear():
    w, x = _case("q5k", 4, 8, 512, seed=14)
    plane = oracle.quantize_q8(x)
    a = w.copy()
    a[..., 2:4] = 0                                   # dmin = 0
    b = a.copy()
    b[..., 0:2] = (a[..., 0:2].copy().view("<f2") * 2).view(np.uint8)
    assert np.array_equal(oracle.matmul(b, "q5k", plane), 2 * oracle.matmul(a, "q5k", plane))
    a = w.copy()
    a[..., 0:2] = 0                                   # d = 0: only the min term is left
    b = a.copy()
    b[..., 2:4] = (a[..., 2:4].copy().view("<f2") * 2).view(np.uint8)
    ya = oracle.matmul(a, "q5k", plane)
    assert np.array_equal(oracle.matmul(b, "q5k", plane), 2 * ya) and np.abs(ya).max() > 0


B32_FMTS = ["q4_0", "q4_1", "q5_0", "q5_1", "q8_0"]


@pytest.mark.parametrize("fmt", B32_FMTS)
@pytest.mark.parametrize("m,n,k", [(8, 16, 256), (3, 7, 512)])
def test_b32_brute_force_dequantized_matmul(fmt, m, n, k):
    r = np.random.default_rng(200 + m + n)
    w = inputs.b32_weights(r, n, k, fmt)
    x = inputs.activations(r, m, k)
    plane = oracle.quantize_q8(x)
    y = oracle.matmul(w, fmt, plane)
    ref = _dequant_plane(plane[0], plane[1]) @ oracle.dequantize(w, fmt).T
    scale = np.linalg.norm(ref, axis=1, keepdims=True)
    assert np.abs(y - ref).max() <= 1e-12 * scale.max()


@pytest.mark.parametrize("fmt", B32_FMTS)
def test_b32_blockdots_recomputed_and_matmul_is_their_scaled_sum(fmt):
    r = np.random.default_rng(21)
    w = inputs.b32_weights(r, 4, 256, fmt)
    x = inputs.activations(r, 3, 256)
    q, d, S = oracle.quantize_q8(x)
    I, _ = oracle.blockdots(w, fmt, q)
    y = oracle.matmul(w, fmt, (q, d, S))
    for n in range(4):
        for mm in range(3):
            acc = 0.0
            for b in range(8):
                dw, mw, iq = oracle.b32_fields(w[n, b], fmt)
                a = q[mm, 32 * b:32 * b + 32].astype(np.int64)
                assert I[mm, n, b] == int((iq * a).sum())
                acc += dw * float(d[mm, b]) * I[mm, n, b] + mw * float(d[mm, b]) * S[mm, b]
            assert abs(acc - y[mm, n]) <= 1e-12 * max(1.0, abs(y[mm, n]))


@pytest.mark.parametrize("fmt", B32_FMTS)
def test_b32_d_and_m_are_linear(fmt):
    r = np.random.default_rng(22)
    w = inputs.b32_weights(r, 5, 512, fmt)
    plane = oracle.quantize_q8(inputs.activations(r, 4, 512))
    a = w.copy()
    if fmt in ("q4_1", "q5_1"):
        a[..., 2:4] = 0                               # m = 0
    b = a.copy()
    b[..., 0:2] = (a[..., 0:2].copy().view("<f2") * 2).view(np.uint8)
    assert np.array_equal(oracle.matmul(b, fmt, plane), 2 * oracle.matmul(a, fmt, plane))
    if fmt in ("q4_1", "q5_1"):
        a = w.copy()
        a[..., 0:2] = 0                               # d = 0: only the offset term is left
        b = a.copy()
        b[..., 2:4] = (a[..., 2:4].copy().view("<f2") * 2).view(np.uint8)
        ya = oracle.matmul(a, fmt, plane)
        assert np.array_equal(oracle.matmul(b, fmt, plane), 2 * ya) and np.abs(ya).max() > 0


def test_b32_blockdot_extremes():
    qa = np.full((1, 32), -128 + 1, np.int8)          # codes at -127
    b = np.zeros((1, 1, 34), np.uint8)
    b[..., 2:] = 0x80                                 # Q8_0 q = -128 everywhere
    I, _ = oracle.blockdots(b, "q8_0", qa)
    assert (I == 128 * 127 * 32).all()
    b = np.zeros((1, 1, 24), np.uint8)
    b[..., 4:] = 0xFF                                 # Q5_1 q = 31 everywhere
    I, _ = oracle.blockdots(b, "q5_1", np.full((1, 32), 127, np.int8))
    assert (I == 31 * 127 * 32).all()
