"""Host model of the RMSNorm producer's f32 evaluation of r = 1/sqrt(mean(x^2) + eps).

The kernel (csrc/mq_quantize.cu, rms_scale_from_pair) sums squares as compensated f32 pairs per
lane, adds the lanes' pairs as f32 pairs, forms t/K + eps as an f32 pair, takes one Newton step
on an rsqrtf estimate and accepts the rounding only when the whole window of 2^-38 around its
estimate rounds to one f32; otherwise it evaluates r in f64.  This replays those steps with
numpy float32 arithmetic (every operation rounded to nearest; the fused multiply-adds through an
exact f64 product, and the rsqrtf estimate perturbed by up to 2 ulp) and checks the two facts the
kernel relies on: the estimate stays within 2^-41 of the f64 evaluation of the same pairs, and an
accepted r always equals that evaluation's rounding.  No GPU, no oracle.
"""
import numpy as np

f32 = np.float32


def _fma(a, b, c):
    return (a.astype(np.float64) * b.astype(np.float64) + c.astype(np.float64)).astype(f32)


def _two_sum(a, b):
    s = a + b
    bv = s - a
    return s, (a - (s - bv)) + (b - bv)


def _pair_add(ah, al, bh, bl):
    s, e = _two_sum(ah, bh)
    e = e + (al + bl)
    h = s + e
    return h, e - (h - s)


def _add_square(v, hi, lo):
    p = v * v
    e = _fma(v, v, -p)
    s = hi + p
    bv = s - hi
    err = (hi - (s - bv)) + (p - bv)
    return s, lo + (err + e)


def test_f32_scale_matches_f64_rounding():
    rng = np.random.default_rng(5)
    T, K = 2000, 3584
    eps = f32(1e-6)
    x = (rng.standard_normal((T, K)) * rng.uniform(0.01, 10, (T, 1))).astype(f32)
    xl = x.reshape(T, K // 256, 32, 8)
    z = np.zeros((T, 32), f32)
    hi0, lo0, hi1, lo1 = z.copy(), z.copy(), z.copy(), z.copy()
    with np.errstate(over="ignore", invalid="ignore"):
        for c in range(K // 256):
            for j in range(8):
                if j % 2 == 0:
                    hi0, lo0 = _add_square(xl[:, c, :, j], hi0, lo0)
                else:
                    hi1, lo1 = _add_square(xl[:, c, :, j], hi1, lo1)
        # the f64 evaluation of the same lane pairs (the kernel's fallback)
        t = (hi0.astype(np.float64) + lo0) + (hi1.astype(np.float64) + lo1)
        for o in (16, 8, 4, 2, 1):
            t = t + t[:, np.arange(32) ^ o]
        y64 = 1.0 / np.sqrt(t[:, 0] / K + np.float64(eps))
        r64 = y64.astype(f32)
        # the f32 evaluation
        th, tl = _pair_add(hi0, lo0, hi1, lo1)
        for o in (16, 8, 4, 2, 1):
            idx = np.arange(32) ^ o
            th, tl = _pair_add(th, tl, th[:, idx], tl[:, idx])
        assert (th == th[:, :1]).all() and (tl == tl[:, :1]).all()      # every lane holds the same pair
        th, tl = th[:, 0], tl[:, 0]
        kf, ik = f32(K), f32(1.0 / K)
        qh = th * ik
        rem = _fma(-qh, np.full_like(qh, kf), th)
        ql = (rem + tl) * ik
        vh, vl = _two_sum(qh, np.full_like(qh, eps))
        vl = vl + ql
        y0 = (1.0 / np.sqrt(vh.astype(np.float64) + vl)).astype(f32)
        y0 = (y0 + np.spacing(y0) * rng.integers(-2, 3, T).astype(f32)).astype(f32)
        p = y0 * y0
        pe = _fma(y0, y0, -p)
        a = _fma(-vh, p, np.ones_like(p))
        c = a - _fma(vh, pe, vl * p)
        yl = (f32(0.5) * y0) * c
        dl = y0 * f32(2.0 ** -38)
        ra, rb = y0 + (yl - dl), y0 + (yl + dl)
    err = np.abs((y0.astype(np.float64) + yl) / y64 - 1)
    assert err.max() < 2.0 ** -41
    ok = ra == rb
    assert ok.mean() > 0.999                     # the f64 path is the rare exception
    assert np.array_equal(ra[ok], r64[ok])
