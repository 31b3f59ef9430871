/*
 * mq_oracle.c -- plain, slow CPU oracle for the Q4_K / Q6_K x Q8 matmul path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (sources: the minfer pages -- "minfer" book print view,
 * sections "Features > GPU -- CUDA" (int8 MMQ over raw Q4_K/Q6_K nibbles with
 * producer-fused Q8 activation quantization) and "Support Matrix > Supported
 * Quantization Formats" (CPU quantizes activations on the fly; Q8_K carries
 * precomputed per-sub-block sums); "Architecture > 6. Quantization & Tensor
 * Layout" (blocks are the GGML ggml-common.h structs); "Architecture > 4.5
 * Core invariants" item 3 (weights [out][in] row-major, activations
 * token-major); "Compute Graph Design > 3.1" (RmsNorm{eps})):
 *
 *   C1  Q4_K super-block decode (GGML layout, 144 bytes)
 *   C1' Q5_K super-block decode (GGML layout, 176 bytes): Q4_K's scales, mins and
 *       nibbles plus one high bit per value ("Support Matrix > CUDA notes": decode
 *       uses the dp4a MMVQ kernels for Q4_K/Q5_K/Q6_K; "Architecture > 6" item on
 *       block layouts: Q4_K/Q5_K/Q6_K are 256-value super-blocks)
 *   C2  Q6_K super-block decode (GGML layout, 210 bytes)
 *   C9  32-value block formats Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 (GGML layouts, 18 / 20 /
 *       22 / 24 / 34 bytes; "Architecture > 6. Quantization & Tensor Layout": the weight
 *       blocks are the GGML structs, these five holding 32 values each) and their block dots
 *   C3  Q8 activation quantization, blocks of 32, round half away from zero
 *   C4  RMSNorm producer y = (x * r) * w,  r = 1/sqrt(mean(x^2) + eps)
 *   C5  integer block dots between decoded weight quants and Q8 codes
 *   C6  float scaling of the block dots into f32 outputs (accumulated in f64)
 *   C7  the per-(token, row, 32-block) integer checkpoint I
 *   C8  SwiGLU producer y = silu(g) * u, silu(g) = g / (1 + exp(-g)), then C3 on y
 *       ("Features > GPU -- CUDA": the swiglu producer emits the q8 plane directly;
 *       "Compute Graph Design > 5": Mul(Silu(X), Y) is rewritten to SwiGLU)
 *
 * The byte layouts are not printed on the pages; they are the public GGML
 * k-quant formats that the pages name.  Rounding of Q8 is half away from zero
 * (C roundf), with d = amax/127 and q = round(x * (1/d)) in IEEE f32.
 *
 * Pins (tests/test_oracle_*.py): hand-built blocks with hand-derived values
 * (tests/golden/), one-hot position maps, numpy's float16 for the fp16 decode,
 * closed forms and exact scaling invariants of C3/C4, dequantize-then-matmul
 * brute force for C5/C6, exact integer recomputation for C7.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared (see build_oracle.py).
 * No FMA contraction, no fast-math: every f32 step rounds once.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OQ_QK 256
#define OQ_Q8 32

/* ---------------------------------------------------------------- fp16 --- */

/* IEEE 754 binary16 -> double, from the format's definition (exact). */
double oq_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                    /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);        /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ----------------------------------------------------------------- C1 --- */

/*
 * Q4_K: bytes [0,2) d, [2,4) dmin, [4,16) scales[12], [16,144) qs[128].
 * Sub-block j (0..7) holds elements 32j..32j+31 with a 6-bit scale sc_j and a
 * 6-bit min m_j.  j < 4: sc = s[j] & 63, m = s[j+4] & 63.  j >= 4: the low
 * four bits come from s[j+4] (sc: low nibble, m: high nibble) and the top two
 * bits from the top two bits of s[j-4] (sc) and s[j] (m).  Element 32j + l
 * is the low nibble of qs[32*(j/2) + l] for even j, the high nibble for odd j.
 * value = d * sc_j * q - dmin * m_j.
 */
void oq_q4k_fields(const uint8_t *blk, double *d, double *dmin,
                   int32_t sc[8], int32_t mn[8], int32_t q[256])
{
    const uint8_t *s = blk + 4;
    const uint8_t *qs = blk + 16;
    *d = oq_half_to_double(rd16(blk));
    *dmin = oq_half_to_double(rd16(blk + 2));
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            mn[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
    for (int j = 0; j < 8; ++j) {
        for (int l = 0; l < 32; ++l) {
            uint8_t b = qs[32 * (j / 2) + l];
            q[32 * j + l] = (j % 2 == 0) ? (b & 15) : (b >> 4);
        }
    }
}

/* ---------------------------------------------------------------- C1' --- */

/*
 * Q5_K: bytes [0,2) d, [2,4) dmin, [4,16) scales[12] (packed exactly as Q4_K's),
 * [16,48) qh[32], [48,176) qs[128].  Element 32j + l of sub-block j (0..7) takes the
 * Q4_K nibble of qs (low nibble of qs[32*(j/2) + l] for even j, high for odd j) as its
 * low four bits and bit j of qh[l] as its fifth: q = nibble + 16 * ((qh[l] >> j) & 1),
 * q in [0, 31].  value = d * sc_j * q - dmin * m_j.
 */
void oq_q5k_fields(const uint8_t *blk, double *d, double *dmin,
                   int32_t sc[8], int32_t mn[8], int32_t q[256])
{
    const uint8_t *s = blk + 4;
    const uint8_t *qh = blk + 16;
    const uint8_t *qs = blk + 48;
    *d = oq_half_to_double(rd16(blk));
    *dmin = oq_half_to_double(rd16(blk + 2));
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            mn[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
    for (int j = 0; j < 8; ++j) {
        for (int l = 0; l < 32; ++l) {
            uint8_t b = qs[32 * (j / 2) + l];
            int nib = (j % 2 == 0) ? (b & 15) : (b >> 4);
            q[32 * j + l] = nib + 16 * ((qh[l] >> j) & 1);
        }
    }
}

/* ----------------------------------------------------------------- C2 --- */

/*
 * Q6_K: bytes [0,128) ql, [128,192) qh, [192,208) scales[16] (int8), [208,210) d.
 * Half h (0, 1) covers elements 128h..128h+127 and uses ql + 64h, qh + 32h.
 * For l in 0..31 with hb = qh[32h + l]:
 *   element 128h + l      : low  nibble of ql[64h + l],      bits (hb >> 0) & 3
 *   element 128h + l + 32 : low  nibble of ql[64h + l + 32], bits (hb >> 2) & 3
 *   element 128h + l + 64 : high nibble of ql[64h + l],      bits (hb >> 4) & 3
 *   element 128h + l + 96 : high nibble of ql[64h + l + 32], bits (hb >> 6) & 3
 * q = (low | high << 4) - 32 in [-32, 31]; element e uses scales[e / 16].
 * value = d * sc * q.
 */
void oq_q6k_fields(const uint8_t *blk, double *d, int32_t sc[16], int32_t q[256])
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *s = (const int8_t *)(blk + 192);
    *d = oq_half_to_double(rd16(blk + 208));
    for (int i = 0; i < 16; ++i) sc[i] = s[i];
    for (int h = 0; h < 2; ++h) {
        for (int l = 0; l < 32; ++l) {
            int hb = qh[32 * h + l];
            int lo0 = ql[64 * h + l] & 15, lo1 = ql[64 * h + l + 32] & 15;
            int hi0 = ql[64 * h + l] >> 4, hi1 = ql[64 * h + l + 32] >> 4;
            q[128 * h + l]      = (lo0 | (((hb >> 0) & 3) << 4)) - 32;
            q[128 * h + l + 32] = (lo1 | (((hb >> 2) & 3) << 4)) - 32;
            q[128 * h + l + 64] = (hi0 | (((hb >> 4) & 3) << 4)) - 32;
            q[128 * h + l + 96] = (hi1 | (((hb >> 6) & 3) << 4)) - 32;
        }
    }
}

/* Dequantize n_rows rows of K values each into out[n_rows][K] (f64, exact products). */
void oq_q4k_dequant(const uint8_t *w, int64_t n_rows, int64_t K, double *out)
{
    int64_t nb = K / OQ_QK;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double d, dmin;
            int32_t sc[8], mn[8], q[256];
            oq_q4k_fields(w + (r * nb + b) * 144, &d, &dmin, sc, mn, q);
            for (int e = 0; e < 256; ++e)
                out[r * K + b * 256 + e] = d * sc[e / 32] * q[e] - dmin * mn[e / 32];
        }
}

void oq_q5k_dequant(const uint8_t *w, int64_t n_rows, int64_t K, double *out)
{
    int64_t nb = K / OQ_QK;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double d, dmin;
            int32_t sc[8], mn[8], q[256];
            oq_q5k_fields(w + (r * nb + b) * 176, &d, &dmin, sc, mn, q);
            for (int e = 0; e < 256; ++e)
                out[r * K + b * 256 + e] = d * sc[e / 32] * q[e] - dmin * mn[e / 32];
        }
}

void oq_q6k_dequant(const uint8_t *w, int64_t n_rows, int64_t K, double *out)
{
    int64_t nb = K / OQ_QK;
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double d;
            int32_t sc[16], q[256];
            oq_q6k_fields(w + (r * nb + b) * 210, &d, sc, q);
            for (int e = 0; e < 256; ++e)
                out[r * K + b * 256 + e] = d * sc[e / 16] * q[e];
        }
}

/* ----------------------------------------------------------------- C4 --- */

/*
 * RMSNorm producer: ms = (sum x^2) / K accumulated in f64 (each x^2 is exact
 * in f64), r = (float)(1 / sqrt(ms + (double)eps)), y = fl32(fl32(x * r) * w).
 */
void oq_rmsnorm(const float *x, int64_t M, int64_t K, const float *w, float eps, float *y)
{
    for (int64_t m = 0; m < M; ++m) {
        const float *xr = x + m * K;
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) ss += (double)xr[k] * (double)xr[k];
        double ms = ss / (double)K;
        float r = (float)(1.0 / sqrt(ms + (double)eps));
        for (int64_t k = 0; k < K; ++k) {
            float t = xr[k] * r;
            y[m * K + k] = t * w[k];
        }
    }
}

/* ----------------------------------------------------------------- C3 --- */

/*
 * Q8 quantization of x[M][K] in blocks of 32 along K:
 *   amax = max |x|,  d = amax / 127 (f32 divide),  id = d ? 1/d : 0 (f32),
 *   q = clamp(roundf(x * id), -127, 127)  (roundf: half away from zero),
 *   S = sum q (int32).
 * Outputs in the oracle's own logical layout: q[M][K], d[M][K/32], S[M][K/32].
 */
/*
 * C8: the pages fix no precision for SwiGLU.  The reading used on both sides: IEEE f32,
 * every step rounded once, and exp(x) evaluated by the textbook reduction written out
 * here -- x = k ln2 + r with k = nearest integer to x / ln2 (ties to even) and
 * |r| <= ln2 / 2, exp(r) by its Taylor series through r^7 (truncation error below
 * 6e-9 relative), times 2^k -- so that the f32 value of y, and with it every Q8 code,
 * is one fixed function of (g, u).  x is clamped to [-86, 88] (exp stays a normal f32;
 * silu(g) is unaffected in f32 beyond that range: 1 + exp(-86) == 1, and for g < -88
 * the result is below 1e-36).
 */
float oq_exp_f32(float x)
{
    if (x > 88.0f) x = 88.0f;
    if (x < -86.0f) x = -86.0f;
    const float k = rintf(x * 1.44269504f);                 /* 1 / ln2 */
    float r = fmaf(-k, 0.693145751953125f, x);               /* ln2, high part (k * hi is exact) */
    r = fmaf(-k, 1.42860677e-06f, r);                        /* ln2, low part */
    float p = 1.98412698e-04f;                               /* 1/7! */
    p = fmaf(p, r, 1.38888889e-03f);                         /* 1/6! */
    p = fmaf(p, r, 8.33333333e-03f);                         /* 1/5! */
    p = fmaf(p, r, 4.16666667e-02f);                         /* 1/4! */
    p = fmaf(p, r, 1.66666667e-01f);                         /* 1/3! */
    p = fmaf(p, r, 0.5f);                                    /* 1/2! */
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    return ldexpf(p, (int)k);
}

void oq_swiglu(const float *g, const float *u, int64_t M, int64_t K, float *y)
{
    for (int64_t i = 0; i < M * K; ++i) {
        const float e = oq_exp_f32(-g[i]);
        const float den = 1.0f + e;
        const float s = g[i] / den;                          /* silu(g) */
        y[i] = s * u[i];
    }
}

void oq_quantize_q8(const float *x, int64_t M, int64_t K, int8_t *q, float *d, int32_t *S)
{
    int64_t nblk = K / OQ_Q8;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nblk; ++b) {
            const float *xb = x + m * K + b * OQ_Q8;
            float amax = 0.0f;
            for (int i = 0; i < OQ_Q8; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float db = amax / 127.0f;
            float id = (db != 0.0f) ? 1.0f / db : 0.0f;
            int32_t s = 0;
            for (int i = 0; i < OQ_Q8; ++i) {
                float v = xb[i] * id;
                float rq = roundf(v);
                if (rq > 127.0f) rq = 127.0f;
                if (rq < -127.0f) rq = -127.0f;
                int8_t qi = (int8_t)rq;
                q[m * K + b * OQ_Q8 + i] = qi;
                s += qi;
            }
            d[m * nblk + b] = db;
            S[m * nblk + b] = s;
        }
}

/* -------------------------------------------------------------- C5, C7 --- */

/* the decoder of a Q4_K-style super-block: d, dmin, sc[8], m[8], q[256] */
typedef void (*oq_kfields_fn)(const uint8_t *, double *, double *, int32_t *, int32_t *, int32_t *);

/*
 * Integer checkpoint for the (token, row) pairs (ms[i], ns[j]).
 * Q4_K / Q5_K, 32-block b of the row (sub-block j = b % 8 of super-block b / 8):
 *   D[b] = sum_{l<32} q_w[32b + l] * q_a[32b + l],   I[b] = sc_j * D[b].
 * Output I and D as [nm][nn][K/32].
 */
static void kq_blockdots(oq_kfields_fn fields, int bytes, const uint8_t *w, int64_t K, const int8_t *qa,
                         const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, int32_t *I, int32_t *D)
{
    int64_t nb = K / OQ_QK, nblk = K / OQ_Q8;
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    int32_t *scw = (int32_t *)malloc(sizeof(int32_t) * nblk);
    for (int64_t jn = 0; jn < nn; ++jn) {
        int64_t n = ns[jn];
        for (int64_t b = 0; b < nb; ++b) {
            double dd, dm;
            int32_t sc[8], mn[8];
            fields(w + (n * nb + b) * bytes, &dd, &dm, sc, mn, qw + b * 256);
            for (int j = 0; j < 8; ++j) scw[b * 8 + j] = sc[j];
        }
        for (int64_t im = 0; im < nm; ++im) {
            const int8_t *a = qa + ms[im] * K;
            for (int64_t blk = 0; blk < nblk; ++blk) {
                int32_t dot = 0;
                for (int l = 0; l < OQ_Q8; ++l) dot += qw[blk * OQ_Q8 + l] * (int32_t)a[blk * OQ_Q8 + l];
                D[(im * nn + jn) * nblk + blk] = dot;
                I[(im * nn + jn) * nblk + blk] = scw[blk] * dot;
            }
        }
    }
    free(qw);
    free(scw);
}

void oq_q4k_blockdots(const uint8_t *w, int64_t N, int64_t K, const int8_t *qa, int64_t M,
                      const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn,
                      int32_t *I, int32_t *D)
{
    (void)N; (void)M;
    kq_blockdots(oq_q4k_fields, 144, w, K, qa, ms, nm, ns, nn, I, D);
}

void oq_q5k_blockdots(const uint8_t *w, int64_t N, int64_t K, const int8_t *qa, int64_t M,
                      const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn,
                      int32_t *I, int32_t *D)
{
    (void)N; (void)M;
    kq_blockdots(oq_q5k_fields, 176, w, K, qa, ms, nm, ns, nn, I, D);
}

/*
 * Q6_K: the 32-block b covers the 16-element sub-blocks s0 = 2b and s1 = 2b + 1
 * (row-global numbering; scales[s % 16] of super-block s / 16):
 *   D[b][t] = sum_{l<16} q_w[16 s_t + l] * q_a[16 s_t + l],
 *   I[b] = sc_{s0} * D[b][0] + sc_{s1} * D[b][1].
 * Output I as [nm][nn][K/32] and D as [nm][nn][K/32][2].
 */
void oq_q6k_blockdots(const uint8_t *w, int64_t N, int64_t K, const int8_t *qa, int64_t M,
                      const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn,
                      int32_t *I, int32_t *D)
{
    (void)N; (void)M;
    int64_t nb = K / OQ_QK, nblk = K / OQ_Q8;
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    int32_t *scw = (int32_t *)malloc(sizeof(int32_t) * (K / 16));
    for (int64_t jn = 0; jn < nn; ++jn) {
        int64_t n = ns[jn];
        for (int64_t b = 0; b < nb; ++b) {
            double dd;
            oq_q6k_fields(w + (n * nb + b) * 210, &dd, scw + b * 16, qw + b * 256);
        }
        for (int64_t im = 0; im < nm; ++im) {
            const int8_t *a = qa + ms[im] * K;
            for (int64_t blk = 0; blk < nblk; ++blk) {
                int32_t acc = 0;
                for (int t = 0; t < 2; ++t) {
                    int64_t s = 2 * blk + t;
                    int32_t dot = 0;
                    for (int l = 0; l < 16; ++l) dot += qw[s * 16 + l] * (int32_t)a[s * 16 + l];
                    D[((im * nn + jn) * nblk + blk) * 2 + t] = dot;
                    acc += scw[s] * dot;
                }
                I[(im * nn + jn) * nblk + blk] = acc;
            }
        }
    }
    free(qw);
    free(scw);
}

/* ----------------------------------------------------------------- C6 --- */

/*
 * Y[ms[i]][ns[j]] for the listed pairs, accumulated in f64:
 *   Q4_K / Q5_K: sum over super-blocks of
 *         d * sum_j sc_j * da[m][j] * D_j  -  dmin * sum_j m_j * da[m][j] * S[m][j]
 *   (the min term uses the integer activation sum S of the Q8 block, as Q8_K's
 *    precomputed sums do).  Output y[nm][nn] (f64).
 */
static void kq_matmul(oq_kfields_fn fields, int bytes, const uint8_t *w, int64_t K,
                      const int8_t *qa, const float *da, const int32_t *Sa,
                      const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, double *y)
{
    int64_t nb = K / OQ_QK, nblk = K / OQ_Q8;
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    int32_t *scw = (int32_t *)malloc(sizeof(int32_t) * nblk);
    int32_t *mnw = (int32_t *)malloc(sizeof(int32_t) * nblk);
    double *dw = (double *)malloc(sizeof(double) * nb);
    double *dmw = (double *)malloc(sizeof(double) * nb);
    for (int64_t jn = 0; jn < nn; ++jn) {
        int64_t n = ns[jn];
        for (int64_t b = 0; b < nb; ++b) {
            int32_t sc[8], mn[8];
            fields(w + (n * nb + b) * bytes, &dw[b], &dmw[b], sc, mn, qw + b * 256);
            for (int j = 0; j < 8; ++j) { scw[b * 8 + j] = sc[j]; mnw[b * 8 + j] = mn[j]; }
        }
        for (int64_t im = 0; im < nm; ++im) {
            int64_t m = ms[im];
            const int8_t *a = qa + m * K;
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double main_part = 0.0, min_part = 0.0;
                for (int j = 0; j < 8; ++j) {
                    int64_t blk = b * 8 + j;
                    int64_t dot = 0;
                    for (int l = 0; l < OQ_Q8; ++l) dot += (int64_t)qw[blk * OQ_Q8 + l] * a[blk * OQ_Q8 + l];
                    double dab = (double)da[m * nblk + blk];
                    main_part += (double)scw[blk] * dab * (double)dot;
                    min_part += (double)mnw[blk] * dab * (double)Sa[m * nblk + blk];
                }
                acc += dw[b] * main_part - dmw[b] * min_part;
            }
            y[im * nn + jn] = acc;
        }
    }
    free(qw); free(scw); free(mnw); free(dw); free(dmw);
}

void oq_q4k_matmul(const uint8_t *w, int64_t N, int64_t K,
                   const int8_t *qa, const float *da, const int32_t *Sa, int64_t M,
                   const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, double *y)
{
    (void)N; (void)M;
    kq_matmul(oq_q4k_fields, 144, w, K, qa, da, Sa, ms, nm, ns, nn, y);
}

void oq_q5k_matmul(const uint8_t *w, int64_t N, int64_t K,
                   const int8_t *qa, const float *da, const int32_t *Sa, int64_t M,
                   const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, double *y)
{
    (void)N; (void)M;
    kq_matmul(oq_q5k_fields, 176, w, K, qa, da, Sa, ms, nm, ns, nn, y);
}

/*
 *   Q6_K: sum over super-blocks of d * sum_s sc_s * da[m][s/2] * D_s
 *   (16-element sub-block s inside the 32-element Q8 block s/2).
 */
void oq_q6k_matmul(const uint8_t *w, int64_t N, int64_t K,
                   const int8_t *qa, const float *da, const int32_t *Sa, int64_t M,
                   const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, double *y)
{
    (void)N; (void)M; (void)Sa;
    int64_t nb = K / OQ_QK, nblk = K / OQ_Q8;
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    int32_t *scw = (int32_t *)malloc(sizeof(int32_t) * (K / 16));
    double *dw = (double *)malloc(sizeof(double) * nb);
    for (int64_t jn = 0; jn < nn; ++jn) {
        int64_t n = ns[jn];
        for (int64_t b = 0; b < nb; ++b)
            oq_q6k_fields(w + (n * nb + b) * 210, &dw[b], scw + b * 16, qw + b * 256);
        for (int64_t im = 0; im < nm; ++im) {
            int64_t m = ms[im];
            const int8_t *a = qa + m * K;
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                double part = 0.0;
                for (int s = 0; s < 16; ++s) {
                    int64_t gs = b * 16 + s;
                    int64_t dot = 0;
                    for (int l = 0; l < 16; ++l) dot += (int64_t)qw[gs * 16 + l] * a[gs * 16 + l];
                    part += (double)scw[gs] * (double)da[m * nblk + gs / 2] * (double)dot;
                }
                acc += dw[b] * part;
            }
            y[im * nn + jn] = acc;
        }
    }
    free(qw); free(scw); free(dw);
}

/* ----------------------------------------------------------------- C9 --- */

/*
 * 32-value block formats.  fmt: 0 = Q4_0, 1 = Q4_1, 2 = Q5_0, 3 = Q5_1, 4 = Q8_0.
 *   Q4_0 (18 B): d fp16 | qs[16]            q_l = low nibble of qs[l], q_{l+16} = high nibble;
 *                                           value = d * (q - 8)
 *   Q4_1 (20 B): d fp16 | m fp16 | qs[16]   nibbles as Q4_0;            value = d * q + m
 *   Q5_0 (22 B): d fp16 | qh[4] | qs[16]    q_l = nibble + 16 * bit l of the little-endian
 *                                           32-bit qh (l = 0..31);       value = d * (q - 16)
 *   Q5_1 (24 B): d fp16 | m fp16 | qh[4] | qs[16]   as Q5_0;            value = d * q + m
 *   Q8_0 (34 B): d fp16 | qs[32] int8       q_l = qs[l];                 value = d * q
 * Outputs the integer of each value in the format's own integer domain, iq[32] = q - off
 * (off = 8, 0, 16, 0, 0), and d, m (m = 0 where the format has none), so value = d * iq + m.
 */
static const int oq_b32_bytes[5] = {18, 20, 22, 24, 34};

int oq_b32_block_bytes(int fmt) { return (fmt >= 0 && fmt < 5) ? oq_b32_bytes[fmt] : 0; }

void oq_b32_fields(int fmt, const uint8_t *blk, double *d, double *m, int32_t iq[32])
{
    *d = oq_half_to_double(rd16(blk));
    *m = (fmt == 1 || fmt == 3) ? oq_half_to_double(rd16(blk + 2)) : 0.0;
    if (fmt == 4) {
        for (int l = 0; l < 32; ++l) iq[l] = (int8_t)blk[2 + l];
        return;
    }
    const int has_m = (fmt == 1 || fmt == 3), five = (fmt == 2 || fmt == 3);
    const uint8_t *after = blk + (has_m ? 4 : 2);
    uint32_t qh = 0;
    if (five) qh = (uint32_t)after[0] | ((uint32_t)after[1] << 8) | ((uint32_t)after[2] << 16) | ((uint32_t)after[3] << 24);
    const uint8_t *qs = after + (five ? 4 : 0);
    const int off = fmt == 0 ? 8 : fmt == 2 ? 16 : 0;
    for (int l = 0; l < 16; ++l) {
        int lo = qs[l] & 15, hi = qs[l] >> 4;
        if (five) {
            lo += 16 * (int)((qh >> l) & 1u);
            hi += 16 * (int)((qh >> (l + 16)) & 1u);
        }
        iq[l] = lo - off;
        iq[l + 16] = hi - off;
    }
}

/* Dequantize: out[r][k] = d * iq + m (f64, exact). */
void oq_b32_dequant(int fmt, const uint8_t *w, int64_t n_rows, int64_t K, double *out)
{
    int64_t nb = K / OQ_Q8;
    int bytes = oq_b32_bytes[fmt];
    for (int64_t r = 0; r < n_rows; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double d, m;
            int32_t iq[32];
            oq_b32_fields(fmt, w + (r * nb + b) * bytes, &d, &m, iq);
            for (int l = 0; l < 32; ++l) out[r * K + b * 32 + l] = d * iq[l] + m;
        }
}

/*
 * Integer checkpoint: I[b] = sum_l iq_w[32b + l] * q_a[32b + l] (the block's dot in the
 * weight format's integer domain), [nm][nn][K/32].
 */
void oq_b32_blockdots(int fmt, const uint8_t *w, int64_t K, const int8_t *qa,
                      const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, int32_t *I)
{
    int64_t nb = K / OQ_Q8;
    int bytes = oq_b32_bytes[fmt];
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    for (int64_t jn = 0; jn < nn; ++jn) {
        for (int64_t b = 0; b < nb; ++b) {
            double d, m;
            oq_b32_fields(fmt, w + (ns[jn] * nb + b) * bytes, &d, &m, qw + b * 32);
        }
        for (int64_t im = 0; im < nm; ++im) {
            const int8_t *a = qa + ms[im] * K;
            for (int64_t b = 0; b < nb; ++b) {
                int32_t dot = 0;
                for (int l = 0; l < 32; ++l) dot += qw[b * 32 + l] * (int32_t)a[b * 32 + l];
                I[(im * nn + jn) * nb + b] = dot;
            }
        }
    }
    free(qw);
}

/*
 * Y[m][n] = sum_b [ d_b * da[m][b] * I_b + m_b * da[m][b] * S[m][b] ]  (f64), where the
 * second term (the block's offset m_b times the Q8 block's value sum da * S) is present for
 * Q4_1 / Q5_1 only.
 */
void oq_b32_matmul(int fmt, const uint8_t *w, int64_t K,
                   const int8_t *qa, const float *da, const int32_t *Sa,
                   const int64_t *ms, int64_t nm, const int64_t *ns, int64_t nn, double *y)
{
    int64_t nb = K / OQ_Q8;
    int bytes = oq_b32_bytes[fmt];
    int32_t *qw = (int32_t *)malloc(sizeof(int32_t) * K);
    double *dw = (double *)malloc(sizeof(double) * nb);
    double *mw = (double *)malloc(sizeof(double) * nb);
    for (int64_t jn = 0; jn < nn; ++jn) {
        for (int64_t b = 0; b < nb; ++b)
            oq_b32_fields(fmt, w + (ns[jn] * nb + b) * bytes, &dw[b], &mw[b], qw + b * 32);
        for (int64_t im = 0; im < nm; ++im) {
            int64_t mm = ms[im];
            const int8_t *a = qa + mm * K;
            double acc = 0.0;
            for (int64_t b = 0; b < nb; ++b) {
                int64_t dot = 0;
                for (int l = 0; l < 32; ++l) dot += (int64_t)qw[b * 32 + l] * a[b * 32 + l];
                double dab = (double)da[mm * nb + b];
                acc += dw[b] * dab * (double)dot + mw[b] * dab * (double)Sa[mm * nb + b];
            }
            y[im * nn + jn] = acc;
        }
    }
    free(qw); free(dw); free(mw);
}
