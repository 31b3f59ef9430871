// mq_quantize.cu -- Q8 activation quantization, plain and RMSNorm-fused.
//
// minfer pages, "Features > GPU -- CUDA": the int8 MMQ path quantizes activations
// itself, and the rms-norm producer emits the q8 plane directly, skipping the
// intermediate f32 write.  "Compute Graph Design > 3.1": RmsNorm{eps}.
//
// One warp quantizes 256 consecutive values of one token per step: lane l holds
// values 8l..8l+7, so lanes 4i..4i+3 form Q8 block i and reduce its amax and code
// sum with two xor-shuffles.  Loads are 2 x 16 B per lane (1 KiB per warp), stores
// are 16 B (f16 codes) + 8 B (int8 codes) per lane; the block scale and sum go to
// the block-major [K/32][M] arrays.  Arithmetic is IEEE f32 with explicit rounding
// intrinsics (no contraction): d = amax/127, q = round_half_away(x * (1/d)).
#include <cuda_fp16.h>

#include <cstring>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// SECT: the plane sections written besides d and S (MQ_PLANE_Q16 | MQ_PLANE_Q8 | MQ_PLANE_DS)
template <unsigned SECT>
__device__ __forceinline__ void quantize8(const float (&v)[8], int lane, const Plane &p, int64_t M, int64_t K,
                                          int64_t m, int64_t k0) {
    Q8Lane q;
    q8_lane(v, q);
    const float(&r)[8] = q.r;
    const float d = q.d;
    const int s = __float2int_rn(q.s);
    const uint2 b8 = q8_bytes(r);
    // f16 codes: each integer is exact in f16, so the packed conversion is exact
    uint4 h;
    __half2 t;
    t = __floats2half2_rn(r[0], r[1]); h.x = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2half2_rn(r[2], r[3]); h.y = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2half2_rn(r[4], r[5]); h.z = *reinterpret_cast<uint32_t *>(&t);
    t = __floats2half2_rn(r[6], r[7]); h.w = *reinterpret_cast<uint32_t *>(&t);

    const int64_t off = m * K + k0;
    if constexpr ((SECT & MQ_PLANE_Q8) != 0) *reinterpret_cast<uint2 *>(p.q8 + off) = b8;
    if constexpr ((SECT & MQ_PLANE_Q16) != 0) *reinterpret_cast<uint4 *>(p.q16 + off) = h;
    if ((lane & 3) == 0) {
        const int64_t b = k0 / kQ8;
        p.d[b * M + m] = d;
        p.s[b * M + m] = s;
        if constexpr ((SECT & MQ_PLANE_DS) != 0) {
            // d*S as a tf32 (hi, lo) pair: operand of the tensor-core Q4_K min term
            const float ds = __fmul_rn(d, (float)s);
            const float hi = tf32_rn(ds);
            const float lo = tf32_rn(__fsub_rn(ds, hi));
            float *row = p.ds + m * (2 * (K / kQ8)) + (b >> 3) * 16 + (b & 7);
            row[0] = hi;
            row[8] = lo;
        }
    }
}

// Two (token, 256-value chunk) items per warp and iteration, both items' loads issued before either
// is quantized (twice the bytes in flight per warp).
template <unsigned SECT>
__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ x, int64_t M, int64_t K, Plane p) {
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const uint32_t nch = (uint32_t)(K / 256);
    const int64_t items = M * (int64_t)nch;
    const int64_t stride = (int64_t)gridDim.x * 8;
    // items < 2^31 * 2^23: the quotient fits 32 bits; divide in 64 bits only when it must
    auto token = [&](int64_t it) { return (it < 0xffffffffll) ? (int64_t)((uint32_t)it / nch) : it / (int64_t)nch; };
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += 2 * stride) {
        const int64_t it2 = it + stride;
        const bool two = it2 < items;
        const int64_t m = token(it), m2 = two ? token(it2) : m;
        const int64_t k0 = (it - m * (int64_t)nch) * 256 + lane * 8;
        const int64_t k02 = two ? (it2 - m2 * (int64_t)nch) * 256 + lane * 8 : k0;
        const float4 *src = reinterpret_cast<const float4 *>(x + m * K + k0);
        const float4 *src2 = reinterpret_cast<const float4 *>(x + m2 * K + k02);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        float4 a2 = make_float4(0.f, 0.f, 0.f, 0.f), b2 = a2;
        if (two) {
            a2 = __ldg(src2);
            b2 = __ldg(src2 + 1);
        }
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        quantize8<SECT>(v, lane, p, M, K, m, k0);
        if (two) {
            const float v2[8] = {a2.x, a2.y, a2.z, a2.w, b2.x, b2.y, b2.z, b2.w};
            quantize8<SECT>(v2, lane, p, M, K, m2, k02);
        }
    }
}

// The plain quantizer over up to 8 independent activations of the same shape [M][K] in one launch
// (the decode sweep's inputs of one layer level); item it belongs to job it / (M * K / 256).
constexpr int kMaxQJobs = 8;
struct QJobs {
    int n;
    const float *x[kMaxQJobs];
    Plane p[kMaxQJobs];
};

template <unsigned SECT>
__global__ void __launch_bounds__(256) quantize_grouped_kernel(const __grid_constant__ QJobs jobs, int64_t M,
                                                               int64_t K) {
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const uint32_t nch = (uint32_t)(K / 256);
    const int64_t per_job = M * (int64_t)nch, items = per_job * jobs.n;
    const int64_t stride = (int64_t)gridDim.x * 8;
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += stride) {
        const int j = (int)(it / per_job);
        const int64_t r = it - (int64_t)j * per_job;
        const int64_t m = r / nch;
        const int64_t k0 = (r - m * (int64_t)nch) * 256 + lane * 8;
        const float *x = jobs.x[0];
        Plane p = jobs.p[0];
#pragma unroll
        for (int i = 1; i < kMaxQJobs; ++i)
            if (i == j) {
                x = jobs.x[i];
                p = jobs.p[i];
            }
        const float4 *src = reinterpret_cast<const float4 *>(x + m * K + k0);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        quantize8<SECT>(v, lane, p, M, K, m, k0);
    }
}

// SwiGLU producer: y = swiglu1(g, u) (mq_device.cuh), then the Q8 quantization of y.
template <unsigned SECT>
__global__ void __launch_bounds__(256) swiglu_quantize_kernel(const float *__restrict__ g, const float *__restrict__ up,
                                                              int64_t M, int64_t K, Plane p) {
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const uint32_t nch = (uint32_t)(K / 256);
    const int64_t items = M * (int64_t)nch;
    const int64_t stride = (int64_t)gridDim.x * 8;
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += stride) {
        const int64_t m = (it < 0xffffffffll) ? (int64_t)((uint32_t)it / nch) : it / (int64_t)nch;
        const int64_t k0 = (it - m * (int64_t)nch) * 256 + lane * 8;
        const float4 *gs = reinterpret_cast<const float4 *>(g + m * K + k0);
        const float4 *us = reinterpret_cast<const float4 *>(up + m * K + k0);
        const float4 ga = __ldg(gs), gb = __ldg(gs + 1), ua = __ldg(us), ub = __ldg(us + 1);
        const float v[8] = {swiglu1(ga.x, ua.x), swiglu1(ga.y, ua.y), swiglu1(ga.z, ua.z), swiglu1(ga.w, ua.w),
                            swiglu1(gb.x, ub.x), swiglu1(gb.y, ub.y), swiglu1(gb.z, ub.z), swiglu1(gb.w, ub.w)};
        quantize8<SECT>(v, lane, p, M, K, m, k0);
    }
}

// Error-free product and sum in f32 (Dekker / Knuth): x * x = p + e exactly (e from one fused
// multiply-add), and the running pair (hi, lo) takes p with Knuth's branch-free two-sum, whose
// rounding error goes to lo.  Every step is an explicitly rounded intrinsic, so the compiler can
// neither contract nor reassociate it.
__device__ __forceinline__ void add_square(float v, float &hi, float &lo) {
    const float p = __fmul_rn(v, v);
    const float e = __fmaf_rn(v, v, -p);
    const float s = __fadd_rn(hi, p);
    const float bv = __fsub_rn(s, hi);
    const float err = __fadd_rn(__fsub_rn(hi, __fsub_rn(s, bv)), __fsub_rn(p, bv));
    hi = s;
    lo = __fadd_rn(lo, __fadd_rn(err, e));
}

// Error-free sum a + b = s + e (Knuth's two-sum, branch-free, any order of magnitudes).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = __fadd_rn(a, b);
    const float bv = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bv)), __fsub_rn(b, bv));
}

// (ah, al) += (bh, bl) for pairs of f32 (a value and its small correction): the high parts add
// error-free, the corrections add rounded, and the result is renormalised (|al| <= ulp(ah) / 2).
// The result does not depend on the order of the operands, so a butterfly over the lanes leaves
// the same pair in every lane.
__device__ __forceinline__ void pair_add(float &ah, float &al, float bh, float bl) {
    float s, e;
    two_sum(ah, bh, s, e);
    e = __fadd_rn(e, __fadd_rn(al, bl));
    ah = __fadd_rn(s, e);
    al = __fsub_rn(e, __fsub_rn(ah, s));
}

// r = 1 / sqrt(t / K + eps) rounded once to f32, from the sum of squares t = th + tl (reduced
// from the lanes' pairs by pair_add), in f32 arithmetic only.  The lanes' pairs add as f32 pairs
// (relative error below 2^-43 for these non-negative sums), t / K is an f32 pair (the remainder
// t - q K of the quotient q is exact for K < 2^22), and one Newton step on rsqrtf's estimate y0
// (error below 2^-21) gives y0 + yl within 2^-41 of the value the same lane pairs give in f64.  When every point within 2^-38 y0 of
// y0 + yl rounds to the same f32, that is r, and it equals the rounding of the f64 evaluation;
// otherwise (about one token in 10^4: the value lies near a rounding boundary) or outside the
// normal range the function returns false and the caller evaluates r in f64.  The f64 pipe of
// this GPU issues ~1.7 operations per clock per SM, so its square root and divide (dozens of
// operations each) cost more than the rest of a token's arithmetic.
__device__ __forceinline__ bool rms_scale_from_pair(float th, float tl, int64_t K, float eps, float &r) {
    const float kf = (float)K;
    const float ik = __frcp_rn(kf);
    const float qh = __fmul_rn(th, ik);
    const float rem = __fmaf_rn(-qh, kf, th);
    const float ql = __fmul_rn(__fadd_rn(rem, tl), ik);
    float vh, vl;
    two_sum(qh, eps, vh, vl);
    vl = __fadd_rn(vl, ql);
    // Newton step for 1/sqrt(v): y1 = y0 + y0 (1 - v y0^2) / 2, with y0^2 = p + pe exactly
    const float y0 = rsqrtf(vh);
    const float p = __fmul_rn(y0, y0);
    const float pe = __fmaf_rn(y0, y0, -p);
    const float a = __fmaf_rn(-vh, p, 1.0f);
    const float c = __fsub_rn(a, __fmaf_rn(vh, pe, __fmul_rn(vl, p)));
    const float yl = __fmul_rn(__fmul_rn(0.5f, y0), c);
    const float dl = __fmul_rn(y0, 0x1p-38f);
    const float ra = __fadd_rn(y0, __fsub_rn(yl, dl));
    const float rb = __fadd_rn(y0, __fadd_rn(yl, dl));
    r = ra;
    return ra == rb && vh >= 0x1p-100f && vh <= 0x1p100f;
}

// the same from the lanes' pairs of one warp (the pair sum over the lanes is the same in every lane)
__device__ __forceinline__ bool rms_scale_f32(float hi0, float lo0, float hi1, float lo1, int64_t K, float eps,
                                              float &r) {
    float th = hi0, tl = lo0;
    pair_add(th, tl, hi1, lo1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float bh = __shfl_xor_sync(kFull, th, o), bl = __shfl_xor_sync(kFull, tl, o);
        pair_add(th, tl, bh, bl);
    }
    return rms_scale_from_pair(th, tl, K, eps, r);
}

// RMSNorm producer: one warp per token.  Pass 1 sums x^2 per lane as an f32 pair (hi, lo)
// carrying about 48 significant bits (every square and every addition's rounding error kept);
// r = 1 / sqrt(sum/K + eps) rounded once to f32 comes from rms_scale_f32, or, when that declines,
// from the lanes' pairs combined in f64 in a fixed order (f64 sums of the same squares in another
// order give the same f32 r but with probability ~1e-7 per token).  Pass 2 re-reads the row
// (cache-resident) and quantizes y = fl(fl(x * r) * w) with the layout of quantize_kernel (lane l
// holds values 8l .. 8l + 7 of each 256-value chunk).
template <unsigned SECT>
__global__ void __launch_bounds__(256) rms_quantize_kernel(const float *__restrict__ x, int64_t M, int64_t K,
                                                           const float *__restrict__ w, float eps, Plane p) {
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t nch = K / 256;
    for (int64_t m = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); m < M; m += (int64_t)gridDim.x * 8) {
        const float *xr = x + m * K + lane * 8;
        float hi0 = 0.0f, lo0 = 0.0f, hi1 = 0.0f, lo1 = 0.0f;
#pragma unroll 4
        for (int64_t c = 0; c < nch; ++c) {
            const float4 a = __ldg(reinterpret_cast<const float4 *>(xr + c * 256));
            const float4 b = __ldg(reinterpret_cast<const float4 *>(xr + c * 256 + 4));
            add_square(a.x, hi0, lo0);
            add_square(a.y, hi1, lo1);
            add_square(a.z, hi0, lo0);
            add_square(a.w, hi1, lo1);
            add_square(b.x, hi0, lo0);
            add_square(b.y, hi1, lo1);
            add_square(b.z, hi0, lo0);
            add_square(b.w, hi1, lo1);
        }
        float r;
        if (!rms_scale_f32(hi0, lo0, hi1, lo1, K, eps, r)) {
            // every lane holds the same f64 sum; one lane takes the square root and divide and
            // broadcasts r
            double t = ((double)hi0 + (double)lo0) + ((double)hi1 + (double)lo1);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
            r = 0.0f;
            if (lane == 0) r = (float)(1.0 / sqrt(t / (double)K + (double)eps));
            r = __shfl_sync(kFull, r, 0);
        }
#pragma unroll 2
        for (int64_t c = 0; c < nch; ++c) {
            const int64_t k0 = c * 256 + lane * 8;
            const float4 *src = reinterpret_cast<const float4 *>(x + m * K + k0);
            const float4 *ws = reinterpret_cast<const float4 *>(w + k0);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            const float4 wa = __ldg(ws), wb = __ldg(ws + 1);
            const float v[8] = {__fmul_rn(__fmul_rn(a.x, r), wa.x), __fmul_rn(__fmul_rn(a.y, r), wa.y),
                                __fmul_rn(__fmul_rn(a.z, r), wa.z), __fmul_rn(__fmul_rn(a.w, r), wa.w),
                                __fmul_rn(__fmul_rn(b.x, r), wb.x), __fmul_rn(__fmul_rn(b.y, r), wb.y),
                                __fmul_rn(__fmul_rn(b.z, r), wb.z), __fmul_rn(__fmul_rn(b.w, r), wb.w)};
            quantize8<SECT>(v, lane, p, M, K, m, k0);
        }
    }
}

// bar.sync on named barrier `id` (1 .. 15) for `threads` threads (whole warps)
__device__ __forceinline__ void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// packed f32 pairs: each component rounded once to nearest, as __fadd_rn / __fsub_rn / __fmul_rn /
// __fmaf_rn on it (one instruction for both)
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "sub.rn.f32x2 rd, ra, rb;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// add_square on two independent (hi, lo) chains at once, chain 0 in .x and chain 1 in .y
__device__ __forceinline__ void add_square2(float2 v, float2 &hi, float2 &lo) {
    const float2 p = __fmul2_rn(v, v);
    const float2 e = __ffma2_rn(v, v, make_float2(-p.x, -p.y));
    const float2 s = __fadd2_rn(hi, p);
    const float2 bv = sub2(s, hi);
    const float2 err = __fadd2_rn(sub2(hi, sub2(s, bv)), sub2(p, bv));
    hi = s;
    lo = __fadd2_rn(lo, __fadd2_rn(err, e));
}

// Q8 quantization of up to four 256-value chunks held by one warp (chunk j: lane l holds values
// 8l .. 8l + 7 of chunk cj = c0 + j * cstep, at columns 256 cj + 8l ..); chunks j >= nvalid are not
// written.  The per-value arithmetic is quantize8's; the per-block arithmetic (d = amax / 127,
// 1 / d, S, d * S and their stores) runs once per block instead of once per lane: the four lanes
// of a block reduce its amax and code sum as in quantize8, then lane 8j + q takes block q of
// chunk j (32 blocks, one per lane) and hands 1 / d back.
template <unsigned SECT>
__device__ __forceinline__ void quantize_chunks4(const float (&v)[4][8], int nvalid, int c0, int cstep, int lane,
                                                 const Plane &p, int64_t M, int64_t K, int64_t m) {
    float am[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        float a = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) a = fmaxf(a, fabsf(v[j][i]));
        a = fmaxf(a, __shfl_xor_sync(kFull, a, 1));
        am[j] = fmaxf(a, __shfl_xor_sync(kFull, a, 2));
    }
    const int jl = lane >> 3, ql = lane & 7;
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float t = __shfl_sync(kFull, am[j], 4 * ql);
        if (jl == j) amax = t;
    }
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    float fsj[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float idj = __shfl_sync(kFull, id, 8 * j + (lane >> 2));
        float r[8];
        float fs = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            r[i] = __fadd_rn(fminf(fmaxf(roundf(__fmul_rn(v[j][i], idj)), -127.0f), 127.0f), 0.0f);
            fs = __fadd_rn(fs, r[i]);
        }
        fs = __fadd_rn(fs, __shfl_xor_sync(kFull, fs, 1));
        fsj[j] = __fadd_rn(fs, __shfl_xor_sync(kFull, fs, 2));
        if (j < nvalid) {
            const int64_t off = m * K + (int64_t)(c0 + j * cstep) * 256 + lane * 8;
            if constexpr ((SECT & MQ_PLANE_Q8) != 0) {
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__fadd_rn(r[i], 12582912.0f));
                uint2 b8;
                b8.x = __byte_perm(__byte_perm(w[0], w[1], 0x0040), __byte_perm(w[2], w[3], 0x0040), 0x5410);
                b8.y = __byte_perm(__byte_perm(w[4], w[5], 0x0040), __byte_perm(w[6], w[7], 0x0040), 0x5410);
                *reinterpret_cast<uint2 *>(p.q8 + off) = b8;
            }
            if constexpr ((SECT & MQ_PLANE_Q16) != 0) {
                uint4 h;
                __half2 t;
                t = __floats2half2_rn(r[0], r[1]); h.x = *reinterpret_cast<uint32_t *>(&t);
                t = __floats2half2_rn(r[2], r[3]); h.y = *reinterpret_cast<uint32_t *>(&t);
                t = __floats2half2_rn(r[4], r[5]); h.z = *reinterpret_cast<uint32_t *>(&t);
                t = __floats2half2_rn(r[6], r[7]); h.w = *reinterpret_cast<uint32_t *>(&t);
                *reinterpret_cast<uint4 *>(p.q16 + off) = h;
            }
        }
    }
    float fs = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float t = __shfl_sync(kFull, fsj[j], 4 * ql);
        if (jl == j) fs = t;
    }
    if (jl < nvalid) {
        const int s = __float2int_rn(fs);
        const int64_t b = (int64_t)(c0 + jl * cstep) * 8 + ql;
        p.d[b * M + m] = d;
        p.s[b * M + m] = s;
        if constexpr ((SECT & MQ_PLANE_DS) != 0) {
            const float ds = __fmul_rn(d, (float)s);
            const float hi = tf32_rn(ds);
            const float lo = tf32_rn(__fsub_rn(ds, hi));
            float *row = p.ds + m * (2 * (K / kQ8)) + (b >> 3) * 16 + (b & 7);
            row[0] = hi;
            row[8] = lo;
        }
    }
}

// RMSNorm producer with the row in registers: a group of WT = 2^wt_log2 warps (the fewest with
// 4 WT >= K / 256 chunks) quantizes one token, warp g of the group holding chunks g, g + WT,
// g + 2 WT, g + 3 WT of it (lane l: values 8l .. 8l + 7 of each) through both passes, so x is read
// from HBM once and never re-read.  Pass 1 runs the two (hi, lo) chains of rms_quantize_kernel as
// packed f32 pairs.  The warps' (hi, lo) sums meet in shared memory and every warp adds them in the
// same order, so all hold the same pair and take the same r.  Pass 2 quantizes with
// quantize_chunks4.  The launch gives every group one token (the block scheduler starts a CTA as
// another finishes, so loads and arithmetic of different CTAs overlap); the loop over further
// tokens only serves grids capped below that.
template <unsigned SECT>
__global__ void __launch_bounds__(256, 3) rms_quantize_regs_kernel(const float *__restrict__ x, int64_t M, int64_t K,
                                                                   const float *__restrict__ w, float eps, Plane p,
                                                                   int wt_log2) {
    __shared__ float2 part[2][8];       // [token parity][warp]: the warp's sum of squares as (hi, lo)
    __shared__ double partd[2][8];      // the same in f64 (the f64 evaluation of r)
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int WT = 1 << wt_log2, grp = warp >> wt_log2, g = warp & (WT - 1), ngrp = 8 >> wt_log2;
    const int first = grp << wt_log2;
    const int nch = (int)(K / 256);
    const int nvalid = min(4, (nch - g + WT - 1) >> wt_log2);    // this warp's chunks
    const int64_t stride = (int64_t)gridDim.x * ngrp;
    int par = 0;
    for (int64_t m = (int64_t)blockIdx.x * ngrp + grp; m < M; m += stride, par ^= 1) {
        const float *xr = x + m * K + lane * 8;
        float v[4][8];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
            if (j < nvalid) {
                a = __ldg(reinterpret_cast<const float4 *>(xr + (g + j * WT) * 256));
                b = __ldg(reinterpret_cast<const float4 *>(xr + (g + j * WT) * 256 + 4));
            }
            v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
            v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
        }
        // pass 1: chain 0 takes the even values of each 8, chain 1 the odd ones
        float2 hi = make_float2(0.f, 0.f), lo = hi;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (j < nvalid) {
#pragma unroll
                for (int i = 0; i < 8; i += 2) add_square2(make_float2(v[j][i], v[j][i + 1]), hi, lo);
            }
        float th = hi.x, tl = lo.x;
        pair_add(th, tl, hi.y, lo.y);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float bh = __shfl_xor_sync(kFull, th, o), bl = __shfl_xor_sync(kFull, tl, o);
            pair_add(th, tl, bh, bl);
        }
        if (WT > 1) {
            if (lane == 0) part[par][warp] = make_float2(th, tl);
            named_bar(1 + grp, WT * 32);
            th = part[par][first].x;
            tl = part[par][first].y;
            for (int k = 1; k < WT; ++k) pair_add(th, tl, part[par][first + k].x, part[par][first + k].y);
        }
        float r;
        if (!rms_scale_from_pair(th, tl, K, eps, r)) {
            double t = ((double)hi.x + (double)lo.x) + ((double)hi.y + (double)lo.y);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
            if (WT > 1) {
                if (lane == 0) partd[par][warp] = t;
                named_bar(1 + grp, WT * 32);
                t = partd[par][first];
                for (int k = 1; k < WT; ++k) t += partd[par][first + k];
            }
            r = 0.0f;
            if (lane == 0) r = (float)(1.0 / sqrt(t / (double)K + (double)eps));
            r = __shfl_sync(kFull, r, 0);
        }
        // pass 2 from the registers: y = fl(fl(x * r) * w)
        const float2 r2 = make_float2(r, r);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float4 wa = make_float4(0.f, 0.f, 0.f, 0.f), wb = wa;
            if (j < nvalid) {
                const float4 *ws = reinterpret_cast<const float4 *>(w + (g + j * WT) * 256 + lane * 8);
                wa = __ldg(ws);
                wb = __ldg(ws + 1);
            }
            const float wv[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                const float2 y = __fmul2_rn(__fmul2_rn(make_float2(v[j][i], v[j][i + 1]), r2),
                                            make_float2(wv[i], wv[i + 1]));
                v[j][i] = y.x;
                v[j][i + 1] = y.y;
            }
        }
        quantize_chunks4<SECT>(v, nvalid, g, WT, lane, p, M, K, m);
    }
}

}  // namespace

// the kernel of each section mask (1 .. 7)
#define MQ_SECT_SWITCH(KERNEL, sections, ...)                               \
    switch (sections) {                                                    \
    case 1: e = launch_pdl(KERNEL<1>, __VA_ARGS__); break;                 \
    case 2: e = launch_pdl(KERNEL<2>, __VA_ARGS__); break;                 \
    case 3: e = launch_pdl(KERNEL<3>, __VA_ARGS__); break;                 \
    case 4: e = launch_pdl(KERNEL<4>, __VA_ARGS__); break;                 \
    case 5: e = launch_pdl(KERNEL<5>, __VA_ARGS__); break;                 \
    case 6: e = launch_pdl(KERNEL<6>, __VA_ARGS__); break;                 \
    default: e = launch_pdl(KERNEL<7>, __VA_ARGS__); break;                \
    }

int launch_quantize(const float *x, int64_t M, int64_t K, const float *rms_w, float eps, unsigned sections,
                    const Plane &p, unsigned int *err, cudaStream_t stream) {
    (void)err;
    const int nsm = sm_count();
    cudaError_t e;
    if (rms_w == nullptr) {
        const int64_t warps = M * (K / 256);
        int64_t ctas = (warps + 7) / 8;
        const int64_t cap = (int64_t)nsm * 8;
        if (ctas > cap) ctas = cap;
        MQ_SECT_SWITCH(quantize_kernel, sections, dim3((unsigned)ctas), dim3(256), 0, stream, x, M, K, p)
    } else if (K <= 256 * 4 * 8) {
        // rows in registers: WT = 2^wl warps per token (4 chunks each at most), 8 / WT tokens per CTA,
        // one token per group of warps
        int wl = 0;
        while ((4 << wl) < (int)(K / 256)) ++wl;
        const int64_t ctas = (M + (8 >> wl) - 1) / (8 >> wl);
        MQ_SECT_SWITCH(rms_quantize_regs_kernel, sections, dim3((unsigned)ctas), dim3(256), 0, stream, x, M, K, rms_w,
                       eps, p, wl)
    } else {
        int64_t ctas = (M + 7) / 8;                 // a warp per token, eight per CTA
        const int64_t cap = (int64_t)nsm * 8;
        if (ctas > cap) ctas = cap;
        MQ_SECT_SWITCH(rms_quantize_kernel, sections, dim3((unsigned)ctas), dim3(256), 0, stream, x, M, K, rms_w, eps, p)
    }
    return cuda_error(e, "quantize launch");
}

int launch_swiglu_quantize(const float *g, const float *up, int64_t M, int64_t K, unsigned sections, const Plane &p,
                           cudaStream_t stream) {
    const int nsm = sm_count();
    const int64_t warps = M * (K / 256);
    int64_t ctas = (warps + 7) / 8;
    const int64_t cap = (int64_t)nsm * 8;
    if (ctas > cap) ctas = cap;
    cudaError_t e;
    MQ_SECT_SWITCH(swiglu_quantize_kernel, sections, dim3((unsigned)ctas), dim3(256), 0, stream, g, up, M, K, p)
    return cuda_error(e, "swiglu quantize launch");
}

int launch_quantize_grouped(int nj, const float *const *x, const Plane *p, int64_t M, int64_t K, unsigned sections,
                            cudaStream_t stream) {
    if (nj < 1 || nj > kMaxQJobs) return set_error(MQ_ERR_ARG, "grouped quantize: %d jobs (1 .. %d)", nj, kMaxQJobs);
    QJobs jobs;
    memset(&jobs, 0, sizeof jobs);
    jobs.n = nj;
    for (int i = 0; i < nj; ++i) {
        jobs.x[i] = x[i];
        jobs.p[i] = p[i];
    }
    const int nsm = sm_count();
    const int64_t warps = nj * M * (K / 256);
    int64_t ctas = (warps + 7) / 8;
    const int64_t cap = (int64_t)nsm * 8;
    if (ctas > cap) ctas = cap;
    cudaError_t e;
    MQ_SECT_SWITCH(quantize_grouped_kernel, sections, dim3((unsigned)ctas), dim3(256), 0, stream, jobs, M, K)
    return cuda_error(e, "grouped quantize launch");
}

}  // namespace mq
