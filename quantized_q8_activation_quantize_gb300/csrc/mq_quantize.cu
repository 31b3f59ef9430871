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

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr unsigned kFull = 0xffffffffu;

__device__ __forceinline__ void quantize8(const float (&v)[8], int lane, const Plane &p, int64_t M, int64_t K,
                                          int64_t m, int64_t k0) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    int q[8];
    int s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        float r = roundf(__fmul_rn(v[i], id));            // half away from zero
        r = fminf(fmaxf(r, -127.0f), 127.0f);
        q[i] = __float2int_rz(r);
        s += q[i];
    }
    s += __shfl_xor_sync(kFull, s, 1);
    s += __shfl_xor_sync(kFull, s, 2);

    uint2 b8;
    b8.x = (uint32_t)(q[0] & 0xff) | ((uint32_t)(q[1] & 0xff) << 8) | ((uint32_t)(q[2] & 0xff) << 16) |
           ((uint32_t)(q[3] & 0xff) << 24);
    b8.y = (uint32_t)(q[4] & 0xff) | ((uint32_t)(q[5] & 0xff) << 8) | ((uint32_t)(q[6] & 0xff) << 16) |
           ((uint32_t)(q[7] & 0xff) << 24);
    uint4 h;
    __half2 t;
    t = __halves2half2(__int2half_rn(q[0]), __int2half_rn(q[1])); h.x = *reinterpret_cast<uint32_t *>(&t);
    t = __halves2half2(__int2half_rn(q[2]), __int2half_rn(q[3])); h.y = *reinterpret_cast<uint32_t *>(&t);
    t = __halves2half2(__int2half_rn(q[4]), __int2half_rn(q[5])); h.z = *reinterpret_cast<uint32_t *>(&t);
    t = __halves2half2(__int2half_rn(q[6]), __int2half_rn(q[7])); h.w = *reinterpret_cast<uint32_t *>(&t);

    const int64_t off = m * K + k0;
    *reinterpret_cast<uint2 *>(p.q8 + off) = b8;
    *reinterpret_cast<uint4 *>(p.q16 + off) = h;
    if ((lane & 3) == 0) {
        const int64_t b = k0 / kQ8;
        p.d[b * M + m] = d;
        p.s[b * M + m] = s;
        // d*S as a tf32 (hi, lo) pair: operand of the tensor-core Q4_K min term
        const float ds = __fmul_rn(d, (float)s);
        const float hi = tf32_rn(ds);
        const float lo = tf32_rn(__fsub_rn(ds, hi));
        float *row = p.ds + m * (2 * (K / kQ8)) + (b >> 3) * 16 + (b & 7);
        row[0] = hi;
        row[8] = lo;
    }
}

__global__ void __launch_bounds__(256) quantize_kernel(const float *__restrict__ x, int64_t M, int64_t K, Plane p) {
    grid_dep_launch();
    grid_dep_wait();
    const int lane = threadIdx.x & 31;
    const uint32_t nch = (uint32_t)(K / 256);
    const int64_t items = M * (int64_t)nch;
    const int64_t stride = (int64_t)gridDim.x * 8;
    for (int64_t it = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); it < items; it += stride) {
        // items < 2^31 * 2^23: the quotient fits 32 bits; divide in 64 bits only when it must
        const int64_t m = (it < 0xffffffffll) ? (int64_t)((uint32_t)it / nch) : it / (int64_t)nch;
        const int64_t k0 = (it - m * (int64_t)nch) * 256 + lane * 8;
        const float4 *src = reinterpret_cast<const float4 *>(x + m * K + k0);
        const float4 a = __ldg(src), b = __ldg(src + 1);
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        quantize8(v, lane, p, M, K, m, k0);
    }
}

// SwiGLU producer: y = swiglu1(g, u) (mq_device.cuh), then the Q8 quantization of y.
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
        quantize8(v, lane, p, M, K, m, k0);
    }
}

// RMSNorm producer: one CTA per token.  Pass 1 sums x^2 in f64 (each square is exact
// in f64); r = (float)(1 / sqrt(sum/K + eps)) is rounded once; pass 2 re-reads the row
// (L2-resident) and quantizes y = fl(fl(x * r) * w).
__global__ void __launch_bounds__(256) rms_quantize_kernel(const float *__restrict__ x, int64_t M, int64_t K,
                                                           const float *__restrict__ w, float eps, Plane p) {
    __shared__ double red[8];
    __shared__ float r_sh;
    grid_dep_launch();
    grid_dep_wait();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t nch = K / 256;
    for (int64_t m = blockIdx.x; m < M; m += gridDim.x) {
        const float *xr = x + m * K;
        double ss = 0.0;
        for (int64_t k = (int64_t)tid * 4; k < K; k += 1024) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(xr + k));
            ss = fma((double)v.x, (double)v.x, ss);
            ss = fma((double)v.y, (double)v.y, ss);
            ss = fma((double)v.z, (double)v.z, ss);
            ss = fma((double)v.w, (double)v.w, ss);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (tid == 0) {
            double t = 0.0;
            for (int i = 0; i < 8; ++i) t += red[i];
            const double ms = t / (double)K;
            r_sh = (float)(1.0 / sqrt(ms + (double)eps));
        }
        __syncthreads();
        const float r = r_sh;
        for (int64_t c = warp; c < nch; c += 8) {
            const int64_t k0 = c * 256 + lane * 8;
            const float4 *src = reinterpret_cast<const float4 *>(xr + k0);
            const float4 *ws = reinterpret_cast<const float4 *>(w + k0);
            const float4 a = __ldg(src), b = __ldg(src + 1);
            const float4 wa = __ldg(ws), wb = __ldg(ws + 1);
            const float v[8] = {__fmul_rn(__fmul_rn(a.x, r), wa.x), __fmul_rn(__fmul_rn(a.y, r), wa.y),
                                __fmul_rn(__fmul_rn(a.z, r), wa.z), __fmul_rn(__fmul_rn(a.w, r), wa.w),
                                __fmul_rn(__fmul_rn(b.x, r), wb.x), __fmul_rn(__fmul_rn(b.y, r), wb.y),
                                __fmul_rn(__fmul_rn(b.z, r), wb.z), __fmul_rn(__fmul_rn(b.w, r), wb.w)};
            quantize8(v, lane, p, M, K, m, k0);
        }
        __syncthreads();   // red / r_sh are reused by the next token
    }
}

}  // namespace

int launch_quantize(const float *x, int64_t M, int64_t K, const float *rms_w, float eps, const Plane &p,
                    unsigned int *err, cudaStream_t stream) {
    (void)err;
    const int nsm = sm_count();
    cudaError_t e;
    if (rms_w == nullptr) {
        const int64_t warps = M * (K / 256);
        int64_t ctas = (warps + 7) / 8;
        const int64_t cap = (int64_t)nsm * 8;
        if (ctas > cap) ctas = cap;
        e = launch_pdl(quantize_kernel, dim3((unsigned)ctas), dim3(256), 0, stream, x, M, K, p);
    } else {
        int64_t ctas = M;
        const int64_t cap = (int64_t)nsm * 8;
        if (ctas > cap) ctas = cap;
        e = launch_pdl(rms_quantize_kernel, dim3((unsigned)ctas), dim3(256), 0, stream, x, M, K, rms_w, eps, p);
    }
    return cuda_error(e, "quantize launch");
}

int launch_swiglu_quantize(const float *g, const float *up, int64_t M, int64_t K, const Plane &p, cudaStream_t stream) {
    const int nsm = sm_count();
    const int64_t warps = M * (K / 256);
    int64_t ctas = (warps + 7) / 8;
    const int64_t cap = (int64_t)nsm * 8;
    if (ctas > cap) ctas = cap;
    return cuda_error(launch_pdl(swiglu_quantize_kernel, dim3((unsigned)ctas), dim3(256), 0, stream, g, up, M, K, p),
                      "swiglu quantize launch");
}

}  // namespace mq
