// mq_gemv.cuh -- decode GEMV (MMVQ): raw Q4_K / Q5_K / Q6_K / Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0
// weight bytes x Q8 codes with dp4a.
//
// minfer pages, "Support Matrix > CUDA notes": decode (nt == 1) uses the dp4a MMVQ
// kernels; "Roadmap > 0": the decode path streams the weights once per token.
//
// Design (HBM-bound): every weight byte is read from HBM exactly once per group of up
// to 8 (4 for Q6_K) tokens.  The 32-value formats enter as groups of eight blocks (256
// values, 144 .. 272 bytes, all multiples of 16), so they share the super-block machinery.  The weight matrix is one flat stream of super-blocks
// (row-major, rows contiguous).  Each CTA owns a contiguous range of whole rows and walks
// it in units of TU super-blocks (a unit may start or end inside a row):
//   * a producer warp refills a 2-4 stage shared-memory ring with ONE large 1-D bulk copy
//     (TMA engine) per unit -- the 16-byte aligned superset of the unit's bytes, so the
//     2-byte aligned 210-byte Q6_K block needs no special load path.  A few large copies
//     per SM keep the copy engine streaming at full HBM rate, where many small per-warp
//     copies stall it;
//   * 8 consumer warps take each super-block with 2 threads, one 128-value half each, so
//     the per-unit hand-offs and the scale decoding amortize over many values: dp4a
//     against the int8 codes, f32 scaling per 32-value block, a lane-pair reduction, and
//     one partial per (token, super-block) into a ring of partial buffers;
//   * a reducer warp sums each row's partials in a fixed order (a row that continues
//     into the next unit carries its running sum), so results are deterministic, and
//     writes Y.  Consumers wait for the reducer only when the partial ring is full.
// The shared-memory data pipe is the scarce resource once the weights stream at full
// rate: when the tokens' activations fit, each CTA first stages them in shared memory
// (codes in a padded layout that spreads every lane pattern below over distinct bank
// groups, plus per-block scale data: (d_a, d_a * S) for Q4_K; d_a and the -32 code
// offset as -32 * S16 per 16-value half block for Q6_K, which seeds the dp4a chain), so
// the inner loop reads 4 wavefronts per 512 bytes instead of one scattered L1 line per lane.
//
// Kernel and launcher templates; mq_gemv_kq.cu instantiates the k-quants (and holds the entry
// point), mq_gemv_b32.cu the 32-value formats, so the two compile in parallel.
#pragma once

#include <cuda_fp16.h>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int kPartBufs = 4;
constexpr unsigned kFull = 0xffffffffu;

template <int FMT>
struct GvCfg {
    static constexpr int BB = block_bytes(FMT);
    static constexpr int CW = 8;                               // consumer warps
    static constexpr int TPS = 2;                              // consumer threads per super-block
    static constexpr int THREADS = (CW + 2) * 32;              // + producer warp + reducer warp
    static constexpr int PRODUCER = CW, REDUCER = CW + 1;
    static constexpr int SB_PER_PASS = CW * 32 / TPS;          // 128
    static constexpr int PASSES = 1;
    static constexpr int TU = SB_PER_PASS * PASSES;            // super-blocks per unit
    static constexpr int STAGES = FMT == FMT_Q6K ? 3 : 4;  // at most; a launch may use fewer (GvArgs::nst)
    // tokens per pass over the weights (Q6_K: the staged activations of 8 tokens would leave
    // room for too few CTAs per SM; two passes of 4 measure faster)
    static constexpr int MAX_MT = FMT == FMT_Q6K ? 4 : 8;
    // CTAs per SM the launch aims for (registers: 64K / (THREADS * this))
    static constexpr int ctas_per_sm(int mt) { return mt <= 2 ? 3 : 2; }
    // unit bytes + up to 15 leading and 15 trailing alignment bytes, + 16 bytes of slack
    static constexpr int STAGE = ((TU * BB + 30 + 15) / 16) * 16 + 16;
    static constexpr int part_bytes(int mt) { return kPartBufs * mt * TU * 4; }
    // Staged activations, per token: one record per half super-block, its 128 int8 codes and
    // then its four 32-value blocks' scale data.  Q4_K: (d_a, d_a * S) per block, 32 B; half
    // stride HALF = 176 B (3 mod 8 bank groups of 16 B), super-block stride 416 B (2 mod 8), so
    // a quarter-warp's 8 lanes -- four consecutive super-blocks x two halves -- read 8 distinct
    // groups.  Q6_K: (d_a, -32 S16 of the first and second 16 values) per block, 64 B; half
    // stride 208 B (5 mod 8), super-block stride 464 B (5 mod 8): distinct groups for its
    // quarter-warps of four super-blocks two apart x two halves.  (Away from row ends.)
    static constexpr uint32_t SB_STRIDE = FMT == FMT_Q6K ? 464 : 416;
    static constexpr uint32_t HALF = FMT == FMT_Q6K ? 208 : 176;
    static int64_t act_bytes(int mt, int64_t K) { return (int64_t)mt * (K / kQK) * SB_STRIDE; }
};
constexpr int kSmemMax = 200 * 1024;                 // stage activations while the CTA fits in this
// the largest dynamic shared memory per CTA that leaves room for n CTAs per SM
constexpr int per_cta_smem(int n) { return n >= 4 ? 55 * 1024 : n == 3 ? 74 * 1024 : 112 * 1024; }

__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
__device__ __forceinline__ void sts64u(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1,%2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float half_bits_to_float(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)bits));
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t ma, uint32_t b, uint32_t mb) {
    return (a & ma) | (b & mb);
}
__device__ __forceinline__ int dot16(const uint4 &w, const uint4 &a, int c = 0) {
    return __dp4a((int)w.w, (int)a.w, __dp4a((int)w.z, (int)a.z, __dp4a((int)w.y, (int)a.y, __dp4a((int)w.x, (int)a.x, c))));
}
__device__ __forceinline__ int dot16w(const uint32_t *w, const uint4 &a, int c) {
    return __dp4a((int)w[3], (int)a.w, __dp4a((int)w[2], (int)a.z, __dp4a((int)w[1], (int)a.y, __dp4a((int)w[0], (int)a.x, c))));
}

// x / d (and x % d in rem) for 0 <= x < 2^24 through a float reciprocal (inv_d = 1/d rounded):
// the estimate is within one of the quotient, and one correction each way makes it exact.
__device__ __forceinline__ uint32_t divmod_small(uint32_t x, uint32_t d, float inv_d, uint32_t &rem) {
    uint32_t q = __float2uint_rz(__uint2float_rz(x) * inv_d);
    int r = (int)x - (int)(q * d);
    if (r < 0) { --q; r += (int)d; }
    if (r >= (int)d) { ++q; r -= (int)d; }
    rem = (uint32_t)r;
    return q;
}

struct GvArgs {
    const uint8_t *w;
    int64_t N, K;
    Plane p;
    int64_t M, t0;
    int mt;
    int nst;                     // ring stages this launch uses (2 .. STAGES)
    float *y;
    Dump dump;
    unsigned int *err;
    // M = 1 only: the token's f32 activation, quantized by every CTA into its staged records
    // (instead of the plane p, which is then not read)
    const float *x = nullptr;
};

// A grouped launch: up to kMaxJobs independent matrices of the same format and K, each with its own
// plane and output, in one grid; job j takes CTAs [cta0[j], cta0[j + 1]).  A plain launch is one job.
constexpr int kMaxJobs = 8;
struct GvJobs {
    int n;
    int cta0[kMaxJobs + 1];
    const uint8_t *w[kMaxJobs];
    int64_t N[kMaxJobs];
    Plane p[kMaxJobs];
    float *y[kMaxJobs];
    const float *x[kMaxJobs];    // GvArgs::x of each job
};

// shared-memory addresses of the staged activations (ACT kernels): codes [MT][K], table
struct GvAct {
    uint32_t codes;              // token 0's records
    uint32_t ck;                 // per-token stride of the records
};

// A thread's raw weight bytes of one super-block quarter, read from the stage before the
// stage is handed back to the producer (the math runs on these registers afterwards).
// Q4_K: half h of a super-block -- the 16-byte header (d, dmin, 12 scale bytes) and the
// qs bytes [64h, 64h+64) holding sub-blocks 4h .. 4h+3.
struct Q4Half {
    uint4 hd;
    uint32_t q[16];
};
// Q5_K: the same header and qs half as Q4_K (qs at byte 48 here) plus all 32 qh bytes,
// whose bit j is the fifth bit of sub-block j.
struct Q5Half {
    uint4 hd;
    uint32_t qh[8], q[16];
};
// Q6_K: half h of a super-block -- ql bytes [64h, 64h+64), qh bytes [128+32h, 128+32h+32),
// the eight int8 scales 8h .. 8h+7 and the fp16 d.
struct Q6Half {
    uint32_t ql[16], qh[8], sc[2], dbits;
};

// Q4_K: loads half h of the super-block at shared address `blk` (144-byte blocks keep every
// block 16-byte aligned inside a unit, so these are plain 16-byte reads).
__device__ __forceinline__ void q4k_load_half(uint32_t blk, int h, Q4Half &r) {
    r.hd = lds128(blk);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 v = lds128(blk + 16 + 64 * h + 16 * k);
        r.q[4 * k] = v.x;
        r.q[4 * k + 1] = v.y;
        r.q[4 * k + 2] = v.z;
        r.q[4 * k + 3] = v.w;
    }
}

// Q5_K: loads half h of the 176-byte super-block at `blk` (16-byte aligned, as for Q4_K).
__device__ __forceinline__ void q5k_load_half(uint32_t blk, int h, Q5Half &r) {
    r.hd = lds128(blk);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const uint4 v = lds128(blk + 16 + 16 * k);
        r.qh[4 * k] = v.x;
        r.qh[4 * k + 1] = v.y;
        r.qh[4 * k + 2] = v.z;
        r.qh[4 * k + 3] = v.w;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint4 v = lds128(blk + 48 + 64 * h + 16 * k);
        r.q[4 * k] = v.x;
        r.q[4 * k + 1] = v.y;
        r.q[4 * k + 2] = v.z;
        r.q[4 * k + 3] = v.w;
    }
}

// Q4_K / Q5_K math of one half (row n, super-block sbi of the row).  Sub-block j = 4h + i
// (i < 4) is the 32-value Q8 block 8 sbi + j: the low (i even) or high (i odd) nibbles of
// the qs words 8 (i / 2) .. 8 (i / 2) + 7, and for Q5_K bit j of each qh byte on top
// (+16).  Its integer dot I = sc_j D_j is exact; the row's two scalings are summed
// separately, d * sum_j d_a I_j - dmin * sum_j m_j (d_a S)_j.  qh is unused for Q4_K.
template <int FMT, int MT, bool ACT, bool DUMP>
__device__ __forceinline__ void kq_half(const GvArgs &a, const GvAct &at, const uint4 hd, const uint32_t (&qw)[16],
                                        const uint32_t *qh, int64_t n, uint32_t sbi, int h, bool valid,
                                        float (&part)[MT]) {
    using C = GvCfg<FMT>;
    const float d = half_bits_to_float(hd.x & 0xffff), dmin = half_bits_to_float(hd.x >> 16);
    // the four 6-bit scales and mins of sub-blocks 4h .. 4h+3, one byte each
    const uint32_t scw = h == 0 ? (hd.y & 0x3f3f3f3fu) : ((hd.w & 0x0f0f0f0fu) | ((hd.y >> 2) & 0x30303030u));
    const uint32_t mw = h == 0 ? (hd.z & 0x3f3f3f3fu) : (((hd.w >> 4) & 0x0f0f0f0fu) | ((hd.z >> 2) & 0x30303030u));
    float acc1[MT], acc2[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) { acc1[t] = 0.0f; acc2[t] = 0.0f; }
    const uint32_t rec = at.codes + sbi * C::SB_STRIDE + C::HALF * (uint32_t)h;    // token 0's record
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            v[e] = ((i & 1) ? (qw[8 * (i >> 1) + e] >> 4) : qw[8 * (i >> 1) + e]) & 0x0f0f0f0fu;
            if constexpr (FMT == FMT_Q5K) v[e] |= ((qh[e] >> (4 * h + i)) & 0x01010101u) << 4;
        }
        const int sc = (int)((scw >> (8 * i)) & 0xff);
        const float mf = (float)((mw >> (8 * i)) & 0xff);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int64_t m = a.t0 + t;
            const bool act = t < a.mt && valid;
            int I = 0;
            if (act) {
                if constexpr (ACT) {
                    const uint32_t rt = rec + (uint32_t)t * at.ck;
                    const uint4 a0 = lds128(rt + 32u * i), a1 = lds128(rt + 32u * i + 16u);
                    const float4 tb = lds128f(rt + 128u + 16u * (i >> 1));    // (d_a, d_a S) of two blocks
                    const float da = (i & 1) ? tb.z : tb.x, dS = (i & 1) ? tb.w : tb.y;
                    I = sc * dot16w(v + 4, a1, dot16w(v, a0, 0));
                    acc1[t] = fmaf(da, (float)I, acc1[t]);
                    acc2[t] = fmaf(mf, dS, acc2[t]);
                } else {
                    const int64_t b = (int64_t)sbi * 8 + 4 * h + i;          // the Q8 block
                    const uint4 *q = reinterpret_cast<const uint4 *>(a.p.q8 + m * a.K + 32 * b);
                    I = sc * dot16w(v + 4, __ldg(q + 1), dot16w(v, __ldg(q), 0));
                    const float da = __ldg(a.p.d + b * a.M + m);
                    acc1[t] = fmaf(da, (float)I, acc1[t]);
                    acc2[t] = fmaf(mf, da * (float)__ldg(a.p.s + b * a.M + m), acc2[t]);
                }
            }
            if constexpr (DUMP) {
                const Dump &dp = a.dump;
                if (act && m >= dp.m0 && m < dp.m0 + dp.m_cnt && n >= dp.n0 && n < dp.n0 + dp.n_cnt)
                    dp.out[((m - dp.m0) * dp.n_cnt + (n - dp.n0)) * (a.K / kQ8) + (int64_t)sbi * 8 + 4 * h + i] = I;
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) part[t] = fmaf(d, acc1[t], -dmin * acc2[t]);
}

// Q6_K: loads half h of the super-block at shared address `blk`.  A 210-byte block sits at
// a 4-byte or a 2-byte aligned address; AL4 picks the aligned reads, else every word is
// funnel-shifted out of two aligned neighbours (all reads stay inside the block).
template <bool AL4>
__device__ __forceinline__ void q6k_load_half(uint32_t blk, int h, Q6Half &r) {
    if constexpr (AL4) {
#pragma unroll
        for (int k = 0; k < 16; ++k) r.ql[k] = lds32(blk + 64 * h + 4 * k);
#pragma unroll
        for (int k = 0; k < 8; ++k) r.qh[k] = lds32(blk + 128 + 32 * h + 4 * k);
        r.sc[0] = lds32(blk + 192 + 8 * h);
        r.sc[1] = lds32(blk + 196 + 8 * h);
        r.dbits = lds16(blk + 208);
    } else {
        const uint32_t b = blk - 2;     // 4-byte aligned: byte i of the block is byte i + 2 here
        uint32_t w0 = lds32(b + 64 * h);
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            const uint32_t w1 = lds32(b + 64 * h + 4 * k + 4);
            r.ql[k] = __funnelshift_r(w0, w1, 16);
            w0 = w1;
        }
        w0 = lds32(b + 128 + 32 * h);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w1 = lds32(b + 128 + 32 * h + 4 * k + 4);
            r.qh[k] = __funnelshift_r(w0, w1, 16);
            w0 = w1;
        }
        const uint32_t s0 = lds32(b + 192 + 8 * h), s1 = lds32(b + 196 + 8 * h), s2 = lds32(b + 200 + 8 * h);
        r.sc[0] = __funnelshift_r(s0, s1, 16);
        r.sc[1] = __funnelshift_r(s1, s2, 16);
        r.dbits = lds32(b + 208) >> 16;
    }
}

// Q6_K math of one half (row n, super-block sbi of the row).  Group g = 0..3 of the half is
// the 32-value Q8 block 8 sbi + 4h + g: value 32g + l (l < 32) takes the low (g < 2) or high
// (g >= 2) nibble of ql[32 (g & 1) + l] and the bits (qh[l] >> 2g) & 3 as its high bits; its
// two 16-value sub-blocks have the scales 2g and 2g + 1 of the half.  The 6-bit codes are
// q + 32, so each 16-value dot starts from -32 * S16 (S16: sum of the 16 activation codes)
// and comes out as the exact sum (q * a); I = sc * x0 + sc' * x1 is the block's integer dot.
template <int MT, bool ACT, bool DUMP>
__device__ __forceinline__ void q6k_half(const GvArgs &a, const GvAct &at, const Q6Half &r, int64_t n,
                                         uint32_t sbi, int h, bool valid, float (&part)[MT]) {
    using C = GvCfg<FMT_Q6K>;
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
    const uint32_t rec = at.codes + sbi * C::SB_STRIDE + C::HALF * (uint32_t)h;   // token 0's record
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint32_t *L = (g & 1) ? r.ql + 8 : r.ql;
        uint32_t v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t H = r.qh[e];
            const uint32_t lo = (g < 2) ? L[e] : (L[e] >> 4);
            const uint32_t hb = (g == 0) ? (H << 4) : (g == 1) ? (H << 2) : (g == 2) ? H : (H >> 2);
            v[e] = lop3_and_or(lo, 0x0f0f0f0fu, hb, 0x30303030u);
        }
        const uint32_t sw = r.sc[g >> 1] >> (16 * (g & 1));
        const int sc0 = (int)(int8_t)(sw & 0xff), sc1 = (int)(int8_t)((sw >> 8) & 0xff);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int64_t m = a.t0 + t;
            const bool act = t < a.mt && valid;
            int I = 0;
            if (act) {
                if constexpr (ACT) {
                    const uint32_t rt = rec + (uint32_t)t * at.ck;
                    const uint4 a0 = lds128(rt + 32u * g), a1 = lds128(rt + 32u * g + 16u);
                    const uint4 tb = lds128(rt + 128u + 16u * g);        // d_a, -32 S16, -32 S16'
                    const int x0 = dot16w(v, a0, (int)tb.y), x1 = dot16w(v + 4, a1, (int)tb.z);
                    I = sc0 * x0 + sc1 * x1;
                    acc[t] = fmaf(__uint_as_float(tb.x), (float)I, acc[t]);
                } else {
                    const int8_t *q = a.p.q8 + m * a.K + (int64_t)sbi * kQK + 128 * h + 32 * g;
                    const uint4 a0 = __ldg(reinterpret_cast<const uint4 *>(q));
                    const uint4 a1 = __ldg(reinterpret_cast<const uint4 *>(q + 16));
                    const uint4 c32 = make_uint4(0x20202020u, 0x20202020u, 0x20202020u, 0x20202020u);
                    const int x0 = dot16w(v, a0, -dot16(c32, a0)), x1 = dot16w(v + 4, a1, -dot16(c32, a1));
                    I = sc0 * x0 + sc1 * x1;
                    acc[t] = fmaf(__ldg(a.p.d + ((int64_t)sbi * 8 + 4 * h + g) * a.M + m), (float)I, acc[t]);
                }
            }
            if constexpr (DUMP) {
                const Dump &dp = a.dump;
                if (act && m >= dp.m0 && m < dp.m0 + dp.m_cnt && n >= dp.n0 && n < dp.n0 + dp.n_cnt)
                    dp.out[((m - dp.m0) * dp.n_cnt + (n - dp.n0)) * (a.K / kQ8) + (int64_t)sbi * 8 + 4 * h + g] = I;
            }
        }
    }
    const float d = half_bits_to_float(r.dbits);
#pragma unroll
    for (int t = 0; t < MT; ++t) part[t] = d * acc[t];
}

// 32-value formats: half h of a group of eight blocks is blocks 4h .. 4h+3, HB = 4 x the
// block size bytes (72 / 80 / 88 / 96 / 136) starting at byte h * HB of the group.  Groups are
// 16-byte aligned in a unit (sizes 144 .. 272), so a half is 8-byte aligned, and 16-byte
// aligned where HB is a multiple of 16; it is read with the widest aligned loads.  With
// consecutive slots, a quarter-warp's four groups x two halves hit 8 distinct bank groups for
// all but Q5_1 (192-byte groups: 2-way).
template <int FMT>
struct B32Half {
    static constexpr int HB = 4 * b32_bytes(FMT);
    static constexpr int NW = HB / 4;
    uint32_t w[NW];
};

template <int FMT>
__device__ __forceinline__ void b32_load_half(uint32_t blk, int h, B32Half<FMT> &r) {
    constexpr int HB = B32Half<FMT>::HB;
    const uint32_t base = blk + (uint32_t)(HB * h);
    if constexpr (HB % 16 == 0) {
#pragma unroll
        for (int k = 0; k < HB / 16; ++k) {
            const uint4 v = lds128(base + 16 * k);
            r.w[4 * k] = v.x;
            r.w[4 * k + 1] = v.y;
            r.w[4 * k + 2] = v.z;
            r.w[4 * k + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < HB / 8; ++k) {
            const uint2 v = lds64(base + 8 * k);
            r.w[2 * k] = v.x;
            r.w[2 * k + 1] = v.y;
        }
    }
}

// the 4 bytes at byte offset o (a multiple of 2, known at compile time once unrolled) of a
// half held in registers
__device__ __forceinline__ uint32_t word_at(const uint32_t *w, int o) {
    return (o & 3) ? __funnelshift_r(w[o >> 2], w[(o >> 2) + 1], 16) : w[o >> 2];
}
__device__ __forceinline__ uint32_t half_at(const uint32_t *w, int o) {
    return (o & 3) ? (w[o >> 2] >> 16) : (w[o >> 2] & 0xffffu);
}

// 32-value formats, math of one half (row n, group sbi of the row).  Block g = 0..3 of the
// half is the Q8 block 8 sbi + 4h + g.  Its quants, as bytes in the order of the 32 values:
// Q8_0 the int8 quants themselves; the others the low nibbles of qs[0..15] (values 0..15)
// and the high nibbles (values 16..31), plus 16 x bit l of the 32-bit qh for value l in the
// five-bit formats (four qh bits spread to bit 4 of four bytes by one multiply: the shifted
// copies of a 4-bit field at 4, 11, 18 and 25 never overlap).  The quants' offset (8 for
// Q4_0, 16 for Q5_0) enters as the seed -off * S of the dp4a chain, so I = sum (q - off) a
// exactly; then y += (d d_a) I [+ m (d_a S)].
template <int FMT, int MT, bool ACT, bool DUMP>
__device__ __forceinline__ void b32_half(const GvArgs &a, const GvAct &at, const B32Half<FMT> &r, int64_t n,
                                         uint32_t sbi, int h, bool valid, float (&part)[MT]) {
    using C = GvCfg<FMT>;
    constexpr int BS = b32_bytes(FMT), OFF = b32_off(FMT);
    constexpr bool HAS_M = b32_has_m(FMT), FIVE = b32_five(FMT);
    constexpr int QH = HAS_M ? 4 : 2, QS = 2 + (HAS_M ? 2 : 0) + (FIVE ? 4 : 0);
    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;
    const uint32_t rec = at.codes + sbi * C::SB_STRIDE + C::HALF * (uint32_t)h;    // token 0's record
#pragma unroll
    for (int gp = 0; gp < 2; ++gp) {                // blocks 2 gp and 2 gp + 1: one table read
        float d[2], mw[2];
        uint32_t v[2][8];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int o = BS * (2 * gp + k);
            d[k] = half_bits_to_float(half_at(r.w, o));
            mw[k] = HAS_M ? half_bits_to_float(half_at(r.w, o + 2)) : 0.0f;
            if constexpr (FMT == FMT_Q8_0) {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[k][e] = word_at(r.w, o + 2 + 4 * e);
            } else {
                const uint32_t qh = FIVE ? word_at(r.w, o + QH) : 0u;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t qs = word_at(r.w, o + QS + 4 * e);
                    v[k][e] = qs & 0x0f0f0f0fu;
                    v[k][4 + e] = (qs >> 4) & 0x0f0f0f0fu;
                    if constexpr (FIVE) {
                        v[k][e] |= (((qh >> (4 * e)) & 0xfu) * 0x02040810u) & 0x10101010u;
                        v[k][4 + e] |= (((qh >> (16 + 4 * e)) & 0xfu) * 0x02040810u) & 0x10101010u;
                    }
                }
            }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int64_t m = a.t0 + t;
            const bool act = t < a.mt && valid;
            int I[2] = {0, 0};
            if (act) {
                if constexpr (ACT) {
                    const uint32_t rt = rec + (uint32_t)t * at.ck;
                    // (d_a, -off S) per block, or (d_a, d_a S) where the format has m
                    const uint4 tb = lds128(rt + 128u + 16u * gp);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t ca = rt + 32u * (2 * gp + k);
                        const uint4 a0 = lds128(ca), a1 = lds128(ca + 16u);
                        const float da = __uint_as_float(k ? tb.z : tb.x);
                        const uint32_t x = k ? tb.w : tb.y;
                        I[k] = dot16w(v[k] + 4, a1, dot16w(v[k], a0, OFF ? (int)x : 0));
                        acc[t] = fmaf(d[k] * da, (float)I[k], acc[t]);
                        if constexpr (HAS_M) acc[t] = fmaf(mw[k], __uint_as_float(x), acc[t]);
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const int64_t b = (int64_t)sbi * 8 + 4 * h + 2 * gp + k;     // the Q8 block
                        const uint4 *q = reinterpret_cast<const uint4 *>(a.p.q8 + m * a.K + 32 * b);
                        const float da = __ldg(a.p.d + b * a.M + m);
                        const int S = (OFF || HAS_M) ? __ldg(a.p.s + b * a.M + m) : 0;
                        I[k] = dot16w(v[k] + 4, __ldg(q + 1), dot16w(v[k], __ldg(q), -OFF * S));
                        acc[t] = fmaf(d[k] * da, (float)I[k], acc[t]);
                        if constexpr (HAS_M) acc[t] = fmaf(mw[k], da * (float)S, acc[t]);
                    }
                }
            }
            if constexpr (DUMP) {
                const Dump &dp = a.dump;
                if (act && m >= dp.m0 && m < dp.m0 + dp.m_cnt && n >= dp.n0 && n < dp.n0 + dp.n_cnt)
#pragma unroll
                    for (int k = 0; k < 2; ++k)
                        dp.out[((m - dp.m0) * dp.n_cnt + (n - dp.n0)) * (a.K / kQ8) + (int64_t)sbi * 8 + 4 * h +
                               2 * gp + k] = I[k];
            }
        }
    }
#pragma unroll
    for (int t = 0; t < MT; ++t) part[t] = acc[t];
}

// One token (M = 1): its f32 activation x quantized straight into the staged records with the
// arithmetic of mq_quantize_q8 (q8_lane), so the records hold exactly what staging its plane
// would give.  Warp w takes super-blocks w, w + CW, ...; lane l holds values 8l .. 8l + 7 of one:
// half l / 16, block (l / 4) % 4 of the half, bytes 8 (l % 16) .. of the half's codes.  The block
// entries: (d_a, d_a S) for Q4_K / Q5_K, (d_a, -32 S16, -32 S16') for Q6_K.
template <int FMT>
__device__ __forceinline__ void stage_x_one(const float (&v)[8], const GvAct &at, uint32_t sbi, int lane) {
    using C = GvCfg<FMT>;
    Q8Lane q;
    q8_lane(v, q);
    const uint2 b8 = q8_bytes(q.r);
    const uint32_t rec = at.codes + sbi * C::SB_STRIDE + C::HALF * (uint32_t)(lane >> 4);
    sts64u(rec + 8u * (uint32_t)(lane & 15), b8.x, b8.y);
    const uint32_t g = (uint32_t)(lane >> 2) & 3u;
    if constexpr (FMT == FMT_Q6K) {
        const uint32_t ent = rec + 128u + 16u * g;
        const uint32_t o32 = (uint32_t)(-32 * __float2int_rn(q.s16));
        if ((lane & 3) == 0)
            sts64u(ent, __float_as_uint(q.d), o32);
        else if ((lane & 3) == 2)
            sts32(ent + 8u, o32);
    } else {
        if ((lane & 3) == 0) sts64u(rec + 128u + 8u * g, __float_as_uint(q.d), __float_as_uint(q.d * q.s));
    }
}

// (two super-blocks' loads in flight per warp before either is quantized)
template <int FMT>
__device__ __forceinline__ void stage_x(const float *__restrict__ x, const GvAct &at, uint32_t nb, int warp,
                                        int lane) {
    using C = GvCfg<FMT>;
    for (uint32_t sbi = (uint32_t)warp; sbi < nb; sbi += 2 * C::CW) {
        const bool two = sbi + C::CW < nb;
        const float4 *src = reinterpret_cast<const float4 *>(x + (int64_t)sbi * kQK + lane * 8);
        const float4 p0 = __ldg(src), p1 = __ldg(src + 1);
        float4 p2 = make_float4(0.f, 0.f, 0.f, 0.f), p3 = p2;
        if (two) {
            p2 = __ldg(src + C::CW * kQK / 4);
            p3 = __ldg(src + C::CW * kQK / 4 + 1);
        }
        const float v0[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        stage_x_one<FMT>(v0, at, sbi, lane);
        if (two) {
            const float v1[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
            stage_x_one<FMT>(v1, at, sbi + C::CW, lane);
        }
    }
}

// Hand a ring stage back to the producer once this warp's reads of it are done.  Every lane
// first waits for its own shared-memory loads to complete (membar.cta): the loaded registers
// are consumed only after the release, and without the fence a lane's loads could still be
// in flight when lane 0's arrival lets the next bulk copy overwrite the stage (observed as
// wrong partials of whole warps on the GPU).
__device__ __forceinline__ void release_stage(uint64_t *bar, int lane) {
    __threadfence_block();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

template <int FMT, int MT, bool ACT, bool DUMP>
__global__ void __launch_bounds__(GvCfg<FMT>::THREADS, GvCfg<FMT>::ctas_per_sm(MT))
    gemv_kernel(GvArgs a0, const __grid_constant__ GvJobs jobs) {
    using C = GvCfg<FMT>;
    // this CTA's matrix: the launch's own (a0), or in a grouped launch its job's (selected with
    // compile-time indices, so the job table stays in parameter space)
    GvArgs a = a0;
    int cta = blockIdx.x, ncta = gridDim.x;
    if (jobs.n > 1) {
#pragma unroll
        for (int i = 0; i < kMaxJobs; ++i)
            if (i < jobs.n && (int)blockIdx.x >= jobs.cta0[i] && (int)blockIdx.x < jobs.cta0[i + 1]) {
                a.w = jobs.w[i];
                a.N = jobs.N[i];
                a.p = jobs.p[i];
                a.y = jobs.y[i];
                a.x = jobs.x[i];
                cta = blockIdx.x - jobs.cta0[i];
                ncta = jobs.cta0[i + 1] - jobs.cta0[i];
            }
    }
    const int S = a.nst;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[C::STAGES], empty[C::STAGES], pfull[kPartBufs], pempty[kPartBufs];
    __shared__ float carry[2][MT];
    __shared__ int abort_flag;
    float *partbuf = reinterpret_cast<float *>(smem + S * C::STAGE);   // [kPartBufs][MT][TU]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int i = 0; i < S; ++i) { mbar_init(&full[i], 1); mbar_init(&empty[i], C::CW); }
        for (int i = 0; i < kPartBufs; ++i) { mbar_init(&pfull[i], C::CW); mbar_init(&pempty[i], 1); }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    grid_dep_launch();

    // this CTA's rows [row_begin, row_end) and their flat super-block range
    const uint32_t nb = (uint32_t)(a.K / kQK);
    const int64_t row_begin = a.N * cta / ncta, row_end = a.N * (cta + 1) / ncta;
    const int64_t sb_begin = row_begin * nb, sb_total = (row_end - row_begin) * nb;
    const int units = (int)((sb_total + C::TU - 1) / C::TU);
    const float inv_nb = 1.0f / (float)nb;
    volatile int *abort = &abort_flag;

    // the 16-byte aligned superset of unit j's bytes: [a0, a1)
    auto unit_bytes = [&](int j, int64_t &a0, int64_t &a1) {
        const int64_t sb0 = sb_begin + (int64_t)j * C::TU;
        const int64_t nsb = min((int64_t)C::TU, sb_begin + sb_total - sb0);
        a0 = (sb0 * C::BB) & ~(int64_t)15;
        a1 = ((sb0 + nsb) * C::BB + 15) & ~(int64_t)15;
    };

    if (warp == C::PRODUCER) {
        if (lane != 0) return;
        // while the predecessor on the stream finishes: pull the first units into L2 (a hint,
        // safe whatever the predecessor writes), then wait for it before the real copies
        for (int j = 0; j < units && j < S; ++j) {
            int64_t a0, a1;
            unit_bytes(j, a0, a1);
            prefetch_l2_bulk(a.w + a0, (uint32_t)(a1 - a0));
        }
        grid_dep_wait();
        int s = 0, issued = 0;
        uint32_t ph = 0;
        for (int j = 0; j < units; ++j) {
            if (j >= S && !mbar_wait(&empty[s], ph ^ 1u, a.err, ERR_GEMV_FULL, abort)) break;
            int64_t a0, a1;
            unit_bytes(j, a0, a1);
            mbar_arrive_expect_tx(&full[s], (uint32_t)(a1 - a0));
            bulk_copy_g2s(smem + s * C::STAGE, a.w + a0, (uint32_t)(a1 - a0), &full[s]);
            ++issued;
            if (++s == S) { s = 0; ph ^= 1u; }
        }
        // after a failed wait: wait (bounded) for the copies still in flight before leaving
        if (*abort)
            for (int j = max(0, issued - S); j < issued; ++j)
                mbar_wait(&full[j % S], (uint32_t)((j / S) & 1), a.err, ERR_GEMV_DRAIN, nullptr);
        return;
    }

    if (warp == C::REDUCER) {
        // unit j covers flat super-blocks [sb0, sb0 + nsb); its first row is r_row0 and the
        // unit starts r_sbi0 super-blocks into it
        uint32_t r_sbi0 = 0;
        int64_t r_row0 = row_begin;
        int pb = 0;
        uint32_t pph = 0;
        for (int j = 0; j < units; ++j) {
            if (!mbar_wait(&pfull[pb], pph, a.err, ERR_GEMV_FULL, abort)) break;
            const int nsb = (int)min((int64_t)C::TU, sb_total - (int64_t)j * C::TU);
            const float *pbuf = partbuf + pb * MT * C::TU;
            const uint32_t nrows_u = (r_sbi0 + (uint32_t)nsb + nb - 1) / nb;   // rows touching this unit
            for (int t = 0; t < a.mt; ++t) {
                for (uint32_t rr = lane; rr < nrows_u; rr += 32) {
                    const int i0 = max(0, (int)(rr * nb) - (int)r_sbi0);
                    const int i1 = min(nsb, (int)((rr + 1) * nb) - (int)r_sbi0);
                    float sum = (rr == 0 && r_sbi0 > 0) ? carry[(j + 1) & 1][t] : 0.0f;
                    for (int i = i0; i < i1; ++i) sum += pbuf[t * C::TU + i];
                    if ((int)((rr + 1) * nb) - (int)r_sbi0 > nsb)
                        carry[j & 1][t] = sum;                                  // the row continues
                    else
                        a.y[(a.t0 + t) * a.N + r_row0 + rr] = sum;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&pempty[pb]);
            uint32_t adv;
            r_row0 += divmod_small(r_sbi0 + (uint32_t)nsb, nb, inv_nb, adv);
            r_sbi0 = adv;
            if (++pb == kPartBufs) { pb = 0; pph ^= 1u; }
        }
        return;
    }

    // consumer warps (the reducer writes y only after them, so after the predecessor too)
    grid_dep_wait();
    GvAct at{0, 0};
    if constexpr (ACT) {
        // stage the tokens' codes (padded layout) and their scale data
        at.codes = smem_u32(partbuf) + (uint32_t)C::part_bytes(MT);
        at.ck = nb * C::SB_STRIDE;
        bool staged = false;
        if constexpr (MT == 1 && !is_b32(FMT)) {
            if (a.x != nullptr) {
                stage_x<FMT>(a.x, at, nb, warp, lane);
                staged = true;
            }
        }
        const uint32_t nch = staged ? 0u : nb * 16u;  // 16-byte chunks of codes per token
        for (int t = 0; t < a.mt; ++t) {
            const int64_t m = a.t0 + t;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.p.q8 + m * a.K);
            const uint32_t cbase = at.codes + (uint32_t)t * at.ck;
            // all of an iteration's global loads go out before its stores (one latency round)
            for (uint32_t c = tid; c < nch; c += C::CW * 32) {
                const uint4 v = __ldg(src + c);
                const uint32_t sbi = c >> 4, r = c & 15u;     // chunk r of super-block sbi
                // chunk r: half r >> 3, block g = (r >> 1) & 3 of it, 16-value piece r & 1
                const uint32_t rec = cbase + sbi * C::SB_STRIDE + C::HALF * (r >> 3);
                sts128(rec + 16u * (r & 7u), v);
                if constexpr (FMT == FMT_Q6K) {
                    // the block's entry holds (d_a, -32 S16, -32 S16') at 128 + 16 g
                    const int s16 = dot16(v, make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u));
                    const uint32_t ent = rec + 128u + 16u * ((r >> 1) & 3u);
                    if (r & 1u) {
                        sts32(ent + 8u, (uint32_t)(-32 * s16));
                    } else {
                        const float da = __ldg(a.p.d + (int64_t)(c >> 1) * a.M + m);
                        sts32(ent, __float_as_uint(da));
                        sts32(ent + 4u, (uint32_t)(-32 * s16));
                    }
                } else if ((r & 1u) == 0) {
                    // the block's entry at 128 + 8 g: (d_a, d_a * S) for the formats with a min or
                    // offset m; (d_a, -off * S) for Q4_0 / Q5_0, the seed of their dp4a chains
                    const int64_t b = c >> 1;
                    const float da = __ldg(a.p.d + b * a.M + m);
                    const int S = __ldg(a.p.s + b * a.M + m);
                    const uint32_t x = (is_b32(FMT) && !b32_has_m(FMT)) ? (uint32_t)(-b32_off(FMT) * S)
                                                                        : __float_as_uint(da * (float)S);
                    sts64u(rec + 128u + 8u * ((r >> 1) & 3u), __float_as_uint(da), x);
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(C::CW * 32) : "memory");
    }

    // super-block slot within the unit, and the thread's half u = lane % 2 of it: Q4_K / Q5_K
    // slot 16 warp + lane / 2; Q6_K warps alternate between even and odd slots (so a warp's
    // 210-byte blocks share one alignment mod 4): slot 2 (16 (warp / 2) + lane / 2) + warp % 2
    const int u = lane & 1;
    const int slot = FMT != FMT_Q6K ? 16 * warp + (lane >> 1) : 2 * (16 * (warp >> 1) + (lane >> 1)) + (warp & 1);
    // this thread's super-block of each pass: offset in its row (and the row, for the dump);
    // both advance by TU super-blocks per unit
    const uint32_t tu_mod = (uint32_t)C::TU % nb, tu_div = (uint32_t)C::TU / nb;
    uint32_t t_sbi[C::PASSES];
    int64_t t_row[C::PASSES];
#pragma unroll
    for (int ps = 0; ps < C::PASSES; ++ps) {
        uint32_t r;
        t_row[ps] = row_begin + divmod_small((uint32_t)(ps * C::SB_PER_PASS + slot), nb, inv_nb, r);
        t_sbi[ps] = r;
    }
    const uint32_t off15 = (uint32_t)((sb_begin * C::BB) & 15);   // units start 16-byte aligned after that
    const int last = units - 1;
    const int nsb_last = (int)(sb_total - (int64_t)last * C::TU);
    const uint32_t ring = smem_u32(smem) + off15;
    // the stage base and 210 * (even slot) are multiples of 4, so a Q6_K warp's blocks are all
    // 4-byte aligned or all 2 mod 4
    const bool al4 = ((off15 + 2u * (uint32_t)(warp & 1)) & 2u) == 0;
    int s = 0, pb = 0;
    uint32_t ph = 0, pph = 0;
    for (int j = 0; j < units; ++j) {
        const bool got = mbar_wait(&full[s], ph, a.err, ERR_GEMV_FULL, abort);
        if (!__all_sync(kFull, got)) break;           // leave together: the shuffles below need every lane
        const int nsb = j == last ? nsb_last : C::TU;
        const uint32_t sbase = ring + (uint32_t)(s * C::STAGE);
        float part[C::PASSES][MT];
        // read this thread's weight bytes, hand the stage back to the producer, then do the
        // math on registers (the refill overlaps the dp4a work)
        static_assert(C::PASSES == 1, "one pass per unit");
        if constexpr (FMT == FMT_Q6K) {
            Q6Half raw;
            const uint32_t blk = sbase + (uint32_t)(slot * C::BB);
            if (al4)
                q6k_load_half<true>(blk, u, raw);
            else
                q6k_load_half<false>(blk, u, raw);
            release_stage(&empty[s], lane);
            q6k_half<MT, ACT, DUMP>(a, at, raw, t_row[0], t_sbi[0], u, slot < nsb, part[0]);
        } else {
            if constexpr (is_b32(FMT)) {
                B32Half<FMT> raw;
                b32_load_half<FMT>(sbase + (uint32_t)(slot * C::BB), u, raw);
                release_stage(&empty[s], lane);
                b32_half<FMT, MT, ACT, DUMP>(a, at, raw, t_row[0], t_sbi[0], u, slot < nsb, part[0]);
            } else if constexpr (FMT == FMT_Q4K) {
                Q4Half raw;
                q4k_load_half(sbase + (uint32_t)(slot * C::BB), u, raw);
                release_stage(&empty[s], lane);
                kq_half<FMT, MT, ACT, DUMP>(a, at, raw.hd, raw.q, nullptr, t_row[0], t_sbi[0], u, slot < nsb, part[0]);
            } else {
                Q5Half raw;
                q5k_load_half(sbase + (uint32_t)(slot * C::BB), u, raw);
                release_stage(&empty[s], lane);
                kq_half<FMT, MT, ACT, DUMP>(a, at, raw.hd, raw.q, raw.qh, t_row[0], t_sbi[0], u, slot < nsb, part[0]);
            }
        }
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps)
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                part[ps][t] += __shfl_xor_sync(kFull, part[ps][t], 1);
                if constexpr (C::TPS == 4) part[ps][t] += __shfl_xor_sync(kFull, part[ps][t], 2);
            }
        const bool pgot = j < kPartBufs || mbar_wait(&pempty[pb], pph ^ 1u, a.err, ERR_GEMV_FULL, abort);
        if (!__all_sync(kFull, pgot)) break;
        if (u == 0) {
            float *pbuf = partbuf + pb * MT * C::TU;
#pragma unroll
            for (int ps = 0; ps < C::PASSES; ++ps)
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    if (t < a.mt) pbuf[t * C::TU + ps * C::SB_PER_PASS + slot] = part[ps][t];
        }
        release_stage(&pfull[pb], lane);              // partials written: the reducer may read them
#pragma unroll
        for (int ps = 0; ps < C::PASSES; ++ps) {
            t_sbi[ps] += tu_mod;
            t_row[ps] += tu_div;
            if (t_sbi[ps] >= nb) { t_sbi[ps] -= nb; ++t_row[ps]; }
        }
        if (++s == S) { s = 0; ph ^= 1u; }
        if (++pb == kPartBufs) { pb = 0; pph ^= 1u; }
    }
}

// shared memory of one CTA with `nst` ring stages
template <int FMT, int MT, bool ACT>
int64_t gemv_smem(int nst, int64_t K) {
    using C = GvCfg<FMT>;
    return (int64_t)nst * C::STAGE + C::part_bytes(MT) + (ACT ? C::act_bytes(MT, K) : 0);
}

template <int FMT, int MT, bool ACT, bool DUMP>
int launch_one(GvArgs a, int nsm, cudaStream_t stream) {
    using C = GvCfg<FMT>;
    auto kern = gemv_kernel<FMT, MT, ACT, DUMP>;
    // the most CTAs per SM (up to what the registers allow, GvCfg::ctas_per_sm) whose shared
    // memory still fits with a 2-stage ring, then the deepest ring that keeps that many
    int budget = kSmemMax;
    for (int n = C::ctas_per_sm(MT); n >= 2; --n)
        if (gemv_smem<FMT, MT, ACT>(2, a.K) <= per_cta_smem(n)) { budget = per_cta_smem(n); break; }
    a.nst = C::STAGES;
    while (a.nst > 2 && gemv_smem<FMT, MT, ACT>(a.nst, a.K) > budget) --a.nst;
    const int smem = (int)gemv_smem<FMT, MT, ACT>(a.nst, a.K);
    constexpr int slot = 16 + FMT * 16 + (ACT ? 8 : 0) + (MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : 3) * 2 + (DUMP ? 1 : 0);
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), ACT ? kSmemMax : smem, slot);
    if (rc != MQ_OK) return rc;
    int per_sm = 0;
    rc = resident_ctas(reinterpret_cast<const void *>(kern), C::THREADS, smem, slot, &per_sm);
    if (rc != MQ_OK) return rc;
    int64_t ctas = (int64_t)nsm * per_sm;
    // at least one full unit of super-blocks per CTA: a small matrix (a 512-row k_proj is 56
    // units) then leaves most of the GPU to kernels running beside it on other streams
    const int64_t units = (a.N * (a.K / kQK) + C::TU - 1) / C::TU;
    if (ctas > units) ctas = units;
    if (ctas > a.N) ctas = a.N;                      // every CTA owns at least one row
    GvJobs none;
    none.n = 1;
    return cuda_error(launch_pdl(kern, dim3((unsigned)ctas), dim3(C::THREADS), smem, stream, a, none), "gemv launch");
}

// A grouped launch of jobs.n matrices (same format, K and tokens): one wave of CTAs, shared by the
// jobs in proportion to their weight bytes (at least one CTA each, at most one per unit or row).
template <int FMT, int MT, bool ACT>
int launch_group(GvArgs a, GvJobs jobs, int nsm, cudaStream_t stream) {
    using C = GvCfg<FMT>;
    auto kern = gemv_kernel<FMT, MT, ACT, false>;
    int budget = kSmemMax;
    for (int n = C::ctas_per_sm(MT); n >= 2; --n)
        if (gemv_smem<FMT, MT, ACT>(2, a.K) <= per_cta_smem(n)) { budget = per_cta_smem(n); break; }
    a.nst = C::STAGES;
    while (a.nst > 2 && gemv_smem<FMT, MT, ACT>(a.nst, a.K) > budget) --a.nst;
    const int smem = (int)gemv_smem<FMT, MT, ACT>(a.nst, a.K);
    constexpr int slot = 16 + FMT * 16 + (ACT ? 8 : 0) + (MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : 3) * 2;
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), ACT ? kSmemMax : smem, slot);
    if (rc != MQ_OK) return rc;
    int per_sm = 0;
    rc = resident_ctas(reinterpret_cast<const void *>(kern), C::THREADS, smem, slot, &per_sm);
    if (rc != MQ_OK) return rc;
    const int64_t wave = (int64_t)nsm * per_sm;
    const int64_t nb = a.K / kQK;
    int64_t total = 0;
    for (int i = 0; i < jobs.n; ++i) total += jobs.N[i] * nb;
    int c = 0;
    for (int i = 0; i < jobs.n; ++i) {
        jobs.cta0[i] = c;
        int64_t n = (wave * jobs.N[i] * nb + total - 1) / total;
        const int64_t units = (jobs.N[i] * nb + C::TU - 1) / C::TU;
        if (n > units) n = units;
        if (n > jobs.N[i]) n = jobs.N[i];
        if (n < 1) n = 1;
        c += (int)n;
    }
    jobs.cta0[jobs.n] = c;
    return cuda_error(launch_pdl(kern, dim3((unsigned)c), dim3(C::THREADS), smem, stream, a, jobs), "gemv launch");
}

template <int FMT, int MT, bool DUMP>
int launch_mt(const GvArgs &a, int nsm, cudaStream_t stream) {
    if (gemv_smem<FMT, MT, true>(2, a.K) <= kSmemMax) return launch_one<FMT, MT, true, DUMP>(a, nsm, stream);
    return launch_one<FMT, MT, false, DUMP>(a, nsm, stream);
}

template <int FMT, bool DUMP>
int launch_fmt(GvArgs a, int nsm, cudaStream_t stream) {
    constexpr int G = GvCfg<FMT>::MAX_MT;
    for (int64_t t0 = 0; t0 < a.M; t0 += G) {
        a.t0 = t0;
        a.mt = (int)((a.M - t0) < G ? (a.M - t0) : G);
        int rc;
        if (a.mt == 1)
            rc = launch_mt<FMT, 1, DUMP>(a, nsm, stream);
        else if (a.mt == 2)
            rc = launch_mt<FMT, 2, DUMP>(a, nsm, stream);
        else if (a.mt <= 4)
            rc = launch_mt<FMT, 4, DUMP>(a, nsm, stream);
        else
            rc = launch_mt<FMT, 8, DUMP>(a, nsm, stream);
        if (rc != MQ_OK) return rc;
    }
    return MQ_OK;
}

template <int FMT>
int launch_group_fmt(GvArgs a, const GvJobs &jobs, int nsm, cudaStream_t stream) {
    constexpr int G = GvCfg<FMT>::MAX_MT;
    for (int64_t t0 = 0; t0 < a.M; t0 += G) {
        a.t0 = t0;
        a.mt = (int)((a.M - t0) < G ? (a.M - t0) : G);
        int rc;
        const bool act = gemv_smem<FMT, 8, true>(2, a.K) <= kSmemMax;
        if (a.mt == 1)
            rc = gemv_smem<FMT, 1, true>(2, a.K) <= kSmemMax ? launch_group<FMT, 1, true>(a, jobs, nsm, stream)
                                                             : launch_group<FMT, 1, false>(a, jobs, nsm, stream);
        else if (a.mt == 2)
            rc = gemv_smem<FMT, 2, true>(2, a.K) <= kSmemMax ? launch_group<FMT, 2, true>(a, jobs, nsm, stream)
                                                             : launch_group<FMT, 2, false>(a, jobs, nsm, stream);
        else if (a.mt <= 4)
            rc = gemv_smem<FMT, 4, true>(2, a.K) <= kSmemMax ? launch_group<FMT, 4, true>(a, jobs, nsm, stream)
                                                             : launch_group<FMT, 4, false>(a, jobs, nsm, stream);
        else
            rc = act ? launch_group<FMT, 8, true>(a, jobs, nsm, stream) : launch_group<FMT, 8, false>(a, jobs, nsm, stream);
        if (rc != MQ_OK) return rc;
    }
    return MQ_OK;
}

}  // namespace

}  // namespace mq
