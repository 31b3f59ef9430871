// mq_gemv.cu -- decode GEMV (MMVQ): raw Q4_K / Q6_K weight bytes x Q8 codes with dp4a.
//
// minfer pages, "Support Matrix > CUDA notes": decode (nt == 1) uses the dp4a MMVQ
// kernels; "Roadmap > 0": the decode path streams the weights once per token.
//
// Design (HBM-bound): every weight byte is read from HBM exactly once per group of up
// to 8 (Q4_K) or 4 (Q6_K) tokens.  The weight matrix is one flat stream of super-blocks
// (row-major, rows contiguous).  Each CTA owns a contiguous range of whole rows and walks
// it in units of TU super-blocks (a unit may start or end inside a row):
//   * a producer warp refills a 2-5 stage shared-memory ring with ONE large 1-D bulk copy
//     (TMA engine) per unit -- the 16-byte aligned superset of the unit's bytes, so the
//     2-byte aligned 210-byte Q6_K block needs no special load path.  A few large copies
//     per SM keep the copy engine streaming at full HBM rate, where many small per-warp
//     copies stall it;
//   * consumer warps take a super-block with 4 threads (Q4_K, 64 values each) or 2 threads
//     (Q6_K, one 128-value half each), so the per-unit hand-offs and the scale decoding
//     amortize over many values: dp4a against the int8 codes, f32 scaling per 32-value
//     block, a lane reduction, and one partial per (token, super-block) into a ring of
//     partial buffers;
//   * a reducer warp sums each row's partials in a fixed order (a row that continues
//     into the next unit carries its running sum), so results are deterministic, and
//     writes Y.  Consumers wait for the reducer only when the partial ring is full.
// The shared-memory data pipe is the scarce resource once the weights stream at full
// rate: when the tokens' activations fit, each CTA first stages them in shared memory
// (codes in a padded layout that spreads every lane pattern below over distinct bank
// groups, plus per-block scale data: (d_a, d_a * S) for Q4_K; d_a and the -32 code
// offset as -32 * S16 per 16-value half block for Q6_K, which seeds the dp4a chain), so
// the inner loop reads 4 wavefronts per 512 bytes instead of one scattered L1 line per lane.
#include <cuda_fp16.h>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int kPartBufs = 4;
constexpr unsigned kFull = 0xffffffffu;

template <int FMT>
struct GvCfg {
    static constexpr int BB = FMT == FMT_Q4K ? 144 : 210;
    static constexpr int CW = FMT == FMT_Q4K ? 8 : 4;          // consumer warps
    static constexpr int TPS = FMT == FMT_Q4K ? 4 : 2;         // consumer threads per super-block
    static constexpr int THREADS = (CW + 2) * 32;              // + producer warp + reducer warp
    static constexpr int PRODUCER = CW, REDUCER = CW + 1;
    static constexpr int SB_PER_PASS = CW * 32 / TPS;          // 64
    static constexpr int PASSES = FMT == FMT_Q4K ? 2 : 1;
    static constexpr int TU = SB_PER_PASS * PASSES;            // super-blocks per unit
    static constexpr int STAGES = FMT == FMT_Q4K ? 4 : 5;  // at most; a launch may use fewer (GvArgs::nst)
    // tokens per pass over the weights (Q6_K: the staged activations of 8 tokens would leave
    // room for too few CTAs per SM; two passes of 4 measure faster)
    static constexpr int MAX_MT = FMT == FMT_Q4K ? 8 : 4;
    // CTAs per SM the launch aims for (registers: 64K / (THREADS * this))
    static constexpr int ctas_per_sm(int mt) { return FMT == FMT_Q4K ? (mt <= 2 ? 3 : 2) : (mt <= 2 ? 4 : 3); }
    // unit bytes + up to 15 leading and 15 trailing alignment bytes, + 16 bytes of slack
    static constexpr int STAGE = ((TU * BB + 30 + 15) / 16) * 16 + 16;
    static constexpr int part_bytes(int mt) { return kPartBufs * mt * TU * 4; }
    // Staged activations, per token.  Q4_K: int8 codes with each super-block's two 128-value
    // halves padded apart (half stride 160 B = 10 bank groups of 16 B, super-block stride 304 B
    // = 19 groups) so that the 8 lanes of every quarter-warp -- two consecutive super-blocks x
    // four quarters -- read 8 distinct 16-byte bank groups; then a float2 (d_a, d_a * S) table
    // per block (TAB_SB = 64 B per super-block).  Q6_K: one record per half super-block, the
    // 128 codes then 4 x 16 B of scale data ((d_a, -32 S16 of the first and second 16 values),
    // one entry per 32-value block); half stride HALF = 208 B (5 mod 8 groups), super-block
    // stride 464 B (5 mod 8 groups): a quarter-warp's 8 lanes -- four super-blocks two apart x
    // two halves -- then hit 8 distinct groups (away from row ends).
    static constexpr uint32_t SB_STRIDE = FMT == FMT_Q6K ? 464 : 304;
    static constexpr uint32_t HALF = 208;
    static constexpr uint32_t TAB_SB = FMT == FMT_Q6K ? 0 : 64;
    static int64_t act_bytes(int mt, int64_t K) { return (int64_t)mt * (K / kQK) * (SB_STRIDE + TAB_SB); }
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
__device__ __forceinline__ void sts64(uint32_t addr, float a, float b) {
    asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ float4 lds128f(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}
// 16 bytes at a 2-byte aligned shared address (five aligned words, funnel-shifted)
__device__ __forceinline__ uint4 lds128_a2(uint32_t addr) {
    const uint32_t b = addr & ~3u, sh = (addr & 3u) * 8u;
    const uint32_t w0 = lds32(b), w1 = lds32(b + 4), w2 = lds32(b + 8), w3 = lds32(b + 12), w4 = lds32(b + 16);
    return make_uint4(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh), __funnelshift_r(w2, w3, sh),
                      __funnelshift_r(w3, w4, sh));
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
};

// shared-memory addresses of the staged activations (ACT kernels): codes [MT][K], table
struct GvAct {
    uint32_t codes, tab;         // token 0's codes and table
    uint32_t ck, tk;             // per-token strides of codes and table
};

// A thread's raw weight bytes of one super-block quarter, read from the stage before the
// stage is handed back to the producer (the math runs on these registers afterwards).
struct Q4Raw {
    uint4 hd, q0, q1;
};
// Q6_K: half h of a super-block -- ql bytes [64h, 64h+64), qh bytes [128+32h, 128+32h+32),
// the eight int8 scales 8h .. 8h+7 and the fp16 d.
struct Q6Half {
    uint32_t ql[16], qh[8], sc[2], dbits;
};

// Q4_K: quarter u of the super-block at shared address `blk`: its header and qs bytes
// [32u, 32u+32), whose low nibbles are sub-block 2u and high nibbles 2u+1.
__device__ __forceinline__ Q4Raw q4k_load(uint32_t blk, int u, bool valid) {
    Q4Raw r{make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
    if (valid) {
        r.hd = lds128(blk);
        r.q0 = lds128(blk + 16 + 32 * u);
        r.q1 = lds128(blk + 32 + 32 * u);
    }
    return r;
}

// Q4_K quarter math (row n, super-block sbi of the row) on the loaded bytes
template <int MT, bool ACT, bool DUMP>
__device__ __forceinline__ void q4k_quarter(const GvArgs &a, const GvAct &at, const Q4Raw &raw, int64_t n,
                                            uint32_t sbi, int u, bool valid, float (&part)[MT]) {
    using C = GvCfg<FMT_Q4K>;
    const uint4 hd = raw.hd, q0 = raw.q0, q1 = raw.q1;
    const float d = half_bits_to_float(hd.x & 0xffff), dmin = half_bits_to_float(hd.x >> 16);
    // the 12 scale bytes: s[0..3] = hd.y, s[4..7] = hd.z, s[8..11] = hd.w; sub-blocks 2u, 2u+1
    int sc0, m0, sc1, m1;
    if (u < 2) {
        const uint32_t x = hd.y >> (16 * u), z = hd.z >> (16 * u);
        sc0 = x & 63; sc1 = (x >> 8) & 63; m0 = z & 63; m1 = (z >> 8) & 63;
    } else {
        const uint32_t lo = hd.w >> (16 * (u - 2));                                 // s[j+4], j = 2u, 2u+1
        const uint32_t ts = hd.y >> (16 * (u - 2)), tm = hd.z >> (16 * (u - 2));   // s[j-4], s[j]
        sc0 = (lo & 15) | (((ts >> 6) & 3) << 4);
        sc1 = ((lo >> 8) & 15) | (((ts >> 14) & 3) << 4);
        m0 = ((lo >> 4) & 15) | (((tm >> 6) & 3) << 4);
        m1 = ((lo >> 12) & 15) | (((tm >> 14) & 3) << 4);
    }
    const uint4 lo0 = make_uint4(q0.x & 0x0f0f0f0fu, q0.y & 0x0f0f0f0fu, q0.z & 0x0f0f0f0fu, q0.w & 0x0f0f0f0fu);
    const uint4 lo1 = make_uint4(q1.x & 0x0f0f0f0fu, q1.y & 0x0f0f0f0fu, q1.z & 0x0f0f0f0fu, q1.w & 0x0f0f0f0fu);
    const uint4 hi0 = make_uint4((q0.x >> 4) & 0x0f0f0f0fu, (q0.y >> 4) & 0x0f0f0f0fu, (q0.z >> 4) & 0x0f0f0f0fu,
                                 (q0.w >> 4) & 0x0f0f0f0fu);
    const uint4 hi1 = make_uint4((q1.x >> 4) & 0x0f0f0f0fu, (q1.y >> 4) & 0x0f0f0f0fu, (q1.z >> 4) & 0x0f0f0f0fu,
                                 (q1.w >> 4) & 0x0f0f0f0fu);
    const int64_t k0 = (int64_t)sbi * kQK + 64 * u;    // values 64u .. 64u+63 of the super-block
    const int64_t b0 = (int64_t)sbi * 8 + 2 * u, b1 = b0 + 1;   // their two Q8 blocks
    const float dsc0 = d * (float)sc0, dsc1 = d * (float)sc1, dm0 = dmin * (float)m0, dm1 = dmin * (float)m1;
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int64_t m = a.t0 + t;
        const bool act = t < a.mt && valid;
        int D0 = 0, D1 = 0;
        part[t] = 0.0f;
        if (act) {
            if constexpr (ACT) {
                // codes 64u .. 64u+63 of the super-block (half u/2, offset 64 (u&1) in it);
                // table: (d, d*S) of blocks 2u, 2u+1
                const uint32_t cb = at.codes + (uint32_t)t * at.ck + sbi * C::SB_STRIDE +
                                    160u * ((uint32_t)u >> 1) + 64u * ((uint32_t)u & 1u);
                const uint4 x0 = lds128(cb), x1 = lds128(cb + 16), x2 = lds128(cb + 32), x3 = lds128(cb + 48);
                D0 = dot16(lo0, x0) + dot16(lo1, x1);
                D1 = dot16(hi0, x2) + dot16(hi1, x3);
                const float4 tb = lds128f(at.tab + (uint32_t)t * at.tk + sbi * C::TAB_SB + 16u * (uint32_t)u);
                part[t] = fmaf(dsc0, tb.x * (float)D0, -dm0 * tb.y) + fmaf(dsc1, tb.z * (float)D1, -dm1 * tb.w);
            } else {
                const uint4 *q = reinterpret_cast<const uint4 *>(a.p.q8 + m * a.K + k0);
                D0 = dot16(lo0, __ldg(q)) + dot16(lo1, __ldg(q + 1));
                D1 = dot16(hi0, __ldg(q + 2)) + dot16(hi1, __ldg(q + 3));
                const float da0 = __ldg(a.p.d + b0 * a.M + m), da1 = __ldg(a.p.d + b1 * a.M + m);
                const float s0 = (float)__ldg(a.p.s + b0 * a.M + m), s1 = (float)__ldg(a.p.s + b1 * a.M + m);
                part[t] = da0 * (dsc0 * (float)D0 - dm0 * s0) + da1 * (dsc1 * (float)D1 - dm1 * s1);
            }
        }
        if constexpr (DUMP) {
            const Dump &dp = a.dump;
            if (act && m >= dp.m0 && m < dp.m0 + dp.m_cnt && n >= dp.n0 && n < dp.n0 + dp.n_cnt) {
                int32_t *o = dp.out + ((m - dp.m0) * dp.n_cnt + (n - dp.n0)) * (a.K / kQ8);
                o[b0] = sc0 * D0;
                o[b1] = sc1 * D1;
            }
        }
    }
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

template <int FMT, int MT, bool ACT, bool DUMP>
__global__ void __launch_bounds__(GvCfg<FMT>::THREADS, GvCfg<FMT>::ctas_per_sm(MT)) gemv_kernel(GvArgs a) {
    using C = GvCfg<FMT>;
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
    const int64_t row_begin = a.N * blockIdx.x / gridDim.x, row_end = a.N * (blockIdx.x + 1) / gridDim.x;
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
    GvAct at{0, 0, 0, 0};
    if constexpr (ACT) {
        // stage the tokens' codes (padded layout) and their scale data
        at.codes = smem_u32(partbuf) + (uint32_t)C::part_bytes(MT);
        at.ck = nb * C::SB_STRIDE;
        at.tab = at.codes + MT * at.ck;
        at.tk = nb * C::TAB_SB;
        const uint32_t nch = nb * 16u;                // 16-byte chunks of codes per token
        for (int t = 0; t < a.mt; ++t) {
            const int64_t m = a.t0 + t;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.p.q8 + m * a.K);
            const uint32_t cbase = at.codes + (uint32_t)t * at.ck, tbase = at.tab + (uint32_t)t * at.tk;
            // all of an iteration's global loads go out before its stores (one latency round)
            for (uint32_t c = tid; c < nch; c += C::CW * 32) {
                const uint4 v = __ldg(src + c);
                const uint32_t sbi = c >> 4, r = c & 15u;     // chunk r of super-block sbi
                if constexpr (FMT == FMT_Q6K) {
                    // chunk r: half r >> 3, block g = (r >> 1) & 3 of it, its 16-value sub-block
                    // r & 1; the block's entry holds (d_a, -32 S16, -32 S16') at 128 + 16 g
                    const uint32_t rec = cbase + sbi * C::SB_STRIDE + C::HALF * (r >> 3);
                    sts128(rec + 16u * (r & 7u), v);
                    const int s16 = dot16(v, make_uint4(0x01010101u, 0x01010101u, 0x01010101u, 0x01010101u));
                    const uint32_t ent = rec + 128u + 16u * ((r >> 1) & 3u);
                    if (r & 1u) {
                        sts32(ent + 8u, (uint32_t)(-32 * s16));
                    } else {
                        const float da = __ldg(a.p.d + (int64_t)(c >> 1) * a.M + m);
                        sts32(ent, __float_as_uint(da));
                        sts32(ent + 4u, (uint32_t)(-32 * s16));
                    }
                } else {
                    // block c (< K/32): (d_a, d_a * S)
                    const bool blk = c < nb * 8u;
                    const float da = blk ? __ldg(a.p.d + (int64_t)c * a.M + m) : 0.0f;
                    const float sa = blk ? (float)__ldg(a.p.s + (int64_t)c * a.M + m) : 0.0f;
                    sts128(cbase + sbi * C::SB_STRIDE + 160u * (r >> 3) + 16u * (r & 7u), v);
                    if (blk) sts64(tbase + 8u * c, da, da * sa);
                }
            }
        }
        asm volatile("bar.sync 1, %0;" ::"n"(C::CW * 32) : "memory");
    }

    // super-block slot within a pass, and the thread's part of it: Q4_K quarter u = tid % 4 of
    // slot tid / 4; Q6_K half u = lane % 2, warps alternating between even and odd slots (so a
    // warp's blocks share one alignment mod 4): slot 2 (16 (warp / 2) + lane / 2) + warp % 2
    const int u = FMT == FMT_Q4K ? (tid & 3) : (lane & 1);
    const int slot = FMT == FMT_Q4K ? (tid >> 2) : 2 * (16 * (warp >> 1) + (lane >> 1)) + (warp & 1);
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
        if constexpr (FMT == FMT_Q6K) {
            // one pass: read this thread's weight bytes, hand the stage back to the producer,
            // then do the math on registers (the refill overlaps the dp4a work)
            static_assert(C::PASSES == 1, "Q6_K takes one pass per unit");
            Q6Half raw;
            const uint32_t blk = sbase + (uint32_t)(slot * C::BB);
            if (al4)
                q6k_load_half<true>(blk, u, raw);
            else
                q6k_load_half<false>(blk, u, raw);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);   // stage read: the producer may refill it
            q6k_half<MT, ACT, DUMP>(a, at, raw, t_row[0], t_sbi[0], u, slot < nsb, part[0]);
        } else {
            // two passes, each loading and computing in turn (fewer live registers); the stage
            // goes back after the last one
#pragma unroll
            for (int ps = 0; ps < C::PASSES; ++ps) {
                const int idx = ps * C::SB_PER_PASS + slot;
                const Q4Raw raw = q4k_load(sbase + (uint32_t)(idx * C::BB), u, idx < nsb);
                q4k_quarter<MT, ACT, DUMP>(a, at, raw, t_row[ps], t_sbi[ps], u, idx < nsb, part[ps]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);   // stage fully read: the producer may refill it
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
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[pb]);
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
    if (ctas > a.N) ctas = a.N;                      // every CTA owns at least one row
    return cuda_error(launch_pdl(kern, dim3((unsigned)ctas), dim3(C::THREADS), smem, stream, a), "gemv launch");
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

}  // namespace

int launch_gemv(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream) {
    const int nsm = sm_count();
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    GvArgs a{w, N, K, p, M, 0, 0, 0, y, dump, err};
    if (fmt == FMT_Q4K)
        return dmp ? launch_fmt<FMT_Q4K, true>(a, nsm, stream) : launch_fmt<FMT_Q4K, false>(a, nsm, stream);
    return dmp ? launch_fmt<FMT_Q6K, true>(a, nsm, stream) : launch_fmt<FMT_Q6K, false>(a, nsm, stream);
}

}  // namespace mq
