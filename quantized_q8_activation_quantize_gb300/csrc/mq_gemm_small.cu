// mq_gemm_small.cu -- the small-M band (1 <= M <= 32 tokens) on the tensor cores: raw Q4_K / Q5_K /
// Q6_K weights x Q8 plane, every weight byte streamed from HBM once for all the tokens.
//
// minfer pages, "Support Matrix > CUDA notes": decode (nt == 1) runs the dp4a MMVQ kernels and
// prefill (nt >= 16) the MMQ GEMM, the band in between general kernels; "Features > Continuous
// batching": several sequences decoded together.  This kernel gives the band its own path: the
// roles of the prefill GEMM are swapped, so a CTA's 128 unpacked weight rows are the MMA's M = 128
// operand and the tokens, padded to NT = 16 or 32, its N side.  One pass over W then serves every
// token, and the MMA work per weight byte is small enough that the kernel runs at the pace of the
// weight stream and its unpacking.  The integer block dots are the exact f16-operand / f32-accumulator
// integers of the prefill GEMM (q8 codes and sc*q are exact in f16, every 32-value sum below 2^24):
// one TMEM accumulator of NT columns per 32-value block, the two blocks of a 64-value stage side by
// side in one ring entry (four entries), so the block-dot checkpoint is bit-exact.  Every barrier
// probe costs a shared-memory round trip even when the phase is complete, so the MMA issuer probes a
// stage's three conditions at once and the epilogue and unpackers probe one step ahead.
//
// CTA = 16 warps: 0 TMA producer of the token code tiles, 1 MMA issuer (and TMEM owner),
// 2 activation-scale stager, 3 TMA producer of the raw weights and token d*S tiles, 4-11 unpackers (two threads per
// weight row, one 32-value block each per 64-value stage), 12-15 epilogue (one weight row per
// thread, all tokens).
#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int SW = 128, SBK = 64;              // weight rows per CTA (MMA M), K per stage
constexpr int kSmThreads = 512;
constexpr int kSmWarpTma = 0, kSmWarpMma = 1, kSmWarpDa = 2, kSmWarpRaw = 3, kSmWarpUnpack0 = 4, kSmWarpEpi0 = 12;
constexpr int kEnt = 4;                        // TMEM ring entries: one per 64-value stage (two block accumulators)
constexpr unsigned kAll = 0xffffffffu;
constexpr int kWTile = SW * SBK * 2;           // one 128 x 64 f16 weight tile (16 KB)

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

__host__ __device__ constexpr int sm_align(int x, int a) { return (x + a - 1) / a * a; }

template <int FMT, int NT>
struct SmCfg {
    static constexpr bool KQ = FMT == FMT_Q4K || FMT == FMT_Q5K;       // Q4_K-style header and min term
    static constexpr bool MIN = KQ;
    static constexpr bool TMW = FMT != FMT_Q6K;                         // raw rows by TMA
    static constexpr bool CORR = FMT == FMT_Q6K;                        // odd |sc| > 64 correction tile
    static constexpr int BB = block_bytes(FMT);
    static constexpr int S = 4;                                          // 64-value stages in flight
    static constexpr int R = FMT == FMT_Q6K ? 2 : 3;                     // raw super-block slots
    static constexpr int RAW_ROW = TMW ? BB : 240;                       // Q6_K: 16-B aligned superset
    static constexpr int XTILE = NT * SBK * 2;                           // token codes of one stage
    // the token tiles have their own, deeper ring: they come from L2 with a latency of a few stages
    static constexpr int XS = NT == 16 ? 16 : 6;
    static constexpr int MIN_W = SW * 64, MIN_X = NT * 64;               // tf32 (hi, lo) x 8 per row
    static constexpr int TMEM_COLS = (2 * kEnt + 1) * NT <= 256 ? 256 : 512;
    static constexpr uint32_t MIN_COL = 2 * kEnt * NT;
    static constexpr int OFF_W = 0;
    static constexpr int OFF_WC = OFF_W + S * kWTile;
    static constexpr int OFF_X = OFF_WC + (CORR ? S * kWTile : 0);
    static constexpr int OFF_WMIN = sm_align(OFF_X + XS * XTILE, 1024);
    static constexpr int OFF_XMIN = OFF_WMIN + (MIN ? 2 * MIN_W : 0);
    static constexpr int OFF_RAW = sm_align(OFF_XMIN + (MIN ? 2 * MIN_X : 0), 1024);
    static constexpr int OFF_INFO = OFF_RAW + R * SW * RAW_ROW;          // d per weight row [2][128]
    // the tokens' activation scales d_a [DAS][8 blocks][NT tokens]: a deep ring, since each slot is
    // filled by plain global loads (the plane's d section has a row stride of M floats)
    static constexpr int DAS = NT == 16 ? 8 : 4;
    static constexpr int OFF_DA = OFF_INFO + 2 * SW * 4;
    static constexpr int OFF_FLAG = OFF_DA + DAS * 8 * NT * 4;           // Q6_K correction flags [S][8]
    static constexpr int OFF_BAR = sm_align(OFF_FLAG + S * 8 * 4, 8);
    // w_full[S] w_empty[S] x_full[XS] x_empty[XS] raw_full[R] raw_empty[R] info_full[2] info_empty[2]
    // xmin_full[2] xmin_empty[2] acc_full[4] acc_empty[4] da_full[DAS] da_empty[DAS] min_final
    static constexpr int NBARS = 2 * S + 2 * XS + 2 * R + 8 + 2 * kEnt + 2 * DAS + 1;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA exceeds the per-CTA limit");
    static_assert(NT == 16 || NT == 32, "token tile: 16 or 32");
};

struct SmBars {
    uint64_t *w_full, *wx_empty, *x_full, *x_empty, *raw_full, *raw_empty, *info_full, *info_empty, *xmin_full, *xmin_empty;
    uint64_t *acc_full, *acc_empty, *da_full, *da_empty, *min_final;
};

__device__ __forceinline__ uint32_t sm_lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 sm_lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ void sm_sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// NW words starting r bytes (r even, < 16) past the 16-byte aligned shared address base (16-byte
// loads, the word offset chosen by selects, the half-word offset by a funnel shift)
template <int NW>
__device__ __forceinline__ void sm_words_r(uint32_t base, uint32_t r, uint32_t (&out)[NW]) {
    constexpr int NC = (NW + 4 + 3) / 4;
    uint32_t w[4 * NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 t = sm_lds128(base + 16u * c);
        w[4 * c] = t.x;
        w[4 * c + 1] = t.y;
        w[4 * c + 2] = t.z;
        w[4 * c + 3] = t.w;
    }
    const bool s1 = (r & 4u) != 0, s2 = (r & 8u) != 0;
    const uint32_t sh = (r & 2u) * 8u;
    uint32_t x[NW + 3];
#pragma unroll
    for (int i = 0; i < NW + 3; ++i) x[i] = s1 ? w[i + 1] : w[i];
    uint32_t v[NW + 1];
#pragma unroll
    for (int i = 0; i < NW + 1; ++i) v[i] = s2 ? x[i + 2] : x[i];
#pragma unroll
    for (int i = 0; i < NW; ++i) out[i] = __funnelshift_r(v[i], v[i + 1], sh);
}
__device__ __forceinline__ uint32_t sm_h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 sm_u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }
// four quant bytes (each < 64) -> two f16x2 words holding 1024 + byte
__device__ __forceinline__ void sm_bytes_biased(uint32_t v, uint32_t &lo, uint32_t &hi) {
    lo = __byte_perm(v, 0x64646464u, 0x4140);
    hi = __byte_perm(v, 0x64646464u, 0x4342);
}
// 128-byte / 64-byte swizzled address of 16-byte chunk c of row r in a K-major tile
__device__ __forceinline__ uint32_t sm_sw128(uint32_t tile, int r, int c) {
    return tile + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
__device__ __forceinline__ uint32_t sm_sw64(uint32_t tile, int r, int c) {
    return tile + (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}
// 32 lanes x 16 consecutive columns
__device__ __forceinline__ void sm_tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
template <int NT>
__device__ __forceinline__ void sm_tmem_ld(uint32_t taddr, uint32_t (&v)[NT]) {
    if constexpr (NT == 32) {
        tmem_ld32(taddr, v);
    } else {
        sm_tmem_ld16(taddr, v);
    }
}

template <int FMT, int NT, bool DUMP>
__global__ void __launch_bounds__(kSmThreads, 1)
    small_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmXS,
                 const __grid_constant__ CUtensorMap tmW, const uint8_t *__restrict__ w, int64_t N, int64_t K, Plane p,
                 int64_t M, float *__restrict__ y, Dump dump, unsigned int *err) {
    using C = SmCfg<FMT, NT>;
    constexpr int S = C::S, R = C::R;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar0 = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    SmBars bars;
    bars.w_full = bar0;
    bars.wx_empty = bars.w_full + S;
    bars.x_full = bars.wx_empty + S;
    bars.x_empty = bars.x_full + C::XS;
    bars.raw_full = bars.x_empty + C::XS;
    bars.raw_empty = bars.raw_full + R;
    bars.info_full = bars.raw_empty + R;
    bars.info_empty = bars.info_full + 2;
    bars.xmin_full = bars.info_empty + 2;
    bars.xmin_empty = bars.xmin_full + 2;
    bars.acc_full = bars.xmin_empty + 2;
    bars.acc_empty = bars.acc_full + kEnt;
    bars.da_full = bars.acc_empty + kEnt;
    bars.da_empty = bars.da_full + C::DAS;
    bars.min_final = bars.da_empty + C::DAS;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);
    volatile uint32_t *corr_flags = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_FLAG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t n0 = (int64_t)blockIdx.x * SW;
    const int nsb = (int)(K / kQK);
    const int nstages = nsb * 4;
    const int64_t row_bytes = (int64_t)nsb * C::BB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars.w_full[s], 8);                   // the unpack warps
            mbar_init(&bars.wx_empty[s], 1);
        }
        for (int s = 0; s < C::XS; ++s) {
            mbar_init(&bars.x_full[s], 1);
            mbar_init(&bars.x_empty[s], 1);
        }
        for (int r = 0; r < R; ++r) {
            mbar_init(&bars.raw_full[r], C::TMW ? 1 : SW);  // TMA, or one bulk copy per row
            mbar_init(&bars.raw_empty[r], 8);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.info_full[i], 8);
            mbar_init(&bars.info_empty[i], C::MIN ? 5 : 4);  // epilogue warps (+ the min MMA)
            mbar_init(&bars.xmin_full[i], 1);
            mbar_init(&bars.xmin_empty[i], 1);
        }
        for (int i = 0; i < kEnt; ++i) {
            mbar_init(&bars.acc_full[i], 1);
            mbar_init(&bars.acc_empty[i], 4);
        }
        for (int i = 0; i < C::DAS; ++i) {
            mbar_init(&bars.da_full[i], 1);
            mbar_init(&bars.da_empty[i], 4);
        }
        mbar_init(bars.min_final, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kSmWarpMma) tmem_alloc(tmem_holder, C::TMEM_COLS);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    grid_dep_launch();
    grid_dep_wait();

    if (warp == kSmWarpTma) {
        // ------------------------------------------------------------ TMA producer: token code tiles
        if (lane == 0) {
            prefetch_tmap(&tmX);
            int st = 0;
            for (; st < nstages && !*abort_flag; ++st) {
                const int s = st % C::XS;
                if (!mbar_wait(&bars.x_empty[s], ((st / C::XS) & 1) ^ 1, err, ERR_GEMM_AB_EMPTY, abort_flag)) break;
                mbar_arrive_expect_tx(&bars.x_full[s], C::XTILE);
                tma_load_2d(sm + C::OFF_X + s * C::XTILE, &tmX, st * SBK, 0, &bars.x_full[s]);
            }
            if (*abort_flag) {   // leave no copy in flight
                for (int i = st - 1; i >= 0 && i >= st - C::XS; --i)
                    mbar_wait(&bars.x_full[i % C::XS], (i / C::XS) & 1, err, ERR_GEMM_A_FULL, nullptr);
            }
        }
    } else if (warp == kSmWarpRaw) {
        // ------------------------------------------------------------ TMA producer: raw weights, token d*S tiles
        // (its own thread, so a slot that the unpackers have not yet handed back never holds up the
        // token tiles)
        if (lane == 0 && (C::TMW || C::MIN)) {
            if constexpr (C::MIN) prefetch_tmap(&tmXS);
            if constexpr (C::TMW) prefetch_tmap(&tmW);
            int raw_issued = 0, xs_issued = 0;
            for (int sb = 0; sb < nsb && !*abort_flag; ++sb) {
                if constexpr (C::TMW) {
                    const int slot = sb % R;
                    if (!mbar_wait(&bars.raw_empty[slot], ((sb / R) & 1) ^ 1, err, ERR_GEMM_RAW_FULL, abort_flag)) break;
                    mbar_arrive_expect_tx(&bars.raw_full[slot], SW * C::RAW_ROW);
                    tma_load_2d(sm + C::OFF_RAW + slot * SW * C::RAW_ROW, &tmW, sb * C::BB, (int32_t)n0,
                                &bars.raw_full[slot]);
                    raw_issued = sb + 1;
                }
                if constexpr (C::MIN) {
                    if (!mbar_wait(&bars.xmin_empty[sb & 1], ((sb >> 1) & 1) ^ 1, err, ERR_GEMM_MIN, abort_flag)) break;
                    mbar_arrive_expect_tx(&bars.xmin_full[sb & 1], C::MIN_X);
                    tma_load_2d(sm + C::OFF_XMIN + (sb & 1) * C::MIN_X, &tmXS, sb * 16, 0, &bars.xmin_full[sb & 1]);
                    xs_issued = sb + 1;
                }
            }
            if (*abort_flag) {
                for (int sb = xs_issued - 1; sb >= 0 && sb >= xs_issued - 2; --sb)
                    mbar_wait(&bars.xmin_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_MIN, nullptr);
                for (int sb = raw_issued - 1; sb >= 0 && sb >= raw_issued - R; --sb)
                    mbar_wait(&bars.raw_full[sb % R], (sb / R) & 1, err, ERR_GEMM_RAW_FULL, nullptr);
            }
        }
    } else if (warp == kSmWarpMma) {
        // ------------------------------------------------------------ MMA issuer (whole warp, one elected lane issues)
        constexpr uint32_t idesc = idesc_f16_f32(SW, NT);
        constexpr uint32_t idesc_min = idesc_tf32_f32(SW, NT);
        const uint64_t w_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_W));
        const uint64_t wc_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_WC));
        const uint64_t x_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_X));
        const uint32_t wmin_base = smem_u32(sm + C::OFF_WMIN), xmin_base = smem_u32(sm + C::OFF_XMIN);
        auto wait_all = [&](uint64_t *bar, uint32_t ph, uint32_t code) {
            return __all_sync(kAll, mbar_wait_prompt(bar, ph, err, code, abort_flag));
        };
        // the min term of super-block x into its own TMEM columns, summed over the whole K:
        // (-dmin m_j) x (d_a S), both operands tf32 (hi, lo) pairs: hi*hi + lo*hi + hi*lo
        auto issue_min = [&](int x) -> bool {
            const uint32_t ph = (x >> 1) & 1;
            if (!wait_all(&bars.xmin_full[x & 1], ph, ERR_GEMM_MIN) ||
                !wait_all(&bars.info_full[x & 1], ph, ERR_GEMM_INFO_FULL))
                return false;
            tc_fence_after();
            const uint32_t wt = wmin_base + (x & 1) * C::MIN_W, xt = xmin_base + (x & 1) * C::MIN_X;
            mma_tf32_warp(tmem + C::MIN_COL, sw64_kmajor_desc(wt), sw64_kmajor_desc(xt), idesc_min, x > 0 ? 1u : 0u);
            mma_tf32_warp(tmem + C::MIN_COL, sw64_kmajor_desc(wt + 32), sw64_kmajor_desc(xt), idesc_min, 1u);
            mma_tf32_warp(tmem + C::MIN_COL, sw64_kmajor_desc(wt), sw64_kmajor_desc(xt + 32), idesc_min, 1u);
            mma_commit_warp(&bars.xmin_empty[x & 1]);
            mma_commit_warp(&bars.info_empty[x & 1]);
            return true;
        };
        const uint32_t w_full0 = smem_u32(bars.w_full), x_full0 = smem_u32(bars.x_full);
        const uint32_t acc_empty0 = smem_u32(bars.acc_empty);
        bool ok = true;
        for (int st = 0; st < nstages && ok; ++st) {
            const int s = st % S, e = st % kEnt, xs = st % C::XS;
            const uint32_t ph = (st / S) & 1, eph = ((st / kEnt) & 1) ^ 1, xph = (st / C::XS) & 1;
            // the stage's three conditions probed at once (their round trips overlap)
            const bool ready = __all_sync(kAll, mbar_test_wait(w_full0 + 8u * s, ph) &
                                                     mbar_test_wait(x_full0 + 8u * xs, xph) &
                                                     mbar_test_wait(acc_empty0 + 8u * e, eph));
            if (!ready && (!wait_all(&bars.w_full[s], ph, ERR_GEMM_B_FULL) || !wait_all(&bars.x_full[xs], xph, ERR_GEMM_A_FULL) ||
                           !wait_all(&bars.acc_empty[e], eph, ERR_GEMM_ACC_EMPTY))) {
                ok = false;
                break;
            }
            tc_fence_after();
            bool corr = false;
            if constexpr (C::CORR) {
                uint32_t f = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) f |= corr_flags[8 * s + i];
                corr = f != 0;
            }
            const uint64_t woff = (uint64_t)((s * kWTile) >> 4), xoff = (uint64_t)((xs * C::XTILE) >> 4);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const uint32_t d_tmem = tmem + (uint32_t)((2 * e + h) * NT);
#pragma unroll
                for (int kk = 0; kk < 2; ++kk) {
                    const uint64_t koff = (uint64_t)((2 * h + kk) * 2);
                    mma_f16_warp(d_tmem, w_desc0 + woff + koff, x_desc0 + xoff + koff, idesc, kk);
                    if (corr) mma_f16_warp(d_tmem, wc_desc0 + woff + koff, x_desc0 + xoff + koff, idesc, 1);
                }
            }
            mma_commit_warp(&bars.acc_full[e]);
            mma_commit_warp(&bars.wx_empty[s]);
            mma_commit_warp(&bars.x_empty[xs]);
            if constexpr (C::MIN) {
                // the previous super-block's min term, after this super-block's first stage
                if ((st & 3) == 0 && st > 0 && !issue_min((st >> 2) - 1)) ok = false;
            }
        }
        if constexpr (C::MIN) {
            if (ok && issue_min(nsb - 1)) mma_commit_warp(bars.min_final);
        }
    } else if (warp == kSmWarpDa) {
        // ------------------------------------------------------------ activation-scale stager
        float *da0 = reinterpret_cast<float *>(sm + C::OFF_DA);
        for (int sb = 0; sb < nsb; ++sb) {
            if (!__all_sync(kAll, mbar_wait(&bars.da_empty[sb % C::DAS], ((sb / C::DAS) & 1) ^ 1, err, ERR_GEMM_DA, abort_flag)))
                break;
            float *dst = da0 + (sb % C::DAS) * 8 * NT;
#pragma unroll
            for (int i = 0; i < 8 * NT / 32; ++i) {
                const int idx = i * 32 + lane, j = idx / NT, t = idx % NT;
                dst[idx] = t < M ? __ldg(p.d + (int64_t)(8 * sb + j) * M + t) : 0.0f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.da_full[sb % C::DAS]);
        }
    } else if (warp >= kSmWarpUnpack0 && warp < kSmWarpEpi0) {
        // ------------------------------------------------------------ unpackers: two threads per row
        const int u = threadIdx.x - 32 * kSmWarpUnpack0;
        const int r = u >> 1, t = u & 1;             // weight row in the tile, 32-value block of the stage
        const int64_t n = n0 + r;
        const bool valid = n < N;
        const uint8_t *wrow = w + (valid ? n : 0) * row_bytes;
        uint8_t *raw_row0 = sm + C::OFF_RAW + r * C::RAW_ROW;
        const uint32_t w_tile0 = smem_u32(sm + C::OFF_W), wc_tile0 = smem_u32(sm + C::OFF_WC);
        const uint32_t wmin_tile0 = smem_u32(sm + C::OFF_WMIN);
        float *info0 = reinterpret_cast<float *>(sm + C::OFF_INFO);
        const int uw = warp - kSmWarpUnpack0;

        // Q6_K: the row's block as its 16-byte aligned superset, one bulk copy per row (thread t = 0)
        auto issue_raw = [&](int sb) {
            const int slot = sb % R;
            if (t != 0) return;
            if (valid) {
                const uint8_t *src = wrow + (int64_t)sb * C::BB;
                const uint8_t *a0 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15));
                const uint32_t nbytes = (uint32_t)(((reinterpret_cast<uintptr_t>(src) + C::BB + 15) & ~uintptr_t(15)) -
                                                   reinterpret_cast<uintptr_t>(a0));
                mbar_arrive_expect_tx(&bars.raw_full[slot], nbytes);
                bulk_copy_g2s(raw_row0 + slot * SW * C::RAW_ROW, a0, nbytes, &bars.raw_full[slot]);
            } else {
                mbar_arrive(&bars.raw_full[slot]);
            }
        };
        int issued = 0;
        if constexpr (!C::TMW) {
            for (int sb = 0; sb < R && sb < nsb; ++sb) issue_raw(sb);
            issued = R < nsb ? R : nsb;
        }
        uint32_t dirty = (1u << S) - 1;              // Q6_K correction chunks that may hold non-zero data
        const uint32_t wx_empty0 = smem_u32(bars.wx_empty);
        // the next round's slots probed one round ahead (a fresh barrier's parity-1 phase counts as complete)
        bool wpre = __all_sync(kAll, mbar_test_wait(wx_empty0, 1) & mbar_test_wait(wx_empty0 + 8u, 1));
        int sb = 0;
        for (; sb < nsb; ++sb) {
            const int slot = sb % R;
            if (!__all_sync(kAll, mbar_wait(&bars.raw_full[slot], (sb / R) & 1, err, ERR_GEMM_RAW_FULL, abort_flag)))
                break;
            const uint32_t blk_a = smem_u32(raw_row0 + slot * SW * C::RAW_ROW);
            const uint32_t blk_r =
                valid && !C::TMW ? (uint32_t)(reinterpret_cast<uintptr_t>(wrow + (int64_t)sb * C::BB) & 15) : 0u;
            // ---- super-block header
            float d = 0.0f, dmin = 0.0f;
            int sc[16];
            int mn[8];
            uint32_t se2[8], bigm = 0;                // Q6_K: this thread's scales as f16 pairs, big-scale mask
            bool wbig = false;                        // Q6_K: some row of the warp has a big scale
            if constexpr (C::KQ) {
                const uint4 hd = valid ? sm_lds128(blk_a) : make_uint4(0, 0, 0, 0);
                d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xffff)));
                dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
                uint32_t sbytes[12];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    sbytes[i] = (hd.y >> (8 * i)) & 0xff;
                    sbytes[4 + i] = (hd.z >> (8 * i)) & 0xff;
                    sbytes[8 + i] = (hd.w >> (8 * i)) & 0xff;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    sc[j] = sbytes[j] & 63;
                    mn[j] = sbytes[j + 4] & 63;
                    sc[j + 4] = (sbytes[j + 8] & 15) | ((sbytes[j] >> 6) << 4);
                    mn[j + 4] = (sbytes[j + 8] >> 4) | ((sbytes[j + 4] >> 6) << 4);
                }
            } else {
                uint32_t tail[5];                     // bytes 192..211: scales[16], d
                if (valid) {
                    sm_words_r<5>(blk_a + 192, blk_r, tail);
                } else {
#pragma unroll
                    for (int i = 0; i < 5; ++i) tail[i] = 0;
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) sc[i] = (int)(int8_t)((tail[i >> 2] >> (8 * (i & 3))) & 0xff);
                d = __half2float(__ushort_as_half((unsigned short)(tail[4] & 0xffff)));
                // the eight 16-value scales this thread applies, sc[8h + 4a + 2t + b] at index 4h + 2a + b,
                // as f16 pairs; an odd |sc| > 64 (13 bits with q) keeps sc - 1 here and marks the
                // correction tile, which then carries q
                bigm = 0;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                    for (int a = 0; a < 2; ++a)
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            const int idx = 4 * hh + 2 * a + b;
                            const int scv = valid ? (t ? sc[8 * hh + 4 * a + 2 + b] : sc[8 * hh + 4 * a + b]) : 0;
                            const bool big = (scv > 64 || scv < -64) && (scv & 1);
                            se2[idx] = sm_h2u(__float2half2_rn((float)(big ? (scv & ~1) : scv)));
                            bigm |= (uint32_t)big << idx;
                        }
                wbig = __any_sync(kAll, bigm != 0);
            }
            // ---- per-row factors: d for the epilogue; the min tile row (-dmin m_j as tf32 hi | lo)
            if (!__all_sync(kAll, mbar_wait(&bars.info_empty[sb & 1], ((sb >> 1) & 1) ^ 1, err, ERR_GEMM_INFO_EMPTY,
                                            abort_flag)))
                break;
            if (t == 0) info0[(sb & 1) * SW + r] = d;
            if constexpr (C::MIN) {
                // -dmin*m_j has at most 17 significant bits: an exact tf32 pair; thread t writes
                // the hi (t = 0) or lo (t = 1) half of the row
                uint32_t wv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float v = -(dmin * (float)mn[j]);
                    const float vh = tf32_rn(v);
                    wv[j] = __float_as_uint(t == 0 ? vh : v - vh);
                }
                const uint32_t bt = wmin_tile0 + (sb & 1) * C::MIN_W;
                sm_sts128(sm_sw64(bt, r, 2 * t), make_uint4(wv[0], wv[1], wv[2], wv[3]));
                sm_sts128(sm_sw64(bt, r, 2 * t + 1), make_uint4(wv[4], wv[5], wv[6], wv[7]));
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.info_full[sb & 1]);

            // ---- four 64-value stages, two per round (one wait, fence and hand-off round per two
            // stages); thread t writes each stage's 32-value block t (chunks 4t .. 4t+3)
            bool ok = true;
            uint32_t ql[8], qh[8];                    // Q6_K: this thread's low / high bits of the half
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int st = sb * 4 + q, s = st % S;
                if ((q & 1) == 0) {
                    const int s1 = (st + 1) % S;
                    if (!wpre &&
                        (!__all_sync(kAll, mbar_wait(&bars.wx_empty[s], ((st / S) & 1) ^ 1, err, ERR_GEMM_AB_EMPTY,
                                                     abort_flag)) ||
                         !__all_sync(kAll, mbar_wait(&bars.wx_empty[s1], (((st + 1) / S) & 1) ^ 1, err,
                                                     ERR_GEMM_AB_EMPTY, abort_flag)))) {
                        ok = false;
                        break;
                    }
                }
                const uint32_t wtile = w_tile0 + s * kWTile;
                if constexpr (C::KQ) {
                    // sub-block j = 2q + t: low (t = 0) or high (t = 1) nibbles of qs[32q .. 32q+32); Q5_K:
                    // qs at byte 48, bit j of qh[l] is the fifth bit of element l of sub-block j
                    constexpr uint32_t QS = FMT == FMT_Q5K ? 48 : 16;
                    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = q0, h0v = q0, h1v = q0;
                    if (valid) {
                        q0 = sm_lds128(blk_a + QS + 32 * q);
                        q1 = sm_lds128(blk_a + QS + 32 * q + 16);
                        if constexpr (FMT == FMT_Q5K) {
                            h0v = sm_lds128(blk_a + 16);
                            h1v = sm_lds128(blk_a + 32);
                        }
                    }
                    const uint32_t wq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    const uint32_t wh[8] = {h0v.x, h0v.y, h0v.z, h0v.w, h1v.x, h1v.y, h1v.z, h1v.w};
                    const int j = 2 * q + t;
                    const float scf = (float)(t ? sc[2 * q + 1] : sc[2 * q]);
                    const __half2 sc2 = __float2half2_rn(scf);
                    const __half2 neg = __float2half2_rn(-1024.0f * scf);
                    const uint32_t nsh = 4u * (uint32_t)t;
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        uint32_t va = (wq[2 * cc] >> nsh) & 0x0f0f0f0fu;
                        uint32_t vb = (wq[2 * cc + 1] >> nsh) & 0x0f0f0f0fu;
                        if constexpr (FMT == FMT_Q5K) {
                            va |= ((wh[2 * cc] >> j) & 0x01010101u) << 4;
                            vb |= ((wh[2 * cc + 1] >> j) & 0x01010101u) << 4;
                        }
                        uint32_t h0, h1, h2, h3;
                        sm_bytes_biased(va, h0, h1);
                        sm_bytes_biased(vb, h2, h3);
                        uint4 o;
                        // (1024 + q) sc - 1024 sc in one fused op: exact, sc q <= 63 * 31 < 2048
                        o.x = sm_h2u(__hfma2(sm_u2h(h0), sc2, neg));
                        o.y = sm_h2u(__hfma2(sm_u2h(h1), sc2, neg));
                        o.z = sm_h2u(__hfma2(sm_u2h(h2), sc2, neg));
                        o.w = sm_h2u(__hfma2(sm_u2h(h3), sc2, neg));
                        sm_sts128(sm_sw128(wtile, r, 4 * t + cc), o);
                    }
                } else {
                    // half h = q / 2, group g = 2 (q % 2) + t: ql bytes 32t .. 32t+31 of the half (low
                    // nibbles for q even, high for q odd) and qh bits 2g .. 2g+1
                    const int h = q >> 1;
                    if ((q & 1) == 0) {
                        if (valid) {
                            sm_words_r<8>(blk_a + 64 * h + 32 * t, blk_r, ql);
                            sm_words_r<8>(blk_a + 128 + 32 * h, blk_r, qh);
                        } else {
#pragma unroll
                            for (int i = 0; i < 8; ++i) ql[i] = qh[i] = 0;
                        }
                    }
                    const int nsh = (q & 1) ? 4 : 0;
                    const uint32_t hsh = (uint32_t)(4 * (q & 1) + 2 * t);
                    const __half2 bias = __float2half2_rn(1056.0f);
                    const uint32_t wct = wc_tile0 + s * kWTile;
                    // the correction chunks are written while the warp has big scales in this super-block,
                    // and once more (zeros) after it, warp-uniformly
                    const bool corr_w = wbig || ((dirty >> s) & 1);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        // values l = 8c .. 8c+7 of the group; scale index 4h + 2(q % 2) + (l >= 16)
                        const int idx = 4 * h + 2 * (q & 1) + (c >> 1);
                        const __half2 s2 = sm_u2h(se2[idx]);
                        uint32_t o[4], tq[4];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t lw = ql[2 * c + e], hw = qh[2 * c + e];
                            const uint32_t v = ((lw >> nsh) & 0x0f0f0f0fu) | (((hw >> hsh) & 0x03030303u) << 4);
                            uint32_t b0, b1;
                            sm_bytes_biased(v, b0, b1);
                            const __half2 t0 = __hsub2(sm_u2h(b0), bias);   // q - 32, exact
                            const __half2 t1 = __hsub2(sm_u2h(b1), bias);
                            o[2 * e] = sm_h2u(__hmul2(t0, s2));
                            o[2 * e + 1] = sm_h2u(__hmul2(t1, s2));
                            tq[2 * e] = sm_h2u(t0);
                            tq[2 * e + 1] = sm_h2u(t1);
                        }
                        sm_sts128(sm_sw128(wtile, r, 4 * t + c), make_uint4(o[0], o[1], o[2], o[3]));
                        if (corr_w) {
                            const bool big = (bigm >> idx) & 1u;
                            sm_sts128(sm_sw128(wct, r, 4 * t + c),
                                      big ? make_uint4(tq[0], tq[1], tq[2], tq[3]) : make_uint4(0, 0, 0, 0));
                        }
                    }
                    if (wbig) dirty |= 1u << s; else dirty &= ~(1u << s);
                    if (lane == 0) corr_flags[8 * s + uw] = wbig ? 1u : 0u;
                }
                if (q & 1) {
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&bars.w_full[(st - 1) % S]);
                        mbar_arrive(&bars.w_full[s]);
                    }
                    // the next round's two slots, probed ahead
                    wpre = st + 2 < nstages &&
                           __all_sync(kAll, mbar_test_wait(wx_empty0 + 8u * (uint32_t)((st + 1) % S),
                                                           ((uint32_t)((st + 1) / S) & 1u) ^ 1u) &
                                                mbar_test_wait(wx_empty0 + 8u * (uint32_t)((st + 2) % S),
                                                               ((uint32_t)((st + 2) / S) & 1u) ^ 1u));
                }
            }
            if (!ok) break;
            // every lane's reads of this raw slot are done before it is refilled
            fence_proxy_async_smem();
            __syncwarp();
            if constexpr (C::TMW) {
                if (lane == 0) mbar_arrive(&bars.raw_empty[slot]);
            } else if (sb + R < nsb) {
                issue_raw(sb + R);
                ++issued;
            }
        }
        if (*abort_flag && t == 0) {   // wait (bounded) for this row's copies still in flight
            for (int i = sb; i < issued; ++i)
                mbar_wait(&bars.raw_full[i % R], (i / R) & 1, err, ERR_GEMM_RAW_FULL, nullptr);
        }
    } else if (warp >= kSmWarpEpi0) {
        // ------------------------------------------------------------ epilogue: thread = weight row
        const int qd = warp & 3;
        const int r = 32 * qd + lane;
        const int64_t n = n0 + r;
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
        const int64_t nblk32 = K / kQ8;
        const float *info0 = reinterpret_cast<const float *>(sm + C::OFF_INFO);
        const float *da0 = reinterpret_cast<const float *>(sm + C::OFF_DA);
        float2 acc[NT / 2], part[NT / 2];
#pragma unroll
        for (int i = 0; i < NT / 2; ++i) {
            acc[i] = make_float2(0.0f, 0.0f);
            part[i] = make_float2(0.0f, 0.0f);
        }
        const uint32_t acc_full0 = smem_u32(bars.acc_full), da_full0 = smem_u32(bars.da_full);
        auto probe_acc = [&](int st) {
            return mbar_test_wait(acc_full0 + 8u * (uint32_t)(st % kEnt), (uint32_t)(st / kEnt) & 1u);
        };
        bool ok = true;
        bool pre = probe_acc(0), da_pre = mbar_test_wait(da_full0, 0);
        for (int sb = 0; sb < nsb && ok; ++sb) {
            if (!da_pre && !mbar_wait(&bars.da_full[sb % C::DAS], (sb / C::DAS) & 1, err, ERR_GEMM_DA, abort_flag)) break;
            const float4 *da_sb = reinterpret_cast<const float4 *>(da0 + (sb % C::DAS) * 8 * NT);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                // one ring entry per stage: blocks 2q and 2q + 1 side by side, one wait and one release
                const int st = sb * 4 + q, e = st % kEnt;
                if (!pre && !mbar_wait(&bars.acc_full[e], (st / kEnt) & 1, err, ERR_GEMM_ACC_FULL, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // NT = 16: both blocks in one 32-column load; NT = 32: one block at a time (fewer
                // live registers), the entry released after the second load
                uint32_t v[32];
                if constexpr (NT == 16) {
                    tmem_ld32(trow + (uint32_t)(2 * e * NT), v);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.acc_empty[e]);
                }
                auto probe_next = [&]() {
                    // the next probes go out ahead of the FMAs
                    pre = st + 1 < nstages ? probe_acc(st + 1) : true;
                    if (q == 3)
                        da_pre = sb + 1 < nsb && mbar_test_wait(da_full0 + 8u * (uint32_t)((sb + 1) % C::DAS),
                                                                (uint32_t)((sb + 1) / C::DAS) & 1u);
                };
                if constexpr (NT == 16) probe_next();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j = 2 * q + h, gb = sb * 8 + j;
                    if constexpr (NT == 32) {
                        tmem_ld32(trow + (uint32_t)((2 * e + h) * NT), v);
                        tmem_ld_wait();
                        if (h == 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars.acc_empty[e]);
                            probe_next();
                        }
                    }
                    const int vo = NT == 16 ? h * NT : 0;      // this block's first column in v
                    // part[t] (+)= I[t] d_a[t]: the tokens' scales of block j (same for every lane)
#pragma unroll
                    for (int i4 = 0; i4 < NT / 4; ++i4) {
                        const float4 da = da_sb[(j * NT) / 4 + i4];
                        const float2 x0 = make_float2(__uint_as_float(v[vo + 4 * i4]), __uint_as_float(v[vo + 4 * i4 + 1]));
                        const float2 x1 =
                            make_float2(__uint_as_float(v[vo + 4 * i4 + 2]), __uint_as_float(v[vo + 4 * i4 + 3]));
                        if (j == 0) {
                            part[2 * i4] = __fmul2_rn(x0, make_float2(da.x, da.y));
                            part[2 * i4 + 1] = __fmul2_rn(x1, make_float2(da.z, da.w));
                        } else {
                            part[2 * i4] = __ffma2_rn(x0, make_float2(da.x, da.y), part[2 * i4]);
                            part[2 * i4 + 1] = __ffma2_rn(x1, make_float2(da.z, da.w), part[2 * i4 + 1]);
                        }
                    }
                    if constexpr (DUMP) {
                        if (n >= dump.n0 && n < dump.n0 + dump.n_cnt && n < N) {
#pragma unroll
                            for (int tt = 0; tt < NT; ++tt) {
                                if (tt >= dump.m0 && tt < dump.m0 + dump.m_cnt && tt < M)
                                    dump.out[((tt - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32 + gb] =
                                        __float2int_rn(__uint_as_float(v[vo + tt]));
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            // ---- super-block end: acc += d * part (d: this row's fp16 factor)
            if (!mbar_wait(&bars.info_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_INFO_FULL, abort_flag)) break;
            const float dr = info0[(sb & 1) * SW + r];
            const float2 d2 = make_float2(dr, dr);
#pragma unroll
            for (int i = 0; i < NT / 2; ++i) acc[i] = __ffma2_rn(part[i], d2, acc[i]);
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.info_empty[sb & 1]);
                mbar_arrive(&bars.da_empty[sb % C::DAS]);
            }
        }
        if (ok && !*abort_flag) {
            if constexpr (C::MIN) {
                if (mbar_wait(bars.min_final, 0, err, ERR_GEMM_MIN, abort_flag)) {
                    tc_fence_after();
                    uint32_t v[NT];
                    sm_tmem_ld<NT>(trow + C::MIN_COL, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < NT / 2; ++i)
                        acc[i] = __fadd2_rn(acc[i], make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])));
                } else {
                    ok = false;
                }
            }
            if (ok && n < N) {
                // token t's row of Y: the warp's 32 lanes store 32 consecutive outputs
#pragma unroll
                for (int i = 0; i < NT / 2; ++i) {
                    if (2 * i < M) y[(int64_t)(2 * i) * N + n] = acc[i].x;
                    if (2 * i + 1 < M) y[(int64_t)(2 * i + 1) * N + n] = acc[i].y;
                }
            }
        }
    }

    __syncthreads();
    if (warp == kSmWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

template <int FMT, int NT, bool DUMP>
int launch_small_fmt(const CUtensorMap &tmx, const CUtensorMap &tmxs, const CUtensorMap &tmw, const uint8_t *w,
                     int64_t N, int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump, unsigned int *err,
                     cudaStream_t stream) {
    using C = SmCfg<FMT, NT>;
    auto kern = small_kernel<FMT, NT, DUMP>;
    const int fi = FMT == FMT_Q4K ? 0 : FMT == FMT_Q6K ? 1 : 2;
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM,
                              kAttrSlotSmall + 2 * (2 * fi + (NT == 32 ? 1 : 0)) + (DUMP ? 1 : 0));
    if (rc != MQ_OK) return rc;
    const dim3 grid((unsigned)((N + SW - 1) / SW));
    return cuda_error(launch_pdl(kern, grid, dim3(kSmThreads), C::SMEM, stream, tmx, tmxs, tmw, w, N, K, p, M, y, dump,
                                 err),
                      "small-M gemm launch");
}

template <int FMT, int NT>
int launch_small_nt(const CUtensorMap &tmx, const CUtensorMap &tmxs, const CUtensorMap &tmw, const uint8_t *w,
                    int64_t N, int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump, unsigned int *err,
                    cudaStream_t stream) {
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    return dmp ? launch_small_fmt<FMT, NT, true>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream)
               : launch_small_fmt<FMT, NT, false>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream);
}

}  // namespace

int launch_gemm_small(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                      const Dump &dump, unsigned int *err, cudaStream_t stream) {
    EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
    if (enc == nullptr) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    if (fmt != FMT_Q4K && fmt != FMT_Q5K && fmt != FMT_Q6K)
        return set_error(MQ_ERR_ARG, "small-M GEMM: Q4_K, Q5_K and Q6_K weights only");
    if (M < 1 || M > 32) return set_error(MQ_ERR_SHAPE, "small-M GEMM: M=%lld not in 1 .. 32", (long long)M);
    const uint32_t nt = M <= 16 ? 16 : 32;
    const cuuint32_t estr[2] = {1, 1};
    CUtensorMap tmx, tmxs, tmw;
    // token codes: f16 [M][K] in 64 x NT boxes (128-byte swizzle); rows past M read as zeros
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {SBK, nt};
        const CUresult r = enc(&tmx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.q16, dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled (small-M codes) failed (%d)", (int)r);
    }
    // the tokens' d*S tf32 pairs [M][2*K/32], one 16-value x NT box per super-block (64-byte swizzle)
    {
        const cuuint64_t dims[2] = {(cuuint64_t)(2 * (K / kQ8)), (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)(2 * (K / kQ8)) * 4};
        const cuuint32_t box[2] = {16, nt};
        const CUresult r = enc(&tmxs, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.ds, dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled (small-M d*S) failed (%d)", (int)r);
    }
    // raw weights (Q4_K / Q5_K): one block-bytes x 128-row box per super-block
    memset(&tmw, 0, sizeof tmw);
    if (fmt != FMT_Q6K) {
        const cuuint64_t bb = (cuuint64_t)block_bytes(fmt);
        const cuuint64_t dims[2] = {(cuuint64_t)(K / kQK) * bb, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)(K / kQK) * bb};
        const cuuint32_t box[2] = {(cuuint32_t)bb, SW};
        const CUresult r = enc(&tmw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(w), dims, strides, box, estr,
                               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled (small-M weights) failed (%d)", (int)r);
    }
    if (fmt == FMT_Q4K)
        return nt == 16 ? launch_small_nt<FMT_Q4K, 16>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream)
                        : launch_small_nt<FMT_Q4K, 32>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream);
    if (fmt == FMT_Q5K)
        return nt == 16 ? launch_small_nt<FMT_Q5K, 16>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream)
                        : launch_small_nt<FMT_Q5K, 32>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream);
    return nt == 16 ? launch_small_nt<FMT_Q6K, 16>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream)
                    : launch_small_nt<FMT_Q6K, 32>(tmx, tmxs, tmw, w, N, K, p, M, y, dump, err, stream);
}

}  // namespace mq
