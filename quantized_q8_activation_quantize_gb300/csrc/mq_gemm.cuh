// mq_gemm.cuh -- prefill GEMM (MMQ): raw Q4_K / Q5_K / Q6_K and Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0
// weights x Q8 plane on tcgen05 tensor cores.
//
// minfer pages, "Features > GPU -- CUDA": raw-nibble int8 GEMMs for q4_K and q6_K
// over the producer-written q8 plane; "Support Matrix > CUDA notes": prefill
// (nt >= 16) takes the MMQ path.  The pages' kernel (mma.m16n8k32 with weight
// planes expanded at registration) targets GB10; this one is written for sm_103a:
//
//  * sm_103a has no tcgen05 int8 MMA kind, so the integer block dots run as
//    kind::f16 MMAs on exact small integers: codes q_a in [-127, 127], Q4_K
//    sc*q in [0, 945], Q6_K sc*q in [-2048, 2048] are all exact in f16, products are
//    exact, and every 32-value block sum stays below 2^24, so the f32 TMEM
//    accumulator holds the exact integer I.  Q6_K scales with |sc| > 64 and odd
//    would need 13 bits: those rows take sc - 1 (even, exact) in the main tile and
//    q * 1 in a correction tile that is multiplied only when the stage has such rows.
//  * A (tokens, f16 codes) is a TMA 2-D tile with the 128-byte swizzle; B (weights)
//    is unpacked from raw block bytes (staged by 1-D bulk copies of each row's
//    16-byte-aligned superset) straight into the same swizzled K-major layout.
//  * Each 32-value block's product goes to its own TMEM accumulator (a ring of 3 slots, 4
//    for Q6_K, which has no min-term region);
//    the epilogue warps drain it and apply the activation scale per block with packed
//    f32x2 FMAs; once per super-block they fold the fp16 d into a running sum kept
//    in a fourth TMEM region.
//  * The Q4_K min term dmin * sum_j m_j d_a[j] S[j] runs on the tensor pipe: per
//    super-block three tf32 MMAs (K = 8) of the plane's d_a*S and of -dmin*m_j, each held
//    as a tf32 (hi, lo) pair (hi*hi + lo*hi + hi*lo, error below 2^-21 relative),
//    accumulate straight into the running sum.
//
// CTA = 16 warps: 0 TMA producer, 1 MMA issuer (+ TMEM owner), 2-3 idle, 4-7 unpackers
// (one weight row per thread), 8-15 epilogue (2 per TMEM lane quadrant, 64 columns
// each); setmaxnreg moves registers from the first two warpgroups to the epilogue.
// Tile: 128 tokens x 128 weight rows, K staged 64 at a time.
//
// Kernel and launcher templates; mq_gemm_kq.cu instantiates the k-quants (and holds the entry
// point, which encodes the tensor maps), mq_gemm_b32.cu the 32-value formats.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int BM = 128, BN = 128, BK = 64;
constexpr int kThreads = 512;   // 4 warpgroups: {TMA, MMA, -, -}, unpack, epilogue x2
constexpr int kWarpTma = 0, kWarpMma = 1, kWarpUnpack0 = 4, kWarpEpi0 = 8;

constexpr int kMaxAccSlots = 4;
// 3 block slots + the min-term sum at column 384, or (formats without a min term) 4 block slots
constexpr uint32_t kTmemCols = 512, kMinCol = 384;
constexpr int kTile = BM * BK * 2;       // one 128 x 64 f16 operand tile
constexpr unsigned kFull = 0xffffffffu;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int FMT>
struct GmCfg {
    // Q4_K and Q5_K share the header (d, dmin, 12 packed scale / min bytes) and the min term;
    // Q5_K adds 32 bytes of fifth bits.  The 32-value formats (B32) come as groups of eight
    // blocks per 256 values, each block with its own fp16 d (and m for Q4_1 / Q5_1).  Every
    // format but Q6_K has a 16-byte multiple per 256 values and takes its raw rows by TMA (TMW).
    static constexpr bool KQ = FMT == FMT_Q4K || FMT == FMT_Q5K;
    static constexpr bool B32 = is_b32(FMT);
    static constexpr bool TMW = FMT != FMT_Q6K;
    static constexpr int BB = block_bytes(FMT);
    static constexpr int TMW_ELEM = B32 ? 2 : 1;                  // bytes per tensor-map element (box <= 256)
    static constexpr int STAGES = TMW ? 4 : 3;
    static constexpr int RAW_STAGES = FMT == FMT_Q4K ? 3 : 2;
    // TMA-fed formats: the block itself; Q6_K: the 16-B aligned superset of one block (224 B at most)
    // at a 240-byte row stride, so that the 16-byte loads of eight consecutive rows hit eight
    // distinct bank groups
    static constexpr int RAW_ROW = TMW ? BB : 240;
    static constexpr bool CORR = FMT == FMT_Q6K;                  // Q6_K odd |sc| > 64 correction tile
    // the min / offset term on the tensor pipe: Q4_K / Q5_K -dmin m_j, Q4_1 / Q5_1 the block offset m
    static constexpr bool MIN = KQ || b32_has_m(FMT);
    // TMEM accumulator slots of 128 columns.  Q6_K has no min-term region and takes a fourth slot
    // (measured -1 % on its GEMMs); the 32-value formats without a min term measured 4-5 %
    // slower with four, so they keep three
    static constexpr int ACC = FMT == FMT_Q6K ? 4 : 3;
    static constexpr int MIN_TILE = BM * 64;                      // 128 rows x 16 tf32 (64 B, 64-B swizzle)
    // Q4_K / Q5_K: the activation scales staged token-major, so the epilogue loads a token's eight
    // once per super-block instead of one per block (measured -3 %; Q6_K and the 32-value formats,
    // with other register pressure in the epilogue, measured slower and keep the block-major table)
    static constexpr bool DA_TOK = KQ;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + STAGES * kTile;
    static constexpr int OFF_BC = OFF_B + STAGES * kTile;
    static constexpr int OFF_AMIN = OFF_BC + (CORR ? STAGES * kTile : 0);
    static constexpr int OFF_BMIN = OFF_AMIN + (MIN ? 2 * MIN_TILE : 0);
    static constexpr int OFF_RAW = OFF_BMIN + (MIN ? 2 * MIN_TILE : 0);
    // row factors, 2 slots: the super-block d per weight row, or (B32) each block's d [8][128]
    static constexpr int OFF_INFO = OFF_RAW + RAW_STAGES * BN * RAW_ROW;
    static constexpr int OFF_DA = OFF_INFO + 2 * BN * 4 * (B32 ? 8 : 1);    // d_a [2][8 blocks][128 tokens] (or token-major)
    static constexpr int OFF_FLAG = OFF_DA + 2 * 8 * BM * 4;
    static constexpr int OFF_BAR = align_up(OFF_FLAG + STAGES * 4 * 4, 8);
    // a_full[S] b_full[S] ab_empty[S] raw_full[R] raw_empty[R] info_full[2] info_empty[2] acc_full[3]
    // acc_empty[3] amin_full[2] amin_empty[2] min_final[1] da_full[2] da_empty[2]
    static constexpr int NBARS = 3 * STAGES + 2 * RAW_STAGES + 4 + 2 * kMaxAccSlots + 5 + 4;
    static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
    static constexpr int SMEM = OFF_MISC + 16 + 1024;             // + slack to align the base to 1 KiB
    static_assert(SMEM <= 227 * 1024, "shared memory of one CTA exceeds the per-CTA limit");
    // per-warpgroup register budgets (launch: 512 x 128 = the whole 64K register file), chosen
    // per format by measurement (spill reloads in a pipeline loop cost an L2 trip each)
    static constexpr int REGS_CTL = TMW ? 56 : 48;
    static constexpr int REGS_UNPACK = TMW ? 72 : 112;
    static constexpr int REGS_EPI = TMW ? 192 : 176;
    static_assert(128 * REGS_CTL + 128 * REGS_UNPACK + 256 * REGS_EPI <= 65536, "register split exceeds the launch pool");
};

struct Bars {
    uint64_t *a_full, *b_full, *ab_empty, *raw_full, *raw_empty, *info_full, *info_empty, *acc_full, *acc_empty;
    uint64_t *amin_full, *amin_empty, *min_final, *da_full, *da_empty;
};

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
__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// NW consecutive 32-bit words starting r bytes (r even, < 16) past the 16-byte aligned shared address
// base: 16-byte loads of the aligned chunks, then the word offset r / 4 selected by two levels of
// selects and the half-word offset by a funnel shift (no per-lane indexing into a register array)
template <int NW>
__device__ __forceinline__ void lds_words_r(uint32_t base, uint32_t r, uint32_t (&out)[NW]) {
    constexpr int NC = (NW + 4 + 3) / 4;             // chunks: words 0 .. NW + 3
    uint32_t w[4 * NC];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const uint4 t = lds128(base + 16u * c);
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

__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u32_as_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// four quant bytes (each < 64) -> two f16x2 words holding 1024 + byte
__device__ __forceinline__ void bytes_to_h2_biased(uint32_t v, uint32_t &lo, uint32_t &hi) {
    lo = __byte_perm(v, 0x64646464u, 0x4140);
    hi = __byte_perm(v, 0x64646464u, 0x4342);
}

// swizzled (128 B) address of 16-byte chunk c of row r in a K-major operand tile
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t tile, int r, int c) {
    return tile + (uint32_t)(r * 128 + ((c ^ (r & 7)) << 4));
}
// swizzled (64 B) address of 16-byte chunk c of row r
__device__ __forceinline__ uint32_t sw64_chunk(uint32_t tile, int r, int c) {
    return tile + (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

// SWIGLU: the fused gate|up GEMM.  The tile's 128 weight rows are 64 gate rows (tmW) and the
// same 64 rows of up (tmW2); each epilogue thread holds gate and up of 32 outputs of its token,
// forms silu(gate) * up and writes it as one Q8 block of the output plane `po` (no Y).
template <int FMT, bool DUMP, bool SWIGLU>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmDS,
                const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmW2,
                const uint8_t *__restrict__ w, int64_t N, int64_t K, Plane p, int64_t M, float *__restrict__ y,
                Plane po, Dump dump, unsigned int *err) {
    static_assert(!SWIGLU || (GmCfg<FMT>::TMW && !DUMP), "the fused gate|up GEMM takes TMA-fed formats, no dump");
    using C = GmCfg<FMT>;
    constexpr int S = C::STAGES, R = C::RAW_STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bar0 = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    Bars bars;
    bars.a_full = bar0;
    bars.b_full = bars.a_full + S;
    bars.ab_empty = bars.b_full + S;
    bars.raw_full = bars.ab_empty + S;
    bars.raw_empty = bars.raw_full + R;
    bars.info_full = bars.raw_empty + R;
    bars.info_empty = bars.info_full + 2;
    bars.acc_full = bars.info_empty + 2;
    bars.acc_empty = bars.acc_full + kMaxAccSlots;
    bars.amin_full = bars.acc_empty + kMaxAccSlots;
    bars.amin_empty = bars.amin_full + 2;
    bars.min_final = bars.amin_empty + 2;
    bars.da_full = bars.min_final + 1;
    bars.da_empty = bars.da_full + 2;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(sm + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + C::OFF_MISC + 4);
    volatile uint32_t *corr_flags = reinterpret_cast<volatile uint32_t *>(sm + C::OFF_FLAG);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // n0: the tile's first weight row (SWIGLU: of gate and of up, 64 each).  SWIGLU walks the
    // token tiles fastest (grid x), so the CTAs in flight share a few weight tiles while the
    // tokens' A tiles stay in L2: gate + up of the 7B FFN (76 MB) re-streamed once per token
    // tile would not stay in L2
    const int64_t m0 = (int64_t)(SWIGLU ? blockIdx.x : blockIdx.y) * BM;
    const int64_t n0 = (int64_t)(SWIGLU ? blockIdx.y : blockIdx.x) * (SWIGLU ? BN / 2 : BN);
    const int nsb = (int)(K / kQK);
    const int nstages = nsb * 4;
    const int64_t row_bytes = (int64_t)(K / kQK) * C::BB;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars.a_full[s], 1);
            mbar_init(&bars.b_full[s], 4);
            mbar_init(&bars.ab_empty[s], 1);
        }
        for (int r = 0; r < R; ++r) {
            // TMA-fed formats: one tensor copy per super-block (producer); Q6_K: one bulk copy per row (unpackers)
            mbar_init(&bars.raw_full[r], C::TMW ? 1 : 128);
            mbar_init(&bars.raw_empty[r], 4);                  // unpack warps (TMA-fed formats only)
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.info_full[i], 4);
            mbar_init(&bars.info_empty[i], C::MIN ? 9 : 8);    // epilogue warps (+ the min MMA)
            mbar_init(&bars.amin_full[i], 1);
            mbar_init(&bars.amin_empty[i], 1);
        }
        mbar_init(bars.min_final, 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars.da_full[i], 2);                    // the two stager warps
            mbar_init(&bars.da_empty[i], 8);                   // the epilogue warps
        }
        for (int i = 0; i < C::ACC; ++i) {
            mbar_init(&bars.acc_full[i], 1);
            mbar_init(&bars.acc_empty[i], 8);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kWarpMma) tmem_alloc(tmem_holder, kTmemCols);
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    // set-up above overlaps the predecessor on the stream; every global access below follows it
    grid_dep_launch();
    grid_dep_wait();

    // Each warpgroup first rebalances the register file (all four of its warps execute the
    // setmaxnreg), so the code of every role is compiled under its own budget.
    if (warp < kWarpUnpack0) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_CTL));
      if (warp == kWarpTma) {
        // ------------------------------------------------------------ A / d*S producer
        if (lane == 0) {
            prefetch_tmap(&tmA);
            if constexpr (C::MIN) prefetch_tmap(&tmDS);
            if constexpr (C::TMW) prefetch_tmap(&tmW);
            if constexpr (SWIGLU) prefetch_tmap(&tmW2);
            int st = 0, sb_issued = 0, raw_issued = 0;
            // raw blocks of the tile's 128 rows for one super-block (256 values): a BB-byte x 128 box
            auto issue_raw = [&](int sb) -> bool {
                const int slot = sb % R;
                if (!mbar_wait(&bars.raw_empty[slot], ((sb / R) & 1) ^ 1, err, ERR_GEMM_RAW_FULL, abort_flag))
                    return false;
                mbar_arrive_expect_tx(&bars.raw_full[slot], BN * C::RAW_ROW);
                tma_load_2d(sm + C::OFF_RAW + slot * BN * C::RAW_ROW, &tmW, sb * (C::BB / C::TMW_ELEM), (int32_t)n0,
                            &bars.raw_full[slot]);
                if constexpr (SWIGLU)      // up rows n0 .. n0+63 into tile rows 64 .. 127
                    tma_load_2d(sm + C::OFF_RAW + slot * BN * C::RAW_ROW + (BN / 2) * C::RAW_ROW, &tmW2,
                                sb * (C::BB / C::TMW_ELEM), (int32_t)n0, &bars.raw_full[slot]);
                raw_issued = sb + 1;
                return true;
            };
            if constexpr (C::TMW) {
                for (int sb = 0; sb < R - 1 && sb < nsb; ++sb)
                    if (!issue_raw(sb)) break;
            }
            for (; st < nstages && !*abort_flag; ++st) {
                const int s = st % S;
                if constexpr (C::TMW) {
                    // keep raw weights R-1 super-blocks ahead of the A stages
                    if ((st & 3) == 0 && (st >> 2) + R - 1 < nsb)
                        if (!issue_raw((st >> 2) + R - 1)) break;
                }
                if constexpr (C::MIN) {
                    if ((st & 3) == 0) {
                        const int sb = st >> 2;
                        if (!mbar_wait(&bars.amin_empty[sb & 1], ((sb >> 1) & 1) ^ 1, err, ERR_GEMM_MIN, abort_flag))
                            break;
                        mbar_arrive_expect_tx(&bars.amin_full[sb & 1], C::MIN_TILE);
                        tma_load_2d(sm + C::OFF_AMIN + (sb & 1) * C::MIN_TILE, &tmDS, sb * 16, (int32_t)m0,
                                    &bars.amin_full[sb & 1]);
                        sb_issued = sb + 1;
                    }
                }
                if (!mbar_wait(&bars.ab_empty[s], ((st / S) & 1) ^ 1, err, ERR_GEMM_AB_EMPTY, abort_flag)) break;
                mbar_arrive_expect_tx(&bars.a_full[s], kTile);
                tma_load_2d(sm + C::OFF_A + s * kTile, &tmA, st * BK, (int32_t)m0, &bars.a_full[s]);
            }
            if (*abort_flag) {   // leave no copy in flight: wait (bounded) for the last ones issued
                for (int i = st - 1; i >= 0 && i >= st - S; --i)
                    mbar_wait(&bars.a_full[i % S], (i / S) & 1, err, ERR_GEMM_A_FULL, nullptr);
                for (int sb = sb_issued - 1; sb >= 0 && sb >= sb_issued - 2; --sb)
                    mbar_wait(&bars.amin_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_MIN, nullptr);
                for (int sb = raw_issued - 1; sb >= 0 && sb >= raw_issued - R; --sb)
                    mbar_wait(&bars.raw_full[sb % R], (sb / R) & 1, err, ERR_GEMM_RAW_FULL, nullptr);
            }
        }
    } else if (warp == kWarpMma) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the loop (warp-uniform control flow and operands); one elected
        // lane issues each MMA and commit.
        {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            constexpr uint32_t idesc_min = idesc_tf32_f32(BM, BN);
            // stage-0 descriptors; a stage adds kTile >> 4 and a K=16 step 32 B >> 4 to the
            // start-address field (which stays below 2^14)
            const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_A));
            const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_B));
            const uint64_t bc_desc0 = sw128_kmajor_desc(smem_u32(sm + C::OFF_BC));
            const uint32_t amin_base = smem_u32(sm + C::OFF_AMIN), bmin_base = smem_u32(sm + C::OFF_BMIN);
            const uint32_t a_full0 = smem_u32(bars.a_full), b_full0 = smem_u32(bars.b_full);
            const uint32_t acc_empty0 = smem_u32(bars.acc_empty);
            // a blocking wait the whole warp leaves together
            auto wait_all = [&](uint64_t *bar, uint32_t ph, uint32_t code) {
                return __all_sync(kFull, mbar_wait(bar, ph, err, code, abort_flag));
            };
            // Q4_K min term of super-block x, summed over the whole K in its own TMEM region:
            // MIN (+)= (d_a S) x (-dmin m_j), both operands tf32 (hi, lo) pairs, three MMAs of K = 8
            auto issue_min = [&](int x) -> bool {
                const uint32_t ph = (x >> 1) & 1;
                const bool ready = __all_sync(kFull, mbar_test_wait(smem_u32(&bars.amin_full[x & 1]), ph) &
                                                         mbar_test_wait(smem_u32(&bars.info_full[x & 1]), ph));
                if (!ready && (!wait_all(&bars.amin_full[x & 1], ph, ERR_GEMM_MIN) ||
                               !wait_all(&bars.info_full[x & 1], ph, ERR_GEMM_INFO_FULL)))
                    return false;
                tc_fence_after();
                const uint32_t at = amin_base + (x & 1) * C::MIN_TILE, bt = bmin_base + (x & 1) * C::MIN_TILE;
                // (hi + lo)(d_a S) x (hi + lo)(-dmin m): hi*hi + lo*hi + hi*lo (lo*lo is below 2^-22)
                mma_tf32_warp(tmem + kMinCol, sw64_kmajor_desc(at), sw64_kmajor_desc(bt), idesc_min, x > 0 ? 1u : 0u);
                mma_tf32_warp(tmem + kMinCol, sw64_kmajor_desc(at + 32), sw64_kmajor_desc(bt), idesc_min, 1u);
                mma_tf32_warp(tmem + kMinCol, sw64_kmajor_desc(at), sw64_kmajor_desc(bt + 32), idesc_min, 1u);
                mma_commit_warp(&bars.amin_empty[x & 1]);
                mma_commit_warp(&bars.info_empty[x & 1]);
                return true;
            };
            int gb = 0;
            bool ok = true;
            for (int sb = 0; sb < nsb && ok; ++sb) {
                for (int q = 0; q < 4 && ok; ++q) {
                    const int st = sb * 4 + q, s = st % S;
                    const uint32_t ph = (st / S) & 1;
                    const int slot0 = gb % C::ACC, slot1 = (gb + 1) % C::ACC;
                    const uint32_t eph0 = ((gb / C::ACC) & 1) ^ 1, eph1 = (((gb + 1) / C::ACC) & 1) ^ 1;
                    // All four conditions of the stage probed at once (their latencies overlap);
                    // only a stage that is not ready yet falls back to the blocking waits.
                    const bool ready = __all_sync(kFull, mbar_test_wait(a_full0 + 8u * s, ph) &
                                                             mbar_test_wait(b_full0 + 8u * s, ph) &
                                                             mbar_test_wait(acc_empty0 + 8u * slot0, eph0) &
                                                             mbar_test_wait(acc_empty0 + 8u * slot1, eph1));
                    if (!ready && (!wait_all(&bars.a_full[s], ph, ERR_GEMM_A_FULL) ||
                                   !wait_all(&bars.b_full[s], ph, ERR_GEMM_B_FULL))) {
                        ok = false;
                        break;
                    }
                    bool corr = false;
                    if constexpr (C::CORR)
                        corr = (corr_flags[4 * s] | corr_flags[4 * s + 1] | corr_flags[4 * s + 2] |
                                corr_flags[4 * s + 3]) != 0;
                    const uint64_t soff = (uint64_t)((s * kTile) >> 4);
                    if (ready) tc_fence_after();
                    for (int h = 0; h < 2; ++h) {
                        const int slot = h ? slot1 : slot0;
                        if (!ready) {
                            if (!wait_all(&bars.acc_empty[slot], h ? eph1 : eph0, ERR_GEMM_ACC_EMPTY)) {
                                ok = false;
                                break;
                            }
                            tc_fence_after();
                        }
                        const uint32_t d_tmem = tmem + (uint32_t)(slot * BN);
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t koff = soff + (uint64_t)((2 * h + kk) * 2);
                            mma_f16_warp(d_tmem, a_desc0 + koff, b_desc0 + koff, idesc, kk);
                            if (corr) mma_f16_warp(d_tmem, a_desc0 + koff, bc_desc0 + koff, idesc, 1);
                        }
                        mma_commit_warp(&bars.acc_full[slot]);
                        ++gb;
                    }
                    if (!ok) break;
                    mma_commit_warp(&bars.ab_empty[s]);
                    if constexpr (C::MIN) {
                        // the previous super-block's min term goes after this super-block's first
                        // stage, so it never delays the block MMAs the epilogue is waiting for
                        if (q == 0 && sb > 0 && !issue_min(sb - 1)) ok = false;
                    }
                }
            }
            if constexpr (C::MIN) {
                if (ok && issue_min(nsb - 1)) mma_commit_warp(bars.min_final);
            }
        }
      } else {
        // ------------------------------------------------------------ activation-scale stager
        // warps 2-3: d_a of the tile's 128 tokens for each super-block's 8 blocks into shared
        // memory (two slots), so the epilogue reads them there instead of from L2
        const int t = threadIdx.x - 64;                  // 0..63: tokens t and t + 64
        float *da_tile0 = reinterpret_cast<float *>(sm + C::OFF_DA);
        for (int sb = 0; sb < nsb; ++sb) {
            const int slot = sb & 1;
            if (!__all_sync(kFull, mbar_wait(&bars.da_empty[slot], ((sb >> 1) & 1) ^ 1, err, ERR_GEMM_DA, abort_flag)))
                break;
            float v[16];
#pragma unroll
            for (int j = 0; j < 8; ++j)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int64_t m = m0 + t + 64 * h;
                    v[2 * j + h] = m < M ? __ldg(p.d + (int64_t)(8 * sb + j) * M + m) : 0.0f;
                }
            float *dst = da_tile0 + slot * 8 * BM;
            if constexpr (C::DA_TOK) {
                // token-major [128 tokens][8 blocks]: an epilogue thread reads its token's eight
                // scales with two 16-byte loads per super-block
                float4 *d4 = reinterpret_cast<float4 *>(dst);
                d4[2 * t] = make_float4(v[0], v[2], v[4], v[6]);
                d4[2 * t + 1] = make_float4(v[8], v[10], v[12], v[14]);
                d4[2 * (t + 64)] = make_float4(v[1], v[3], v[5], v[7]);
                d4[2 * (t + 64) + 1] = make_float4(v[9], v[11], v[13], v[15]);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    dst[j * BM + t] = v[2 * j];
                    dst[j * BM + t + 64] = v[2 * j + 1];
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.da_full[slot]);
        }
      }
    } else if (warp < kWarpEpi0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REGS_UNPACK));
        // ------------------------------------------------------------ unpackers
        const int r = threadIdx.x - 32 * kWarpUnpack0;     // weight row in the tile
        const int64_t n = n0 + (SWIGLU ? (r & (BN / 2 - 1)) : r);
        const bool valid = n < N;
        const uint8_t *wrow = w + (valid ? n : 0) * row_bytes;
        uint8_t *raw_row0 = sm + C::OFF_RAW + r * C::RAW_ROW;
        const uint32_t b_tile0 = smem_u32(sm + C::OFF_B), bc_tile0 = smem_u32(sm + C::OFF_BC);
        const uint32_t bmin_tile0 = smem_u32(sm + C::OFF_BMIN);
        float *info0 = reinterpret_cast<float *>(sm + C::OFF_INFO);

        // Q6_K: this row's block (210 B, 2-byte aligned) as the 16-byte aligned superset (224 B at
        // most), one bulk copy per row: rows of K/256 x 210 bytes fit no TMA tensor map
        auto issue_raw = [&](int sb) {
            const int slot = sb % R;
            if (valid) {
                const uint8_t *src = wrow + (int64_t)sb * C::BB;
                const uint8_t *a0 = reinterpret_cast<const uint8_t *>(reinterpret_cast<uintptr_t>(src) & ~uintptr_t(15));
                const uint32_t nbytes = (uint32_t)(((reinterpret_cast<uintptr_t>(src) + C::BB + 15) & ~uintptr_t(15)) -
                                                   reinterpret_cast<uintptr_t>(a0));
                // one bulk copy of the row's aligned superset (<= RAW_ROW bytes; the bytes past
                // the block stay in the 16-byte granule of its last byte)
                mbar_arrive_expect_tx(&bars.raw_full[slot], nbytes);
                bulk_copy_g2s(raw_row0 + slot * BN * C::RAW_ROW, a0, nbytes, &bars.raw_full[slot]);
            } else {
                mbar_arrive(&bars.raw_full[slot]);
            }
        };
        if constexpr (FMT == FMT_Q6K) {
            for (int sb = 0; sb < R && sb < nsb; ++sb) issue_raw(sb);
        }

        uint32_t dirty = (1u << S) - 1;      // Q6_K: stage slots whose correction rows may hold non-zero data (per warp)
        int issued = (FMT == FMT_Q6K) ? (R < nsb ? R : nsb) : 0;
        int sb = 0;
        for (; sb < nsb; ++sb) {
            const int slot = sb % R;
            // waits are warp-uniform (all lanes leave together): the warp-level arrivals below need it
            if (!__all_sync(kFull, mbar_wait(&bars.raw_full[slot], (sb / R) & 1, err, ERR_GEMM_RAW_FULL, abort_flag)))
                break;
            // Q6_K: the block starts blk_r bytes into its row's 16-byte aligned copy at blk_a
            const uint32_t blk_a = smem_u32(raw_row0 + slot * BN * C::RAW_ROW);
            const uint32_t blk_r = valid ? (uint32_t)(reinterpret_cast<uintptr_t>(wrow + (int64_t)sb * C::BB) & 15) : 0u;
            const uint32_t blk = blk_a + blk_r;
            // ---- super-block header
            float d = 0.0f, dmin = 0.0f;
            int sc[16];
            int mn[8];
            float dw[8], mw[8];          // 32-value formats: each block's d and m (m = 0 without one)
            bool wbig = false;           // Q6_K: some row of the warp has a big scale in this super-block
            // Q6_K: the 16 int8 scales (big ones made even) and the correction factors (1 where the
            // scale is big, else 0), four per word
            uint32_t scw[4], cw[4];
            if constexpr (C::B32) {
                // block j's fp16 d at byte BS j of the group (2-byte aligned), m right after it
                constexpr int BS = b32_bytes(FMT);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const uint32_t o = (uint32_t)(BS * j);
                    const uint32_t wd = valid ? lds32(blk + (o & ~3u)) : 0u;
                    const uint32_t dbits = (o & 2u) ? (wd >> 16) : (wd & 0xffffu);
                    dw[j] = __half2float(__ushort_as_half((unsigned short)dbits));
                    mw[j] = 0.0f;
                    if constexpr (b32_has_m(FMT))      // Q4_1 / Q5_1 blocks are 4-byte aligned: d | m << 16
                        mw[j] = __half2float(__ushort_as_half((unsigned short)(wd >> 16)));
                }
            } else if constexpr (C::KQ) {
                const uint4 hd = valid ? lds128(blk) : make_uint4(0, 0, 0, 0);
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
                uint32_t tail[5];                 // bytes 192..211: scales[16], d
                if (valid) {
                    lds_words_r<5>(blk_a + 192, blk_r, tail);
                } else {
#pragma unroll
                    for (int i = 0; i < 5; ++i) tail[i] = 0;
                }
                d = __half2float(__ushort_as_half((unsigned short)(tail[4] & 0xffff)));
                // an odd |sc| > 64 (13 bits with q - 32) keeps sc - 1 in the main tile and marks the
                // correction tile, which then carries q - 32 itself.  For an int8 byte that is bit 0
                // and (bit 6 xor bit 7): 65..127 and -128..-65 are the bytes whose bits 6 and 7 differ.
                uint32_t any = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    cw[i] = tail[i] & ((tail[i] >> 6) ^ (tail[i] >> 7)) & 0x01010101u;
                    scw[i] = tail[i] & ~cw[i];
                    any |= cw[i];
                }
                wbig = __any_sync(kFull, any != 0);
            }
            // ---- per-row factors of this super-block: d for the epilogue, -dmin m_j for the min MMA
            if (!__all_sync(kFull, mbar_wait(&bars.info_empty[sb & 1], ((sb >> 1) & 1) ^ 1, err, ERR_GEMM_INFO_EMPTY,
                                             abort_flag)))
                break;
            if constexpr (C::B32) {
#pragma unroll
                for (int j = 0; j < 8; ++j) info0[((sb & 1) * 8 + j) * BN + r] = dw[j];
            } else {
                info0[(sb & 1) * BN + r] = d;
            }
            if constexpr (C::MIN) {
                // -dmin*m_j has at most 17 significant bits (exact in f32); it splits exactly into
                // a tf32 pair: row = [hi_0..hi_7 | lo_0..lo_7].  The fp16 block offset m of Q4_1 /
                // Q5_1 is exact in tf32 itself (lo = 0).
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float v = C::B32 ? mw[j] : -(dmin * (float)mn[j]);
                    const float vh = tf32_rn(v);
                    wh[j] = __float_as_uint(vh);
                    wl[j] = __float_as_uint(v - vh);
                }
                const uint32_t bt = bmin_tile0 + (sb & 1) * C::MIN_TILE;
                sts128(sw64_chunk(bt, r, 0), make_uint4(wh[0], wh[1], wh[2], wh[3]));
                sts128(sw64_chunk(bt, r, 1), make_uint4(wh[4], wh[5], wh[6], wh[7]));
                sts128(sw64_chunk(bt, r, 2), make_uint4(wl[0], wl[1], wl[2], wl[3]));
                sts128(sw64_chunk(bt, r, 3), make_uint4(wl[4], wl[5], wl[6], wl[7]));
                fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.info_full[sb & 1]);      // one arrival per unpack warp

            // ---- four 64-value stages of this super-block (unrolled: sc[] stays in registers)
            bool ok = true;
            uint32_t ql[16], qh[8];      // Q6_K: the current half's low / high bits, read once per half
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int st = sb * 4 + q, s = st % S;
                if (!__all_sync(kFull, mbar_wait(&bars.ab_empty[s], ((st / S) & 1) ^ 1, err, ERR_GEMM_AB_EMPTY,
                                                 abort_flag))) {
                    ok = false;
                    break;
                }
                const uint32_t btile = b_tile0 + s * kTile;
                if constexpr (C::B32) {
                    // blocks 2q and 2q+1 of the group: 32 values each, as the exact f16 integers
                    // q - off (Q8_0: the int8 quant) -- 1024 + byte by a byte permute, minus 1024 + off
                    constexpr int BS = b32_bytes(FMT), OFF = b32_off(FMT);
                    constexpr bool HAS_M = b32_has_m(FMT), FIVE = b32_five(FMT), Q8 = FMT == FMT_Q8_0;
                    constexpr int QH = HAS_M ? 4 : 2, QS = 2 + (HAS_M ? 2 : 0) + (FIVE ? 4 : 0);
                    const __half2 bias = __float2half2_rn(1024.0f + (Q8 ? 128.0f : (float)OFF));
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        // the block's 16-byte aligned superset (2 or 3 reads, inside the group)
                        const int o0 = BS * (2 * q + k), a0 = o0 & ~15, nu = (o0 + BS - a0 + 15) >> 4;
                        uint32_t wv[12];
#pragma unroll
                        for (int u = 0; u < 3; ++u) {
                            uint4 t = make_uint4(0, 0, 0, 0);
                            if (u < nu && valid) t = lds128(blk + (uint32_t)(a0 + 16 * u));
                            wv[4 * u] = t.x;
                            wv[4 * u + 1] = t.y;
                            wv[4 * u + 2] = t.z;
                            wv[4 * u + 3] = t.w;
                        }
                        const int b = o0 - a0;           // the block's first byte in wv (even)
                        auto word = [&](int o) -> uint32_t {   // 4 bytes at byte b + o of the block
                            const int x = b + o;
                            return (x & 3) ? __funnelshift_r(wv[x >> 2], wv[(x >> 2) + 1], 16) : wv[x >> 2];
                        };
                        const uint32_t qhw = FIVE ? word(QH) : 0u;
#pragma unroll
                        for (int c = 0; c < 4; ++c) {    // values 8c .. 8c+7 of the block
                            uint32_t o[4];
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                uint32_t v;
                                if constexpr (Q8) {
                                    v = word(2 + 8 * c + 4 * e) ^ 0x80808080u;      // int8 -> q + 128
                                } else {
                                    // values 8c + 4e .. +3: nibbles of qs word 2 (c & 1) + e, low for c < 2
                                    const int ew = 2 * (c & 1) + e;
                                    v = (word(QS + 4 * ew) >> (4 * (c >> 1))) & 0x0f0f0f0fu;
                                    if constexpr (FIVE)
                                        v |= (((qhw >> (16 * (c >> 1) + 4 * ew)) & 0xfu) * 0x02040810u) & 0x10101010u;
                                }
                                uint32_t h0, h1;
                                bytes_to_h2_biased(v, h0, h1);
                                o[2 * e] = h2_as_u32(__hsub2(u32_as_h2(h0), bias));
                                o[2 * e + 1] = h2_as_u32(__hsub2(u32_as_h2(h1), bias));
                            }
                            sts128(sw128_chunk(btile, r, 4 * k + c), make_uint4(o[0], o[1], o[2], o[3]));
                        }
                    }
                } else if constexpr (C::KQ) {
                    // sub-blocks 2q (low nibbles of qs[32q..32q+32)) and 2q+1 (high nibbles); Q5_K:
                    // qs at byte 48, and bit j of qh[l] is the fifth bit of element l of sub-block j
                    constexpr uint32_t QS = FMT == FMT_Q5K ? 48 : 16;
                    uint4 q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
                    uint4 h0v = make_uint4(0, 0, 0, 0), h1v = make_uint4(0, 0, 0, 0);
                    if (valid) {
                        q0 = lds128(blk + QS + 32 * q);
                        q1 = lds128(blk + QS + 32 * q + 16);
                        if constexpr (FMT == FMT_Q5K) {
                            h0v = lds128(blk + 16);
                            h1v = lds128(blk + 32);
                        }
                    }
                    const uint32_t wq[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    const uint32_t wh[8] = {h0v.x, h0v.y, h0v.z, h0v.w, h1v.x, h1v.y, h1v.z, h1v.w};
#pragma unroll
                    for (int hn = 0; hn < 2; ++hn) {
                        const float scf = (float)sc[2 * q + hn];
                        const __half2 sc2 = __float2half2_rn(scf);
                        const __half2 neg = __float2half2_rn(-1024.0f * scf);
#pragma unroll
                        for (int cc = 0; cc < 4; ++cc) {
                            uint32_t va = (wq[2 * cc] >> (4 * hn)) & 0x0f0f0f0fu;
                            uint32_t vb = (wq[2 * cc + 1] >> (4 * hn)) & 0x0f0f0f0fu;
                            if constexpr (FMT == FMT_Q5K) {             // + 16 * bit (2q + hn) of qh[l]
                                va |= ((wh[2 * cc] >> (2 * q + hn)) & 0x01010101u) << 4;
                                vb |= ((wh[2 * cc + 1] >> (2 * q + hn)) & 0x01010101u) << 4;
                            }
                            uint32_t h0, h1, h2, h3;
                            bytes_to_h2_biased(va, h0, h1);
                            bytes_to_h2_biased(vb, h2, h3);
                            uint4 o;
                            // (1024 + q) sc - 1024 sc in one fused op: exact, sc q <= 63 * 31 < 2048
                            o.x = h2_as_u32(__hfma2(u32_as_h2(h0), sc2, neg));
                            o.y = h2_as_u32(__hfma2(u32_as_h2(h1), sc2, neg));
                            o.z = h2_as_u32(__hfma2(u32_as_h2(h2), sc2, neg));
                            o.w = h2_as_u32(__hfma2(u32_as_h2(h3), sc2, neg));
                            sts128(sw128_chunk(btile, r, 4 * hn + cc), o);
                        }
                    }
                } else {
                    // half h = q/2, groups g = 2(q%2), 2(q%2)+1; chunk c -> g = g0 + c/4, l = 8(c%4)
                    const int h = q >> 1, g0 = 2 * (q & 1);
                    if ((q & 1) == 0) {
                        if (valid) {
                            lds_words_r<16>(blk_a + 64 * h, blk_r, ql);
                            lds_words_r<8>(blk_a + 128 + 32 * h, blk_r, qh);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) ql[i] = 0;
#pragma unroll
                            for (int i = 0; i < 8; ++i) qh[i] = 0;
                        }
                    }
                    const int nsh = (g0 >= 2) ? 4 : 0;
                    const __half2 bias = __float2half2_rn(1056.0f);
                    const uint32_t bct = bc_tile0 + s * kTile;
                    // the 8 values of chunk c as (q - 32) pairs
                    auto chunk_t = [&](int c, __half2 (&t)[4]) {
                        const int g = g0 + (c >> 2), l = 8 * (c & 3);
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const uint32_t lw = ql[8 * (g & 1) + (l >> 2) + e];
                            const uint32_t hw = qh[(l >> 2) + e];
                            const uint32_t v = ((lw >> nsh) & 0x0f0f0f0fu) | (((hw >> (2 * g)) & 0x03030303u) << 4);
                            uint32_t b0, b1;
                            bytes_to_h2_biased(v, b0, b1);
                            t[2 * e] = __hsub2(u32_as_h2(b0), bias);      // q - 32, exact
                            t[2 * e + 1] = __hsub2(u32_as_h2(b1), bias);
                        }
                    };
                    auto chunk_si = [&](int c) { return 8 * h + 2 * (g0 + (c >> 2)) + ((c & 3) >= 2 ? 1 : 0); };
                    // pass 0 writes the main tile, (q - 32) times the scale (made even if big); pass 1
                    // (only while the warp has big scales in this super-block, and once more after it,
                    // to zero its rows) the correction tile, (q - 32) times 1 where the scale is big, else 0
                    const int npass = (wbig || ((dirty >> s) & 1)) ? 2 : 1;
#pragma unroll 1
                    for (int pass = 0; pass < npass; ++pass) {
                        uint32_t fw[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) fw[i] = pass ? cw[i] : scw[i];
                        const uint32_t tile = pass ? bct : btile;
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const int si = chunk_si(c);
                            const __half2 s2 = __float2half2_rn((float)(int)(int8_t)(fw[si >> 2] >> (8 * (si & 3))));
                            __half2 t[4];
                            chunk_t(c, t);
                            sts128(sw128_chunk(tile, r, c),
                                   make_uint4(h2_as_u32(__hmul2(t[0], s2)), h2_as_u32(__hmul2(t[1], s2)),
                                              h2_as_u32(__hmul2(t[2], s2)), h2_as_u32(__hmul2(t[3], s2))));
                        }
                    }
                    if (wbig) dirty |= 1u << s; else dirty &= ~(1u << s);
                    if (lane == 0) corr_flags[4 * s + (warp - kWarpUnpack0)] = wbig ? 1u : 0u;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars.b_full[s]);          // one arrival per unpack warp
            }
            if (!ok) break;
            if constexpr (C::TMW) {
                __syncwarp();                               // the warp's 32 rows of this slot are read
                if (lane == 0) mbar_arrive(&bars.raw_empty[slot]);
            } else if (sb + R < nsb) {
                issue_raw(sb + R);
                ++issued;
            }
        }
        if (*abort_flag) {   // wait (bounded) for this row's copies still in flight
            for (int i = sb; i < issued; ++i)
                mbar_wait(&bars.raw_full[i % R], (i / R) & 1, err, ERR_GEMM_RAW_FULL, nullptr);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REGS_EPI));
        // ------------------------------------------------------------ epilogue
        const int e = warp - kWarpEpi0, qd = warp & 3, hf = e >> 2;
        const int64_t m = m0 + 32 * qd + lane;
        const bool valid_m = m < M;
        const uint32_t trow = tmem + ((uint32_t)(32 * qd) << 16);
        const int col0 = hf * 64;
        // TMEM column of this thread's 32-column half hh: plain, 64 hf + 32 hh; SWIGLU, gate
        // columns 32 hf .. (hh = 0) and the matching up columns 64 + 32 hf .. (hh = 1)
        auto colh = [&](int hh) -> int { return SWIGLU ? 32 * hf + 64 * hh : col0 + 32 * hh; };
        const int64_t nblk32 = K / kQ8;
        const float *info0 = reinterpret_cast<const float *>(sm + C::OFF_INFO);
        // acc: the running sum over super-blocks; part: sum_j d_a[j] I_j of the current super-block
        float2 acc[32], part[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            acc[i] = make_float2(0.0f, 0.0f);
            part[i] = make_float2(0.0f, 0.0f);
        }
        // activation scales: this thread's token in the stager's shared-memory tile
        const float *da_tok = reinterpret_cast<const float *>(sm + C::OFF_DA) + 32 * qd + lane;
        // The waits below decide the same way in every lane: the warp enters each one converged
        // (after a .sync.aligned TMEM op) and its lanes probe the same barrier, read the same abort
        // flag and the same timer in the same instructions, so a failure makes the whole warp leave
        // together and no lane is left at an .aligned TMEM load alone.  (Voting on each result
        // instead measured 10% slower.)
        bool ok = true;
        for (int sb = 0; sb < nsb && ok; ++sb) {
            if (!mbar_wait(&bars.da_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_DA, abort_flag)) break;
            const float *da_sb = da_tok + (sb & 1) * 8 * BM;
            float das[8];
            if constexpr (C::DA_TOK) {
                const float4 *dq = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(sm + C::OFF_DA) +
                                                                    (sb & 1) * 8 * BM + (32 * qd + lane) * 8);
                const float4 dq0 = dq[0], dq1 = dq[1];
                das[0] = dq0.x; das[1] = dq0.y; das[2] = dq0.z; das[3] = dq0.w;
                das[4] = dq1.x; das[5] = dq1.y; das[6] = dq1.z; das[7] = dq1.w;
            }
            // 32-value formats: every block's d per weight row is needed from the first block on
            if constexpr (C::B32)
                if (!mbar_wait(&bars.info_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_INFO_FULL, abort_flag)) break;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int gb = sb * 8 + j;
                const int slot = gb % C::ACC;
                if (!mbar_wait(&bars.acc_full[slot], (gb / C::ACC) & 1, err, ERR_GEMM_ACC_FULL, abort_flag)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float da = C::DA_TOK ? das[j] : da_sb[j * BM];
                const float2 da2 = make_float2(da, da);
                // Q4_K: both 32-column halves in flight together, one wait, then the slot goes back;
                // Q6_K (a smaller epilogue register budget): one half at a time
                constexpr bool kBoth = C::TMW;
                uint32_t vv[kBoth ? 2 : 1][32];
                if constexpr (kBoth) {
                    tmem_ld32(trow + (uint32_t)(slot * BN + colh(0)), vv[0]);
                    tmem_ld32(trow + (uint32_t)(slot * BN + colh(1)), vv[kBoth ? 1 : 0]);
                    tmem_ld_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars.acc_empty[slot]);
                }
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if constexpr (!kBoth) {
                        tmem_ld32(trow + (uint32_t)(slot * BN + colh(hh)), vv[0]);
                        tmem_ld_wait();
                        if (hh == 1) {       // both halves are in registers: hand the slot back to the MMA
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&bars.acc_empty[slot]);
                        }
                    }
                    const uint32_t (&v)[32] = vv[kBoth ? hh : 0];
                    if constexpr (C::B32) {
                        // y += I (d_a d_w): d_w of the 32 weight rows from the unpackers' table
                        const float4 *dwv =
                            reinterpret_cast<const float4 *>(info0 + ((sb & 1) * 8 + j) * BN + colh(hh));
#pragma unroll
                        for (int i4 = 0; i4 < 8; ++i4) {
                            const float4 dv = dwv[i4];
                            const float2 c0 = __fmul2_rn(da2, make_float2(dv.x, dv.y));
                            const float2 c1 = __fmul2_rn(da2, make_float2(dv.z, dv.w));
                            acc[16 * hh + 2 * i4] = __ffma2_rn(
                                make_float2(__uint_as_float(v[4 * i4]), __uint_as_float(v[4 * i4 + 1])), c0,
                                acc[16 * hh + 2 * i4]);
                            acc[16 * hh + 2 * i4 + 1] = __ffma2_rn(
                                make_float2(__uint_as_float(v[4 * i4 + 2]), __uint_as_float(v[4 * i4 + 3])), c1,
                                acc[16 * hh + 2 * i4 + 1]);
                        }
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            part[16 * hh + i] = __ffma2_rn(make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])),
                                                           da2, part[16 * hh + i]);
                    }
                    if constexpr (DUMP) {
                        if (valid_m && m >= dump.m0 && m < dump.m0 + dump.m_cnt) {
#pragma unroll
                            for (int i = 0; i < 32; ++i) {
                                const int64_t n = n0 + colh(hh) + i;
                                if (n >= dump.n0 && n < dump.n0 + dump.n_cnt && n < N)
                                    dump.out[((m - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32 + gb] =
                                        __float2int_rn(__uint_as_float(v[i]));
                            }
                        }
                    }
                }
            }
            if (!ok) break;
            // ---- super-block end: acc += d * part (d: fp16 factor of each weight row)
            if constexpr (C::B32) {
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars.info_empty[sb & 1]);
                    mbar_arrive(&bars.da_empty[sb & 1]);
                }
                continue;
            }
            if (!mbar_wait(&bars.info_full[sb & 1], (sb >> 1) & 1, err, ERR_GEMM_INFO_FULL, abort_flag)) break;
            const float4 *info = reinterpret_cast<const float4 *>(info0 + (sb & 1) * BN);
            // all 16 loads of the 64 row factors first (independent, their latencies overlap), then the FMAs
            float4 dv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) dv[i] = info[colh(i >> 3) / 4 + (i & 7)];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                acc[2 * i] = __ffma2_rn(part[2 * i], make_float2(dv[i].x, dv[i].y), acc[2 * i]);
                acc[2 * i + 1] = __ffma2_rn(part[2 * i + 1], make_float2(dv[i].z, dv[i].w), acc[2 * i + 1]);
                part[2 * i] = make_float2(0.0f, 0.0f);
                part[2 * i + 1] = make_float2(0.0f, 0.0f);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars.info_empty[sb & 1]);
                mbar_arrive(&bars.da_empty[sb & 1]);
            }
        }
        if (ok && !*abort_flag) {
            if constexpr (C::MIN) {
                // the tensor-core min term, summed over all super-blocks
                if (mbar_wait(bars.min_final, 0, err, ERR_GEMM_MIN, abort_flag)) {
                    tc_fence_after();
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v[32];
                        tmem_ld32(trow + kMinCol + (uint32_t)colh(hh), v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            acc[16 * hh + i] = __fadd2_rn(acc[16 * hh + i],
                                                          make_float2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])));
                    }
                } else {
                    ok = false;
                }
            }
            if constexpr (SWIGLU) {
                // outputs n0 + 32 hf .. +31 of token m: silu(gate) * up, one Q8 block of the plane
                // (the plane's K is N, a multiple of 256, so the block is whole)
                const int64_t nb0 = n0 + 32 * hf;
                if (ok && valid_m && nb0 < N) {
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        v[2 * i] = swiglu1(acc[i].x, acc[16 + i].x);
                        v[2 * i + 1] = swiglu1(acc[i].y, acc[16 + i].y);
                    }
                    float d, hi, lo;
                    int sum;
                    quantize_block32(v, po.q8 + m * N + nb0, po.q16 + m * N + nb0, d, sum, hi, lo);
                    const int64_t b = nb0 / kQ8;
                    po.d[b * M + m] = d;
                    po.s[b * M + m] = sum;
                    float *row = po.ds + m * (2 * (N / kQ8)) + (b >> 3) * 16 + (b & 7);
                    row[0] = hi;
                    row[8] = lo;
                }
            } else if (ok && valid_m) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int64_t nb0 = n0 + colh(hh);
                    float *dst = y + m * N + nb0;
                    if (nb0 + 32 <= N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
#pragma unroll
                        for (int i = 0; i < 16; i += 2)
                            *reinterpret_cast<float4 *>(dst + 2 * i) =
                                make_float4(acc[16 * hh + i].x, acc[16 * hh + i].y, acc[16 * hh + i + 1].x,
                                            acc[16 * hh + i + 1].y);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            if (nb0 + 2 * i < N) dst[2 * i] = acc[16 * hh + i].x;
                            if (nb0 + 2 * i + 1 < N) dst[2 * i + 1] = acc[16 * hh + i].y;
                        }
                    }
                }
            }
        }
    }

    __syncthreads();
    if (warp == kWarpMma) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

template <int FMT, bool DUMP>
int launch_fmt(const CUtensorMap &tm, const CUtensorMap &tmds, const CUtensorMap &tmw, const uint8_t *w, int64_t N,
               int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump, unsigned int *err,
               cudaStream_t stream) {
    using C = GmCfg<FMT>;
    auto kern = gemm_kernel<FMT, DUMP, false>;
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, FMT * 2 + (DUMP ? 1 : 0));
    if (rc != MQ_OK) return rc;
    const dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
    return cuda_error(launch_pdl(kern, grid, dim3(kThreads), C::SMEM, stream, tm, tmds, tmw, tmw, w, N, K, p, M, y,
                                 Plane{}, dump, err),
                      "gemm launch");
}

// the fused gate|up GEMM: tmg / tmu are the gate and up weight maps with 64-row boxes; the
// output plane po has K = F
template <int FMT>
int launch_swiglu_fmt(const CUtensorMap &tm, const CUtensorMap &tmds, const CUtensorMap &tmg, const CUtensorMap &tmu,
                      const uint8_t *wg, int64_t F, int64_t K, const Plane &p, int64_t M, const Plane &po,
                      unsigned int *err, cudaStream_t stream) {
    using C = GmCfg<FMT>;
    auto kern = gemm_kernel<FMT, false, true>;
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, kAttrSlotSwiglu + FMT);
    if (rc != MQ_OK) return rc;
    const dim3 grid((unsigned)((M + BM - 1) / BM), (unsigned)((F + BN / 2 - 1) / (BN / 2)));
    return cuda_error(launch_pdl(kern, grid, dim3(kThreads), C::SMEM, stream, tm, tmds, tmg, tmu, wg, F, K, p, M,
                                 static_cast<float *>(nullptr), po, Dump{nullptr, 0, 0, 0, 0}, err),
                      "gemm swiglu launch");
}

}  // namespace

// the 32-value formats' launches (mq_gemm_b32.cu), with the tensor maps launch_gemm encodes
int launch_gemm_b32(Fmt fmt, const CUtensorMap &tm, const CUtensorMap &tmds, const CUtensorMap &tmw,
                    const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump,
                    unsigned int *err, cudaStream_t stream);

}  // namespace mq
