// mq_gemv.cu -- decode GEMV (MMVQ): raw Q4_K / Q6_K weight bytes x Q8 codes with dp4a.
//
// minfer pages, "Support Matrix > CUDA notes": decode (nt == 1) uses the dp4a MMVQ
// kernels; "Roadmap > 0": the decode path streams the weights once per token.
//
// Design (HBM-bound): every weight byte is read from HBM exactly once per group of up
// to 8 tokens.  Each warp owns a private 4-stage ring in shared memory and walks its
// rows in chunks of up to 16 super-blocks; lane 0 refills a stage with one 1-D bulk
// async copy (TMA engine) of the 16-byte-aligned superset of the chunk's bytes, so a
// Q6_K block (210 B, only 2-byte aligned) needs no special load path from HBM.  About
// 80 KiB per SM is in flight.  The math runs from shared memory: 8 lanes per
// super-block, each owning 32 of its 256 values, dp4a against the int8 codes (read
// through L1), f32 scaling per 32-value block, one warp reduction per row.
#include <cuda_fp16.h>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int kWarps = 8;
constexpr int kStages = 4;
constexpr int kChunkBlocks = 16;
constexpr unsigned kFull = 0xffffffffu;

template <int FMT>
struct GvCfg {
    static constexpr int BB = FMT == FMT_Q4K ? 144 : 210;
    // superset of a 16-block chunk + up to 15 leading bytes + 16 bytes of over-read slack
    static constexpr int STAGE = ((kChunkBlocks * BB + 15 + 15) / 16) * 16 + 16;
    static constexpr int SMEM = kWarps * kStages * STAGE;
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
__device__ __forceinline__ uint32_t lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ int lds8s(uint32_t addr) {
    short v;
    asm volatile("ld.shared.s8 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
// 8 bytes at a 2-byte aligned shared address
__device__ __forceinline__ uint2 lds64_a2(uint32_t addr) {
    const uint32_t b = addr & ~3u, sh = (addr & 3u) * 8u;
    const uint32_t w0 = lds32(b), w1 = lds32(b + 4), w2 = lds32(b + 8);
    return make_uint2(__funnelshift_r(w0, w1, sh), __funnelshift_r(w1, w2, sh));
}

__device__ __forceinline__ float half_bits_to_float(uint32_t bits) {
    return __half2float(__ushort_as_half((unsigned short)bits));
}

// byte-wise v - 32 for bytes in [0, 63] (result bytes are the signed values)
__device__ __forceinline__ uint32_t minus32_bytes(uint32_t v) {
    return ((v | 0x80808080u) - 0x20202020u) ^ 0x80808080u;
}

template <int FMT, int MT, bool DUMP>
__global__ void __launch_bounds__(kWarps * 32) gemv_kernel(const uint8_t *__restrict__ w, int64_t N, int64_t K,
                                                           Plane p, int64_t M, int64_t t0, int mt,
                                                           float *__restrict__ y, Dump dump, unsigned int *err) {
    using C = GvCfg<FMT>;
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ __align__(8) uint64_t bars[kWarps][kStages];

    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint8_t *ring = smem + warp * kStages * C::STAGE;
    const uint32_t ring_s = smem_u32(ring);
    uint64_t *bar = bars[warp];

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bar[s], 1);
        mbar_init_fence();
    }
    __syncwarp();

    const int64_t nb = K / kQK;                         // super-blocks per row
    const int64_t nch = (nb + kChunkBlocks - 1) / kChunkBlocks;
    const int64_t row_bytes = nb * C::BB;
    const int64_t nblk32 = K / kQ8;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, GW = (int64_t)gridDim.x * kWarps;
    const int64_t nrows = gw < N ? (N - gw + GW - 1) / GW : 0;
    const int64_t items = nrows * nch;

    auto item_range = [&](int64_t item, int64_t &n, int64_t &c, int64_t &start, int64_t &end) {
        const int64_t r = item / nch;
        c = item - r * nch;
        n = gw + r * GW;
        start = n * row_bytes + c * kChunkBlocks * C::BB;
        end = start + kChunkBlocks * C::BB;
        if (end > (n + 1) * row_bytes) end = (n + 1) * row_bytes;
    };
    auto issue = [&](int64_t item) {
        int64_t n, c, start, end;
        item_range(item, n, c, start, end);
        const int64_t a0 = start & ~(int64_t)15, a1 = (end + 15) & ~(int64_t)15;
        const int s = (int)(item % kStages);
        mbar_arrive_expect_tx(&bar[s], (uint32_t)(a1 - a0));
        bulk_copy_g2s(ring + s * C::STAGE, w + a0, (uint32_t)(a1 - a0), &bar[s]);
    };

    if (lane == 0)
        for (int64_t i = 0; i < items && i < kStages; ++i) issue(i);

    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;

    const int u = lane & 7;          // the 32-value unit of the super-block this lane owns
    bool ok = true;
    int64_t item = 0;
    for (; item < items; ++item) {
        const int s = (int)(item % kStages);
        const bool got = mbar_wait(&bar[s], (uint32_t)((item / kStages) & 1), err, ERR_GEMV_FULL, nullptr);
        if (!__all_sync(kFull, got)) {   // leave the loop together (shuffles below need every lane)
            ok = false;
            break;
        }
        int64_t n, c, start, end;
        item_range(item, n, c, start, end);
        const int nblk_c = (int)((end - start) / C::BB);
        const uint32_t base = ring_s + s * C::STAGE + (uint32_t)(start & 15);

#pragma unroll
        for (int g4 = 0; g4 < kChunkBlocks / 4; ++g4) {
            const int lb = (lane >> 3) + 4 * g4;                 // block of the chunk
            const bool valid = lb < nblk_c;                      // uniform over the 8 lanes of a block
            if (!__any_sync(kFull, valid)) break;
            const int64_t sbi = c * kChunkBlocks + lb;           // super-block index in the row
            const uint32_t blk = base + (uint32_t)(lb * C::BB);
            if constexpr (FMT == FMT_Q4K) {
                // unit u: qs bytes [16u, 16u+16): low nibbles -> sub-block j0 = u & ~1,
                // values 32*j0 + 16*(u&1) + i; high nibbles -> j1 = j0 + 1.
                uint4 hd = make_uint4(0, 0, 0, 0), qv = make_uint4(0, 0, 0, 0);
                if (valid) {
                    hd = lds128(blk);
                    qv = lds128(blk + 16 + 16 * u);
                }
                const float d = half_bits_to_float(hd.x & 0xffff), dmin = half_bits_to_float(hd.x >> 16);
                const int j0 = u & ~1, j1 = j0 + 1;
                // the 12 scale bytes: s[0..3] = hd.y, s[4..7] = hd.z, s[8..11] = hd.w
                auto sb = [&](int i) -> int {
                    const uint32_t wv = i < 4 ? hd.y : (i < 8 ? hd.z : hd.w);
                    return (int)((wv >> (8 * (i & 3))) & 0xff);
                };
                int sc0, m0, sc1, m1;
                if (j0 < 4) {
                    sc0 = sb(j0) & 63; m0 = sb(j0 + 4) & 63;
                    sc1 = sb(j1) & 63; m1 = sb(j1 + 4) & 63;
                } else {
                    sc0 = (sb(j0 + 4) & 15) | ((sb(j0 - 4) >> 6) << 4);
                    m0 = (sb(j0 + 4) >> 4) | ((sb(j0) >> 6) << 4);
                    sc1 = (sb(j1 + 4) & 15) | ((sb(j1 - 4) >> 6) << 4);
                    m1 = (sb(j1 + 4) >> 4) | ((sb(j1) >> 6) << 4);
                }
                const uint32_t lo[4] = {qv.x & 0x0f0f0f0fu, qv.y & 0x0f0f0f0fu, qv.z & 0x0f0f0f0fu,
                                        qv.w & 0x0f0f0f0fu};
                const uint32_t hi[4] = {(qv.x >> 4) & 0x0f0f0f0fu, (qv.y >> 4) & 0x0f0f0f0fu,
                                        (qv.z >> 4) & 0x0f0f0f0fu, (qv.w >> 4) & 0x0f0f0f0fu};
                const int64_t k_lo = sbi * kQK + 32 * j0 + 16 * (u & 1);
                const int64_t b0 = sbi * 8 + j0, b1 = b0 + 1;     // Q8 block indices
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    const int64_t m = t0 + t;
                    const bool act = t < mt && valid;
                    int D0 = 0, D1 = 0;
                    if (act) {
                        const int8_t *a = p.q8 + m * K;
                        const uint4 a0 = __ldg(reinterpret_cast<const uint4 *>(a + k_lo));
                        const uint4 a1 = __ldg(reinterpret_cast<const uint4 *>(a + k_lo + 32));
                        D0 = __dp4a((int)lo[0], (int)a0.x, 0);
                        D0 = __dp4a((int)lo[1], (int)a0.y, D0);
                        D0 = __dp4a((int)lo[2], (int)a0.z, D0);
                        D0 = __dp4a((int)lo[3], (int)a0.w, D0);
                        D1 = __dp4a((int)hi[0], (int)a1.x, 0);
                        D1 = __dp4a((int)hi[1], (int)a1.y, D1);
                        D1 = __dp4a((int)hi[2], (int)a1.z, D1);
                        D1 = __dp4a((int)hi[3], (int)a1.w, D1);
                        const float da0 = __ldg(p.d + b0 * M + m), da1 = __ldg(p.d + b1 * M + m);
                        float v = d * ((float)(sc0 * D0) * da0 + (float)(sc1 * D1) * da1);
                        if ((u & 1) == 0) {   // the min term of a 32-value block is taken once
                            const float s0 = (float)__ldg(p.s + b0 * M + m), s1 = (float)__ldg(p.s + b1 * M + m);
                            v -= dmin * ((float)m0 * da0 * s0 + (float)m1 * da1 * s1);
                        }
                        acc[t] += v;
                    }
                    if constexpr (DUMP) {
                        // a 32-value block's dot is split over lanes u and u^1
                        D0 += __shfl_xor_sync(kFull, D0, 1);
                        D1 += __shfl_xor_sync(kFull, D1, 1);
                        if (act && (u & 1) == 0 && m >= dump.m0 && m < dump.m0 + dump.m_cnt &&
                            n >= dump.n0 && n < dump.n0 + dump.n_cnt) {
                            int32_t *o = dump.out + ((m - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32;
                            o[b0] = sc0 * D0;
                            o[b1] = sc1 * D1;
                        }
                    }
                }
            } else {
                // unit u: half h = u >> 2, l0 = 8*(u & 3); values 128h + 32g + l0 + i (g = 0..3,
                // i = 0..7).  Group g: low (g < 2) / high (g >= 2) nibble of ql[64h + 32(g&1) + l0 + i],
                // high bits (qh[32h + l0 + i] >> 2g) & 3; scale index 8h + 2g + (l0 >= 16).
                const int h = u >> 2, l0 = 8 * (u & 3);
                uint2 ql0 = make_uint2(0, 0), ql1 = make_uint2(0, 0), qh = make_uint2(0, 0);
                float d = 0.0f;
                int scg[4] = {0, 0, 0, 0};
                if (valid) {
                    ql0 = lds64_a2(blk + 64 * h + l0);
                    ql1 = lds64_a2(blk + 64 * h + 32 + l0);
                    qh = lds64_a2(blk + 128 + 32 * h + l0);
                    d = half_bits_to_float(lds16(blk + 208));
#pragma unroll
                    for (int g = 0; g < 4; ++g) scg[g] = lds8s(blk + 192 + 8 * h + 2 * g + (l0 >> 4));
                }
                uint32_t qs[4][2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const uint32_t a = e ? ql0.y : ql0.x, b = e ? ql1.y : ql1.x, hb = e ? qh.y : qh.x;
                    qs[0][e] = minus32_bytes((a & 0x0f0f0f0fu) | ((hb & 0x03030303u) << 4));
                    qs[1][e] = minus32_bytes((b & 0x0f0f0f0fu) | (((hb >> 2) & 0x03030303u) << 4));
                    qs[2][e] = minus32_bytes(((a >> 4) & 0x0f0f0f0fu) | (((hb >> 4) & 0x03030303u) << 4));
                    qs[3][e] = minus32_bytes(((b >> 4) & 0x0f0f0f0fu) | (((hb >> 6) & 0x03030303u) << 4));
                }
                const int64_t kb = sbi * kQK + 128 * h + l0;
                const int64_t bq = sbi * 8 + 4 * h;                // Q8 block of group 0
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    int Dg[4] = {0, 0, 0, 0};
                    const int64_t m = t0 + t;
                    if (t < mt && valid) {
                        const int8_t *a = p.q8 + m * K + kb;
                        float v = 0.0f;
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            const uint2 av = __ldg(reinterpret_cast<const uint2 *>(a + 32 * g));
                            Dg[g] = __dp4a((int)qs[g][0], (int)av.x, __dp4a((int)qs[g][1], (int)av.y, 0));
                            v += (float)(scg[g] * Dg[g]) * __ldg(p.d + (bq + g) * M + m);
                        }
                        acc[t] += d * v;
                    }
                    if constexpr (DUMP) {
                        int I[4];
#pragma unroll
                        for (int g = 0; g < 4; ++g) {
                            I[g] = scg[g] * Dg[g];
                            I[g] += __shfl_xor_sync(kFull, I[g], 1);
                            I[g] += __shfl_xor_sync(kFull, I[g], 2);
                        }
                        if (t < mt && valid && (u & 3) == 0 && m >= dump.m0 && m < dump.m0 + dump.m_cnt &&
                            n >= dump.n0 && n < dump.n0 + dump.n_cnt) {
                            int32_t *o = dump.out + ((m - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32;
#pragma unroll
                            for (int g = 0; g < 4; ++g) o[bq + g] = I[g];
                        }
                    }
                }
            }
        }

        if (c == nch - 1) {
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                float v = acc[t];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
                if (lane == 0 && t < mt) y[(t0 + t) * N + n] = v;
                acc[t] = 0.0f;
            }
        }
        __syncwarp();
        if (lane == 0 && item + kStages < items) issue(item + kStages);
    }

    if (!ok && lane == 0) {
        // a copy never arrived: wait (bounded) for the ones still in flight before leaving
        for (int64_t i = item + 1; i < items && i < item + kStages; ++i)
            mbar_wait(&bar[i % kStages], (uint32_t)((i / kStages) & 1), err, ERR_GEMV_DRAIN, nullptr);
    }
}

template <int FMT, int MT, bool DUMP>
int launch_one(const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, int64_t t0, int mt, float *y,
               const Dump &dump, unsigned int *err, int nsm, cudaStream_t stream) {
    using C = GvCfg<FMT>;
    auto kern = gemv_kernel<FMT, MT, DUMP>;
    constexpr int slot = 16 + FMT * 8 + (MT == 1 ? 0 : MT == 2 ? 1 : MT == 4 ? 2 : 3) * 2 + (DUMP ? 1 : 0);
    int rc = ensure_smem_attr(reinterpret_cast<const void *>(kern), C::SMEM, slot);
    if (rc != MQ_OK) return rc;
    int64_t ctas = (N + kWarps - 1) / kWarps;
    const int64_t cap = (int64_t)nsm * 2;
    if (ctas > cap) ctas = cap;
    kern<<<(unsigned)ctas, kWarps * 32, C::SMEM, stream>>>(w, N, K, p, M, t0, mt, y, dump, err);
    return cuda_error(cudaGetLastError(), "gemv launch");
}

template <int FMT, bool DUMP>
int launch_fmt(const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump,
               unsigned int *err, int nsm, cudaStream_t stream) {
    for (int64_t t0 = 0; t0 < M; t0 += 8) {
        const int mt = (int)((M - t0) < 8 ? (M - t0) : 8);
        int rc;
        if (mt == 1)
            rc = launch_one<FMT, 1, DUMP>(w, N, K, p, M, t0, mt, y, dump, err, nsm, stream);
        else if (mt == 2)
            rc = launch_one<FMT, 2, DUMP>(w, N, K, p, M, t0, mt, y, dump, err, nsm, stream);
        else if (mt <= 4)
            rc = launch_one<FMT, 4, DUMP>(w, N, K, p, M, t0, mt, y, dump, err, nsm, stream);
        else
            rc = launch_one<FMT, 8, DUMP>(w, N, K, p, M, t0, mt, y, dump, err, nsm, stream);
        if (rc != MQ_OK) return rc;
    }
    return MQ_OK;
}

}  // namespace

int launch_gemv(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream) {
    const int nsm = sm_count();
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    if (fmt == FMT_Q4K)
        return dmp ? launch_fmt<FMT_Q4K, true>(w, N, K, p, M, y, dump, err, nsm, stream)
                   : launch_fmt<FMT_Q4K, false>(w, N, K, p, M, y, dump, err, nsm, stream);
    return dmp ? launch_fmt<FMT_Q6K, true>(w, N, K, p, M, y, dump, err, nsm, stream)
               : launch_fmt<FMT_Q6K, false>(w, N, K, p, M, y, dump, err, nsm, stream);
}

}  // namespace mq
