// mq_gemv.cu -- decode GEMV (MMVQ): raw Q4_K / Q6_K weight bytes x Q8 codes with dp4a.
//
// minfer pages, "Support Matrix > CUDA notes": decode (nt == 1) uses the dp4a MMVQ
// kernels; "Roadmap > 0": the decode path streams the weights once per token.
//
// Design (HBM-bound): every weight byte is read from HBM exactly once per group of up
// to 8 tokens.  Each warp owns a private 3-stage ring in shared memory and walks its
// rows in chunks of up to 8 super-blocks; lane 0 refills a stage with one 1-D bulk
// async copy (TMA engine) of the 16-byte-aligned superset of the chunk's bytes, so a
// Q6_K block (210 B, only 2-byte aligned) needs no special load path from HBM.  Four
// 8-warp CTAs per SM keep ~160 KB in flight.  The math runs from shared memory: 4 lanes
// per super-block, each owning 64 of its 256 values (so scale decoding and the float
// work of a block amortize over 64 values), dp4a against the int8 codes (read through
// L1), f32 scaling per 32-value block, one warp reduction per row.
#include <cuda_fp16.h>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {
namespace {

constexpr int kWarps = 8;
constexpr int kStages = 3;
constexpr int kChunkBlocks = 8;        // super-blocks per staged chunk: 32 lanes x 64 values
constexpr unsigned kFull = 0xffffffffu;

template <int FMT>
struct GvCfg {
    static constexpr int BB = FMT == FMT_Q4K ? 144 : 210;
    // superset of an 8-block chunk + up to 15 leading bytes + 16 bytes of over-read slack
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
__device__ __forceinline__ int dot16(const uint4 &w, const uint4 &a) {
    return __dp4a((int)w.w, (int)a.w, __dp4a((int)w.z, (int)a.z, __dp4a((int)w.y, (int)a.y, __dp4a((int)w.x, (int)a.x, 0))));
}

// Each warp owns a kStages ring in shared memory and walks its rows in chunks of up to 8
// super-blocks (one bulk copy of the chunk's 16-byte aligned superset per stage).  Lane l
// takes super-block l/4 of the chunk and a 64-value quarter u = l%4 of it.
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

    const int nb = (int)(K / kQK);                      // super-blocks per row
    const int nch = (nb + kChunkBlocks - 1) / kChunkBlocks;
    const int64_t row_bytes = (int64_t)nb * C::BB;
    const int64_t nblk32 = K / kQ8;
    const int64_t gw = (int64_t)blockIdx.x * kWarps + warp, GW = (int64_t)gridDim.x * kWarps;
    const int nrows = gw < N ? (int)((N - gw + GW - 1) / GW) : 0;
    const int items = nrows * nch;

    // items run row-major over (row r of this warp, chunk c); positions advance incrementally
    auto chunk_bytes = [&](int r, int c, int64_t &start, int &nblk) {
        const int64_t n = gw + (int64_t)r * GW;
        start = n * row_bytes + (int64_t)c * (kChunkBlocks * C::BB);
        nblk = min(kChunkBlocks, nb - c * kChunkBlocks);
    };
    int ri = 0, ci = 0, si = 0;                         // next item to issue, and its stage
    auto issue = [&]() {
        int64_t start;
        int nblk;
        chunk_bytes(ri, ci, start, nblk);
        const int64_t a0 = start & ~(int64_t)15, a1 = (start + nblk * C::BB + 15) & ~(int64_t)15;
        mbar_arrive_expect_tx(&bar[si], (uint32_t)(a1 - a0));
        bulk_copy_g2s(ring + si * C::STAGE, w + a0, (uint32_t)(a1 - a0), &bar[si]);
        if (++ci == nch) { ci = 0; ++ri; }
        if (++si == kStages) si = 0;
    };

    if (lane == 0)
        for (int i = 0; i < items && i < kStages; ++i) issue();

    float acc[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t] = 0.0f;

    const int u = lane & 3;          // the 64-value quarter of the super-block this lane owns
    const int lb = lane >> 2;        // the super-block of the chunk this lane owns
    bool ok = true;
    int item = 0, r = 0, c = 0, s = 0;
    uint32_t phase = 0;
    for (; item < items; ++item) {
        const bool got = mbar_wait(&bar[s], phase, err, ERR_GEMV_FULL, nullptr);
        if (!__all_sync(kFull, got)) {   // leave the loop together (shuffles below need every lane)
            ok = false;
            break;
        }
        int64_t start;
        int nblk_c;
        chunk_bytes(r, c, start, nblk_c);
        const int64_t n = gw + (int64_t)r * GW;
        const bool valid = lb < nblk_c;                  // uniform over the 4 lanes of a block
        const int64_t sbi = c * kChunkBlocks + lb;       // super-block index in the row
        const uint32_t blk = ring_s + s * C::STAGE + (uint32_t)(start & 15) + (uint32_t)(lb * C::BB);
        if constexpr (FMT == FMT_Q4K) {
            // quarter u: qs bytes [32u, 32u+32): low nibbles -> sub-block j0 = 2u, high -> j1 = 2u+1
            uint4 hd = make_uint4(0, 0, 0, 0), q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
            if (valid) {
                hd = lds128(blk);
                q0 = lds128(blk + 16 + 32 * u);
                q1 = lds128(blk + 32 + 32 * u);
            }
            const float d = half_bits_to_float(hd.x & 0xffff), dmin = half_bits_to_float(hd.x >> 16);
            // the 12 scale bytes: s[0..3] = hd.y, s[4..7] = hd.z, s[8..11] = hd.w; sub-blocks 2u, 2u+1
            int sc0, m0, sc1, m1;
            if (u < 2) {
                const uint32_t a = hd.y >> (16 * u), b = hd.z >> (16 * u);
                sc0 = a & 63; sc1 = (a >> 8) & 63; m0 = b & 63; m1 = (b >> 8) & 63;
            } else {
                const uint32_t lo = hd.w >> (16 * (u - 2));                  // s[j+4] for j = 2u, 2u+1
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
            const int64_t k0 = sbi * kQK + 64 * u;             // values 64u .. 64u+63 of the super-block
            const int64_t b0 = sbi * 8 + 2 * u, b1 = b0 + 1;   // their two Q8 blocks
            const float dsc0 = d * (float)sc0, dsc1 = d * (float)sc1, dm0 = dmin * (float)m0, dm1 = dmin * (float)m1;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int64_t m = t0 + t;
                const bool act = t < mt && valid;
                int D0 = 0, D1 = 0;
                if (act) {
                    const uint4 *a = reinterpret_cast<const uint4 *>(p.q8 + m * K + k0);
                    D0 = dot16(lo0, __ldg(a)) + dot16(lo1, __ldg(a + 1));
                    D1 = dot16(hi0, __ldg(a + 2)) + dot16(hi1, __ldg(a + 3));
                    const float da0 = __ldg(p.d + b0 * M + m), da1 = __ldg(p.d + b1 * M + m);
                    const float s0 = (float)__ldg(p.s + b0 * M + m), s1 = (float)__ldg(p.s + b1 * M + m);
                    acc[t] += da0 * (dsc0 * (float)D0 - dm0 * s0) + da1 * (dsc1 * (float)D1 - dm1 * s1);
                }
                if constexpr (DUMP) {
                    if (act && m >= dump.m0 && m < dump.m0 + dump.m_cnt && n >= dump.n0 && n < dump.n0 + dump.n_cnt) {
                        int32_t *o = dump.out + ((m - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32;
                        o[b0] = sc0 * D0;
                        o[b1] = sc1 * D1;
                    }
                }
            }
        } else {
            // quarter u: half h = u/2, l0 = 16*(u%2); values 128h + 32g + l0 + i (g = 0..3, i = 0..15).
            // group g: low (g < 2) / high (g >= 2) nibble of ql[64h + 32(g&1) + l0 + i], high bits
            // (qh[32h + l0 + i] >> 2g) & 3; each group is one 16-value sub-block 8h + 2g + u%2.
            const int h = u >> 1, l0 = 16 * (u & 1);
            uint4 ql0 = make_uint4(0, 0, 0, 0), ql1 = make_uint4(0, 0, 0, 0), qh = make_uint4(0, 0, 0, 0);
            float d = 0.0f;
            uint32_t scw = 0, scw2 = 0;
            if (valid) {
                ql0 = lds128_a2(blk + 64 * h + l0);
                ql1 = lds128_a2(blk + 64 * h + 32 + l0);
                qh = lds128_a2(blk + 128 + 32 * h + l0);
                d = half_bits_to_float(lds16(blk + 208));
                // scales 8h + (u&1) + {0, 2, 4, 6}: the 8 bytes at 192 + 8h, even or odd ones
                const uint32_t sa = (lds16(blk + 192 + 8 * h) | (lds16(blk + 194 + 8 * h) << 16));
                const uint32_t sb2 = (lds16(blk + 196 + 8 * h) | (lds16(blk + 198 + 8 * h) << 16));
                const uint32_t sel = (u & 1) ? 0x7531u : 0x6420u;
                scw = __byte_perm(sa, sb2, sel);                // 4 int8 scales of groups 0..3
                scw2 = 0;
            }
            (void)scw2;
            // 6-bit codes (q + 32) of the four groups
            uint4 v[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const uint32_t *L = reinterpret_cast<const uint32_t *>((g & 1) ? &ql1 : &ql0);
                const uint32_t *H = reinterpret_cast<const uint32_t *>(&qh);
                uint32_t o[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t lo = (g < 2) ? L[e] : (L[e] >> 4);
                    const uint32_t hb = (g == 0) ? (H[e] << 4) : (g == 1) ? (H[e] << 2) : (g == 2) ? H[e] : (H[e] >> 2);
                    o[e] = lop3_and_or(lo, 0x0f0f0f0fu, hb, 0x30303030u);
                }
                v[g] = make_uint4(o[0], o[1], o[2], o[3]);
            }
            const int64_t kb = sbi * kQK + 128 * h + l0;
            const int64_t bq = sbi * 8 + 4 * h;                // Q8 block of group 0
            float dsc[4];
#pragma unroll
            for (int g = 0; g < 4; ++g) dsc[g] = d * (float)(int8_t)((scw >> (8 * g)) & 0xff);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int64_t m = t0 + t;
                const bool act = t < mt && valid;
                int Dg[4] = {0, 0, 0, 0};
                if (act) {
                    const int8_t *a = p.q8 + m * K + kb;
                    float vsum = 0.0f;
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        const uint4 av = __ldg(reinterpret_cast<const uint4 *>(a + 32 * g));
                        // sum (code - 32) a = sum code*a - 32 sum a
                        Dg[g] = dot16(v[g], av) - dot16(make_uint4(0x20202020u, 0x20202020u, 0x20202020u, 0x20202020u), av);
                        vsum += dsc[g] * (float)Dg[g] * __ldg(p.d + (bq + g) * M + m);
                    }
                    acc[t] += vsum;
                }
                if constexpr (DUMP) {
                    int I[4];
#pragma unroll
                    for (int g = 0; g < 4; ++g) {
                        I[g] = (int)(int8_t)((scw >> (8 * g)) & 0xff) * Dg[g];
                        I[g] += __shfl_xor_sync(kFull, I[g], 1);       // the two 16-value halves of the Q8 block
                    }
                    if (act && (u & 1) == 0 && m >= dump.m0 && m < dump.m0 + dump.m_cnt && n >= dump.n0 &&
                        n < dump.n0 + dump.n_cnt) {
                        int32_t *o = dump.out + ((m - dump.m0) * dump.n_cnt + (n - dump.n0)) * nblk32;
#pragma unroll
                        for (int g = 0; g < 4; ++g) o[bq + g] = I[g];
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
        if (lane == 0 && item + kStages < items) issue();
        if (++c == nch) { c = 0; ++r; }
        if (++s == kStages) { s = 0; phase ^= 1u; }
    }

    if (!ok && lane == 0) {
        // a copy never arrived: wait (bounded) for the ones still in flight before leaving
        for (int i = item + 1; i < items && i < item + kStages; ++i)
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
    const int64_t cap = (int64_t)nsm * 4;    // four 8-warp CTAs per SM (registers; 41.5 KB of stages each)
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
