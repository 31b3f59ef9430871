// mq_gemm_kq.cu -- the prefill GEMM entry point (tensor maps, format dispatch) and its k-quant
// instantiations (Q4_K, Q5_K, Q6_K); the 32-value formats are instantiated in mq_gemm_b32.cu.
#include "mq_gemm.cuh"

namespace mq {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

}  // namespace

void *tensor_map_encoder() { return reinterpret_cast<void *>(encode_tiled_fn()); }

// the activation maps: f16 codes [M][K] in 64 x 128 boxes (128-byte swizzle) and the d*S tf32
// pairs [M][2*K/32] f32, one 16-value x 128-token box per super-block (64-byte swizzle)
static int encode_act_maps(EncodeTiledFn enc, const Plane &p, int64_t M, int64_t K, CUtensorMap *tm,
                           CUtensorMap *tmds) {
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {BK, BM};
    const CUresult r = enc(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, p.q16, dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for M=%lld K=%lld", (int)r,
                                            (long long)M, (long long)K);
    const cuuint64_t dims2[2] = {(cuuint64_t)(2 * (K / kQ8)), (cuuint64_t)M};
    const cuuint64_t strides2[1] = {(cuuint64_t)(2 * (K / kQ8)) * 4};
    const cuuint32_t box2[2] = {16, BM};
    const CUresult r2 = enc(tmds, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, p.ds, dims2, strides2, box2, estr,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r2 != CUDA_SUCCESS)
        return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled (d*S) failed (%d) for M=%lld K=%lld", (int)r2,
                         (long long)M, (long long)K);
    return MQ_OK;
}

// raw weights of every format but Q6_K: [N][K/256 * bb] bytes, one bb-byte x `rows` box per
// 256 values (bb = 144 .. 272: a multiple of 16 bytes, so every box starts 16-byte aligned);
// the 32-value formats use 2-byte elements, which keeps Q8_0's 272 bytes within the
// 256-element box limit
static int encode_weight_map(EncodeTiledFn enc, Fmt fmt, const uint8_t *w, int64_t N, int64_t K, uint32_t rows,
                             CUtensorMap *tmw) {
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t el = is_b32(fmt) ? 2 : 1;
    const cuuint64_t bb = (cuuint64_t)block_bytes(fmt);
    const cuuint64_t dims3[2] = {(cuuint64_t)(K / kQK) * bb / el, (cuuint64_t)N};
    const cuuint64_t strides3[1] = {(cuuint64_t)(K / kQK) * bb};
    const cuuint32_t box3[2] = {(cuuint32_t)(bb / el), rows};
    const CUresult r3 = enc(tmw, el == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                            const_cast<uint8_t *>(w), dims3, strides3, box3, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r3 != CUDA_SUCCESS)
        return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled (weights) failed (%d) for N=%lld K=%lld", (int)r3,
                         (long long)N, (long long)K);
    return MQ_OK;
}

int launch_gemm(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    if ((M + BM - 1) / BM > 65535) return set_error(MQ_ERR_SHAPE, "M=%lld: more than 65535 token tiles", (long long)M);
    CUtensorMap tm, tmds, tmw;
    int rc = encode_act_maps(enc, p, M, K, &tm, &tmds);
    if (rc != MQ_OK) return rc;
    memset(&tmw, 0, sizeof tmw);
    if (fmt != FMT_Q6K) {
        rc = encode_weight_map(enc, fmt, w, N, K, BN, &tmw);
        if (rc != MQ_OK) return rc;
    }
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    if (fmt == FMT_Q4K)
        return dmp ? launch_fmt<FMT_Q4K, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q4K, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    if (fmt == FMT_Q5K)
        return dmp ? launch_fmt<FMT_Q5K, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q5K, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    if (is_b32(fmt)) return launch_gemm_b32(fmt, tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    return dmp ? launch_fmt<FMT_Q6K, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
               : launch_fmt<FMT_Q6K, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
}

int launch_gemm_swiglu(Fmt fmt, const uint8_t *wg, const uint8_t *wu, int64_t F, int64_t K, const Plane &p, int64_t M,
                       const Plane &po, unsigned int *err, cudaStream_t stream) {
    EncodeTiledFn enc = encode_tiled_fn();
    if (enc == nullptr) return set_error(MQ_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
    if (fmt != FMT_Q4K) return set_error(MQ_ERR_ARG, "fused gate|up GEMM: Q4_K weights only");
    if ((F + BN / 2 - 1) / (BN / 2) > 65535)
        return set_error(MQ_ERR_SHAPE, "F=%lld: more than 65535 weight tiles", (long long)F);
    CUtensorMap tm, tmds, tmg, tmu;
    int rc = encode_act_maps(enc, p, M, K, &tm, &tmds);
    if (rc == MQ_OK) rc = encode_weight_map(enc, fmt, wg, F, K, BN / 2, &tmg);
    if (rc == MQ_OK) rc = encode_weight_map(enc, fmt, wu, F, K, BN / 2, &tmu);
    if (rc != MQ_OK) return rc;
    return launch_swiglu_fmt<FMT_Q4K>(tm, tmds, tmg, tmu, wg, F, K, p, M, po, err, stream);
}

}  // namespace mq
