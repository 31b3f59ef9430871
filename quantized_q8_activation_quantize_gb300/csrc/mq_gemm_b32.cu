// mq_gemm_b32.cu -- prefill GEMM instantiations for the 32-value block formats (Q4_0, Q4_1,
// Q5_0, Q5_1, Q8_0); reached through launch_gemm (mq_gemm_kq.cu).
#include "mq_gemm.cuh"

namespace mq {

int launch_gemm_b32(Fmt fmt, const CUtensorMap &tm, const CUtensorMap &tmds, const CUtensorMap &tmw,
                    const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y, const Dump &dump,
                    unsigned int *err, cudaStream_t stream) {
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    if (fmt == FMT_Q4_0)
        return dmp ? launch_fmt<FMT_Q4_0, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q4_0, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    if (fmt == FMT_Q4_1)
        return dmp ? launch_fmt<FMT_Q4_1, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q4_1, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    if (fmt == FMT_Q5_0)
        return dmp ? launch_fmt<FMT_Q5_0, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q5_0, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    if (fmt == FMT_Q5_1)
        return dmp ? launch_fmt<FMT_Q5_1, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
                   : launch_fmt<FMT_Q5_1, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
    return dmp ? launch_fmt<FMT_Q8_0, true>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream)
               : launch_fmt<FMT_Q8_0, false>(tm, tmds, tmw, w, N, K, p, M, y, dump, err, stream);
}

}  // namespace mq
