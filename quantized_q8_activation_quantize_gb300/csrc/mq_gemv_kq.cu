// mq_gemv_kq.cu -- the decode GEMV entry point and its k-quant instantiations (Q4_K, Q5_K,
// Q6_K); the 32-value formats are instantiated in mq_gemv_b32.cu.
#include "mq_gemv.cuh"

namespace mq {

int launch_gemv(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream) {
    if (is_b32(fmt)) return launch_gemv_b32(fmt, w, N, K, p, M, y, dump, err, stream);
    const int nsm = sm_count();
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    GvArgs a{w, N, K, p, M, 0, 0, 0, y, dump, err};
    if (fmt == FMT_Q4K)
        return dmp ? launch_fmt<FMT_Q4K, true>(a, nsm, stream) : launch_fmt<FMT_Q4K, false>(a, nsm, stream);
    if (fmt == FMT_Q5K)
        return dmp ? launch_fmt<FMT_Q5K, true>(a, nsm, stream) : launch_fmt<FMT_Q5K, false>(a, nsm, stream);
    return dmp ? launch_fmt<FMT_Q6K, true>(a, nsm, stream) : launch_fmt<FMT_Q6K, false>(a, nsm, stream);
}

}  // namespace mq
