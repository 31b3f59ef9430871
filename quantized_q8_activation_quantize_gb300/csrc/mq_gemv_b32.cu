// mq_gemv_b32.cu -- decode GEMV instantiations for the 32-value block formats (Q4_0, Q4_1,
// Q5_0, Q5_1, Q8_0); reached through launch_gemv (mq_gemv_kq.cu).
#include "mq_gemv.cuh"

namespace mq {

int launch_gemv_b32(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                    const Dump &dump, unsigned int *err, cudaStream_t stream) {
    const int nsm = sm_count();
    const bool dmp = dump.m_cnt > 0 && dump.n_cnt > 0;
    GvArgs a{w, N, K, p, M, 0, 0, 0, y, dump, err};
    if (fmt == FMT_Q4_0)
        return dmp ? launch_fmt<FMT_Q4_0, true>(a, nsm, stream) : launch_fmt<FMT_Q4_0, false>(a, nsm, stream);
    if (fmt == FMT_Q4_1)
        return dmp ? launch_fmt<FMT_Q4_1, true>(a, nsm, stream) : launch_fmt<FMT_Q4_1, false>(a, nsm, stream);
    if (fmt == FMT_Q5_0)
        return dmp ? launch_fmt<FMT_Q5_0, true>(a, nsm, stream) : launch_fmt<FMT_Q5_0, false>(a, nsm, stream);
    if (fmt == FMT_Q5_1)
        return dmp ? launch_fmt<FMT_Q5_1, true>(a, nsm, stream) : launch_fmt<FMT_Q5_1, false>(a, nsm, stream);
    return dmp ? launch_fmt<FMT_Q8_0, true>(a, nsm, stream) : launch_fmt<FMT_Q8_0, false>(a, nsm, stream);
}

}  // namespace mq
