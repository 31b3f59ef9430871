// mq_gemv_kq.cu -- the decode GEMV entry point and its k-quant instantiations (Q4_K, Q5_K,
// Q6_K); the 32-value formats are instantiated in mq_gemv_b32.cu.
#include <cstring>

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

int launch_gemv_grouped(Fmt fmt, int nj, const uint8_t *const *w, const int64_t *N, const Plane *p, float *const *y,
                        int64_t K, int64_t M, unsigned int *err, cudaStream_t stream, const float *const *x) {
    if (nj < 1 || nj > kMaxJobs) return set_error(MQ_ERR_ARG, "grouped GEMV: %d jobs (1 .. %d)", nj, kMaxJobs);
    const int nsm = sm_count();
    GvJobs jobs;
    memset(&jobs, 0, sizeof jobs);
    jobs.n = nj;
    for (int i = 0; i < nj; ++i) {
        jobs.w[i] = w[i];
        jobs.N[i] = N[i];
        jobs.p[i] = p[i];
        jobs.y[i] = y[i];
        jobs.x[i] = x ? x[i] : nullptr;
    }
    GvArgs a{w[0], N[0], K, p[0], M, 0, 0, 0, y[0], Dump{nullptr, 0, 0, 0, 0}, err, jobs.x[0]};
    if (x != nullptr) {
        // the activation is quantized inside the kernel: one token, staged in shared memory
        if (M != 1) return set_error(MQ_ERR_SHAPE, "grouped GEMV from f32 activations: M=%lld must be 1", (long long)M);
        const bool fits = fmt == FMT_Q4K   ? gemv_smem<FMT_Q4K, 1, true>(2, K) <= kSmemMax
                          : fmt == FMT_Q5K ? gemv_smem<FMT_Q5K, 1, true>(2, K) <= kSmemMax
                                           : gemv_smem<FMT_Q6K, 1, true>(2, K) <= kSmemMax;
        if (!fits) return set_error(MQ_ERR_SHAPE, "grouped GEMV from f32 activations: K=%lld too large to stage", (long long)K);
    }
    if (fmt == FMT_Q4K) return launch_group_fmt<FMT_Q4K>(a, jobs, nsm, stream);
    if (fmt == FMT_Q5K) return launch_group_fmt<FMT_Q5K>(a, jobs, nsm, stream);
    if (fmt == FMT_Q6K) return launch_group_fmt<FMT_Q6K>(a, jobs, nsm, stream);
    return set_error(MQ_ERR_ARG, "grouped GEMV: k-quant weights (Q4_K, Q5_K, Q6_K) only");
}

}  // namespace mq
