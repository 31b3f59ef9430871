// mq_abi.cu -- the C ABI (include/mq.h): argument validation, plane layout, per-device
// state, status reporting.  Every check happens on the host before any launch; an
// invalid call launches nothing and returns a negative mq_status.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "mq_device.cuh"
#include "mq_internal.h"

namespace mq {

namespace {
thread_local char g_msg[512] = "";

// One error word per device (module globals are instantiated per device).
__device__ unsigned int g_err_word;

constexpr int kMaxDevices = 64;
struct DevState {
    bool ready = false;
    int status = MQ_OK;
    unsigned int *err = nullptr;
};
DevState g_dev[kMaxDevices];
std::mutex g_dev_mu;

// a bounded wait on a barrier that nothing will ever complete (test hook)
__global__ void forced_timeout_kernel(unsigned int *err, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    mbar_init_fence();
    const uint32_t a = smem_u32(&bar);
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(a, 0)) {
        if (global_timer_ns() - t0 > timeout_ns) {
            atomicOr(err, ERR_TEST_FORCED);
            return;
        }
    }
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// whether the byte ranges [a, a + na) and [b, b + nb) share a byte
bool overlaps(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return na != 0 && nb != 0 && a0 < b0 + nb && b0 < a0 + na;
}

constexpr int64_t kMaxDim = (int64_t)1 << 31;
// the tensor-core GEMMs put their token tiles (128 tokens) in grid.y, the fused gate|up GEMM its
// output tiles (64 rows of gate and of up) there; CUDA caps grid.y at 65535
constexpr int64_t kMaxGemmM = (int64_t)65535 * 128;
constexpr int64_t kMaxSwigluF = (int64_t)65535 * 64;
}  // namespace

int set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return code;
}

namespace {
int g_sm_count[kMaxDevices] = {0};
constexpr int kAttrSlots = kAttrSlotSmall + 16;     // GEMM below 16; GEMV 16 + 16 per format; fused GEMM; small-M GEMM
bool g_attr_done[kMaxDevices][kAttrSlots] = {};
}  // namespace

int sm_count() {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices) return 1;
    if (g_sm_count[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        g_sm_count[dev] = n > 0 ? n : 1;
    }
    return g_sm_count[dev];
}

int ensure_smem_attr(const void *kernel, int bytes, int slot) {
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kAttrSlots)
        return set_error(MQ_ERR_CUDA, "ensure_smem_attr: bad device %d / slot %d", dev, slot);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_attr_done[dev][slot]) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
        if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(max dynamic shared memory)");
        g_attr_done[dev][slot] = true;
    }
    return MQ_OK;
}

int resident_ctas(const void *kernel, int threads, int smem_bytes, int slot, int *out) {
    // per (device, slot): a few (shared-memory size, answer) pairs, replaced round-robin
    constexpr int kWays = 4;
    static int cache_smem[kMaxDevices][kAttrSlots][kWays] = {};
    static int cache_n[kMaxDevices][kAttrSlots][kWays] = {};
    static int cache_next[kMaxDevices][kAttrSlots] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= kMaxDevices || slot < 0 || slot >= kAttrSlots)
        return set_error(MQ_ERR_CUDA, "resident_ctas: bad device %d / slot %d", dev, slot);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    for (int i = 0; i < kWays; ++i)
        if (cache_n[dev][slot][i] > 0 && cache_smem[dev][slot][i] == smem_bytes) {
            *out = cache_n[dev][slot][i];
            return MQ_OK;
        }
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem_bytes);
    if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
    if (n < 1) return set_error(MQ_ERR_CUDA, "kernel in slot %d cannot be resident (%d B shared memory)", slot, smem_bytes);
    const int i = cache_next[dev][slot];
    cache_next[dev][slot] = (i + 1) % kWays;
    cache_smem[dev][slot][i] = smem_bytes;
    cache_n[dev][slot][i] = n;
    *out = n;
    return MQ_OK;
}

int cuda_error(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return MQ_OK;
    return set_error(MQ_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Current device must be compute capability 10.3; resolves its error-word address once.
static int device_state(unsigned int **err) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return set_error(MQ_ERR_DEVICE, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DevState &st = g_dev[dev];
    if (!st.ready) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        if (major != 10 || minor != 3) {
            st.status = set_error(MQ_ERR_DEVICE, "device %d is compute capability %d.%d; this library is built for 10.3 (sm_103a)",
                                  dev, major, minor);
        } else {
            void *ptr = nullptr;
            e = cudaGetSymbolAddress(&ptr, g_err_word);
            if (e != cudaSuccess) {
                st.status = cuda_error(e, "cudaGetSymbolAddress(error word)");
            } else {
                st.err = static_cast<unsigned int *>(ptr);
                st.status = MQ_OK;
            }
        }
        st.ready = true;
    }
    if (st.status != MQ_OK) {
        if (st.status == MQ_ERR_DEVICE) set_error(MQ_ERR_DEVICE, "device %d is not compute capability 10.3 (sm_103a)", dev);
        return st.status;
    }
    *err = st.err;
    return MQ_OK;
}

static int plane_from(void *base, int64_t M, int64_t K, Plane *p) {
    mq_plane_layout L;
    int rc = mq_q8_plane_layout(M, K, &L);
    if (rc != MQ_OK) return rc;
    uint8_t *b = static_cast<uint8_t *>(base);
    p->q16 = reinterpret_cast<uint16_t *>(b + L.off_q16);
    p->q8 = reinterpret_cast<int8_t *>(b + L.off_q8);
    p->d = reinterpret_cast<float *>(b + L.off_d);
    p->s = reinterpret_cast<int32_t *>(b + L.off_s);
    p->ds = reinterpret_cast<float *>(b + L.off_ds);
    return MQ_OK;
}

static int check_k(int64_t K) {
    if (K <= 0 || K % kQK != 0 || K >= kMaxDim)
        return set_error(MQ_ERR_SHAPE, "K=%lld must be a positive multiple of 256 below 2^31", (long long)K);
    return MQ_OK;
}

enum MatmulKind { KIND_GEMV = 0, KIND_GEMM = 1, KIND_SMALL = 2 };

// shared validation of the matmul entry points (bb: weight bytes per 256 values of a row)
static int check_matmul(const char *fn, int kind, int bb, const void *w, int64_t N, int64_t K, const void *plane,
                        int64_t M, const float *y) {
    if (M < 0 || N < 0) return set_error(MQ_ERR_ARG, "%s: negative size M=%lld N=%lld", fn, (long long)M, (long long)N);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    if (M >= kMaxDim || N >= kMaxDim)
        return set_error(MQ_ERR_SHAPE, "%s: M=%lld N=%lld must be below 2^31", fn, (long long)M, (long long)N);
    if (kind == KIND_GEMM && M > kMaxGemmM)
        return set_error(MQ_ERR_SHAPE, "%s: M=%lld exceeds the GEMM limit of %lld tokens", fn, (long long)M,
                         (long long)kMaxGemmM);
    if (kind == KIND_SMALL && M > 32)
        return set_error(MQ_ERR_SHAPE, "%s: M=%lld exceeds the small-M limit of 32 tokens", fn, (long long)M);
    if (M == 0 || N == 0) return MQ_OK;
    if (!w || !plane || !y) return set_error(MQ_ERR_ARG, "%s: NULL pointer (w=%p plane=%p y=%p)", fn, w, plane, (const void *)y);
    if (!aligned(w, 16)) return set_error(MQ_ERR_ALIGN, "%s: weights %p not 16-byte aligned", fn, w);
    if (!aligned(plane, 256)) return set_error(MQ_ERR_ALIGN, "%s: plane %p not 256-byte aligned", fn, plane);
    if (!aligned(y, 4)) return set_error(MQ_ERR_ALIGN, "%s: y %p not 4-byte aligned", fn, (const void *)y);
    const size_t yb = (size_t)M * (size_t)N * 4, wb = (size_t)N * (size_t)(K / kQK) * (size_t)bb;
    if (overlaps(y, yb, plane, mq_q8_plane_bytes(M, K)) || overlaps(y, yb, w, wb))
        return set_error(MQ_ERR_ARG, "%s: output y %p overlaps the plane %p or the weights %p", fn, (const void *)y,
                         plane, w);
    return MQ_OK;
}

constexpr int kMatmulOps = 19;

static int run_matmul(int op, const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y,
                      const Dump &dump, mq_stream_t stream) {
    // the matmul entry points by op number (the debug hook's numbering)
    static const struct {
        const char *name;
        Fmt fmt;
        int kind;
    } ops[kMatmulOps] = {{"mq_gemm_q4k", FMT_Q4K, KIND_GEMM},   {"mq_gemm_q6k", FMT_Q6K, KIND_GEMM},
                         {"mq_gemv_q4k", FMT_Q4K, KIND_GEMV},   {"mq_gemv_q6k", FMT_Q6K, KIND_GEMV},
                         {"mq_gemv_q5k", FMT_Q5K, KIND_GEMV},   {"mq_gemm_q5k", FMT_Q5K, KIND_GEMM},
                         {"mq_gemv_q4_0", FMT_Q4_0, KIND_GEMV}, {"mq_gemv_q4_1", FMT_Q4_1, KIND_GEMV},
                         {"mq_gemv_q5_0", FMT_Q5_0, KIND_GEMV}, {"mq_gemv_q5_1", FMT_Q5_1, KIND_GEMV},
                         {"mq_gemv_q8_0", FMT_Q8_0, KIND_GEMV}, {"mq_gemm_q4_0", FMT_Q4_0, KIND_GEMM},
                         {"mq_gemm_q4_1", FMT_Q4_1, KIND_GEMM}, {"mq_gemm_q5_0", FMT_Q5_0, KIND_GEMM},
                         {"mq_gemm_q5_1", FMT_Q5_1, KIND_GEMM}, {"mq_gemm_q8_0", FMT_Q8_0, KIND_GEMM},
                         {"mq_gemm_small_q4k", FMT_Q4K, KIND_SMALL}, {"mq_gemm_small_q6k", FMT_Q6K, KIND_SMALL},
                         {"mq_gemm_small_q5k", FMT_Q5K, KIND_SMALL}};
    int rc = check_matmul(ops[op].name, ops[op].kind, block_bytes(ops[op].fmt), w, N, K, plane, M, y);
    if (rc != MQ_OK || M == 0 || N == 0) return rc;
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    Plane p;
    plane_from(const_cast<void *>(plane), M, K, &p);
    const uint8_t *wb = static_cast<const uint8_t *>(w);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (ops[op].kind == KIND_GEMM) return launch_gemm(ops[op].fmt, wb, N, K, p, M, y, dump, err, s);
    if (ops[op].kind == KIND_SMALL) return launch_gemm_small(ops[op].fmt, wb, N, K, p, M, y, dump, err, s);
    return launch_gemv(ops[op].fmt, wb, N, K, p, M, y, dump, err, s);
}

}  // namespace mq

using namespace mq;

extern "C" {

const char *mq_last_error(void) { return g_msg; }

int mq_q8_plane_layout(int64_t M, int64_t K, mq_plane_layout *out) {
    if (out == nullptr) return set_error(MQ_ERR_ARG, "mq_q8_plane_layout: NULL output");
    if (M < 0 || M >= kMaxDim) return set_error(MQ_ERR_SHAPE, "M=%lld out of range", (long long)M);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    const size_t m = (size_t)M, k = (size_t)K, nblk = k / kQ8;
    out->off_q16 = 0;
    out->off_q8 = align256(2 * m * k);
    out->off_d = align256(out->off_q8 + m * k);
    out->off_s = align256(out->off_d + 4 * nblk * m);
    out->off_ds = align256(out->off_s + 4 * nblk * m);
    out->total_bytes = align256(out->off_ds + 8 * nblk * m);
    return MQ_OK;
}

size_t mq_q8_plane_bytes(int64_t M, int64_t K) {
    mq_plane_layout L;
    if (M < 0 || M >= kMaxDim || K <= 0 || K % kQK != 0 || K >= kMaxDim) return 0;
    mq_q8_plane_layout(M, K, &L);
    return L.total_bytes;
}

int mq_quantize_q8(const float *x, int64_t M, int64_t K, const float *rms_w, float eps, void *plane,
                   mq_stream_t stream) {
    return mq_quantize_q8_ex(x, M, K, rms_w, eps, MQ_PLANE_ALL, plane, stream);
}

int mq_quantize_q8_ex(const float *x, int64_t M, int64_t K, const float *rms_w, float eps, unsigned sections,
                      void *plane, mq_stream_t stream) {
    if (sections == 0 || sections > MQ_PLANE_ALL)
        return set_error(MQ_ERR_ARG, "mq_quantize_q8: sections=0x%x not a non-empty MQ_PLANE_* mask", sections);
    if (M < 0) return set_error(MQ_ERR_ARG, "mq_quantize_q8: negative M=%lld", (long long)M);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    if (M >= kMaxDim) return set_error(MQ_ERR_SHAPE, "mq_quantize_q8: M=%lld must be below 2^31", (long long)M);
    if (rms_w != nullptr && !(std::isfinite(eps) && eps >= 0.0f))
        return set_error(MQ_ERR_ARG, "mq_quantize_q8: eps=%g must be finite and >= 0", (double)eps);
    if (M == 0) return MQ_OK;
    if (!x || !plane) return set_error(MQ_ERR_ARG, "mq_quantize_q8: NULL pointer (x=%p plane=%p)", (const void *)x, plane);
    if (!aligned(x, 16)) return set_error(MQ_ERR_ALIGN, "mq_quantize_q8: x %p not 16-byte aligned", (const void *)x);
    if (rms_w && !aligned(rms_w, 16))
        return set_error(MQ_ERR_ALIGN, "mq_quantize_q8: rms_w %p not 16-byte aligned", (const void *)rms_w);
    if (!aligned(plane, 256)) return set_error(MQ_ERR_ALIGN, "mq_quantize_q8: plane %p not 256-byte aligned", plane);
    const size_t pb = mq_q8_plane_bytes(M, K);
    if (overlaps(plane, pb, x, (size_t)M * (size_t)K * 4) || (rms_w && overlaps(plane, pb, rms_w, (size_t)K * 4)))
        return set_error(MQ_ERR_ARG, "mq_quantize_q8: plane %p overlaps x %p or rms_w %p", plane, (const void *)x,
                         (const void *)rms_w);
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    Plane p;
    plane_from(plane, M, K, &p);
    return launch_quantize(x, M, K, rms_w, eps, sections, p, err, reinterpret_cast<cudaStream_t>(stream));
}

int mq_quantize_swiglu_q8(const float *gate, const float *up, int64_t M, int64_t K, void *plane, mq_stream_t stream) {
    return mq_quantize_swiglu_q8_ex(gate, up, M, K, MQ_PLANE_ALL, plane, stream);
}

int mq_quantize_swiglu_q8_ex(const float *gate, const float *up, int64_t M, int64_t K, unsigned sections, void *plane,
                             mq_stream_t stream) {
    if (sections == 0 || sections > MQ_PLANE_ALL)
        return set_error(MQ_ERR_ARG, "mq_quantize_swiglu_q8: sections=0x%x not a non-empty MQ_PLANE_* mask", sections);
    if (M < 0) return set_error(MQ_ERR_ARG, "mq_quantize_swiglu_q8: negative M=%lld", (long long)M);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    if (M >= kMaxDim) return set_error(MQ_ERR_SHAPE, "mq_quantize_swiglu_q8: M=%lld must be below 2^31", (long long)M);
    if (M == 0) return MQ_OK;
    if (!gate || !up || !plane)
        return set_error(MQ_ERR_ARG, "mq_quantize_swiglu_q8: NULL pointer (gate=%p up=%p plane=%p)", (const void *)gate,
                         (const void *)up, plane);
    if (!aligned(gate, 16) || !aligned(up, 16))
        return set_error(MQ_ERR_ALIGN, "mq_quantize_swiglu_q8: gate %p / up %p not 16-byte aligned", (const void *)gate,
                         (const void *)up);
    if (!aligned(plane, 256))
        return set_error(MQ_ERR_ALIGN, "mq_quantize_swiglu_q8: plane %p not 256-byte aligned", plane);
    {
        const size_t pb = mq_q8_plane_bytes(M, K), xb = (size_t)M * (size_t)K * 4;
        if (overlaps(plane, pb, gate, xb) || overlaps(plane, pb, up, xb))
            return set_error(MQ_ERR_ARG, "mq_quantize_swiglu_q8: plane %p overlaps gate %p or up %p", plane,
                             (const void *)gate, (const void *)up);
    }
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    Plane p;
    plane_from(plane, M, K, &p);
    return launch_swiglu_quantize(gate, up, M, K, sections, p, reinterpret_cast<cudaStream_t>(stream));
}

int mq_gemm_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(0, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(1, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(2, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(3, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

int mq_gemv_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(4, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

int mq_gemm_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(5, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

int mq_gemv_q4_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(6, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q4_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(7, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q5_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(8, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q5_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(9, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemv_q8_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(10, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

int mq_gemm_q4_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(11, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_q4_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(12, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_q5_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(13, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_q5_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(14, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_q8_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y, mq_stream_t stream) {
    return run_matmul(15, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

// the grouped GEMV: every job validated as a GEMV call, and no output may overlap any input or
// other output of the call
static int run_gemv_grouped(const char *fn, Fmt fmt, const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M,
                            mq_stream_t stream) {
    if (n_jobs < 0 || n_jobs > 8) return set_error(MQ_ERR_ARG, "%s: n_jobs=%d not in 0 .. 8", fn, n_jobs);
    if (n_jobs == 0) return MQ_OK;
    if (jobs == nullptr) return set_error(MQ_ERR_ARG, "%s: NULL job table", fn);
    const uint8_t *w[8];
    int64_t N[8];
    Plane p[8];
    float *y[8];
    int nj = 0;
    const size_t pb = mq_q8_plane_bytes(M, K);
    for (int i = 0; i < n_jobs; ++i) {
        int rc = check_matmul(fn, KIND_GEMV, block_bytes(fmt), jobs[i].w, jobs[i].N, K, jobs[i].plane, M, jobs[i].y);
        if (rc != MQ_OK) return rc;
        if (M == 0) return MQ_OK;
        const size_t yb = (size_t)M * (size_t)jobs[i].N * 4;
        for (int k = 0; k < n_jobs; ++k) {
            if (k == i || jobs[k].N == 0) continue;
            const size_t wb = (size_t)jobs[k].N * (size_t)(K / kQK) * (size_t)block_bytes(fmt);
            if (overlaps(jobs[i].y, yb, jobs[k].w, wb) || overlaps(jobs[i].y, yb, jobs[k].plane, pb) ||
                overlaps(jobs[i].y, yb, jobs[k].y, (size_t)M * (size_t)jobs[k].N * 4))
                return set_error(MQ_ERR_ARG, "%s: output of job %d overlaps an input or output of job %d", fn, i, k);
        }
        if (jobs[i].N == 0) continue;                 // an empty job launches nothing
        w[nj] = static_cast<const uint8_t *>(jobs[i].w);
        N[nj] = jobs[i].N;
        plane_from(const_cast<void *>(jobs[i].plane), M, K, &p[nj]);
        y[nj] = jobs[i].y;
        ++nj;
    }
    if (nj == 0) return MQ_OK;
    unsigned int *err = nullptr;
    int rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    return launch_gemv_grouped(fmt, nj, w, N, p, y, K, M, err, reinterpret_cast<cudaStream_t>(stream));
}

int mq_gemv_grouped_q4k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream) {
    return run_gemv_grouped("mq_gemv_grouped_q4k", FMT_Q4K, jobs, n_jobs, K, M, stream);
}
int mq_gemv_grouped_q5k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream) {
    return run_gemv_grouped("mq_gemv_grouped_q5k", FMT_Q5K, jobs, n_jobs, K, M, stream);
}
int mq_gemv_grouped_q6k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream) {
    return run_gemv_grouped("mq_gemv_grouped_q6k", FMT_Q6K, jobs, n_jobs, K, M, stream);
}

// the grouped GEMV from f32 activations (M = 1): every job validated as a GEMV call with x in place of
// the plane, and no output may overlap any input or other output of the call
static int run_gemv_grouped_x(const char *fn, Fmt fmt, const mq_gemv_xjob *jobs, int n_jobs, int64_t K,
                              mq_stream_t stream) {
    if (n_jobs < 0 || n_jobs > 8) return set_error(MQ_ERR_ARG, "%s: n_jobs=%d not in 0 .. 8", fn, n_jobs);
    if (n_jobs == 0) return MQ_OK;
    if (jobs == nullptr) return set_error(MQ_ERR_ARG, "%s: NULL job table", fn);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    const uint8_t *w[8];
    int64_t N[8];
    Plane p[8];
    float *y[8];
    const float *x[8];
    int nj = 0;
    for (int i = 0; i < n_jobs; ++i) {
        const mq_gemv_xjob &j = jobs[i];
        if (j.N < 0) return set_error(MQ_ERR_ARG, "%s: job %d: negative N=%lld", fn, i, (long long)j.N);
        if (j.N >= kMaxDim) return set_error(MQ_ERR_SHAPE, "%s: job %d: N=%lld must be below 2^31", fn, i, (long long)j.N);
        if (j.N == 0) continue;                      // an empty job launches nothing
        if (!j.w || !j.x || !j.y)
            return set_error(MQ_ERR_ARG, "%s: job %d: NULL pointer (w=%p x=%p y=%p)", fn, i, j.w, (const void *)j.x,
                             (const void *)j.y);
        if (!aligned(j.w, 16)) return set_error(MQ_ERR_ALIGN, "%s: job %d: weights %p not 16-byte aligned", fn, i, j.w);
        if (!aligned(j.x, 16)) return set_error(MQ_ERR_ALIGN, "%s: job %d: x %p not 16-byte aligned", fn, i, (const void *)j.x);
        if (!aligned(j.y, 4)) return set_error(MQ_ERR_ALIGN, "%s: job %d: y %p not 4-byte aligned", fn, i, (const void *)j.y);
        const size_t yb = (size_t)j.N * 4;
        for (int k = 0; k < n_jobs; ++k) {
            if (jobs[k].N <= 0) continue;
            const size_t wb = (size_t)jobs[k].N * (size_t)(K / kQK) * (size_t)block_bytes(fmt);
            if (overlaps(j.y, yb, jobs[k].w, wb) || overlaps(j.y, yb, jobs[k].x, (size_t)K * 4) ||
                (k != i && overlaps(j.y, yb, jobs[k].y, (size_t)jobs[k].N * 4)))
                return set_error(MQ_ERR_ARG, "%s: output of job %d overlaps an input or output of job %d", fn, i, k);
        }
        w[nj] = static_cast<const uint8_t *>(j.w);
        N[nj] = j.N;
        memset(&p[nj], 0, sizeof p[nj]);
        y[nj] = j.y;
        x[nj] = j.x;
        ++nj;
    }
    if (nj == 0) return MQ_OK;
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    return launch_gemv_grouped(fmt, nj, w, N, p, y, K, 1, err, reinterpret_cast<cudaStream_t>(stream), x);
}

int mq_gemv_grouped_x_q4k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream) {
    return run_gemv_grouped_x("mq_gemv_grouped_x_q4k", FMT_Q4K, jobs, n_jobs, K, stream);
}
int mq_gemv_grouped_x_q5k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream) {
    return run_gemv_grouped_x("mq_gemv_grouped_x_q5k", FMT_Q5K, jobs, n_jobs, K, stream);
}
int mq_gemv_grouped_x_q6k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream) {
    return run_gemv_grouped_x("mq_gemv_grouped_x_q6k", FMT_Q6K, jobs, n_jobs, K, stream);
}

int mq_quantize_q8_grouped(const mq_quantize_job *jobs, int n_jobs, int64_t M, int64_t K, unsigned sections,
                           mq_stream_t stream) {
    const char *fn = "mq_quantize_q8_grouped";
    if (n_jobs < 0 || n_jobs > 8) return set_error(MQ_ERR_ARG, "%s: n_jobs=%d not in 0 .. 8", fn, n_jobs);
    if (sections == 0 || sections > MQ_PLANE_ALL)
        return set_error(MQ_ERR_ARG, "%s: sections=0x%x not a non-empty MQ_PLANE_* mask", fn, sections);
    if (M < 0) return set_error(MQ_ERR_ARG, "%s: negative M=%lld", fn, (long long)M);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    if (M >= kMaxDim) return set_error(MQ_ERR_SHAPE, "%s: M=%lld must be below 2^31", fn, (long long)M);
    if (n_jobs == 0 || M == 0) return MQ_OK;
    if (jobs == nullptr) return set_error(MQ_ERR_ARG, "%s: NULL job table", fn);
    const size_t pb = mq_q8_plane_bytes(M, K), xb = (size_t)M * (size_t)K * 4;
    const float *x[8];
    Plane p[8];
    for (int i = 0; i < n_jobs; ++i) {
        if (!jobs[i].x || !jobs[i].plane)
            return set_error(MQ_ERR_ARG, "%s: NULL pointer in job %d", fn, i);
        if (!aligned(jobs[i].x, 16) || !aligned(jobs[i].plane, 256))
            return set_error(MQ_ERR_ALIGN, "%s: job %d: x needs 16-byte, the plane 256-byte alignment", fn, i);
        for (int k = 0; k < n_jobs; ++k)
            if (overlaps(jobs[i].plane, pb, jobs[k].x, xb) || (k != i && overlaps(jobs[i].plane, pb, jobs[k].plane, pb)))
                return set_error(MQ_ERR_ARG, "%s: the plane of job %d overlaps an input or plane of job %d", fn, i, k);
        x[i] = jobs[i].x;
        plane_from(jobs[i].plane, M, K, &p[i]);
    }
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    return launch_quantize_grouped(n_jobs, x, p, M, K, sections, reinterpret_cast<cudaStream_t>(stream));
}

int mq_gemm_small_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y,
                      mq_stream_t stream) {
    return run_matmul(16, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_small_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y,
                      mq_stream_t stream) {
    return run_matmul(17, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}
int mq_gemm_small_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y,
                      mq_stream_t stream) {
    return run_matmul(18, w, N, K, plane, M, y, Dump{nullptr, 0, 0, 0, 0}, stream);
}

int mq_gemm_q4k_swiglu(const void *w_gate, const void *w_up, int64_t F, int64_t K, const void *plane_in, int64_t M,
                       void *plane_out, mq_stream_t stream) {
    const char *fn = "mq_gemm_q4k_swiglu";
    if (M < 0 || F < 0) return set_error(MQ_ERR_ARG, "%s: negative size M=%lld F=%lld", fn, (long long)M, (long long)F);
    int rc = check_k(K);
    if (rc != MQ_OK) return rc;
    if (F % kQK != 0 || F > kMaxSwigluF)
        return set_error(MQ_ERR_SHAPE, "%s: F=%lld must be a multiple of 256 of at most %lld", fn, (long long)F,
                         (long long)kMaxSwigluF);
    if (M >= kMaxDim) return set_error(MQ_ERR_SHAPE, "%s: M=%lld must be below 2^31", fn, (long long)M);
    if (M == 0 || F == 0) return MQ_OK;
    if (!w_gate || !w_up || !plane_in || !plane_out)
        return set_error(MQ_ERR_ARG, "%s: NULL pointer (w_gate=%p w_up=%p plane_in=%p plane_out=%p)", fn, w_gate, w_up,
                         plane_in, plane_out);
    if (!aligned(w_gate, 16) || !aligned(w_up, 16))
        return set_error(MQ_ERR_ALIGN, "%s: weights %p / %p not 16-byte aligned", fn, w_gate, w_up);
    if (!aligned(plane_in, 256) || !aligned(plane_out, 256))
        return set_error(MQ_ERR_ALIGN, "%s: planes %p / %p not 256-byte aligned", fn, plane_in, plane_out);
    {
        // the output plane is written while the input plane is read: they must not overlap
        const uintptr_t i0 = reinterpret_cast<uintptr_t>(plane_in), o0 = reinterpret_cast<uintptr_t>(plane_out);
        const uintptr_t i1 = i0 + mq_q8_plane_bytes(M, K), o1 = o0 + mq_q8_plane_bytes(M, F);
        if (i0 < o1 && o0 < i1)
            return set_error(MQ_ERR_ARG, "%s: plane_out %p overlaps plane_in %p", fn, plane_out, plane_in);
        const size_t wb = (size_t)F * (size_t)(K / kQK) * (size_t)block_bytes(FMT_Q4K), ob = o1 - o0;
        if (overlaps(plane_out, ob, w_gate, wb) || overlaps(plane_out, ob, w_up, wb))
            return set_error(MQ_ERR_ARG, "%s: plane_out %p overlaps the weights %p / %p", fn, plane_out, w_gate, w_up);
    }
    unsigned int *err = nullptr;
    rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    Plane pi, po;
    plane_from(const_cast<void *>(plane_in), M, K, &pi);
    plane_from(plane_out, M, F, &po);
    return launch_gemm_swiglu(FMT_Q4K, static_cast<const uint8_t *>(w_gate), static_cast<const uint8_t *>(w_up), F, K,
                              pi, M, po, err, reinterpret_cast<cudaStream_t>(stream));
}

int mq_debug_blockdots(int op, const void *w, int64_t N, int64_t K, const void *plane, int64_t M, float *y,
                       int64_t m0, int64_t m_cnt, int64_t n0, int64_t n_cnt, int32_t *I_out, mq_stream_t stream) {
    if (op < 0 || op >= kMatmulOps)
        return set_error(MQ_ERR_ARG, "mq_debug_blockdots: op=%d not in 0..%d", op, kMatmulOps - 1);
    if (m_cnt <= 0 || n_cnt <= 0 || m0 < 0 || n0 < 0 || m0 + m_cnt > M || n0 + n_cnt > N)
        return set_error(MQ_ERR_ARG, "mq_debug_blockdots: window [%lld,+%lld) x [%lld,+%lld) outside %lld x %lld",
                         (long long)m0, (long long)m_cnt, (long long)n0, (long long)n_cnt, (long long)M, (long long)N);
    if (!I_out || !aligned(I_out, 4)) return set_error(MQ_ERR_ARG, "mq_debug_blockdots: bad I_out %p", (void *)I_out);
    return run_matmul(op, w, N, K, plane, M, y, Dump{I_out, m0, m_cnt, n0, n_cnt}, stream);
}

int mq_device_status(mq_stream_t stream) {
    unsigned int *errp = nullptr;
    int rc = device_state(&errp);
    if (rc != MQ_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_error(e, "mq_device_status: stream synchronize");
    unsigned int v = 0;
    e = cudaMemcpy(&v, errp, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_error(e, "mq_device_status: read error word");
    if (v == 0) return MQ_OK;
    const unsigned int zero = 0;
    e = cudaMemcpy(errp, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_error(e, "mq_device_status: clear error word");
    static const char *names[] = {"gemv stage", "gemm A stage", "gemm B stage", "gemm stage release",
                                  "gemm raw weights", "gemm accumulator", "gemm accumulator release",
                                  "gemm row factors", "gemm row factor release", "gemv drain", "gemm min term",
                                  "gemm activation scales"};
    static_assert(sizeof names / sizeof names[0] == 12 && (ERR_GEMM_DA >> 11) == 1u,
                  "one name per device error bit ERR_GEMV_FULL .. ERR_GEMM_DA");
    char buf[400] = "";
    for (int i = 0; i < (int)(sizeof names / sizeof names[0]); ++i)
        if (v & (1u << i)) {
            strncat(buf, " ", sizeof buf - strlen(buf) - 1);
            strncat(buf, names[i], sizeof buf - strlen(buf) - 1);
        }
    if (v & ERR_TEST_FORCED) strncat(buf, " forced-test-wait", sizeof buf - strlen(buf) - 1);
    return set_error(MQ_ERR_DEVICE_TIMEOUT, "bounded device wait ran out (code 0x%x):%s", v, buf);
}

// Test hook: a kernel whose only wait can never complete; it must give up after
// timeout_us and report through mq_device_status().
int mq_debug_forced_timeout(uint32_t timeout_us, mq_stream_t stream) {
    if (timeout_us == 0 || timeout_us > 1000000)
        return set_error(MQ_ERR_ARG, "mq_debug_forced_timeout: timeout_us=%u not in 1..1000000", timeout_us);
    unsigned int *err = nullptr;
    int rc = device_state(&err);
    if (rc != MQ_OK) return rc;
    forced_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, (uint64_t)timeout_us * 1000ull);
    return cuda_error(cudaGetLastError(), "forced timeout launch");
}

}  // extern "C"
