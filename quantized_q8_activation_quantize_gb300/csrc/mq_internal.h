// mq_internal.h -- host-side declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/mq.h"

namespace mq {

// weight formats: the 256-value k-quants, then the 32-value block formats
enum Fmt : int { FMT_Q4K = 0, FMT_Q6K = 1, FMT_Q5K = 2, FMT_Q4_0 = 3, FMT_Q4_1 = 4, FMT_Q5_0 = 5, FMT_Q5_1 = 6, FMT_Q8_0 = 7 };

constexpr int kQK = 256;     // values per k-quant super-block
constexpr int kQ8 = 32;      // values per Q8 activation block

constexpr bool is_b32(int f) { return f >= FMT_Q4_0; }
// 32-value formats: bytes of one block (fp16 d [, fp16 m] [, 32-bit qh] then the quants),
// whether it has the offset m, whether it has the fifth bit, and the offset its unsigned
// quants carry (value = d * (q - off) [+ m])
constexpr int b32_bytes(int f) { return f == FMT_Q4_0 ? 18 : f == FMT_Q4_1 ? 20 : f == FMT_Q5_0 ? 22 : f == FMT_Q5_1 ? 24 : 34; }
constexpr bool b32_has_m(int f) { return f == FMT_Q4_1 || f == FMT_Q5_1; }
constexpr bool b32_five(int f) { return f == FMT_Q5_0 || f == FMT_Q5_1; }
constexpr int b32_off(int f) { return f == FMT_Q4_0 ? 8 : f == FMT_Q5_0 ? 16 : 0; }
// bytes per 256 values of a row (one k-quant super-block, or eight 32-value blocks)
constexpr int block_bytes(int f) {
    return f == FMT_Q4K ? 144 : f == FMT_Q5K ? 176 : f == FMT_Q6K ? 210 : 8 * b32_bytes(f);
}

// device pointers to the sections of one Q8 plane
struct Plane {
    uint16_t *q16;     // f16 codes [M][K] (binary16 bit patterns)
    int8_t *q8;        // int8 codes [M][K]
    float *d;          // [K/32][M]
    int32_t *s;        // [K/32][M]
    float *ds;         // [M][2*K/32]: per super-block hi[8], lo[8] of tf32(d*S)
};

// window of the integer checkpoint dump (test hook); cnt == 0 disables it
struct Dump {
    int32_t *out;
    int64_t m0, m_cnt, n0, n_cnt;
};

int set_error(int code, const char *fmt, ...);

// SM count of the current device (cached per device)
int sm_count();

// Sets the dynamic shared-memory limit of `kernel` once per device; returns MQ_OK or MQ_ERR_CUDA.
int ensure_smem_attr(const void *kernel, int bytes, int slot);
int cuda_error(cudaError_t e, const char *what);
// CTAs of `kernel` resident per SM at this block size and dynamic shared memory (cached per
// device and slot); returns MQ_OK or MQ_ERR_CUDA.
int resident_ctas(const void *kernel, int threads, int smem_bytes, int slot, int *out);

// Launch with programmatic stream serialization (the kernel may start while its predecessor on
// the stream finishes; every kernel of the library waits on griddepcontrol before it touches
// dependent memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launchers (arguments already validated); return MQ_OK or MQ_ERR_CUDA
// sections: the MQ_PLANE_* mask of the plane sections written besides d and S (1 .. 7)
int launch_quantize(const float *x, int64_t M, int64_t K, const float *rms_w, float eps, unsigned sections,
                    const Plane &p, unsigned int *err, cudaStream_t stream);
int launch_swiglu_quantize(const float *g, const float *up, int64_t M, int64_t K, unsigned sections, const Plane &p,
                           cudaStream_t stream);
int launch_gemv(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream);
int launch_gemv_b32(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                    const Dump &dump, unsigned int *err, cudaStream_t stream);
// the fused gate|up GEMM with the SwiGLU epilogue: plane p (M x K) -> plane po (M x F)
int launch_gemm_swiglu(Fmt fmt, const uint8_t *wg, const uint8_t *wu, int64_t F, int64_t K, const Plane &p, int64_t M,
                       const Plane &po, unsigned int *err, cudaStream_t stream);
// attribute slots (ensure_smem_attr / resident_ctas): GEMM 2 fmt + dump (below 16), GEMV 16 + 16 fmt + ...,
// the fused gate|up GEMM kAttrSlotSwiglu + fmt
constexpr int kAttrSlotSwiglu = 16 + 8 * 16;
int launch_gemm(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                const Dump &dump, unsigned int *err, cudaStream_t stream);
// the small-M tensor-core GEMM (1 <= M <= 32 tokens; k-quant weights)
int launch_gemm_small(Fmt fmt, const uint8_t *w, int64_t N, int64_t K, const Plane &p, int64_t M, float *y,
                      const Dump &dump, unsigned int *err, cudaStream_t stream);
// one launch over nj independent matrices of one format (k-quants) and K, each with its own plane
// (M tokens) and output
// x: nullptr (each job reads its plane p), or each job's f32 activation (M = 1; quantized in the kernel)
int launch_gemv_grouped(Fmt fmt, int nj, const uint8_t *const *w, const int64_t *N, const Plane *p, float *const *y,
                        int64_t K, int64_t M, unsigned int *err, cudaStream_t stream, const float *const *x = nullptr);
// one launch quantizing nj activations [M][K] (plain Q8, no RMSNorm) into their own planes
int launch_quantize_grouped(int nj, const float *const *x, const Plane *p, int64_t M, int64_t K, unsigned sections,
                            cudaStream_t stream);
// cuTensorMapEncodeTiled from the driver (nullptr if unavailable), resolved once
void *tensor_map_encoder();
// attribute slots of the small-M GEMM: kAttrSlotSmall + 2 * (3 fmt + NT/32) + dump
constexpr int kAttrSlotSmall = kAttrSlotSwiglu + 8;

}  // namespace mq
