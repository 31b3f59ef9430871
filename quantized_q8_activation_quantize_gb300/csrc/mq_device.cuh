// mq_device.cuh -- sm_103a device helpers shared by the library's kernels:
// bounded mbarrier waits, bulk / tensor TMA copies, tcgen05 (TMEM + MMA) wrappers.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace mq {

// ------------------------------------------------------------------ error word ---
// Each kernel receives a pointer to a per-device error word.  A wait that runs out
// ORs its site code into it and the kernel winds down without further waiting.
enum : unsigned int {
    ERR_GEMV_FULL = 1u << 0,
    ERR_GEMM_A_FULL = 1u << 1,
    ERR_GEMM_B_FULL = 1u << 2,
    ERR_GEMM_AB_EMPTY = 1u << 3,
    ERR_GEMM_RAW_FULL = 1u << 4,
    ERR_GEMM_ACC_FULL = 1u << 5,
    ERR_GEMM_ACC_EMPTY = 1u << 6,
    ERR_GEMM_INFO_FULL = 1u << 7,
    ERR_GEMM_INFO_EMPTY = 1u << 8,
    ERR_GEMV_DRAIN = 1u << 9,
    ERR_GEMM_MIN = 1u << 10,
    ERR_GEMM_DA = 1u << 11,
    ERR_TEST_FORCED = 1u << 31,
};

// A bounded wait gives up after this much wall time (the longest legitimate wait in
// these kernels is a few microseconds).
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------- mbarrier ---
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// make barrier initialisation visible to the other threads and to the async proxy
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking test of the phase with the given parity (returns at once).  Several of
// these issued back to back overlap their latencies.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Same, but the thread may be suspended for up to `hint_ns` while the phase is incomplete
// (it resumes as soon as the phase completes), so a waiting warp does not spin on the
// issue slots the working warps of its SM sub-partition need.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (after
// recording `code` in *err and raising *abort) if it did not complete within
// kWaitTimeoutNs, or at once if another warp already raised *abort.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned int *err, uint32_t code,
                                          volatile int *abort) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(a, parity, 100000u)) return true;     // sleep up to 100 us
        if (abort != nullptr && *abort) return false;
        if (global_timer_ns() - t0 > kWaitTimeoutNs) {
            atomicOr(err, code);
            if (abort != nullptr) *abort = 1;
            return false;
        }
    }
}

// The same bound and failure handling, but the thread waits in the hardware's default suspend
// (try_wait without a time hint) rather than a long hinted sleep, so it resumes sooner after the
// phase completes; for the one warp whose wake-up latency is on a pipeline's critical path.
__device__ __forceinline__ bool mbar_wait_prompt(uint64_t *bar, uint32_t parity, unsigned int *err, uint32_t code,
                                                 volatile int *abort) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (abort != nullptr && *abort) return false;
            if (global_timer_ns() - t0 > kWaitTimeoutNs) {
                atomicOr(err, code);
                if (abort != nullptr) *abort = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------ programmatic dependent launch ---
// Kernels are launched with programmatic stream serialization: a kernel may be scheduled
// while its predecessor on the stream is still running.  Each kernel calls grid_dep_wait()
// before it touches memory the predecessor may write or read (the plane, activations,
// outputs, weights); only L2 prefetch hints go ahead of it.  grid_dep_launch() lets the
// successor be scheduled early; it is a no-op without a successor.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// hint: bring [p, p + bytes) into L2 (16-byte aligned address and size); never faults the data
__device__ __forceinline__ void prefetch_l2_bulk(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// ----------------------------------------------------------------- bulk copies ---
// 1-D bulk async copy global -> shared, completion counted on `bar` (bytes, 16-B granular).
__device__ __forceinline__ void bulk_copy_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst_smem)),
        "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// 2-D tiled tensor copy global -> shared through a CUtensorMap (x = innermost coordinate).
__device__ __forceinline__ void tma_load_2d(void *dst_smem, const void *tmap, int32_t x, int32_t y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst_smem)),
        "l"(tmap), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// generic-proxy shared-memory writes -> visible to the async proxy (tensor core reads)
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------------- tcgen05 ---
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (f16 operands, f32 accumulator), one CTA.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once every previously issued tcgen05 op of this thread has completed
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns (lane i of the warp reads TMEM lane base+i)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns into r[off .. off+15]
template <int NR>
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[NR], int off) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[off + 0]), "=r"(r[off + 1]), "=r"(r[off + 2]), "=r"(r[off + 3]), "=r"(r[off + 4]), "=r"(r[off + 5]),
          "=r"(r[off + 6]), "=r"(r[off + 7]), "=r"(r[off + 8]), "=r"(r[off + 9]), "=r"(r[off + 10]), "=r"(r[off + 11]),
          "=r"(r[off + 12]), "=r"(r[off + 13]), "=r"(r[off + 14]), "=r"(r[off + 15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor for a K-major operand tile stored with the 128-byte
// swizzle: rows of 128 B (64 f16), 8-row atoms of 1024 B stacked at a 1024-B stride.
// `addr` is the shared address of the tile (1024-B aligned) plus the byte offset of
// the K slice inside the 128-byte row.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);         // start address
    d |= (uint64_t)1 << 16;                        // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;              // stride byte offset: next 8-row atom
    d |= (uint64_t)1 << 46;                        // descriptor version (tcgen05)
    d |= (uint64_t)2 << 61;                        // swizzle mode: 128 B
    return d;
}

// Same for a K-major tile stored with the 64-byte swizzle: rows of 64 B, 8-row atoms of
// 512 B stacked at a 512-B stride (tile base 512-B aligned).
__device__ __forceinline__ uint64_t sw64_kmajor_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(512 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)4 << 61;                        // swizzle mode: 64 B
    return d;
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::tf32 (tf32 operands in f32 containers, f32 accumulator).
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Warp-converged issue: all 32 lanes execute these with identical operands and one elected
// lane (always the same: the lowest) issues the instruction, so the operands and the loop
// around it stay in the uniform datapath.  A commit tracks the elected lane's own MMAs.
__device__ __forceinline__ void mma_f16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint64_t *bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar))
        : "memory");
}

// round an f32 to the nearest tf32 value (10 explicit mantissa bits), kept in f32 format
__device__ __forceinline__ float tf32_rn(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

// Instruction descriptor: kind::tf32, tf32 A and B (K-major), f32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int m, int n) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// Instruction descriptor: kind::f16, f16 A and B (K-major), f32 D, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int m, int n) {
    return (1u << 4)                               // D format f32
           | (0u << 7) | (0u << 10)                // A, B format f16
           | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}


// SwiGLU producer ("Features > GPU -- CUDA": the swiglu producer emits the q8 plane directly;
// "Compute Graph Design > 5": Mul(Silu(X), Y) -> SwiGLU): y = silu(g) * u in IEEE f32, every
// step rounded once, then the Q8 quantization of y.  exp is evaluated by the textbook
// reduction: x = k ln2 + r, k = nearest integer to x / ln2 (ties to even), |r| <= ln2 / 2,
// exp(r) by its Taylor series through r^7, times 2^k; x is clamped to [-86, 88] so the
// result stays a normal f32 (in f32, silu is unaffected outside that range).  Every step is
// an explicitly rounded operation, so y -- and every Q8 code -- is one fixed function of
// (g, u).
__device__ __forceinline__ float exp_f32(float x) {
    x = x > 88.0f ? 88.0f : x;
    x = x < -86.0f ? -86.0f : x;
    const float k = rintf(__fmul_rn(x, 1.44269504f));         // 1 / ln2
    float r = fmaf(-k, 0.693145751953125f, x);                  // ln2, high part (k * hi is exact)
    r = fmaf(-k, 1.42860677e-06f, r);                           // ln2, low part
    float p = 1.98412698e-04f;                                  // 1/7!
    p = fmaf(p, r, 1.38888889e-03f);                            // 1/6!
    p = fmaf(p, r, 8.33333333e-03f);                            // 1/5!
    p = fmaf(p, r, 4.16666667e-02f);                            // 1/4!
    p = fmaf(p, r, 1.66666667e-01f);                            // 1/3!
    p = fmaf(p, r, 0.5f);                                       // 1/2!
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    // p * 2^k with 2^k built from its exponent field: k is in [-124, 127] and p in [0.70, 1.42],
    // so the product is a normal float and the multiply is exact -- the value ldexpf returns
    return __fmul_rn(p, __int_as_float(((int)k + 127) << 23));
}

// g / den is divided as (g 2^-64) / (den 2^-64) when den > 2^64: then g < -44, both scalings
// are exact and the correctly rounded quotient is the same number, but the divide stays off the
// slow path it takes for a huge denominator (measured: 0.34 ms of a 2.7 ms fused FFN GEMM).
// Branch-free (a factor of 1 otherwise, also exact), so independent calls interleave.
__device__ __forceinline__ float swiglu1(float g, float u) {
    const float den = __fadd_rn(1.0f, exp_f32(-g));
    const float sc = den > 0x1p64f ? 0x1p-64f : 1.0f;
    return __fmul_rn(__fdiv_rn(__fmul_rn(g, sc), __fmul_rn(den, sc)), u);
}


// Q8 quantization of a 32-value block held by four consecutive lanes (lane 4i + j holds values
// 8j .. 8j + 7 of block i; every lane of the warp takes part): amax over the block, d = amax / 127
// (IEEE divide), the codes q = clamp(round_half_away(y * (1 / d)), -127, 127) as exact floats (+0
// for a zero code; 0 when d = 0), and the code sums of the lane pair (lane, lane ^ 1: values 0 .. 15
// or 16 .. 31 of the block) and of the whole block -- exact integers, |S| <= 4064.
struct Q8Lane {
    float r[8];
    float d;
    float s16;
    float s;
};
__device__ __forceinline__ void q8_lane(const float (&v)[8], Q8Lane &o) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    o.d = __fdiv_rn(amax, 127.0f);
    const float id = (o.d != 0.0f) ? __fdiv_rn(1.0f, o.d) : 0.0f;
    float fs = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        // half away from zero, clamped; + 0 turns a -0 code into +0 (the f16 code of 0 is 0x0000)
        o.r[i] = __fadd_rn(fminf(fmaxf(roundf(__fmul_rn(v[i], id)), -127.0f), 127.0f), 0.0f);
        fs = __fadd_rn(fs, o.r[i]);
    }
    fs = __fadd_rn(fs, __shfl_xor_sync(0xffffffffu, fs, 1));
    o.s16 = fs;
    o.s = __fadd_rn(fs, __shfl_xor_sync(0xffffffffu, fs, 2));
}

// the int8 bytes of eight codes held as exact floats in [-127, 127], without conversion
// instructions: r + 1.5 * 2^23 holds r in the low mantissa bits, so its low byte is r in two's
// complement
__device__ __forceinline__ uint2 q8_bytes(const float (&r)[8]) {
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(__fadd_rn(r[i], 12582912.0f));
    uint2 b8;
    b8.x = __byte_perm(__byte_perm(w[0], w[1], 0x0040), __byte_perm(w[2], w[3], 0x0040), 0x5410);
    b8.y = __byte_perm(__byte_perm(w[4], w[5], 0x0040), __byte_perm(w[6], w[7], 0x0040), 0x5410);
    return b8;
}

// Q8 quantization of one 32-value block held by one thread, with the same operations as the
// warp-cooperative quantizer (amax, d = amax / 127, q = round_half_away(x * (1 / d)) clamped to
// +-127, S = sum q, and d * S as a tf32 (hi, lo) pair), so equal inputs give equal planes.
// Writes the block's 32 int8 and f16 codes at q8 / q16 (16-byte aligned) and returns d, S and
// the pair through the references.
__device__ __forceinline__ void quantize_block32(const float (&v)[32], int8_t *q8, uint16_t *q16, float &d_out,
                                                 int &s_out, float &hi_out, float &lo_out) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
    const float d = __fdiv_rn(amax, 127.0f);
    const float id = (d != 0.0f) ? __fdiv_rn(1.0f, d) : 0.0f;
    int s = 0;
    uint32_t b8[8], h16[16];
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        float r0 = roundf(__fmul_rn(v[i], id)), r1 = roundf(__fmul_rn(v[i + 1], id));
        r0 = fminf(fmaxf(r0, -127.0f), 127.0f);
        r1 = fminf(fmaxf(r1, -127.0f), 127.0f);
        const int q0 = __float2int_rz(r0), q1 = __float2int_rz(r1);
        s += q0 + q1;
        const uint32_t pair = (uint32_t)(q0 & 0xff) | ((uint32_t)(q1 & 0xff) << 8);
        if ((i & 2) == 0)
            b8[i >> 2] = pair;
        else
            b8[i >> 2] |= pair << 16;
        __half2 t = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
        h16[i >> 1] = *reinterpret_cast<uint32_t *>(&t);
    }
    uint4 *d8 = reinterpret_cast<uint4 *>(q8);
    d8[0] = make_uint4(b8[0], b8[1], b8[2], b8[3]);
    d8[1] = make_uint4(b8[4], b8[5], b8[6], b8[7]);
    uint4 *d16 = reinterpret_cast<uint4 *>(q16);
#pragma unroll
    for (int k = 0; k < 4; ++k) d16[k] = make_uint4(h16[4 * k], h16[4 * k + 1], h16[4 * k + 2], h16[4 * k + 3]);
    const float ds = __fmul_rn(d, (float)s);
    const float hi = tf32_rn(ds);
    d_out = d;
    s_out = s;
    hi_out = hi;
    lo_out = tf32_rn(__fsub_rn(ds, hi));
}

}  // namespace mq
