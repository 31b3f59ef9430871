/*
 * mq.h -- C ABI of the GB300 (sm_103a) quantized matmul library (GGML k-quants and
 * 32-value block formats).
 *
 * The hot path of quantized LLM inference over GGML k-quant weights, as the
 * minfer pages describe it ("minfer" book print view, "Features > GPU -- CUDA";
 * "Support Matrix > CUDA notes"):
 *   1. f32 activations are quantized on the fly into an int8 Q8 plane
 *      (blocks of 32, one f32 scale per block), optionally straight out of an
 *      RMSNorm producer, so the normalized f32 rows are never written;
 *   2. prefill (many tokens) multiplies the plane with raw Q4_K / Q5_K / Q6_K
 *      super-blocks (or Q4_0 .. Q8_0 blocks) on the tensor cores (MMQ);
 *   3. decode (one or a few tokens) streams the raw weight bytes once and
 *      takes integer dots per block on the CUDA cores (MMVQ).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is a DEVICE pointer owned by the caller, unless
 *     stated otherwise.  Nothing is retained after the call returns and the
 *     library never allocates device memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and returns MQ_OK or a negative mq_status.  Argument
 *     errors are detected on the host before anything is launched;
 *     mq_last_error() then names the offending values.  There is no fallback
 *     path: an unsupported device or shape is an error, never a slower route.
 *   - Weights are raw GGML block bytes, row-major [N rows][K/256 super-blocks]
 *     (weight memory layout [out][in], "Architecture > 4.5 Core invariants",
 *     item 3), base aligned to 16 bytes.  K must be a positive multiple of 256.
 *     Weights are copied in 16-byte aligned pieces, so a read may run up to 15
 *     bytes past the last weight byte, never past the 16-byte granule that holds
 *     it; those bytes do not affect any result.
 *   - Activations are token-major f32 [M][K]; outputs are token-major f32 [M][N].
 *     An output must not overlap any input of the same call: every entry point
 *     compares the byte ranges of its output and its inputs on the host and
 *     returns MQ_ERR_ARG if any two share a byte.
 *   - M == 0 or N == 0 is a valid empty call (returns MQ_OK, launches nothing).
 *   - Kernels never wait without bound.  A device-side wait that runs out sets
 *     a per-device error word and the kernel returns early; mq_device_status()
 *     reports it as MQ_ERR_DEVICE_TIMEOUT.
 */
#ifndef MQ_H
#define MQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MQ_API __attribute__((visibility("default")))
#else
#define MQ_API
#endif

typedef struct CUstream_st *mq_stream_t;  /* same type as cudaStream_t */

typedef enum {
    MQ_OK = 0,
    MQ_ERR_ARG = -1,            /* NULL pointer, negative size, bad flag */
    MQ_ERR_SHAPE = -2,          /* K not a positive multiple of 256, size beyond the limits */
    MQ_ERR_ALIGN = -3,          /* a pointer lacks the alignment stated for it */
    MQ_ERR_DEVICE = -4,         /* current device is not compute capability 10.3 (sm_103) */
    MQ_ERR_CUDA = -5,           /* a CUDA runtime/driver call failed; text in mq_last_error() */
    MQ_ERR_DEVICE_TIMEOUT = -6  /* a bounded device-side wait ran out (see mq_device_status) */
} mq_status;

/* Thread-local text describing the last error returned on this thread ("" if none). */
MQ_API const char *mq_last_error(void);

/* ---------------------------------------------------------------- Q8 plane ---
 *
 * The Q8 activation plane is this library's own format (the pages call it the
 * "transposed q8 plane" that the producers emit).  For M tokens and K values
 * per token, nblk = K/32 blocks per token, it holds:
 *   q16 : f16  [M][K]     the codes q in [-127, 127] as f16 (every code is an
 *                          exact f16 value); operand of the tensor-core GEMM
 *   q8  : int8 [M][K]     the same codes as int8; operand of the dp4a GEMV
 *   d   : f32  [nblk][M]  block scale d = amax/127 (block-major: "transposed")
 *   s   : i32  [nblk][M]  block code sum S = sum q (used by the Q4_K min term)
 *   ds  : f32  [M][2*nblk] per super-block of token m, 16 values: the tf32 pair
 *                          (hi[8], lo[8]) of d*S for its eight 32-value blocks,
 *                          hi = tf32(d*S), lo = tf32(d*S - hi) (round to nearest);
 *                          operand of the tensor-core Q4_K min term
 * each section starting on a 256-byte boundary.  The plane base must be
 * 256-byte aligned.  Contents are defined only after mq_quantize_q8 wrote them.
 */
typedef struct {
    size_t off_q16, off_q8, off_d, off_s, off_ds;
    size_t total_bytes;
} mq_plane_layout;

/* Bytes needed for the plane of an M x K activation (0 if the shape is invalid). */
MQ_API size_t mq_q8_plane_bytes(int64_t M, int64_t K);

/* Section offsets of the plane; MQ_ERR_SHAPE for invalid M or K. Host-only, no CUDA call. */
MQ_API int mq_q8_plane_layout(int64_t M, int64_t K, mq_plane_layout *out);

/*
 * mq_quantize_q8 -- activation quantization (MMQ activation quantize; the
 * RMSNorm-fused producer when rms_w != NULL).  "Features > GPU -- CUDA":
 * producer-fused activation quantization; "Compute Graph Design > 3.1": RmsNorm{eps}.
 *
 *   x      f32 [M][K], 16-byte aligned
 *   rms_w  NULL: quantize x itself.
 *          else f32 [K] (16-byte aligned): quantize y = (x * r) * rms_w with
 *          r = 1/sqrt(mean_k(x^2) + eps) per token (sum of squares in f64,
 *          r rounded once to f32, two f32 products).
 *   eps    RMSNorm epsilon (ignored when rms_w == NULL); must be >= 0 and finite
 *   plane  output, mq_q8_plane_bytes(M, K) bytes, 256-byte aligned
 *
 * Per token and 32-block: amax = max|y|, d = amax/127 (IEEE f32 divide),
 * q = clamp(round_half_away_from_zero(y * (1/d)), -127, 127) (0 when d == 0),
 * S = sum q.
 */
MQ_API int mq_quantize_q8(const float *x, int64_t M, int64_t K, const float *rms_w, float eps,
                   void *plane, mq_stream_t stream);

/*
 * Plane sections.  d and S are always written; the other three sections are written on request,
 * so a producer writes only what its consumers read:
 *   mq_gemm_*            read q16, d and (Q4_K, Q5_K, Q4_1, Q5_1) ds      -> MQ_PLANE_FOR_GEMM
 *   mq_gemv_*            read q8, d and S                                  -> MQ_PLANE_FOR_GEMV
 *   mq_gemm_q4k_swiglu   reads q16, d and ds of its input plane            -> MQ_PLANE_FOR_GEMM
 * A section that was not written keeps whatever the buffer held before; a consumer that reads it
 * then computes from those bytes (no error is raised: the plane carries no record of its sections).
 */
enum {
    MQ_PLANE_Q16 = 1u,                    /* f16 codes (tensor-core operand) */
    MQ_PLANE_Q8 = 2u,                     /* int8 codes (dp4a operand) */
    MQ_PLANE_DS = 4u,                     /* tf32 pairs of d*S (tensor-core min term) */
    MQ_PLANE_ALL = 7u,
    MQ_PLANE_FOR_GEMM = 5u,               /* MQ_PLANE_Q16 | MQ_PLANE_DS */
    MQ_PLANE_FOR_GEMV = 2u                /* MQ_PLANE_Q8 */
};

/*
 * mq_quantize_q8_ex -- mq_quantize_q8 writing only the requested sections (a non-empty
 * MQ_PLANE_* mask; MQ_ERR_ARG otherwise) besides d and S.  Every section it writes holds exactly
 * what mq_quantize_q8 writes there; mq_quantize_q8 is this call with MQ_PLANE_ALL.  Per value,
 * MQ_PLANE_ALL writes 3.5 bytes, MQ_PLANE_FOR_GEMM 2.5 and MQ_PLANE_FOR_GEMV 1.25 (the int8 code
 * plus 8 bytes of d and S per 32 values).
 */
MQ_API int mq_quantize_q8_ex(const float *x, int64_t M, int64_t K, const float *rms_w, float eps,
                             unsigned sections, void *plane, mq_stream_t stream);

/*
 * mq_quantize_swiglu_q8 -- the SwiGLU producer of the down projection: writes the Q8 plane
 * of y = silu(gate) * up, silu(g) = g / (1 + exp(-g)), with no f32 intermediate in memory.
 * "Features > GPU -- CUDA": the swiglu producer emits the q8 plane directly; "Compute Graph
 * Design > 5": Mul(Silu(X), Y) is the SwiGLU pattern.
 *
 *   gate, up  f32 [M][K] (token-major), each 16-byte aligned, read only
 *   plane     as for mq_quantize_q8
 *
 * y is computed in IEEE f32 with every step rounded once; exp is the textbook reduction
 * x = k ln2 + r (k nearest to x / ln2, ties to even), exp(r) by its Taylor series through
 * r^7, times 2^k, with x clamped to [-86, 88].  Then the Q8 quantization of mq_quantize_q8
 * applies to y.  Same errors as mq_quantize_q8 (M == 0 is a no-op).
 */
MQ_API int mq_quantize_swiglu_q8(const float *gate, const float *up, int64_t M, int64_t K, void *plane,
                                 mq_stream_t stream);

/* mq_quantize_swiglu_q8_ex -- the same, writing only the requested MQ_PLANE_* sections besides d and S. */
MQ_API int mq_quantize_swiglu_q8_ex(const float *gate, const float *up, int64_t M, int64_t K, unsigned sections,
                                    void *plane, mq_stream_t stream);

/*
 * mq_gemm_q4k / mq_gemm_q6k -- prefill GEMM (MMQ) on the tensor cores.
 * "Features > GPU -- CUDA": raw-nibble GEMMs for q4_K and q6_K over the Q8
 * plane; "Support Matrix > CUDA notes": prefill (nt >= 16) takes this path.
 *
 *   w      raw Q4_K (144 B/block) or Q6_K (210 B/block) bytes [N][K/256], 16-byte aligned
 *   plane  Q8 plane of an M x K activation written by mq_quantize_q8
 *   y      f32 [M][N] output (fully overwritten), 4-byte aligned
 *
 * Y[m][n] = sum over super-blocks of
 *   Q4_K: d * sum_j sc_j * d_a[m][j] * D_j  -  dmin * sum_j m_j * d_a[m][j] * S[m][j]
 *   Q6_K: d * sum_s sc_s * d_a[m][s/2] * D_s
 * with D the exact integer dot of the weight quants and the Q8 codes over a
 * 32-value (Q4_K sub-block) or 16-value (Q6_K sub-block) range.  The integer
 * dots are exact; the float scaling is f32.  Any N >= 0 and any M from 0 to
 * 65535 * 128 = 8388480 (tokens are tiled by 128, the tail is masked); a larger M
 * returns MQ_ERR_SHAPE (split the tokens over several calls).
 */
MQ_API int mq_gemm_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);

/*
 * mq_gemm_small_q4k / mq_gemm_small_q5k / mq_gemm_small_q6k -- the small-M band (1 <= M <= 32
 * tokens) on the tensor cores ("Support Matrix > CUDA notes": the band between decode (nt == 1,
 * dp4a MMVQ) and prefill (nt >= 16, MMQ); "Features > Continuous batching": several sequences
 * decoded together).  Same arguments, layouts, errors and result as mq_gemm_q4k / mq_gemm_q5k /
 * mq_gemm_q6k (the same exact integer block dots, f32 scaling), computed with the weights as the
 * 128-row MMA operand and the tokens as its 16- or 32-wide side, so every weight byte is read
 * from memory once for all M tokens.  M must be at most 32 (MQ_ERR_SHAPE otherwise); M == 0 or
 * N == 0 is a valid empty call.  The plane needs the MQ_PLANE_FOR_GEMM sections.
 */
MQ_API int mq_gemm_small_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                             float *y, mq_stream_t stream);
MQ_API int mq_gemm_small_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                             float *y, mq_stream_t stream);
MQ_API int mq_gemm_small_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                             float *y, mq_stream_t stream);

/*
 * mq_gemm_q4k_swiglu -- the fused gate|up GEMM of a SwiGLU FFN: both Q4_K projections of one
 * input plane in one kernel, whose epilogue writes the Q8 plane of silu(gate) * up for the
 * down projection ("Features > GPU -- CUDA": the FFN's gate and up matmuls share one plane and
 * the swiglu producer emits the q8 plane; "Compute Graph Design > 5": the FusedFFN form).
 *
 *   w_gate, w_up  raw Q4_K bytes [F][K/256] each, 16-byte aligned
 *   plane_in      Q8 plane of the M x K input (mq_quantize_q8)
 *   plane_out     Q8 plane of an M x F activation (mq_q8_plane_bytes(M, F) bytes, 256-byte
 *                 aligned), fully written
 *   F             rows of each projection, a multiple of 256 (the output plane's K) of at most
 *                 65535 * 64 = 4194240; F == 0 (or M == 0) is a valid empty call
 *
 * G and U are what mq_gemm_q4k writes for w_gate and w_up (the same f32 values, bit for bit);
 * the output plane is then what mq_quantize_swiglu_q8(G, U) writes, so the pair
 * (mq_gemm_q4k x 2, mq_quantize_swiglu_q8) and this call give identical planes, without the
 * two f32 [M][F] intermediates.  Same errors as mq_gemm_q4k plus MQ_ERR_SHAPE for F % 256
 * or F beyond the limit and MQ_ERR_ARG if plane_out overlaps plane_in or either weight matrix.
 */
MQ_API int mq_gemm_q4k_swiglu(const void *w_gate, const void *w_up, int64_t F, int64_t K, const void *plane_in,
                              int64_t M, void *plane_out, mq_stream_t stream);

/*
 * mq_gemv_q4k / mq_gemv_q6k -- decode GEMV (MMVQ): streams every weight byte
 * once per group of up to 8 (Q4_K) or 4 (Q6_K) tokens and takes dp4a int8 dots
 * per block ("Support Matrix > CUDA notes": decode (nt == 1) uses the dp4a MMVQ
 * kernels).  Same arguments, same result definition as the GEMMs.  Meant for
 * M < 16 (any M >= 0 is accepted; each further token group streams W again).
 */
MQ_API int mq_gemv_q4k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemv_q6k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);

/*
 * mq_gemv_q5k / mq_gemm_q5k -- decode GEMV and prefill GEMM over Q5_K weights ("Support
 * Matrix > CUDA notes": decode uses the dp4a MMVQ kernels for Q4_K/Q5_K/Q6_K; the
 * tensor-core GEMM is the Q4_K skeleton with the fifth bit unpacked).  Same arguments and
 * errors as mq_gemv_q4k / mq_gemm_q4k; w is raw Q5_K bytes (176 B/block: d, dmin, 12 scale
 * bytes packed as in Q4_K, qh[32], qs[128]) [N][K/256], 16-byte aligned.  The GEMV takes
 * tokens 8 per pass over W.
 *   Y[m][n] = sum over super-blocks of
 *             d * sum_j sc_j * d_a[m][j] * D_j  -  dmin * sum_j m_j * d_a[m][j] * S[m][j]
 * with D_j the exact integer dot of the 5-bit quants q = nibble + 16 * (bit j of qh[l])
 * and the Q8 codes over the 32-value sub-block j.
 */
MQ_API int mq_gemv_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q5k(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);

/*
 * mq_gemv_grouped_q4k / _q5k / _q6k -- several independent decode GEMVs of one format in one launch:
 * the matrices of one level of a decoder layer (q|k|v from the layer input, gate|up from the
 * post-attention input) share the launch's fixed cost instead of paying it each ("Features >
 * GPU -- CUDA": decode streams the weights with the MMVQ kernel; a layer's independent matmuls
 * have no order between them).
 *
 *   jobs     HOST array of n_jobs descriptors {w, N, plane, y}, read during the call and not
 *            retained: each job is exactly the arguments of one mq_gemv_q4k / _q5k / _q6k call
 *   n_jobs   0 .. 8 (0: nothing to do)
 *   K, M     shared by every job: the reduction length and the tokens of every plane
 *
 * Each job's y is what the single call would write, bit for bit.  Errors: as the single call for
 * each job, plus MQ_ERR_ARG for n_jobs outside 0 .. 8, a NULL table, or an output that overlaps any
 * input or other output of the call.
 */
typedef struct {
    const void *w;       /* raw weight blocks [N][K/256], 16-byte aligned (device) */
    int64_t N;           /* rows of this job's weight matrix */
    const void *plane;   /* Q8 plane of the job's M x K activation (device, 256-byte aligned) */
    float *y;            /* f32 [M][N] output (device) */
} mq_gemv_job;

MQ_API int mq_gemv_grouped_q4k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream);
MQ_API int mq_gemv_grouped_q5k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream);
MQ_API int mq_gemv_grouped_q6k(const mq_gemv_job *jobs, int n_jobs, int64_t K, int64_t M, mq_stream_t stream);

/*
 * mq_gemv_grouped_x_q4k / _q5k / _q6k -- the grouped decode GEMV for one token (M = 1) straight from
 * f32 activations: every CTA quantizes its job's x with the arithmetic of mq_quantize_q8 (no
 * RMSNorm) into shared memory and runs the GEMV on those codes, so a layer level takes one launch
 * instead of a quantize launch and a GEMV launch ("Features > GPU -- CUDA": activation quantization
 * fused into the kernels of the path; decode uses the MMVQ weight-streaming kernel).  No plane is
 * written.
 *
 *   jobs     HOST array of n_jobs descriptors {w, N, x, y}, read during the call and not retained:
 *            w, N and y as for mq_gemv_q4k / _q5k / _q6k with M = 1; x f32 [K], 16-byte aligned
 *            (device); jobs may share one x
 *   n_jobs   0 .. 8 (0: nothing to do); a job with N == 0 is skipped
 *   K        shared by every job; one token's staged codes must fit a CTA's shared memory:
 *            K <= 101888 (Q4_K), 96768 (Q5_K), 81920 (Q6_K)
 *
 * Each job's y is, bit for bit, the y of mq_quantize_q8(x) followed by mq_gemv_q4k / _q5k / _q6k
 * on that plane.  Errors: MQ_ERR_ARG for n_jobs outside 0 .. 8, a NULL table or pointer, negative
 * N, or an output overlapping any input or other output; MQ_ERR_ALIGN for a misaligned w, x or y;
 * MQ_ERR_SHAPE for an invalid K, N >= 2^31, or K too large to stage.
 */
typedef struct {
    const void *w;       /* raw weight blocks [N][K/256], 16-byte aligned (device) */
    int64_t N;           /* rows of this job's weight matrix */
    const float *x;      /* f32 [K] activation of the token (device) */
    float *y;            /* f32 [N] output (device) */
} mq_gemv_xjob;

MQ_API int mq_gemv_grouped_x_q4k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream);
MQ_API int mq_gemv_grouped_x_q5k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream);
MQ_API int mq_gemv_grouped_x_q6k(const mq_gemv_xjob *jobs, int n_jobs, int64_t K, mq_stream_t stream);

/*
 * mq_quantize_q8_grouped -- the plain mq_quantize_q8_ex over several independent activations of one
 * shape [M][K] in one launch (the inputs of one level of a decoder layer in the decode sweep).
 *
 *   jobs      HOST array of n_jobs descriptors {x, plane} (read during the call, not retained):
 *             x f32 [M][K] 16-byte aligned, plane 256-byte aligned (device pointers)
 *   n_jobs    0 .. 8; sections a non-empty MQ_PLANE_* mask as for mq_quantize_q8_ex
 *
 * Every plane holds exactly what mq_quantize_q8_ex writes for its x.  Errors: as mq_quantize_q8_ex,
 * plus MQ_ERR_ARG for n_jobs outside 0 .. 8, a NULL table or pointer, or a plane overlapping any x
 * or other plane.
 */
typedef struct {
    const float *x;      /* f32 [M][K] activation (device) */
    void *plane;         /* its Q8 plane (device) */
} mq_quantize_job;

MQ_API int mq_quantize_q8_grouped(const mq_quantize_job *jobs, int n_jobs, int64_t M, int64_t K, unsigned sections,
                                  mq_stream_t stream);

/*
 * mq_gemv_q4_0 / _q4_1 / _q5_0 / _q5_1 / _q8_0 -- decode GEMV over the 32-value GGML block
 * formats ("Architecture > 6. Quantization & Tensor Layout": the weight blocks are the GGML
 * structs; "Support Matrix > CUDA notes": decode runs the dp4a MMVQ kernels).  Same
 * arguments, errors and token grouping (8 per pass over W) as mq_gemv_q4k.  w is raw block
 * bytes [N][K/32], row-major with rows contiguous, 16-byte aligned; K % 256 == 0 (as for
 * every entry point).  Blocks, little-endian:
 *   Q4_0 18 B: d fp16, qs[16]                 q_l = low nibble of qs[l], q_{l+16} = high;  v = d (q - 8)
 *   Q4_1 20 B: d fp16, m fp16, qs[16]         nibbles as Q4_0;                           v = d q + m
 *   Q5_0 22 B: d fp16, qh u32, qs[16]         q_l = nibble + 16 * bit l of qh;            v = d (q - 16)
 *   Q5_1 24 B: d fp16, m fp16, qh u32, qs[16] as Q5_0;                                    v = d q + m
 *   Q8_0 34 B: d fp16, qs[32] int8            q_l = qs[l];                                v = d q
 *   Y[m][n] = sum over blocks b of  d_b * d_a[m][b] * I_b  +  m_b * d_a[m][b] * S[m][b]
 * with I_b the exact integer dot of (q - offset) and the Q8 codes over block b (m_b = 0 for
 * the formats without m).
 */
MQ_API int mq_gemv_q4_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemv_q4_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemv_q5_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemv_q5_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemv_q8_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);

/*
 * mq_gemm_q4_0 / _q4_1 / _q5_0 / _q5_1 / _q8_0 -- prefill GEMM over the same 32-value formats
 * ("Support Matrix > CUDA notes": prefill (nt >= 16) runs the tensor-core MMQ path for
 * Q4_0/Q4_1/Q5_0/Q5_1/Q8_0 as well).  Same arguments, errors and result as the matching
 * mq_gemv_* (w as documented there), computed on the tensor cores like mq_gemm_q4k: the
 * exact integers q - offset of each block multiply the Q8 codes into one accumulator per
 * block, scaled by d * d_a; the Q4_1 / Q5_1 offset term m * d_a * S runs as tf32 MMAs.
 */
MQ_API int mq_gemm_q4_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q4_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q5_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q5_1(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);
MQ_API int mq_gemm_q8_0(const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                float *y, mq_stream_t stream);

/*
 * mq_device_status -- synchronizes `stream`, then reads and clears this
 * device's error word.  MQ_OK if no kernel reported a failed bounded wait
 * since the last call, MQ_ERR_DEVICE_TIMEOUT (with the failing wait named in
 * mq_last_error()) otherwise, MQ_ERR_CUDA if the synchronization failed.
 */
MQ_API int mq_device_status(mq_stream_t stream);

/* ------------------------------------------------------------- test hooks ---
 *
 * mq_debug_blockdots -- runs the same kernel as the named entry point (same
 * launch configuration, same y output) and also writes the integer
 * checkpoint I for the window of tokens [m0, m0+m_cnt) x rows [n0, n0+n_cnt):
 *   I_out int32 [m_cnt][n_cnt][K/32], per 32-value block b:
 *     Q4_K, Q5_K: I = sc_j * D_j                (j = b % 8)
 *     Q6_K: I = sc_2b * D_2b + sc_2b+1 * D_2b+1 (16-value sub-blocks)
 *     32-value formats: I = I_b = sum (q - offset) * code
 * op: 0 = mq_gemm_q4k, 1 = mq_gemm_q6k, 2 = mq_gemv_q4k, 3 = mq_gemv_q6k, 4 = mq_gemv_q5k,
 *     5 = mq_gemm_q5k, 6 = mq_gemv_q4_0, 7 = mq_gemv_q4_1, 8 = mq_gemv_q5_0,
 *     9 = mq_gemv_q5_1, 10 = mq_gemv_q8_0, 11 = mq_gemm_q4_0, 12 = mq_gemm_q4_1,
 *     13 = mq_gemm_q5_0, 14 = mq_gemm_q5_1, 15 = mq_gemm_q8_0, 16 = mq_gemm_small_q4k,
 *     17 = mq_gemm_small_q6k, 18 = mq_gemm_small_q5k.
 * The window must lie inside [0, M) x [0, N).  Test infrastructure: slower
 * than the plain entry points.
 */
MQ_API int mq_debug_blockdots(int op, const void *w, int64_t N, int64_t K, const void *plane, int64_t M,
                       float *y, int64_t m0, int64_t m_cnt, int64_t n0, int64_t n_cnt,
                       int32_t *I_out, mq_stream_t stream);

/*
 * mq_debug_forced_timeout -- launches a one-thread kernel whose only wait is on a
 * barrier that nothing completes.  The wait gives up after timeout_us (1..10^6)
 * and records the failure in the device error word, so the next
 * mq_device_status() returns MQ_ERR_DEVICE_TIMEOUT.  Exercises the bounded-wait
 * and status path without faulting or hanging the GPU.  Test infrastructure.
 */
MQ_API int mq_debug_forced_timeout(uint32_t timeout_us, mq_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MQ_H */
