"""GB300-native (sm_103a) quantized matmul: Q8 activation quantization, then
Q4_K / Q5_K / Q6_K and Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 weights x Q8 on the tensor cores
(prefill GEMM) and with dp4a (decode GEMV).

The compute lives in libmq.so (C ABI, include/mq.h); ``binding`` marshals torch
tensors into it, ``inputs`` makes the seeded synthetic workloads.
"""
from .binding import (MQError, alloc_plane, matmul, mq_debug_blockdots, mq_debug_forced_timeout,  # noqa: F401
                      mq_device_status, mq_gemm_q4_0, mq_gemm_q4_1, mq_gemm_q4k, mq_gemm_q4k_swiglu, mq_gemm_q5_0, mq_gemm_q5_1,
                      mq_gemm_q5k, mq_gemm_q6k, mq_gemm_q8_0, mq_gemv_q4_0, mq_gemv_q4_1,
                      mq_gemv_q4k, mq_gemv_q5_0, mq_gemv_q5_1, mq_gemv_q5k, mq_gemv_q6k, mq_gemv_q8_0,
                      mq_q8_plane_bytes,
                      mq_q8_plane_layout, mq_quantize_q8, mq_quantize_swiglu_q8, plane_views)
