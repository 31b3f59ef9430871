"""GB300-native (sm_103a) quantized k-quant matmul: Q8 activation quantization,
Q4_K / Q5_K / Q6_K x Q8 tensor-core GEMM (prefill) and dp4a GEMV (decode).

The compute lives in libmq.so (C ABI, include/mq.h); ``binding`` marshals torch
tensors into it, ``inputs`` makes the seeded synthetic workloads.
"""
from .binding import (MQError, alloc_plane, matmul, mq_debug_blockdots, mq_debug_forced_timeout,  # noqa: F401
                      mq_device_status, mq_gemm_q4k, mq_gemm_q5k, mq_gemm_q6k, mq_gemv_q4k, mq_gemv_q5k, mq_gemv_q6k,
                      mq_q8_plane_bytes,
                      mq_q8_plane_layout, mq_quantize_q8, mq_quantize_swiglu_q8, plane_views)
