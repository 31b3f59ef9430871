"""Thin ctypes binding over libmq.so (include/mq.h).  Argument marshalling only.

Every function here has the name of the C entry point it calls and forwards device
pointers (torch CUDA tensors or raw integers) plus a CUDA stream.  All arithmetic of
the path runs in the library's CUDA kernels; there is no Python or CPU fallback: if
the library is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libmq.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "mq.h")

MQ_OK, MQ_ERR_ARG, MQ_ERR_SHAPE, MQ_ERR_ALIGN, MQ_ERR_DEVICE, MQ_ERR_CUDA, MQ_ERR_DEVICE_TIMEOUT = 0, -1, -2, -3, -4, -5, -6
STATUS_NAMES = {0: "MQ_OK", -1: "MQ_ERR_ARG", -2: "MQ_ERR_SHAPE", -3: "MQ_ERR_ALIGN", -4: "MQ_ERR_DEVICE",
                -5: "MQ_ERR_CUDA", -6: "MQ_ERR_DEVICE_TIMEOUT"}
OP_GEMM_Q4K, OP_GEMM_Q6K, OP_GEMV_Q4K, OP_GEMV_Q6K = 0, 1, 2, 3
# plane sections (include/mq.h MQ_PLANE_*)
PLANE_Q16, PLANE_Q8, PLANE_DS, PLANE_ALL, PLANE_FOR_GEMM, PLANE_FOR_GEMV = 1, 2, 4, 7, 5, 2


class MQError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class PlaneLayout(ctypes.Structure):
    _fields_ = [("off_q16", ctypes.c_size_t), ("off_q8", ctypes.c_size_t), ("off_d", ctypes.c_size_t),
                ("off_s", ctypes.c_size_t), ("off_ds", ctypes.c_size_t), ("total_bytes", ctypes.c_size_t)]


class GemvJob(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("N", ctypes.c_int64), ("plane", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class GemvXJob(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("N", ctypes.c_int64), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


class QuantizeJob(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("plane", ctypes.c_void_p)]


_lib = None


def header_functions() -> list[str]:
    """Names of the functions include/mq.h declares."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(mq_\w+)\s*\(", text)))


def lib():
    """Load libmq.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} not built; run __graft_entry__.build() "
                               "(or python -m quantized_q8_activation_quantize_gb300.build)")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, I32, U32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_uint32
        L.mq_last_error.restype = ctypes.c_char_p
        L.mq_q8_plane_bytes.argtypes = [I64, I64]
        L.mq_q8_plane_bytes.restype = ctypes.c_size_t
        L.mq_q8_plane_layout.argtypes = [I64, I64, ctypes.POINTER(PlaneLayout)]
        L.mq_quantize_q8.argtypes = [P, I64, I64, P, ctypes.c_float, P, P]
        L.mq_quantize_swiglu_q8.argtypes = [P, P, I64, I64, P, P]
        L.mq_quantize_q8_ex.argtypes = [P, I64, I64, P, ctypes.c_float, ctypes.c_uint, P, P]
        L.mq_quantize_swiglu_q8_ex.argtypes = [P, P, I64, I64, ctypes.c_uint, P, P]
        for name in ("mq_gemm_q4k", "mq_gemm_q6k", "mq_gemv_q4k", "mq_gemv_q6k", "mq_gemv_q5k", "mq_gemm_q5k",
                     "mq_gemv_q4_0", "mq_gemv_q4_1", "mq_gemv_q5_0", "mq_gemv_q5_1", "mq_gemv_q8_0",
                     "mq_gemm_q4_0", "mq_gemm_q4_1", "mq_gemm_q5_0", "mq_gemm_q5_1", "mq_gemm_q8_0",
                     "mq_gemm_small_q4k", "mq_gemm_small_q5k", "mq_gemm_small_q6k"):
            getattr(L, name).argtypes = [P, I64, I64, P, I64, P, P]
        L.mq_gemm_q4k_swiglu.argtypes = [P, P, I64, I64, P, I64, P, P]
        for name in ("mq_gemv_grouped_q4k", "mq_gemv_grouped_q5k", "mq_gemv_grouped_q6k"):
            getattr(L, name).argtypes = [ctypes.POINTER(GemvJob), I32, I64, I64, P]
        for name in ("mq_gemv_grouped_x_q4k", "mq_gemv_grouped_x_q5k", "mq_gemv_grouped_x_q6k"):
            getattr(L, name).argtypes = [ctypes.POINTER(GemvXJob), I32, I64, P]
        L.mq_quantize_q8_grouped.argtypes = [ctypes.POINTER(QuantizeJob), I32, I64, I64, ctypes.c_uint, P]
        L.mq_device_status.argtypes = [P]
        L.mq_debug_blockdots.argtypes = [I32, P, I64, I64, P, I64, P, I64, I64, I64, I64, P, P]
        L.mq_debug_forced_timeout.argtypes = [U32, P]
        for name in header_functions():
            if name not in ("mq_last_error", "mq_q8_plane_bytes"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def last_error() -> str:
    return lib().mq_last_error().decode()


def _check(rc: int):
    if rc != MQ_OK:
        raise MQError(rc, last_error())
    return rc


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ---------------------------------------------------------------------------------- plane ---

def mq_q8_plane_bytes(M: int, K: int) -> int:
    return lib().mq_q8_plane_bytes(M, K)


def mq_q8_plane_layout(M: int, K: int) -> dict:
    out = PlaneLayout()
    _check(lib().mq_q8_plane_layout(M, K, ctypes.byref(out)))
    return {f: getattr(out, f) for f, _ in PlaneLayout._fields_}


def alloc_plane(M: int, K: int, device="cuda"):
    """A uint8 device tensor big enough for the plane (torch blocks are 512-byte aligned)."""
    import torch
    t = torch.empty(max(mq_q8_plane_bytes(M, K), 1), dtype=torch.uint8, device=device)
    assert t.data_ptr() % 256 == 0
    return t


def plane_views(plane, M: int, K: int, with_ds: bool = False):
    """(q16 f16 [M,K], q8 int8 [M,K], d f32 [K/32,M], s int32 [K/32,M][, ds f32 [M,2K/32]]) views."""
    import torch
    L = mq_q8_plane_layout(M, K)
    nb = K // 32
    q16 = plane[L["off_q16"]:L["off_q16"] + 2 * M * K].view(torch.float16).view(M, K)
    q8 = plane[L["off_q8"]:L["off_q8"] + M * K].view(torch.int8).view(M, K)
    d = plane[L["off_d"]:L["off_d"] + 4 * nb * M].view(torch.float32).view(nb, M)
    s = plane[L["off_s"]:L["off_s"] + 4 * nb * M].view(torch.int32).view(nb, M)
    if not with_ds:
        return q16, q8, d, s
    ds = plane[L["off_ds"]:L["off_ds"] + 8 * nb * M].view(torch.float32).view(M, 2 * nb)
    return q16, q8, d, s, ds


# ------------------------------------------------------------------------------ entry points ---

def mq_quantize_q8(x, M: int, K: int, rms_w, eps: float, plane, stream=None):
    return _check(lib().mq_quantize_q8(_ptr(x), M, K, _ptr(rms_w), float(eps), _ptr(plane), _stream(stream)))


def mq_quantize_swiglu_q8(gate, up, M: int, K: int, plane, stream=None):
    return _check(lib().mq_quantize_swiglu_q8(_ptr(gate), _ptr(up), M, K, _ptr(plane), _stream(stream)))


def mq_quantize_q8_ex(x, M: int, K: int, rms_w, eps: float, sections: int, plane, stream=None):
    return _check(lib().mq_quantize_q8_ex(_ptr(x), M, K, _ptr(rms_w), float(eps), sections, _ptr(plane),
                                          _stream(stream)))


def mq_quantize_swiglu_q8_ex(gate, up, M: int, K: int, sections: int, plane, stream=None):
    return _check(lib().mq_quantize_swiglu_q8_ex(_ptr(gate), _ptr(up), M, K, sections, _ptr(plane), _stream(stream)))


def _matmul(name, w, N, K, plane, M, y, stream):
    return _check(getattr(lib(), name)(_ptr(w), N, K, _ptr(plane), M, _ptr(y), _stream(stream)))


def mq_gemm_q4k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q4k", w, N, K, plane, M, y, stream)


def mq_gemm_q6k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q6k", w, N, K, plane, M, y, stream)


def mq_gemv_q4k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q4k", w, N, K, plane, M, y, stream)


def mq_gemv_q6k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q6k", w, N, K, plane, M, y, stream)


def mq_gemv_q5k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q5k", w, N, K, plane, M, y, stream)


def mq_gemm_q5k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q5k", w, N, K, plane, M, y, stream)


def mq_gemv_q4_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q4_0", w, N, K, plane, M, y, stream)


def mq_gemv_q4_1(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q4_1", w, N, K, plane, M, y, stream)


def mq_gemv_q5_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q5_0", w, N, K, plane, M, y, stream)


def mq_gemv_q5_1(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q5_1", w, N, K, plane, M, y, stream)


def mq_gemv_q8_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemv_q8_0", w, N, K, plane, M, y, stream)


def mq_gemm_q4_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q4_0", w, N, K, plane, M, y, stream)


def mq_gemm_q4_1(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q4_1", w, N, K, plane, M, y, stream)


def mq_gemm_q5_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q5_0", w, N, K, plane, M, y, stream)


def mq_gemm_q5_1(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q5_1", w, N, K, plane, M, y, stream)


def mq_gemm_q8_0(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_q8_0", w, N, K, plane, M, y, stream)


def _gemv_grouped(name, jobs, K, M, stream):
    arr = (GemvJob * max(1, len(jobs)))(*[GemvJob(_ptr(w), N, _ptr(p), _ptr(y)) for (w, N, p, y) in jobs])
    return _check(getattr(lib(), name)(arr, len(jobs), K, M, _stream(stream)))


def mq_gemv_grouped_q4k(jobs, K: int, M: int, stream=None):
    """jobs: a list of (w, N, plane, y); one launch for all of them."""
    return _gemv_grouped("mq_gemv_grouped_q4k", jobs, K, M, stream)


def mq_gemv_grouped_q5k(jobs, K: int, M: int, stream=None):
    return _gemv_grouped("mq_gemv_grouped_q5k", jobs, K, M, stream)


def mq_gemv_grouped_q6k(jobs, K: int, M: int, stream=None):
    return _gemv_grouped("mq_gemv_grouped_q6k", jobs, K, M, stream)


def _gemv_grouped_x(name, jobs, K, stream):
    arr = (GemvXJob * max(1, len(jobs)))(*[GemvXJob(_ptr(w), N, _ptr(x), _ptr(y)) for (w, N, x, y) in jobs])
    return _check(getattr(lib(), name)(arr, len(jobs), K, _stream(stream)))


def mq_gemv_grouped_x_q4k(jobs, K: int, stream=None):
    """jobs: a list of (w, N, x, y) for one token (x f32 [K]); the activations are quantized in the
    kernel, one launch for all of them."""
    return _gemv_grouped_x("mq_gemv_grouped_x_q4k", jobs, K, stream)


def mq_gemv_grouped_x_q5k(jobs, K: int, stream=None):
    return _gemv_grouped_x("mq_gemv_grouped_x_q5k", jobs, K, stream)


def mq_gemv_grouped_x_q6k(jobs, K: int, stream=None):
    return _gemv_grouped_x("mq_gemv_grouped_x_q6k", jobs, K, stream)


def mq_quantize_q8_grouped(jobs, M: int, K: int, sections: int, stream=None):
    """jobs: a list of (x, plane); the plain quantizer over all of them in one launch."""
    arr = (QuantizeJob * max(1, len(jobs)))(*[QuantizeJob(_ptr(x), _ptr(p)) for (x, p) in jobs])
    return _check(lib().mq_quantize_q8_grouped(arr, len(jobs), M, K, sections, _stream(stream)))


def mq_gemm_small_q4k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_small_q4k", w, N, K, plane, M, y, stream)


def mq_gemm_small_q5k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_small_q5k", w, N, K, plane, M, y, stream)


def mq_gemm_small_q6k(w, N: int, K: int, plane, M: int, y, stream=None):
    return _matmul("mq_gemm_small_q6k", w, N, K, plane, M, y, stream)


def mq_gemm_q4k_swiglu(w_gate, w_up, F: int, K: int, plane_in, M: int, plane_out, stream=None):
    return _check(lib().mq_gemm_q4k_swiglu(_ptr(w_gate), _ptr(w_up), F, K, _ptr(plane_in), M, _ptr(plane_out),
                                           _stream(stream)))


def mq_device_status(stream=None):
    return _check(lib().mq_device_status(_stream(stream)))


def mq_debug_blockdots(op: int, w, N: int, K: int, plane, M: int, y, m0: int, m_cnt: int, n0: int, n_cnt: int,
                       I_out, stream=None):
    return _check(lib().mq_debug_blockdots(op, _ptr(w), N, K, _ptr(plane), M, _ptr(y), m0, m_cnt, n0, n_cnt,
                                           _ptr(I_out), _stream(stream)))


def mq_debug_forced_timeout(timeout_us: int, stream=None):
    return _check(lib().mq_debug_forced_timeout(timeout_us, _stream(stream)))


# ------------------------------------------------------------------------------- convenience ---

GEMM = {"q4k": mq_gemm_q4k, "q6k": mq_gemm_q6k, "q5k": mq_gemm_q5k, "q4_0": mq_gemm_q4_0, "q4_1": mq_gemm_q4_1,
        "q5_0": mq_gemm_q5_0, "q5_1": mq_gemm_q5_1, "q8_0": mq_gemm_q8_0}
GEMV = {"q4k": mq_gemv_q4k, "q6k": mq_gemv_q6k, "q5k": mq_gemv_q5k, "q4_0": mq_gemv_q4_0, "q4_1": mq_gemv_q4_1,
        "q5_0": mq_gemv_q5_0, "q5_1": mq_gemv_q5_1, "q8_0": mq_gemv_q8_0}
GEMV_GROUPED = {"q4k": mq_gemv_grouped_q4k, "q5k": mq_gemv_grouped_q5k, "q6k": mq_gemv_grouped_q6k}
GEMV_GROUPED_X = {"q4k": mq_gemv_grouped_x_q4k, "q5k": mq_gemv_grouped_x_q5k, "q6k": mq_gemv_grouped_x_q6k}
# the small-M band (1 <= M <= 32) on the tensor cores, k-quant weights
GEMM_SMALL = {"q4k": mq_gemm_small_q4k, "q5k": mq_gemm_small_q5k, "q6k": mq_gemm_small_q6k}
SMALL_MAX_M = 32
# the fewest tokens at which the size dispatch prefers the small-M kernel to the GEMV: measured on a
# 152064 x 3584 LM head (GB300), the GEMV's time grows with its passes over W (8 tokens a pass for
# Q4_K / Q5_K, 4 for Q6_K) while the small-M kernel's is flat up to 32 tokens; Q4_K: GEMV 0.168 ms at
# 5 tokens, 0.256 at 8, small-M 0.213; Q6_K (int8 scales over the whole range): GEMV 0.168 at 4, 0.334
# at 8 (two passes), 0.5 at 9 (three), small-M 0.348
SMALL_MIN_M = {"q4k": 7, "q5k": 7, "q6k": 9}
# debug op of each (kind, format) for mq_debug_blockdots
DEBUG_OP = {("gemm", "q4k"): 0, ("gemm", "q6k"): 1, ("gemv", "q4k"): 2, ("gemv", "q6k"): 3, ("gemv", "q5k"): 4,
            ("gemm", "q5k"): 5, ("gemv", "q4_0"): 6, ("gemv", "q4_1"): 7, ("gemv", "q5_0"): 8, ("gemv", "q5_1"): 9,
            ("gemv", "q8_0"): 10, ("gemm", "q4_0"): 11, ("gemm", "q4_1"): 12, ("gemm", "q5_0"): 13,
            ("gemm", "q5_1"): 14, ("gemm", "q8_0"): 15, ("small", "q4k"): 16, ("small", "q6k"): 17,
            ("small", "q5k"): 18}


def matmul_path(fmt: str, M: int) -> str:
    """The entry point family the size dispatch picks: the pages' gate (MMVQ for one token, MMQ from 16),
    with the band up to 32 tokens on the small-M tensor-core kernel where the format has one and it is
    the faster path (SMALL_MIN_M[fmt] .. 32 tokens)."""
    if fmt in GEMM_SMALL:
        if M < SMALL_MIN_M[fmt]:
            return "gemv"
        return "small" if M <= SMALL_MAX_M else "gemm"
    return "gemv" if M < 16 else "gemm"


def matmul(fmt: str, w, N: int, K: int, plane, M: int, y, stream=None):
    """Size dispatch (matmul_path): k-quants take the GEMV below SMALL_MIN_M tokens, the small-M
    tensor-core GEMM up to 32 tokens and the GEMM beyond; the 32-value formats take the GEMV below
    16 tokens and the GEMM from 16 on."""
    table = {"gemv": GEMV, "gemm": GEMM, "small": GEMM_SMALL}[matmul_path(fmt, M)]
    return table[fmt](w, N, K, plane, M, y, stream)
