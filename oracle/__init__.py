"""CPU oracle for the k-quant (Q4_K / Q5_K / Q6_K) and 32-value block (Q4_0 / Q4_1 / Q5_0 /
Q5_1 / Q8_0) x Q8 matmul path (numpy front end over plain C).

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the bench's ``cpu_baseline`` / ``--impl reference`` legs, never by the
package.  It shares no code with the CUDA library.

Every function here is a thin marshalling layer over ``mq_oracle.c`` (the
arithmetic, and the citation of the passage each step follows, live there), or
a composition of such functions (``gate_up_swiglu_q8``: two matmuls rounded to
f32, then the SwiGLU producer).
Arrays use the oracle's own logical layouts:

* weights: raw GGML block bytes, ``[N, K/256, B]`` with B = 144 (Q4_K), 176 (Q5_K), 210 (Q6_K),
  or ``[N, K/32, b]`` with b = 18 (Q4_0), 20 (Q4_1), 22 (Q5_0), 24 (Q5_1), 34 (Q8_0)
* Q8 plane: ``q`` int8 ``[M, K]``, ``d`` f32 ``[M, K/32]``, ``S`` int32 ``[M, K/32]``
* outputs: f64 ``[len(ms), len(ns)]`` for the listed (token, row) index pairs

Every oracle function is pinned by ``tests/test_oracle_*.py`` against hand-built
blocks, closed forms, invariants and brute force; none is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build_oracle

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = build_oracle.build()
        L = ctypes.CDLL(path)
        P, I64, F32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float
        L.oq_half_to_double.argtypes = [ctypes.c_uint16]
        L.oq_half_to_double.restype = ctypes.c_double
        L.oq_q4k_fields.argtypes = [P, P, P, P, P, P]
        L.oq_q5k_fields.argtypes = [P, P, P, P, P, P]
        L.oq_q5k_dequant.argtypes = [P, I64, I64, P]
        L.oq_q6k_fields.argtypes = [P, P, P, P]
        L.oq_q4k_dequant.argtypes = [P, I64, I64, P]
        L.oq_q6k_dequant.argtypes = [P, I64, I64, P]
        L.oq_rmsnorm.argtypes = [P, I64, I64, P, F32, P]
        L.oq_quantize_q8.argtypes = [P, I64, I64, P, P, P]
        L.oq_exp_f32.argtypes = [F32]
        L.oq_exp_f32.restype = F32
        L.oq_swiglu.argtypes = [P, P, I64, I64, P]
        for f in (L.oq_q4k_blockdots, L.oq_q5k_blockdots, L.oq_q6k_blockdots):
            f.argtypes = [P, I64, I64, P, I64, P, I64, P, I64, P, P]
        for f in (L.oq_q4k_matmul, L.oq_q5k_matmul, L.oq_q6k_matmul):
            f.argtypes = [P, I64, I64, P, P, P, I64, P, I64, P, I64, P]
        C = ctypes.c_int
        L.oq_b32_fields.argtypes = [C, P, P, P, P]
        L.oq_b32_dequant.argtypes = [C, P, I64, I64, P]
        L.oq_b32_blockdots.argtypes = [C, P, I64, P, P, I64, P, I64, P]
        L.oq_b32_matmul.argtypes = [C, P, I64, P, P, P, P, I64, P, I64, P]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


BLOCK_BYTES = {"q4k": 144, "q5k": 176, "q6k": 210}
# the 32-value block formats: bytes per block and their id in mq_oracle.c (C9)
B32 = {"q4_0": (18, 0), "q4_1": (20, 1), "q5_0": (22, 2), "q5_1": (24, 3), "q8_0": (34, 4)}


def _weights(w: np.ndarray, fmt: str):
    w = np.ascontiguousarray(w, dtype=np.uint8)
    n = w.shape[0]
    per_row = w.size // n
    if fmt in B32:
        nb = per_row // B32[fmt][0]
        assert nb * B32[fmt][0] == per_row
        return w, n, nb * 32
    nb = per_row // BLOCK_BYTES[fmt]
    assert nb * BLOCK_BYTES[fmt] == per_row
    return w, n, nb * 256


def half_to_double(bits: int) -> float:
    return lib().oq_half_to_double(int(bits) & 0xFFFF)


def q4k_fields(block: np.ndarray):
    """Decode one 144-byte Q4_K block -> (d, dmin, sc[8], m[8], q[256])."""
    blk = np.ascontiguousarray(block, dtype=np.uint8).reshape(144)
    d, dmin = ctypes.c_double(), ctypes.c_double()
    sc, mn, q = np.zeros(8, np.int32), np.zeros(8, np.int32), np.zeros(256, np.int32)
    lib().oq_q4k_fields(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return d.value, dmin.value, sc, mn, q


def q5k_fields(block: np.ndarray):
    """Decode one 176-byte Q5_K block -> (d, dmin, sc[8], m[8], q[256])."""
    blk = np.ascontiguousarray(block, dtype=np.uint8).reshape(176)
    d, dmin = ctypes.c_double(), ctypes.c_double()
    sc, mn, q = np.zeros(8, np.int32), np.zeros(8, np.int32), np.zeros(256, np.int32)
    lib().oq_q5k_fields(_p(blk), ctypes.byref(d), ctypes.byref(dmin), _p(sc), _p(mn), _p(q))
    return d.value, dmin.value, sc, mn, q


def q6k_fields(block: np.ndarray):
    """Decode one 210-byte Q6_K block -> (d, sc[16], q[256])."""
    blk = np.ascontiguousarray(block, dtype=np.uint8).reshape(210)
    d = ctypes.c_double()
    sc, q = np.zeros(16, np.int32), np.zeros(256, np.int32)
    lib().oq_q6k_fields(_p(blk), ctypes.byref(d), _p(sc), _p(q))
    return d.value, sc, q


def b32_fields(block: np.ndarray, fmt: str):
    """Decode one 32-value block -> (d, m, iq[32]) with value = d * iq + m."""
    nbytes, fid = B32[fmt]
    blk = np.ascontiguousarray(block, dtype=np.uint8).reshape(nbytes)
    d, m = ctypes.c_double(), ctypes.c_double()
    iq = np.zeros(32, np.int32)
    lib().oq_b32_fields(fid, _p(blk), ctypes.byref(d), ctypes.byref(m), _p(iq))
    return d.value, m.value, iq


def dequantize(w: np.ndarray, fmt: str) -> np.ndarray:
    """Dequantized weights [N, K] in f64."""
    w, n, k = _weights(w, fmt)
    out = np.empty((n, k), np.float64)
    if fmt in B32:
        lib().oq_b32_dequant(B32[fmt][1], _p(w), n, k, _p(out))
        return out
    {"q4k": lib().oq_q4k_dequant, "q5k": lib().oq_q5k_dequant, "q6k": lib().oq_q6k_dequant}[fmt](_p(w), n, k, _p(out))
    return out


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    m, k = x.shape
    y = np.empty_like(x)
    lib().oq_rmsnorm(_p(x), m, k, _p(w), float(eps), _p(y))
    return y


def exp_f32(x: float) -> float:
    return float(lib().oq_exp_f32(float(x)))


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    """y = silu(g) * u in f32 (C8)."""
    g = np.ascontiguousarray(g, dtype=np.float32)
    u = np.ascontiguousarray(u, dtype=np.float32)
    assert g.shape == u.shape and g.ndim == 2
    y = np.empty_like(g)
    lib().oq_swiglu(_p(g), _p(u), g.shape[0], g.shape[1], _p(y))
    return y


def quantize_swiglu_q8(g: np.ndarray, u: np.ndarray):
    """Q8 plane of silu(g) * u -> (q, d, S)."""
    return quantize_q8(swiglu(g, u))


def gate_up_swiglu_q8(w_gate: np.ndarray, w_up: np.ndarray, fmt: str, plane, ms=None, threads: int = 1):
    """Q8 plane of silu(G) * U for the FFN's gate and up projections of one plane: G and U are
    C6 matmuls (f64), each rounded once to f32 -- the f32 [M][F] form in which the SwiGLU
    producer (C8) takes them -- then C8.  Rows ``ms`` of the plane (all by default), all F
    outputs -> (q, d, S).  A composition of pinned functions; no arithmetic of its own but
    the f64 -> f32 rounding."""
    g = matmul(w_gate, fmt, plane, ms, None, threads).astype(np.float32)
    u = matmul(w_up, fmt, plane, ms, None, threads).astype(np.float32)
    return quantize_swiglu_q8(g, u)


def quantize_q8(x: np.ndarray, rms_w: np.ndarray | None = None, eps: float = 1e-6):
    """Q8 plane of x (optionally after the RMSNorm producer) -> (q, d, S)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if rms_w is not None:
        x = rmsnorm(x, rms_w, eps)
    m, k = x.shape
    assert k % 32 == 0
    q = np.empty((m, k), np.int8)
    d = np.empty((m, k // 32), np.float32)
    S = np.empty((m, k // 32), np.int32)
    lib().oq_quantize_q8(_p(x), m, k, _p(q), _p(d), _p(S))
    return q, d, S


def _idx(v, limit):
    v = np.ascontiguousarray(np.arange(limit) if v is None else v, dtype=np.int64)
    assert v.ndim == 1 and (v.size == 0 or (v.min() >= 0 and v.max() < limit))
    return v


def blockdots(w: np.ndarray, fmt: str, q: np.ndarray, ms=None, ns=None):
    """Integer checkpoint I[len(ms), len(ns), K/32] (and the raw dots D)."""
    w, n, k = _weights(w, fmt)
    q = np.ascontiguousarray(q, dtype=np.int8)
    m = q.shape[0]
    assert q.shape[1] == k
    ms, ns = _idx(ms, m), _idx(ns, n)
    I = np.zeros((ms.size, ns.size, k // 32), np.int32)
    if fmt in B32:
        lib().oq_b32_blockdots(B32[fmt][1], _p(w), k, _p(q), _p(ms), ms.size, _p(ns), ns.size, _p(I))
        return I, None
    if fmt in ("q4k", "q5k"):
        D = np.zeros_like(I)
        fn = lib().oq_q4k_blockdots if fmt == "q4k" else lib().oq_q5k_blockdots
        fn(_p(w), n, k, _p(q), m, _p(ms), ms.size, _p(ns), ns.size, _p(I), _p(D))
    else:
        D = np.zeros((ms.size, ns.size, k // 32, 2), np.int32)
        lib().oq_q6k_blockdots(_p(w), n, k, _p(q), m, _p(ms), ms.size, _p(ns), ns.size, _p(I), _p(D))
    return I, D


def matmul(w: np.ndarray, fmt: str, plane, ms=None, ns=None, threads: int = 1) -> np.ndarray:
    """Y[len(ms), len(ns)] (f64) from weight bytes and an oracle Q8 plane (q, d, S).

    ``threads`` > 1 splits the row list ``ns`` over Python threads (the C call
    releases the GIL); each thread runs the same plain C loop on its slice.
    """
    w, n, k = _weights(w, fmt)
    q, d, S = (np.ascontiguousarray(a) for a in plane)
    m = q.shape[0]
    assert q.shape == (m, k) and d.shape == (m, k // 32) and S.shape == (m, k // 32)
    assert q.dtype == np.int8 and d.dtype == np.float32 and S.dtype == np.int32
    ms, ns = _idx(ms, m), _idx(ns, n)
    if fmt in B32:
        fid = B32[fmt][1]
        fn = lambda *a: lib().oq_b32_matmul(fid, a[0], a[2], a[3], a[4], a[5], *a[7:])   # no N, M
    else:
        fn = {"q4k": lib().oq_q4k_matmul, "q5k": lib().oq_q5k_matmul, "q6k": lib().oq_q6k_matmul}[fmt]
    if threads <= 1 or ns.size < 2:
        y = np.empty((ms.size, ns.size), np.float64)
        fn(_p(w), n, k, _p(q), _p(d), _p(S), m, _p(ms), ms.size, _p(ns), ns.size, _p(y))
        return y
    parts = np.array_split(ns, min(threads, ns.size))

    def run(part):
        part = np.ascontiguousarray(part)
        yp = np.empty((ms.size, part.size), np.float64)
        fn(_p(w), n, k, _p(q), _p(d), _p(S), m, _p(ms), ms.size, _p(part), part.size, _p(yp))
        return yp

    with ThreadPoolExecutor(len(parts)) as ex:
        return np.concatenate(list(ex.map(run, parts)), axis=1)
