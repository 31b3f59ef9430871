"""Host-side tests of the C ABI: the library loads, exports every symbol include/mq.h
declares, lays out the Q8 plane as documented, and rejects bad arguments before any
CUDA call (these run without a GPU)."""
import ctypes
import subprocess
import sys

import pytest

from quantized_q8_activation_quantize_gb300 import binding as B
from quantized_q8_activation_quantize_gb300 import build as mqbuild


@pytest.fixture(scope="session")
def L():
    mqbuild.build()
    return B.lib()


EXPECTED = {"mq_last_error", "mq_q8_plane_bytes", "mq_q8_plane_layout", "mq_quantize_q8", "mq_quantize_swiglu_q8",
            "mq_gemm_q4k",
            "mq_gemm_q6k", "mq_gemv_q4k", "mq_gemv_q6k", "mq_gemv_q5k", "mq_gemm_q5k", "mq_device_status", "mq_debug_blockdots",
            "mq_debug_forced_timeout", "mq_gemv_q4_0", "mq_gemv_q4_1", "mq_gemv_q5_0", "mq_gemv_q5_1", "mq_gemv_q8_0",
            "mq_gemm_q4_0", "mq_gemm_q4_1", "mq_gemm_q5_0", "mq_gemm_q5_1", "mq_gemm_q8_0", "mq_gemm_q4k_swiglu",
            "mq_quantize_q8_ex", "mq_quantize_swiglu_q8_ex", "mq_gemm_small_q4k", "mq_gemm_small_q5k",
            "mq_gemm_small_q6k", "mq_gemv_grouped_q4k", "mq_gemv_grouped_q5k", "mq_gemv_grouped_q6k",
            "mq_quantize_q8_grouped", "mq_gemv_grouped_x_q4k", "mq_gemv_grouped_x_q5k", "mq_gemv_grouped_x_q6k"}


def test_header_declares_the_boundary():
    assert set(B.header_functions()) == EXPECTED


def test_library_exports_every_declared_symbol(L):
    for name in B.header_functions():
        assert hasattr(L, name), name
    # and nothing else with C linkage leaks out under the mq_ prefix
    out = subprocess.run(["nm", "-D", "--defined-only", B.LIB_PATH], capture_output=True, text=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.split() and ln.split()[-1].startswith("mq_")}
    assert exported == EXPECTED


def test_binding_mirrors_every_entry_point():
    # the Python binding has one function of the same name per C entry point (the error-string
    # accessor is read through MQError instead), and the format / op tables cover the same calls
    for name in B.header_functions():
        if name == "mq_last_error":
            continue
        assert callable(getattr(B, name, None)), name
    assert set(B.GEMM) <= set(B.GEMV)
    tables = {"gemm": (B.GEMM, "mq_gemm_"), "gemv": (B.GEMV, "mq_gemv_"), "small": (B.GEMM_SMALL, "mq_gemm_small_")}
    for (path, fmt), op in B.DEBUG_OP.items():
        table, prefix = tables[path]
        assert table[fmt].__name__ == prefix + fmt, (path, fmt, op)
    assert sorted(B.DEBUG_OP.values()) == list(range(len(B.DEBUG_OP)))


@pytest.mark.parametrize("M,K", [(0, 256), (1, 256), (8, 512), (3314, 3584), (3314, 18944), (7, 768)])
def test_plane_layout(L, M, K):
    lay = B.mq_q8_plane_layout(M, K)
    nb = K // 32
    secs = [("off_q16", 2 * M * K), ("off_q8", M * K), ("off_d", 4 * nb * M), ("off_s", 4 * nb * M),
            ("off_ds", 8 * nb * M)]
    end = 0
    for name, size in secs:
        assert lay[name] % 256 == 0 and lay[name] >= end
        end = lay[name] + size
    assert lay["total_bytes"] >= end and lay["total_bytes"] % 256 == 0 and lay["total_bytes"] - end < 256
    assert B.mq_q8_plane_bytes(M, K) == lay["total_bytes"]


@pytest.mark.parametrize("M,K", [(-1, 256), (4, 0), (4, 100), (4, 300), (4, -256), (1 << 31, 256)])
def test_plane_layout_rejects_bad_shapes(L, M, K):
    assert B.mq_q8_plane_bytes(M, K) == 0
    with pytest.raises(B.MQError) as e:
        B.mq_q8_plane_layout(M, K)
    assert e.value.status == B.MQ_ERR_SHAPE


def _rc(fn, *args):
    return fn(*args)


def test_quantize_argument_errors(L):
    q = L.mq_quantize_q8
    assert q(16, 4, 100, None, 0.0, 256, None) == B.MQ_ERR_SHAPE
    assert q(16, -1, 256, None, 0.0, 256, None) == B.MQ_ERR_ARG
    assert q(16, 0, 256, None, 0.0, 256, None) == B.MQ_OK            # empty: nothing to do
    assert q(None, 4, 256, None, 0.0, 256, None) == B.MQ_ERR_ARG
    assert "NULL" in B.last_error()
    assert q(16, 4, 256, None, 0.0, None, None) == B.MQ_ERR_ARG
    assert q(20, 4, 256, None, 0.0, 256, None) == B.MQ_ERR_ALIGN      # x not 16-byte aligned
    assert q(16, 4, 256, 24, 1e-6, 256, None) == B.MQ_ERR_ALIGN      # rms_w not 16-byte aligned
    assert q(16, 4, 256, None, 0.0, 128, None) == B.MQ_ERR_ALIGN     # plane not 256-byte aligned
    assert q(16, 4, 256, 32, float("nan"), 256, None) == B.MQ_ERR_ARG
    assert q(16, 4, 256, 32, -1.0, 256, None) == B.MQ_ERR_ARG
    assert q(1 << 20, 4, 256, None, 0.0, (1 << 20) + 256, None) == B.MQ_ERR_ARG      # plane over x
    assert q(1 << 20, 4, 256, 1 << 24, 1e-6, (1 << 24) - 256, None) == B.MQ_ERR_ARG  # plane over rms_w


def test_plane_sections_argument_errors(L):
    q, g = L.mq_quantize_q8_ex, L.mq_quantize_swiglu_q8_ex
    for bad in (0, 8, 0xffffffff):
        assert q(16, 4, 256, None, 0.0, bad, 256, None) == B.MQ_ERR_ARG
        assert "sections" in B.last_error()
        assert g(16, 32, 4, 256, bad, 256, None) == B.MQ_ERR_ARG
    assert q(16, 0, 256, None, 0.0, B.PLANE_FOR_GEMV, 256, None) == B.MQ_OK      # empty
    assert q(16, 4, 100, None, 0.0, B.PLANE_FOR_GEMM, 256, None) == B.MQ_ERR_SHAPE
    assert g(16, 32, 0, 256, B.PLANE_ALL, 256, None) == B.MQ_OK
    assert (B.PLANE_FOR_GEMM, B.PLANE_FOR_GEMV) == (B.PLANE_Q16 | B.PLANE_DS, B.PLANE_Q8)


def test_swiglu_quantize_argument_errors(L):
    q = L.mq_quantize_swiglu_q8
    assert q(16, 32, 4, 100, 256, None) == B.MQ_ERR_SHAPE
    assert q(16, 32, -1, 256, 256, None) == B.MQ_ERR_ARG
    assert q(16, 32, 0, 256, 256, None) == B.MQ_OK                     # empty: nothing to do
    assert q(None, 32, 4, 256, 256, None) == B.MQ_ERR_ARG
    assert q(16, None, 4, 256, 256, None) == B.MQ_ERR_ARG
    assert q(16, 32, 4, 256, None, None) == B.MQ_ERR_ARG
    assert q(20, 32, 4, 256, 256, None) == B.MQ_ERR_ALIGN              # gate not 16-byte aligned
    assert q(16, 36, 4, 256, 256, None) == B.MQ_ERR_ALIGN              # up not 16-byte aligned
    assert q(16, 32, 4, 256, 128, None) == B.MQ_ERR_ALIGN              # plane not 256-byte aligned
    assert q(1 << 20, 1 << 24, 4, 256, (1 << 24) + 256, None) == B.MQ_ERR_ARG   # plane over up


@pytest.mark.parametrize("name", ["mq_gemm_q4k", "mq_gemm_q6k", "mq_gemv_q4k", "mq_gemv_q6k", "mq_gemv_q5k",
                                  "mq_gemm_q5k", "mq_gemv_q4_0", "mq_gemv_q4_1", "mq_gemv_q5_0", "mq_gemv_q5_1",
                                  "mq_gemv_q8_0", "mq_gemm_q4_0", "mq_gemm_q4_1", "mq_gemm_q5_0", "mq_gemm_q5_1",
                                  "mq_gemm_q8_0", "mq_gemm_small_q4k", "mq_gemm_small_q5k", "mq_gemm_small_q6k"])
def test_matmul_argument_errors(L, name):
    f = getattr(L, name)
    assert f(16, 8, 300, 256, 4, 16, None) == B.MQ_ERR_SHAPE          # K % 256
    assert f(16, 8, 0, 256, 4, 16, None) == B.MQ_ERR_SHAPE
    assert f(16, -8, 256, 256, 4, 16, None) == B.MQ_ERR_ARG
    assert f(16, 8, 256, 256, -4, 16, None) == B.MQ_ERR_ARG
    assert f(16, 0, 256, 256, 4, 16, None) == B.MQ_OK                 # N == 0: empty
    assert f(16, 8, 256, 256, 0, 16, None) == B.MQ_OK                 # M == 0: empty
    assert f(None, 8, 256, 256, 4, 16, None) == B.MQ_ERR_ARG
    assert f(16, 8, 256, None, 4, 16, None) == B.MQ_ERR_ARG
    assert f(16, 8, 256, 256, 4, None, None) == B.MQ_ERR_ARG
    assert f(8, 8, 256, 256, 4, 16, None) == B.MQ_ERR_ALIGN           # weights need 16 B
    assert f(16, 8, 256, 64, 4, 16, None) == B.MQ_ERR_ALIGN           # plane needs 256 B
    assert f(16, 8, 256, 256, 4, 18, None) == B.MQ_ERR_ALIGN          # y needs 4 B
    assert f(16, 1 << 31, 256, 256, 4, 16, None) == B.MQ_ERR_SHAPE
    # the output may overlap neither the plane nor the weights
    assert f(1 << 20, 8, 256, 1 << 24, 4, (1 << 24) + 64, None) == B.MQ_ERR_ARG
    assert f(1 << 20, 8, 256, 1 << 24, 4, (1 << 20) + 64, None) == B.MQ_ERR_ARG
    if "small" in name:                                                 # the band's limit
        assert f(16, 8, 256, 256, 33, 16, None) == B.MQ_ERR_SHAPE
    elif "gemm" in name:                                                # token tiles in grid.y
        assert f(16, 8, 256, 256, 65535 * 128 + 1, 16, None) == B.MQ_ERR_SHAPE


def test_size_dispatch():
    # the pages' gate: one token -> MMVQ; for the k-quants the GEMV while it is the faster path (below
    # SMALL_MIN_M tokens), then the small-M tensor-core GEMM up to 32 tokens, then MMQ; the 32-value
    # formats: MMVQ below 16 tokens and MMQ from 16
    for fmt in ("q4k", "q5k", "q6k"):
        lo = B.SMALL_MIN_M[fmt]
        assert 2 <= lo <= 16
        for m in range(1, lo):
            assert B.matmul_path(fmt, m) == "gemv"
        for m in range(lo, B.SMALL_MAX_M + 1):
            assert B.matmul_path(fmt, m) == "small"
        assert B.matmul_path(fmt, B.SMALL_MAX_M + 1) == "gemm"
    assert B.matmul_path("q8_0", 8) == "gemv" and B.matmul_path("q8_0", 16) == "gemm"


def test_grouped_argument_errors():
    # host-side validation of the grouped calls (no device needed): job counts, NULL tables, per-job
    # checks, and outputs overlapping another job's inputs or outputs
    L = B.lib()
    J = B.GemvJob
    jobs = (J * 2)(J(1 << 20, 8, 1 << 24, 1 << 28), J(1 << 21, 8, 1 << 25, (1 << 28) + 64))
    assert L.mq_gemv_grouped_q4k(jobs, 9, 256, 4, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_q4k(None, 2, 256, 4, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_q4k(jobs, 0, 256, 4, None) == B.MQ_OK
    assert L.mq_gemv_grouped_q4k(jobs, 2, 300, 4, None) == B.MQ_ERR_SHAPE
    assert L.mq_gemv_grouped_q6k(jobs, 2, 256, 4, None) == B.MQ_ERR_ARG     # job 0's y overlaps job 1's y
    assert "overlaps" in B.last_error()
    bad = (J * 1)(J(8, 8, 1 << 24, 1 << 28))
    assert L.mq_gemv_grouped_q5k(bad, 1, 256, 4, None) == B.MQ_ERR_ALIGN
    X = B.GemvXJob
    xj = (X * 2)(X(1 << 20, 8, 1 << 24, 1 << 28), X(1 << 21, 8, 1 << 25, (1 << 28) + 16))
    assert L.mq_gemv_grouped_x_q4k(xj, 9, 256, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_x_q4k(None, 2, 256, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_x_q4k(xj, 0, 256, None) == B.MQ_OK
    assert L.mq_gemv_grouped_x_q4k(xj, 2, 300, None) == B.MQ_ERR_SHAPE
    assert L.mq_gemv_grouped_x_q6k(xj, 2, 256, None) == B.MQ_ERR_ARG     # job 0's y overlaps job 1's y
    assert "overlaps" in B.last_error()
    over_x = (X * 1)(X(1 << 20, 64, 1 << 28, (1 << 28) + 512))           # y inside x
    assert L.mq_gemv_grouped_x_q5k(over_x, 1, 256, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_x_q5k((X * 1)(X(1 << 20, 8, (1 << 24) + 4, 1 << 28)), 1, 256, None) == B.MQ_ERR_ALIGN
    assert L.mq_gemv_grouped_x_q5k((X * 1)(X(1 << 20, 8, None, 1 << 28)), 1, 256, None) == B.MQ_ERR_ARG
    assert L.mq_gemv_grouped_x_q6k((X * 1)(X(1 << 20, -1, 1 << 24, 1 << 28)), 1, 256, None) == B.MQ_ERR_ARG
    Q = B.QuantizeJob
    q = (Q * 2)(Q(1 << 20, 1 << 24), Q(1 << 21, (1 << 24) + 256))
    assert L.mq_quantize_q8_grouped(q, 9, 4, 256, B.PLANE_ALL, None) == B.MQ_ERR_ARG
    assert L.mq_quantize_q8_grouped(q, 2, 4, 256, 0, None) == B.MQ_ERR_ARG
    assert L.mq_quantize_q8_grouped(q, 2, 4, 256, B.PLANE_ALL, None) == B.MQ_ERR_ARG   # planes overlap
    assert L.mq_quantize_q8_grouped(q, 2, 0, 256, B.PLANE_ALL, None) == B.MQ_OK


def test_debug_window_errors(L):
    d = L.mq_debug_blockdots
    assert d(16, 16, 8, 256, 256, 4, 16, 0, 1, 0, 1, 16, None) == B.MQ_ERR_ARG     # op
    assert d(-1, 16, 8, 256, 256, 4, 16, 0, 1, 0, 1, 16, None) == B.MQ_ERR_ARG
    assert d(0, 16, 8, 256, 256, 4, 16, 3, 2, 0, 1, 16, None) == B.MQ_ERR_ARG      # window past M
    assert d(0, 16, 8, 256, 256, 4, 16, 0, 1, 0, 0, 16, None) == B.MQ_ERR_ARG      # empty window
    assert d(0, 16, 8, 256, 256, 4, 16, 0, 1, 0, 1, None, None) == B.MQ_ERR_ARG
    assert L.mq_debug_forced_timeout(0, None) == B.MQ_ERR_ARG


def test_valid_call_without_a_device_fails_loudly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    rc = L.mq_gemm_q4k(1 << 20, 8, 256, 1 << 24, 4, 1 << 28, None)
    assert rc in (B.MQ_ERR_CUDA, B.MQ_ERR_DEVICE)
    assert B.last_error()
    with pytest.raises(B.MQError):
        B.mq_gemm_q4k(1 << 20, 8, 256, 1 << 24, 4, 1 << 28, stream=0)


def test_product_package_does_not_import_the_oracle():
    code = ("import sys, quantized_q8_activation_quantize_gb300 as p, quantized_q8_activation_quantize_gb300.inputs;"
            "import quantized_q8_activation_quantize_gb300.binding; print('oracle' in sys.modules)")
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, cwd=B.PKG + "/..")
    assert out.stdout.strip() == "False", out.stderr


def test_missing_library_raises(monkeypatch, tmp_path):
    monkeypatch.setattr(B, "_lib", None)
    monkeypatch.setattr(B, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(RuntimeError, match="not built"):
        B.lib()


def test_gate_up_swiglu_argument_errors(L):
    f = L.mq_gemm_q4k_swiglu          # (w_gate, w_up, F, K, plane_in, M, plane_out, stream)
    assert f(16, 16, 300, 256, 256, 4, 256, None) == B.MQ_ERR_SHAPE      # F % 256
    assert f(16, 16, 0, 256, 256, 4, 256, None) == B.MQ_OK            # F == 0: nothing to do
    assert f(16, 16, 65535 * 64 + 256, 256, 256, 4, 256, None) == B.MQ_ERR_SHAPE   # F past the grid limit
    assert f(16, 16, 256, 100, 256, 4, 256, None) == B.MQ_ERR_SHAPE      # K % 256
    assert f(16, 16, -256, 256, 256, 4, 256, None) == B.MQ_ERR_ARG
    assert f(16, 16, 256, 256, 256, -1, 256, None) == B.MQ_ERR_ARG
    assert f(16, 16, 256, 256, 256, 0, 256, None) == B.MQ_OK            # M == 0: nothing to do
    assert f(None, 16, 256, 256, 256, 4, 256, None) == B.MQ_ERR_ARG
    assert f(16, 16, 256, 256, 256, 4, None, None) == B.MQ_ERR_ARG
    assert f(24, 16, 256, 256, 256, 4, 256, None) == B.MQ_ERR_ALIGN     # w_gate not 16-byte aligned
    assert f(16, 24, 256, 256, 256, 4, 256, None) == B.MQ_ERR_ALIGN
    assert f(16, 16, 256, 256, 128, 4, 256, None) == B.MQ_ERR_ALIGN     # plane_in
    assert f(16, 16, 256, 256, 256, 4, 384, None) == B.MQ_ERR_ALIGN     # plane_out
    n_in = B.mq_q8_plane_bytes(4, 256)
    assert f(16, 16, 256, 256, 1 << 20, 4, 1 << 20, None) == B.MQ_ERR_ARG           # the same plane
    assert f(16, 16, 256, 256, 1 << 20, 4, (1 << 20) + 256, None) == B.MQ_ERR_ARG   # overlapping
    assert n_in > 256
    # plane_out over the weights
    assert f(1 << 20, 1 << 24, 256, 256, 1 << 28, 4, (1 << 20) + 256, None) == B.MQ_ERR_ARG
