"""GPU parity of mq_quantize_q8 (plain and RMSNorm-fused) against the oracle: the Q8 plane
must match bit for bit (int8 codes, f16 codes, f32 scales, int32 sums)."""
import numpy as np
import pytest

from quantized_q8_activation_quantize_gb300 import binding as B
from quantized_q8_activation_quantize_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,K", [(1, 256), (3, 512), (8, 512), (1, 18944), (37, 768), (130, 3584)])
def test_plain_quantize_bit_exact(M, K):
    x = inputs.activations(np.random.default_rng(M * 1000 + K), M, K)
    plane, got = G.gpu_plane(x)
    G.assert_plane_equal(got, G.oracle_plane(x))
    G.assert_ds_consistent(plane, M, K)


def test_tiny_and_qproj_planes():
    for cfg in (inputs.tiny_q4k(), inputs.qproj_prefill()):
        _, got = G.gpu_plane(cfg["x"])
        G.assert_plane_equal(got, G.oracle_plane(cfg["x"]))


def test_edge_values():
    # zero blocks, exact ties, the largest element, tiny and huge magnitudes, signed zeros
    M, K = 4, 256
    x = np.zeros((M, K), np.float32)
    x[0, 32:64] = [127.0, 0.5, -0.5, 2.5, -2.5, 1.5, -1.5, 126.5, -126.5, 0.49999997] + [0.0] * 22
    x[1, :] = np.linspace(-1e-30, 1e-30, K, dtype=np.float32)
    x[2, :] = np.linspace(-3e37, 3e37, K, dtype=np.float32)
    x[3, ::2] = -0.0
    x[3, 64:96] = 1.0
    x[3, 96:128] = -1e-45          # subnormal: amax/127 underflows to 0 -> all-zero block
    _, got = G.gpu_plane(x)
    G.assert_plane_equal(got, G.oracle_plane(x))


def test_rms_quantize_bit_exact_small():
    r = np.random.default_rng(3)
    # K <= 8192: rows in registers, 1 / 2 / 4 / 8 warps per token (K = 256 .. 1024, 1280 .. 2048,
    # 2304 .. 4096, 4352 .. 8192); above, the warp-per-token producer
    for M, K in ((1, 3584), (5, 256), (64, 3584), (6, 1536), (3, 2048), (9, 4096), (7, 8192), (2, 18432),
                 (3, 18944)):
        x = inputs.activations(r, M, K)
        w = inputs.rms_weight(r, K)
        plane, got = G.gpu_plane(x, w, 1e-6)
        G.assert_plane_equal(got, G.oracle_plane(x, w, 1e-6))
        G.assert_ds_consistent(plane, M, K)


def test_rms_scale_near_rounding_boundary():
    # Rows whose 1/sqrt(mean(x^2)) lies within 2^-40 of the midpoint between two f32 values: 255 ones
    # and one 1 - 2^-16 give mean 1 - 2^-23 + 2^-40, so r = 1 + 2^-24 - 2^-41 + O(2^-48), just below
    # the midpoint of 1 and 1 + 2^-23; r must round to 1 (the producer's f32 evaluation of r declines
    # such rows and evaluates them in f64).  Scaling a row by 2^k scales r by 2^-k exactly.  The rows
    # sit among random tokens, so the warps that take them also quantize ordinary rows.
    M, K = 40, 256
    r = np.random.default_rng(21)
    x = inputs.activations(r, M, K)
    w = np.ones(K, np.float32)
    near = np.ones(K, np.float32)
    near[100] = np.float32(1 - 2.0 ** -16)
    for i, k in enumerate((0, 3, -5, 10, -20)):
        x[7 * i + 1] = np.ldexp(np.roll(near, 31 * i), k).astype(np.float32)
    plane, got = G.gpu_plane(x, w, 0.0)
    G.assert_plane_equal(got, G.oracle_plane(x, w, 0.0))
    # the codes of a near row are those of the row itself (r rounds to 1, w = 1)
    _, plain = G.gpu_plane(x[1:2])
    assert np.array_equal(got[0][1], plain[0][0]) and np.array_equal(got[2][1], plain[2][0])


def test_ffn_prefill_full_size_planes():
    cfg = inputs.ffn_prefill()
    M = cfg["x_hidden"].shape[0]
    plane, got = G.gpu_plane(cfg["x_hidden"], cfg["rms_w"], float(cfg["eps"]))
    G.assert_plane_equal(got, G.oracle_plane(cfg["x_hidden"], cfg["rms_w"], float(cfg["eps"])))
    G.assert_ds_consistent(plane, M, inputs.HIDDEN)
    plane, got = G.gpu_plane(cfg["x_ffn"])
    G.assert_plane_equal(got, G.oracle_plane(cfg["x_ffn"]))
    G.assert_ds_consistent(plane, M, inputs.FFN)


def test_quantize_is_deterministic_and_reuses_plane():
    x = inputs.activations(np.random.default_rng(4), 33, 512)
    plane, a = G.gpu_plane(x)
    _, b = G.gpu_plane(x, plane=plane)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ---- plane sections (mq_quantize_q8_ex / mq_quantize_swiglu_q8_ex)

def _sections_of(plane, M, K):
    import torch
    q16, q8, d, s, ds = B.plane_views(plane, M, K, with_ds=True)
    return {"q16": q16.view(torch.int16).cpu().numpy(), "q8": q8.cpu().numpy(), "d": d.cpu().numpy().view(np.uint32),
            "s": s.cpu().numpy(), "ds": ds.cpu().numpy().view(np.uint32)}


@pytest.mark.parametrize("producer", ["plain", "rms", "swiglu"])
def test_plane_sections_write_only_what_is_asked(producer):
    import torch
    M, K = 37, 768
    r = np.random.default_rng(11)
    x = inputs.activations(r, M, K)
    w = inputs.rms_weight(r, K)
    g, u = inputs.swiglu_inputs(r, M, K)

    def run(sections, plane):
        if producer == "plain":
            B.mq_quantize_q8_ex(G.dev(x), M, K, None, 0.0, sections, plane)
        elif producer == "rms":
            B.mq_quantize_q8_ex(G.dev(x), M, K, G.dev(w), 1e-6, sections, plane)
        else:
            B.mq_quantize_swiglu_q8_ex(G.dev(g), G.dev(u), M, K, sections, plane)
        torch.cuda.synchronize()
        B.mq_device_status()

    full = B.alloc_plane(M, K)
    run(B.PLANE_ALL, full)
    ref = _sections_of(full, M, K)
    sentinel = _sections_of(torch.full_like(full, 0xA5), M, K)
    for sections in range(1, 8):
        plane = torch.full_like(full, 0xA5)
        run(sections, plane)
        got = _sections_of(plane, M, K)
        want = {"q16": sections & B.PLANE_Q16, "q8": sections & B.PLANE_Q8, "ds": sections & B.PLANE_DS,
                "d": True, "s": True}
        for name, written in want.items():
            expect = ref[name] if written else sentinel[name]
            assert np.array_equal(got[name], expect), (producer, sections, name)


def test_consumers_read_only_their_sections():
    # a GEMM on a MQ_PLANE_FOR_GEMM plane and a GEMV on a MQ_PLANE_FOR_GEMV plane give the same
    # outputs as on a full plane, bit for bit
    import torch
    M, K, N = 20, 512, 256
    r = np.random.default_rng(12)
    x = inputs.activations(r, M, K)
    full, _ = G.gpu_plane(x)
    for fmt in ("q4k", "q6k", "q4_1"):
        wt = inputs.q4k_weights(r, N, K) if fmt == "q4k" else (
            inputs.q6k_weights(r, N, K) if fmt == "q6k" else inputs.b32_weights(r, N, K, fmt))
        wd = G.dev(wt.reshape(N, -1))
        for path, sections in (("gemm", B.PLANE_FOR_GEMM), ("gemv", B.PLANE_FOR_GEMV)):
            part = torch.full_like(full, 0xA5)
            B.mq_quantize_q8_ex(G.dev(x), M, K, None, 0.0, sections, part)
            y_full = torch.empty((M, N), dtype=torch.float32, device="cuda")
            y_part = torch.empty_like(y_full)
            f = (B.GEMM if path == "gemm" else B.GEMV)[fmt]
            f(wd, N, K, full, M, y_full)
            f(wd, N, K, part, M, y_part)
            torch.cuda.synchronize()
            B.mq_device_status()
            assert torch.equal(y_full, y_part), (fmt, path)
