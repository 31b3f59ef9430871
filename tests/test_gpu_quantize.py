"""GPU parity of mq_quantize_q8 (plain and RMSNorm-fused) against the oracle: the Q8 plane
must match bit for bit (int8 codes, f16 codes, f32 scales, int32 sums)."""
import numpy as np
import pytest

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
    for M, K in ((1, 3584), (5, 256), (64, 3584), (3, 18944)):
        x = inputs.activations(r, M, K)
        w = inputs.rms_weight(r, K)
        plane, got = G.gpu_plane(x, w, 1e-6)
        G.assert_plane_equal(got, G.oracle_plane(x, w, 1e-6))
        G.assert_ds_consistent(plane, M, K)


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
