"""GPU parity of the SwiGLU producer (mq_quantize_swiglu_q8) against the oracle: the Q8 plane
of silu(gate) * up must match bit for bit (int8 codes, f16 codes, f32 scales, int32 sums)."""
import numpy as np
import pytest

import oracle
from quantized_q8_activation_quantize_gb300 import binding as B
from quantized_q8_activation_quantize_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _gpu_swiglu_plane(g, u):
    import torch
    M, K = g.shape
    plane = B.alloc_plane(M, K)
    B.mq_quantize_swiglu_q8(G.dev(g), G.dev(u), M, K, plane)
    torch.cuda.synchronize()
    B.mq_device_status()
    q16, q8, d, s = B.plane_views(plane, M, K)
    return (q16.float().cpu().numpy(), q8.cpu().numpy(), d.t().contiguous().cpu().numpy(),
            s.t().contiguous().cpu().numpy())


@pytest.mark.parametrize("M,K", [(1, 256), (3, 512), (8, 3584), (37, 768), (130, 18944)])
def test_swiglu_plane_bit_exact(M, K):
    g, u = inputs.swiglu_inputs(np.random.default_rng(M * 31 + K), M, K)
    G.assert_plane_equal(_gpu_swiglu_plane(g, u), oracle.quantize_swiglu_q8(g, u))


def test_swiglu_edge_values():
    M, K = 4, 256
    g = np.zeros((M, K), np.float32)
    u = np.ones((M, K), np.float32)
    g[0, :16] = [0.0, -0.0, 1e-30, -1e-30, 86.0, -86.0, 88.0, -88.0, 89.0, -89.0, 1e4, -1e4, 0.5, -0.5, 20.0, -20.0]
    g[1, :] = np.linspace(-100, 100, K, dtype=np.float32)
    u[1, :] = np.linspace(-3, 3, K, dtype=np.float32)
    g[2, :] = np.float32(0.6931472) * np.arange(-128, 128, dtype=np.float32)   # near k ln2
    u[3, :] = 0.0                                                               # all-zero blocks
    g[3, :] = 5.0
    G.assert_plane_equal(_gpu_swiglu_plane(g, u), oracle.quantize_swiglu_q8(g, u))


def test_swiglu_full_ffn_size():
    # the down projection's input in the 7B FFN at the 3314-token prompt: 3314 x 18944
    g, u = inputs.swiglu_inputs(inputs.rng(2, 7), inputs.PREFILL_TOKENS, inputs.FFN)
    G.assert_plane_equal(_gpu_swiglu_plane(g, u), oracle.quantize_swiglu_q8(g, u))
