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
    G.assert_ds_consistent(plane, M, K)
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


# ---- the fused gate|up GEMM with the SwiGLU epilogue (mq_gemm_q4k_swiglu)

def _plane_np(plane, M, K):
    """(q16, q8, d, S) in token-major form, then the raw ds section (tf32 pairs of d * S), which the
    fused kernel writes itself and a Q4_K / Q5_K down projection would read."""
    q16, q8, d, s, ds = B.plane_views(plane, M, K, with_ds=True)
    return (q16.float().cpu().numpy(), q8.cpu().numpy(), d.t().contiguous().cpu().numpy(),
            s.t().contiguous().cpu().numpy(), ds.cpu().numpy().view(np.uint32))


def _fused(wgd, wud, plane, M, K, F):
    import torch
    out = B.alloc_plane(M, F)
    B.mq_gemm_q4k_swiglu(wgd, wud, F, K, plane, M, out)
    torch.cuda.synchronize()
    B.mq_device_status()
    return out


def _unfused(wgd, wud, plane, M, K, F):
    # the two plain GEMMs and the SwiGLU producer, all on the GPU
    import torch
    yg = torch.empty((M, F), dtype=torch.float32, device="cuda")
    yu = torch.empty((M, F), dtype=torch.float32, device="cuda")
    B.mq_gemm_q4k(wgd, F, K, plane, M, yg)
    B.mq_gemm_q4k(wud, F, K, plane, M, yu)
    out = B.alloc_plane(M, F)
    B.mq_quantize_swiglu_q8(yg, yu, M, F, out)
    torch.cuda.synchronize()
    B.mq_device_status()
    return out


def _assert_near_oracle(got, wg, wu, ref_plane, ms):
    """The fused plane's rows `ms` against the oracle at the stated bar, in its own form: errors
    relative to the L2 norm of the reference row (as for the matmul outputs).  G and U are f32
    sums in another order than the oracle's f64 ones, and silu's tail turns an absolute error of
    G into the same relative error of y (d silu(G) / silu(G) ~ dG for G << 0), so in blocks whose
    gates are all far below zero (values ~1e-30) the scale can move by ~1e-3 of itself; against
    the row those blocks weigh nothing.  Checked: every code is a correct rounding of the f64
    silu(G) U -- |q d - y| within half a step plus 1e-3 of the row's largest |y| (the bar
    normalised by the row's max, stricter than by its L2 norm; the quantization step itself is
    ~1e-3 of the L2 norm at F = 1024) --, every scale within 1e-3 of the row's largest scale,
    codes within 1 of the oracle's (at most 0.1% of them off), and S and the f16 codes consistent
    with the int8 codes."""
    q16, q8, d, s = (a[ms] for a in got[:4])
    qr, dr, sr = oracle.gate_up_swiglu_q8(wg, wu, "q4k", ref_plane, ms, threads=16)
    assert np.all(np.abs(d.astype(np.float64) - dr) <= 1e-3 * dr.max(axis=1, keepdims=True))
    dq = np.abs(q8.astype(np.int32) - qr.astype(np.int32))
    assert dq.max() <= 1 and (dq != 0).mean() <= 1e-3, (dq.max(), (dq != 0).mean())
    assert np.array_equal(q16, q8.astype(np.float32))
    Mm, F = q8.shape
    assert np.array_equal(s, q8.reshape(Mm, -1, 32).astype(np.int32).sum(axis=2))
    Gm = oracle.matmul(wg, "q4k", ref_plane, ms, None, threads=16)
    Um = oracle.matmul(wu, "q4k", ref_plane, ms, None, threads=16)
    y = Gm / (1.0 + np.exp(-Gm)) * Um
    deq = (q8.reshape(Mm, -1, 32).astype(np.float64) * d[..., None]).reshape(Mm, F)
    half = 0.5 * np.repeat(d.astype(np.float64), 32, axis=1)
    excess = (np.abs(deq - y) - half) / np.abs(y).max(axis=1, keepdims=True)
    assert excess.max() <= G.REL_TOL, excess.max()


@pytest.mark.parametrize("M,K,F", [(1, 256, 256), (16, 512, 256), (130, 512, 512), (200, 1024, 768),
                                   (129, 3584, 1024), (300, 256, 2048)])
def test_gate_up_swiglu_shapes(M, K, F):
    r = np.random.default_rng(M * 131 + K + F)
    wg = inputs.q4k_weights(r, F, K)
    wu = inputs.q4k_weights(r, F, K)
    x = inputs.activations(r, M, K)
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    wgd, wud = G.dev(wg.reshape(F, -1)), G.dev(wu.reshape(F, -1))
    fused = _fused(wgd, wud, plane, M, K, F)
    got = _plane_np(fused, M, F)
    # the same arithmetic as the unfused GPU chain, bit for bit (the ds section included)
    unf = _plane_np(_unfused(wgd, wud, plane, M, K, F), M, F)
    for a, b in zip(got, unf):
        assert np.array_equal(a, b)
    G.assert_ds_consistent(fused, M, F)
    _assert_near_oracle(got, wg, wu, ref_plane, np.arange(M))


def test_gate_up_swiglu_ffn_size():
    # the 7B FFN at the 3314-token prompt: gate / up 18944 x 3584 Q4_K from the RMSNorm plane
    c = inputs.ffn_prefill()
    M, K, F = c["x_hidden"].shape[0], inputs.HIDDEN, inputs.FFN
    plane, _ = G.gpu_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ref_plane = G.oracle_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    wgd, wud = G.dev(c["w_gate"].reshape(F, -1)), G.dev(c["w_up"].reshape(F, -1))
    fused = _fused(wgd, wud, plane, M, K, F)
    got = _plane_np(fused, M, F)
    unf = _plane_np(_unfused(wgd, wud, plane, M, K, F), M, F)
    for a, b in zip(got, unf):
        assert np.array_equal(a, b)
    G.assert_ds_consistent(fused, M, F)
    ms = np.array(sorted({0, 1, 127, 128, 1000, 2047, 2048, M - 2, M - 1} |
                         set(np.random.default_rng(5).choice(M, 15, replace=False).tolist())))
    _assert_near_oracle(got, c["w_gate"], c["w_up"], ref_plane, ms)
