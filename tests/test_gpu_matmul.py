"""GPU parity of the GEMM (tensor-core MMQ) and GEMV (dp4a MMVQ) entry points against the
oracle, on identical seeded bytes:

* the integer checkpoint I (per token, row, 32-value block) must match bit for bit;
* outputs must satisfy max |Y_gpu - Y_ref| / ||Y_ref[m, :]||_2 <= 1e-3 (the stated bar);
  on sampled full-size cases the stricter RMS-normalised form (divide by the RMS of the
  reference row's sampled entries instead of its L2 norm, a factor sqrt(N) stricter) is used.
"""
import numpy as np
import pytest

import oracle
from quantized_q8_activation_quantize_gb300 import binding as B
from quantized_q8_activation_quantize_gb300 import inputs
from tests import gpu_util as G

pytestmark = pytest.mark.gpu


def _weights(fmt, n, k, seed, scale_range=(-64, 63)):
    r = np.random.default_rng(seed)
    if fmt == "q4k":
        return inputs.q4k_weights(r, n, k)
    if fmt == "q5k":
        return inputs.q5k_weights(r, n, k)
    if fmt in inputs.B32_BYTES:
        return inputs.b32_weights(r, n, k, fmt)
    return inputs.q6k_weights(r, n, k, scale_range=scale_range)


def _full_check(path, fmt, M, N, K, seed, scale_range=(-64, 63), dump=True):
    w = _weights(fmt, N, K, seed, scale_range)
    x = inputs.activations(np.random.default_rng(seed + 1), M, K)
    plane, got = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    G.assert_plane_equal(got, ref_plane)
    y, wd = G.run_matmul(path, fmt, w, plane, M, K, N)
    ref = oracle.matmul(w, fmt, ref_plane, threads=8)
    err = G.rel_err(y, ref)
    assert err <= G.REL_TOL, f"rel err {err}"
    if dump:
        I, y2 = G.run_dump(path, fmt, wd, plane, M, K, N, 0, M, 0, N)
        Iref, _ = oracle.blockdots(w, fmt, ref_plane[0])
        assert np.array_equal(I, Iref), f"block dots differ at {np.argwhere(I != Iref)[:5]}"
        assert np.array_equal(y2, y), "the dump variant must produce the same output"
    return err


SHAPES = [(1, 7, 256), (2, 65, 512), (5, 129, 768), (8, 64, 2048), (13, 33, 512), (16, 128, 256),
          (17, 130, 512), (130, 129, 256), (200, 200, 1024), (129, 1, 512)]


@pytest.mark.parametrize("fmt", ["q4k", "q6k"])
@pytest.mark.parametrize("path", ["gemv", "gemm"])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_small_shapes(path, fmt, M, N, K):
    _full_check(path, fmt, M, N, K, seed=M * 7919 + N * 31 + K)


# rows longer than one GEMV unit (rows straddle several units), many short rows per unit,
# and row counts that do not divide among the CTAs
GEMV_SHAPES = [(1, 3, 65536), (3, 5, 33280), (1, 1000, 256), (2, 997, 3584), (9, 77, 18944)]


@pytest.mark.parametrize("fmt", ["q4k", "q6k"])
@pytest.mark.parametrize("M,N,K", GEMV_SHAPES)
def test_gemv_row_layouts(fmt, M, N, K):
    _full_check("gemv", fmt, M, N, K, seed=M * 104729 + N * 17 + K)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_q6k_full_scale_range(path):
    # real GGML Q6_K files use scales up to +-128; odd |sc| > 64 takes the correction tile
    for seed, (M, N, K) in enumerate([(3, 40, 512), (64, 200, 768), (150, 130, 256)]):
        _full_check(path, "q6k", M, N, K, seed=900 + seed, scale_range=(-128, 127))


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_extreme_blocks(path):
    # every quant at its extreme with every code at +-127: the int32 headroom cases
    M, N, K = 16, 16, 512
    x = np.full((M, K), 1.0, np.float32)
    x[1::2] = -1.0
    plane, got = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    for fmt in ("q4k", "q6k"):
        w = _weights(fmt, N, K, 5, (-128, 127))
        if fmt == "q4k":
            w[..., 4:] = 0xFF                  # sc = m = 63, q = 15
        else:
            w[..., 0:192] = 0                  # q = -32
            w[..., 192:208] = 0x80             # sc = -128
        y, wd = G.run_matmul(path, fmt, w, plane, M, K, N)
        ref = oracle.matmul(w, fmt, ref_plane)
        assert G.rel_err(y, ref) <= G.REL_TOL
        I, _ = G.run_dump(path, fmt, wd, plane, M, K, N, 0, M, 0, N)
        Iref, _ = oracle.blockdots(w, fmt, ref_plane[0])
        assert np.array_equal(I, Iref)


@pytest.mark.parametrize("path", ["gemv", "gemm"])
def test_tiny_q4k_case(path):
    c = inputs.tiny_q4k()
    M, K = c["x"].shape
    N = c["w"].shape[0]
    plane, got = G.gpu_plane(c["x"])
    ref_plane = G.oracle_plane(c["x"])
    y, wd = G.run_matmul(path, "q4k", c["w"], plane, M, K, N)
    assert G.rel_err(y, oracle.matmul(c["w"], "q4k", ref_plane)) <= G.REL_TOL
    I, _ = G.run_dump(path, "q4k", wd, plane, M, K, N, 0, M, 0, N)
    assert np.array_equal(I, oracle.blockdots(c["w"], "q4k", ref_plane[0])[0])


def test_qproj_prefill_gemm_full():
    c = inputs.qproj_prefill()
    M, K = c["x"].shape
    N = c["w"].shape[0]
    plane, got = G.gpu_plane(c["x"])
    ref_plane = G.oracle_plane(c["x"])
    G.assert_plane_equal(got, ref_plane)
    y, wd = G.run_matmul("gemm", "q4k", c["w"], plane, M, K, N)
    ref = oracle.matmul(c["w"], "q4k", ref_plane, threads=16)
    assert G.rel_err(y, ref) <= G.REL_TOL
    # integer checkpoint on a window crossing token and row tile borders
    m0, mc, n0, nc = 120, 140, 100, 200
    I, _ = G.run_dump("gemm", "q4k", wd, plane, M, K, N, m0, mc, n0, nc)
    Iref, _ = oracle.blockdots(c["w"], "q4k", ref_plane[0], np.arange(m0, m0 + mc), np.arange(n0, n0 + nc))
    assert np.array_equal(I, Iref)


def _sampled(path, fmt, w, plane, ref_plane, M, K, N, ms, ns, dump_window=None):
    y, wd = G.run_matmul(path, fmt, w, plane, M, K, N)
    ref = oracle.matmul(w, fmt, ref_plane, ms, ns, threads=16)
    got = y[np.ix_(ms, ns)]
    rms = np.sqrt((ref ** 2).mean(axis=1, keepdims=True))
    err = float((np.abs(got - ref) / np.where(rms == 0, 1, rms)).max())
    assert err <= G.REL_TOL, f"RMS-normalised err {err}"
    if dump_window is not None:
        m0, mc, n0, nc = dump_window
        I, _ = G.run_dump(path, fmt, wd, plane, M, K, N, m0, mc, n0, nc)
        Iref, _ = oracle.blockdots(w, fmt, ref_plane[0], np.arange(m0, m0 + mc), np.arange(n0, n0 + nc))
        assert np.array_equal(I, Iref)
    return err


def _sample_idx(total, count, seed, must=()):
    r = np.random.default_rng(seed)
    idx = set(r.choice(total, size=min(count, total), replace=False).tolist()) | set(must)
    return np.array(sorted(i for i in idx if 0 <= i < total))


def test_ffn_prefill_full_size_sampled():
    c = inputs.ffn_prefill()
    M = c["x_hidden"].shape[0]
    plane_h, _ = G.gpu_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ref_h = G.oracle_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ms = _sample_idx(M, 48, 1, must=(0, 127, 128, M - 1))
    for name in ("w_gate", "w_up"):
        N = c[name].shape[0]
        ns = _sample_idx(N, 384, 2, must=(0, N - 1))
        _sampled("gemm", "q4k", c[name], plane_h, ref_h, M, 3584, N, ms, ns,
                 dump_window=(M - 40, 40, N - 70, 70))
    plane_f, _ = G.gpu_plane(c["x_ffn"])
    ref_f = G.oracle_plane(c["x_ffn"])
    ns = _sample_idx(3584, 384, 3, must=(0, 3583))
    _sampled("gemm", "q6k", c["w_down"], plane_f, ref_f, M, 18944, 3584, ms, ns, dump_window=(3200, 114, 0, 40))


def test_decode_sweep_layers():
    # two layers of the decode sweep: layer 0 (Q6_K v and down) and layer 1 (all Q4_K), full rows
    for layer in (0, 1):
        for idx in range(7):
            c = inputs.decode_matrix(layer, idx)
            N, K = c["w"].shape[0], c["x"].shape[1]
            plane, _ = G.gpu_plane(c["x"])
            ref_plane = G.oracle_plane(c["x"])
            y, wd = G.run_matmul("gemv", c["fmt"], c["w"], plane, 1, K, N)
            ref = oracle.matmul(c["w"], c["fmt"], ref_plane, threads=16)
            assert G.rel_err(y, ref) <= G.REL_TOL, (layer, c["name"])
            I, _ = G.run_dump("gemv", c["fmt"], wd, plane, 1, K, N, 0, 1, 0, min(N, 256))
            assert np.array_equal(I, oracle.blockdots(c["w"], c["fmt"], ref_plane[0], None, np.arange(min(N, 256)))[0])


@pytest.fixture(scope="module")
def lm_head():
    return inputs.lm_head_weights()


@pytest.mark.parametrize("M,paths", [(1, ("gemv",)), (4, ("small",)), (16, ("gemv", "gemm", "small")),
                                     (32, ("small",)), (3314, ("gemm",))])
def test_lm_head(lm_head, M, paths):
    x = inputs.lm_head_x(M)
    N, K = lm_head.shape[0], 3584
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    ms = _sample_idx(M, 24, 5, must=(0, M - 1))
    ns = _sample_idx(N, 2048, 6, must=(0, N - 1))
    for path in paths:
        _sampled(path, "q6k", lm_head, plane, ref_plane, M, K, N, ms, ns,
                 dump_window=(0, min(M, 8), N - 100, 100))


# ---- Q5_K (NEXT row): decode GEMV and prefill GEMM on the Q4_K skeletons

@pytest.mark.parametrize("M,N,K", SHAPES + GEMV_SHAPES)
def test_q5k_gemv_shapes(M, N, K):
    _full_check("gemv", "q5k", M, N, K, seed=M * 6151 + N * 13 + K)


def test_q5k_gemv_extreme_blocks():
    # q = 31 with sc = m = 63 and every code at +-127: the int32 / f32 headroom case
    M, N, K = 9, 16, 512
    x = np.full((M, K), 1.0, np.float32)
    x[1::2] = -1.0
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    w = _weights("q5k", N, K, 5)
    w[..., 4:] = 0xFF
    y, wd = G.run_matmul("gemv", "q5k", w, plane, M, K, N)
    assert G.rel_err(y, oracle.matmul(w, "q5k", ref_plane)) <= G.REL_TOL
    I, _ = G.run_dump("gemv", "q5k", wd, plane, M, K, N, 0, M, 0, N)
    assert np.array_equal(I, oracle.blockdots(w, "q5k", ref_plane[0])[0])


def test_q5k_gemv_ffn_size():
    # the 7B FFN gate shape (18944 x 3584) at M = 1, every output and a block-dot window
    M, N, K = 1, 18944, 3584
    err = _full_check("gemv", "q5k", M, N, K, seed=31, dump=False)
    assert err <= G.REL_TOL
    w = _weights("q5k", N, K, 31)
    x = inputs.activations(np.random.default_rng(32), M, K)
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    _, wd = G.run_matmul("gemv", "q5k", w, plane, M, K, N)
    n0, nc = 18000, 300
    I, _ = G.run_dump("gemv", "q5k", wd, plane, M, K, N, 0, 1, n0, nc)
    Iref, _ = oracle.blockdots(w, "q5k", ref_plane[0], ns=np.arange(n0, n0 + nc))
    assert np.array_equal(I, Iref)


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k", "q4_0", "q4_1", "q5_0", "q5_1", "q8_0"])
def test_gemv_repeated_launches_agree(fmt):
    # 18944 x 3584 at M = 1: every CTA wraps its stage ring several times, the case where a
    # stage handed back too early showed up as wrong partials of whole warps.  The reduction
    # order is fixed, so repeated launches must agree bit for bit, and with the oracle.
    import torch
    M, N, K = 1, 18944, 3584
    w = _weights(fmt, N, K, 77)
    x = inputs.activations(np.random.default_rng(78), M, K)
    plane, _ = G.gpu_plane(x)
    ref = oracle.matmul(w, fmt, G.oracle_plane(x), threads=8)
    wd = G.dev(w.reshape(N, -1))
    ys = [torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda") for _ in range(5)]
    for y in ys:
        B.GEMV[fmt](wd, N, K, plane, M, y)
    torch.cuda.synchronize()
    B.mq_device_status()
    first = ys[0].cpu().numpy()
    assert G.rel_err(first, ref) <= G.REL_TOL
    for y in ys[1:]:
        assert np.array_equal(y.cpu().numpy(), first)


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_q5k_gemm_shapes(M, N, K):
    _full_check("gemm", "q5k", M, N, K, seed=M * 7411 + N * 19 + K)


def test_q5k_gemm_extreme_blocks():
    # q = 31 with sc = m = 63 and every code at +-127: sc * q = 1953 must stay exact in f16
    M, N, K = 16, 16, 512
    x = np.full((M, K), 1.0, np.float32)
    x[1::2] = -1.0
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    w = _weights("q5k", N, K, 5)
    w[..., 4:] = 0xFF
    y, wd = G.run_matmul("gemm", "q5k", w, plane, M, K, N)
    assert G.rel_err(y, oracle.matmul(w, "q5k", ref_plane)) <= G.REL_TOL
    I, _ = G.run_dump("gemm", "q5k", wd, plane, M, K, N, 0, M, 0, N)
    assert np.array_equal(I, oracle.blockdots(w, "q5k", ref_plane[0])[0])


def test_q5k_gemm_ffn_size_sampled():
    # the 7B FFN gate shape with Q5_K weights at the 3314-token prompt
    c = inputs.ffn_prefill()
    M, K, N = c["x_hidden"].shape[0], 3584, 18944
    w = _weights("q5k", N, K, 41)
    plane, _ = G.gpu_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ref_plane = G.oracle_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ms = _sample_idx(M, 48, 7, must=(0, 127, 128, M - 1))
    ns = _sample_idx(N, 384, 8, must=(0, N - 1))
    _sampled("gemm", "q5k", w, plane, ref_plane, M, K, N, ms, ns, dump_window=(M - 40, 40, N - 70, 70))


# ---- 32-value block formats Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q8_0 (NEXT row): decode GEMV on the
# k-quant GEMV skeleton, eight blocks to a 256-value group

B32_FMTS = ["q4_0", "q4_1", "q5_0", "q5_1", "q8_0"]


@pytest.mark.parametrize("fmt", B32_FMTS)
@pytest.mark.parametrize("M,N,K", SHAPES + GEMV_SHAPES)
def test_b32_gemv_shapes(fmt, M, N, K):
    _full_check("gemv", fmt, M, N, K, seed=M * 5179 + N * 17 + K + len(fmt) * 3 + ord(fmt[1]) + ord(fmt[3]))


@pytest.mark.parametrize("fmt,fill", [("q4_0", 0xFF), ("q4_0", 0x00), ("q4_1", 0xFF), ("q5_0", 0xFF),
                                      ("q5_0", 0x00), ("q5_1", 0xFF), ("q8_0", 0x80), ("q8_0", 0x7F)])
def test_b32_gemv_extreme_blocks(fmt, fill):
    # every quant at the top or bottom of its range (q - offset = 7 / -8, 15 / -16, 15, 31,
    # -128, 127) against codes at +-127: the int32 headroom and the dp4a seed
    M, N, K = 9, 16, 512
    x = np.full((M, K), 1.0, np.float32)
    x[1::2] = -1.0
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    w = _weights(fmt, N, K, 6)
    w[..., 4 if fmt in ("q4_1", "q5_1") else 2:] = fill
    y, wd = G.run_matmul("gemv", fmt, w, plane, M, K, N)
    assert G.rel_err(y, oracle.matmul(w, fmt, ref_plane)) <= G.REL_TOL
    I, _ = G.run_dump("gemv", fmt, wd, plane, M, K, N, 0, M, 0, N)
    assert np.array_equal(I, oracle.blockdots(w, fmt, ref_plane[0])[0])


@pytest.mark.parametrize("fmt", B32_FMTS)
@pytest.mark.parametrize("M,N,K", [(1, 18944, 3584), (8, 600, 18944), (3, 3584, 18944)])
def test_b32_gemv_model_sizes(fmt, M, N, K):
    # the 7B FFN gate (M = 1, staged activations) and down shapes (K = 18944: at M = 8 the
    # activations no longer fit in shared memory and the kernel reads them from global memory)
    _full_check("gemv", fmt, M, N, K, seed=N + K + M + ord(fmt[1]) * 7 + ord(fmt[3]), dump=M > 1)


@pytest.mark.parametrize("fmt", B32_FMTS)
def test_b32_gemv_vocab_sampled(fmt):
    # the LM-head shape (152064 x 3584) at M = 1, the launch the benchmark times
    w = inputs.b32_vocab_weights(fmt)
    x = inputs.lm_head_x(1)
    N, K = w.shape[0], 3584
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    ns = _sample_idx(N, 2048, 9, must=(0, N - 1))
    _sampled("gemv", fmt, w, plane, ref_plane, 1, K, N, np.array([0]), ns, dump_window=(0, 1, N - 100, 100))


@pytest.mark.parametrize("fmt", B32_FMTS)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_b32_gemm_shapes(fmt, M, N, K):
    _full_check("gemm", fmt, M, N, K, seed=M * 7919 + N * 23 + K + ord(fmt[1]) * 5 + ord(fmt[3]))


@pytest.mark.parametrize("fmt,fill", [("q4_0", 0xFF), ("q4_0", 0x00), ("q4_1", 0xFF), ("q5_0", 0xFF),
                                      ("q5_0", 0x00), ("q5_1", 0xFF), ("q8_0", 0x80), ("q8_0", 0x7F)])
def test_b32_gemm_extreme_blocks(fmt, fill):
    # quants at the ends of their ranges against codes at +-127: the f16 operands (q - offset,
    # Q8_0's -128) and the per-block f32 accumulators stay exact
    M, N, K = 16, 16, 512
    x = np.full((M, K), 1.0, np.float32)
    x[1::2] = -1.0
    plane, _ = G.gpu_plane(x)
    ref_plane = G.oracle_plane(x)
    w = _weights(fmt, N, K, 7)
    w[..., 4 if fmt in ("q4_1", "q5_1") else 2:] = fill
    y, wd = G.run_matmul("gemm", fmt, w, plane, M, K, N)
    assert G.rel_err(y, oracle.matmul(w, fmt, ref_plane)) <= G.REL_TOL
    I, _ = G.run_dump("gemm", fmt, wd, plane, M, K, N, 0, M, 0, N)
    assert np.array_equal(I, oracle.blockdots(w, fmt, ref_plane[0])[0])


@pytest.mark.parametrize("fmt", B32_FMTS)
def test_b32_gemm_ffn_size_sampled(fmt):
    # the 7B FFN gate shape at the 3314-token prompt, synthetic weights of the format
    c = inputs.ffn_prefill()
    M, K, N = c["x_hidden"].shape[0], 3584, 18944
    w = _weights(fmt, N, K, 43 + ord(fmt[1]) + ord(fmt[3]))
    plane, _ = G.gpu_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ref_plane = G.oracle_plane(c["x_hidden"], c["rms_w"], float(c["eps"]))
    ms = _sample_idx(M, 32, 11, must=(0, 127, 128, M - 1))
    ns = _sample_idx(N, 256, 12, must=(0, N - 1))
    _sampled("gemm", fmt, w, plane, ref_plane, M, K, N, ms, ns, dump_window=(M - 30, 30, N - 50, 50))


@pytest.mark.parametrize("fmt", B32_FMTS)
def test_b32_size_dispatch_agrees(fmt):
    # matmul() takes the GEMV below 16 tokens and the GEMM from 16 on; at M = 16 both paths
    # must meet the bar against the oracle
    M, N, K = 16, 300, 1024
    w = _weights(fmt, N, K, 91)
    x = inputs.activations(np.random.default_rng(92), M, K)
    plane, _ = G.gpu_plane(x)
    ref = oracle.matmul(w, fmt, G.oracle_plane(x))
    for path in ("gemv", "gemm"):
        y, _ = G.run_matmul(path, fmt, w, plane, M, K, N)
        assert G.rel_err(y, ref) <= G.REL_TOL, path


# ---- the small-M band on the tensor cores (mq_gemm_small_*): weights as the 128-row MMA operand,
# tokens (padded to 16 or 32) as its N side; the same exact block dots and the same bar

SMALL_SHAPES = [(1, 7, 256), (2, 65, 512), (5, 129, 768), (9, 300, 2048), (15, 33, 512), (16, 128, 256),
                (17, 130, 512), (31, 257, 1024), (32, 1000, 3584), (4, 129, 18944)]


@pytest.mark.parametrize("fmt", ["q4k", "q5k", "q6k"])
@pytest.mark.parametrize("M,N,K", SMALL_SHAPES)
def test_small_m_shapes(fmt, M, N, K):
    _full_check("small", fmt, M, N, K, seed=M * 6007 + N * 37 + K + len(fmt))


def test_small_m_q6k_full_scale_range():
    # scales up to +-128: odd |sc| > 64 takes the correction tile (now an A operand)
    for seed, (M, N, K) in enumerate([(3, 40, 512), (16, 200, 768), (32, 130, 256)]):
        _full_check("small", "q6k", M, N, K, seed=700 + seed, scale_range=(-128, 127))


def test_small_m_extreme_blocks():
    # every quant at its extreme with every code at +-127: the int32 headroom cases
    for M in (5, 32):
        N, K = 16, 512
        x = np.full((M, K), 1.0, np.float32)
        x[1::2] = -1.0
        plane, _ = G.gpu_plane(x)
        ref_plane = G.oracle_plane(x)
        for fmt in ("q4k", "q5k", "q6k"):
            w = _weights(fmt, N, K, 5, (-128, 127))
            if fmt == "q6k":
                w[..., 0:192] = 0                  # q = -32
                w[..., 192:208] = 0x80             # sc = -128
            else:
                w[..., 4:] = 0xFF                  # sc = m = 63, q = 15 (Q5_K: 31)
            y, wd = G.run_matmul("small", fmt, w, plane, M, K, N)
            assert G.rel_err(y, oracle.matmul(w, fmt, ref_plane)) <= G.REL_TOL
            I, _ = G.run_dump("small", fmt, wd, plane, M, K, N, 0, M, 0, N)
            assert np.array_equal(I, oracle.blockdots(w, fmt, ref_plane[0])[0]), (M, fmt)


def test_small_m_decode_shapes():
    # a layer of the 7B decode stack batched over 8 sequences: q (Q4_K), v and down (Q6_K), gate (Q4_K)
    for idx in (0, 2, 4, 6):
        c = inputs.decode_matrix(0, idx)
        N, K = c["w"].shape[0], c["x"].shape[1]
        x = inputs.activations(np.random.default_rng(300 + idx), 8, K)
        plane, _ = G.gpu_plane(x)
        ref_plane = G.oracle_plane(x)
        ms, ns = np.arange(8), _sample_idx(N, 512, 301 + idx, must=(0, N - 1))
        _sampled("small", c["fmt"], c["w"], plane, ref_plane, 8, K, N, ms, ns, dump_window=(0, 8, N - 64, 64))


@pytest.mark.parametrize("M", [2, 5, 7, 8, 16, 32])
def test_small_m_size_dispatch_agrees(M):
    # matmul() routes the band to the GEMV or the small-M kernel (matmul_path): the path it picks meets
    # the bar against the oracle, and every path on the same inputs meets it too
    import torch
    N, K = 300, 1024
    for fmt in ("q4k", "q6k"):
        w = _weights(fmt, N, K, 93)
        x = inputs.activations(np.random.default_rng(94 + M), M, K)
        plane, _ = G.gpu_plane(x)
        ref = oracle.matmul(w, fmt, G.oracle_plane(x))
        assert B.matmul_path(fmt, M) == ("small" if M >= B.SMALL_MIN_M[fmt] else "gemv")
        y = torch.empty((M, N), dtype=torch.float32, device="cuda")
        B.matmul(fmt, G.dev(w.reshape(N, -1)), N, K, plane, M, y)
        torch.cuda.synchronize()
        B.mq_device_status()
        assert G.rel_err(y.cpu().numpy(), ref) <= G.REL_TOL
        for path in ("gemv", "gemm", "small"):
            y2, _ = G.run_matmul(path, fmt, w, plane, M, K, N)
            assert G.rel_err(y2, ref) <= G.REL_TOL, path


# ---- grouped decode GEMV and grouped quantize (one launch per layer level of the decode sweep)

@pytest.mark.parametrize("M", [1, 3])
def test_grouped_gemv_matches_single_calls(M):
    # the level shapes of a decoder layer: q|k|v (3584, 512, 512 rows, K = 3584), gate|up (18944 rows
    # each), and Q6_K matrices of different heights; every job's output equals its single call bit for
    # bit, and meets the bar against the oracle
    import torch
    cases = [("q4k", 3584, [3584, 512, 512]), ("q4k", 3584, [18944, 18944]), ("q6k", 18944, [3584, 1000]),
             ("q5k", 512, [7, 300, 129])]
    for fmt, K, Ns in cases:
        r = np.random.default_rng(K + len(Ns) + M)
        ws = [_weights(fmt, n, K, 500 + i + K) for i, n in enumerate(Ns)]
        xs = [inputs.activations(r, M, K) for _ in Ns]
        planes = [G.gpu_plane(x)[0] for x in xs]
        wds = [G.dev(w.reshape(n, -1)) for w, n in zip(ws, Ns)]
        ys = [torch.full((M, n), float("nan"), dtype=torch.float32, device="cuda") for n in Ns]
        B.GEMV_GROUPED[fmt]([(wd, n, p, y) for wd, n, p, y in zip(wds, Ns, planes, ys)], K, M)
        torch.cuda.synchronize()
        B.mq_device_status()
        for i, n in enumerate(Ns):
            y1 = torch.empty((M, n), dtype=torch.float32, device="cuda")
            B.GEMV[fmt](wds[i], n, K, planes[i], M, y1)
            torch.cuda.synchronize()
            assert torch.equal(ys[i], y1), (fmt, K, n, M)
            ref = oracle.matmul(ws[i], fmt, G.oracle_plane(xs[i]), threads=8)
            assert G.rel_err(ys[i].cpu().numpy(), ref) <= G.REL_TOL


def test_grouped_gemv_from_f32_activations():
    # one token, the activation quantized inside the GEMV (mq_gemv_grouped_x_*): every job's output
    # equals, bit for bit, the plane quantizer followed by the grouped GEMV, and meets the bar against
    # the oracle; jobs may share an x (q|k|v of a layer), and ragged, edge-valued and zero activations
    # take the same codes as the plane quantizer
    import torch
    cases = [("q4k", 3584, [3584, 512, 512], True), ("q4k", 3584, [18944, 18944], False),
             ("q6k", 18944, [3584, 1000], False), ("q6k", 3584, [512, 7], True), ("q5k", 512, [7, 300, 129], False),
             ("q4k", 256, [33], False)]
    for fmt, K, Ns, shared in cases:
        r = np.random.default_rng(K * 7 + len(Ns))
        ws = [_weights(fmt, n, K, 900 + i + K) for i, n in enumerate(Ns)]
        x0 = inputs.activations(r, 1, K)
        xs = [x0 if shared else inputs.activations(r, 1, K) for _ in Ns]
        if not shared:
            xs[0][0, :32] = 0.0                                   # an all-zero block: d = 0, codes 0
            xs[0][0, 32:40] = [0.5, -0.5, 2.5, -2.5, 126.5, -126.5, 127.0, 0.49999997]
        xds = [G.dev(x.reshape(-1)) for x in xs]
        wds = [G.dev(w.reshape(n, -1)) for w, n in zip(ws, Ns)]
        ys = [torch.full((1, n), float("nan"), dtype=torch.float32, device="cuda") for n in Ns]
        B.GEMV_GROUPED_X[fmt]([(wd, n, xd, y) for wd, n, xd, y in zip(wds, Ns, xds, ys)], K)
        torch.cuda.synchronize()
        B.mq_device_status()
        planes = [G.gpu_plane(x)[0] for x in xs]
        yp = [torch.empty((1, n), dtype=torch.float32, device="cuda") for n in Ns]
        B.GEMV_GROUPED[fmt]([(wd, n, p, y) for wd, n, p, y in zip(wds, Ns, planes, yp)], K, 1)
        torch.cuda.synchronize()
        for i, n in enumerate(Ns):
            assert torch.equal(ys[i], yp[i]), (fmt, K, n)
            ref = oracle.matmul(ws[i], fmt, G.oracle_plane(xs[i]), threads=8)
            assert G.rel_err(ys[i].cpu().numpy(), ref) <= G.REL_TOL


def test_grouped_gemv_from_f32_staging_limit():
    # the largest K whose staged codes fit one CTA, per format (include/mq.h); one super-block more
    # is MQ_ERR_SHAPE before any launch
    import torch
    for fmt, kmax, bb in (("q4k", 101888, 144), ("q5k", 96768, 176), ("q6k", 81920, 210)):
        K = kmax + 256
        x = torch.zeros(K, dtype=torch.float32, device="cuda")
        w = torch.zeros(K // 256 * bb, dtype=torch.uint8, device="cuda")
        y = torch.zeros(8, dtype=torch.float32, device="cuda")
        with pytest.raises(B.MQError) as e:
            B.GEMV_GROUPED_X[fmt]([(w, 1, x, y)], K)
        assert e.value.status == B.MQ_ERR_SHAPE, (fmt, e.value)
    r = np.random.default_rng(77)
    K = 81920
    wt = _weights("q6k", 3, K, 78)
    xk = inputs.activations(r, 1, K)
    wd, xd = G.dev(wt.reshape(3, -1)), G.dev(xk.reshape(-1))
    yx = torch.full((1, 3), float("nan"), dtype=torch.float32, device="cuda")
    B.GEMV_GROUPED_X["q6k"]([(wd, 3, xd, yx)], K)
    torch.cuda.synchronize()
    yp = torch.empty_like(yx)
    B.GEMV["q6k"](wd, 3, K, G.gpu_plane(xk)[0], 1, yp)
    torch.cuda.synchronize()
    assert torch.equal(yx, yp)


def test_grouped_quantize_matches_single_calls():
    import torch
    for M, K, n in ((1, 3584, 3), (1, 18944, 1), (5, 512, 8)):
        r = np.random.default_rng(M * 100 + K + n)
        xs = [inputs.activations(r, M, K) for _ in range(n)]
        xds = [G.dev(x) for x in xs]
        for sections in (B.PLANE_ALL, B.PLANE_FOR_GEMV):
            planes = [torch.full((B.mq_q8_plane_bytes(M, K),), 0x5A, dtype=torch.uint8, device="cuda") for _ in xs]
            B.mq_quantize_q8_grouped(list(zip(xds, planes)), M, K, sections)
            torch.cuda.synchronize()
            B.mq_device_status()
            for x, xd, plane in zip(xs, xds, planes):
                single = torch.full_like(plane, 0x5A)
                B.mq_quantize_q8_ex(xd, M, K, None, 0.0, sections, single)
                torch.cuda.synchronize()
                assert torch.equal(plane, single)
                q16, q8, d, s = B.plane_views(plane, M, K)
                G.assert_plane_equal((q16.float().cpu().numpy() if sections & B.PLANE_Q16 else
                                      q8.cpu().numpy().astype(np.float32), q8.cpu().numpy(),
                                      d.t().contiguous().cpu().numpy(), s.t().contiguous().cpu().numpy()),
                                     G.oracle_plane(x))
