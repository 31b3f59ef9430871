"""Seeded synthetic inputs for the Q4_K / Q6_K x Q8 matmul path.

This module draws random numbers and lays out random bytes.  It holds none of
the method's arithmetic: nothing here decodes a block, quantizes an
activation or multiplies anything.  The CUDA path (through the tests and the
bench) and the CPU oracle both consume exactly the arrays made here, so the
two sides always see identical bytes.

Workloads follow the 7B q4_K_m shapes of the minfer pages (Qwen2.5-7B: hidden
3584, 28 query heads and 4 KV heads of dim 128, FFN 18944, vocab 152064;
3314-token prefill prompt).  Seeds are ``20261202 + 100 * case + stream`` with case
0 = the tiny Q4_K GEMM, 1 = the q_proj prefill, 2 = the FFN prefill, 3 = the decode
sweep, 4 = the LM head (and the synthetic-format matrices of its shape), and stream
0 = weights, 1 = activations, 2 = RMSNorm weight, 3 = outlier channel choice; matrices
of one workload that need separate streams add their (layer, matrix) index to the numpy
``SeedSequence``.

Block sizes (GGML k-quant super-blocks of 256 values): Q4_K = 144 bytes
(fp16 d, fp16 dmin, 12 bytes of packed 6-bit scales/mins, 128 bytes of 4-bit
quants); Q6_K = 210 bytes (128 bytes low 4 bits, 64 bytes high 2 bits,
16 int8 scales, fp16 d).  Only the positions of the fp16 and int8 scale
fields matter here, so that their value ranges can be drawn as stated.
"""
from __future__ import annotations

import numpy as np

SEED_BASE = 20261202
STREAM_W, STREAM_X, STREAM_RMS_W, STREAM_OUTLIERS = 0, 1, 2, 3
STREAM_SWIGLU = 4            # gate / up inputs of the SwiGLU producer

QK_K = 256             # values per k-quant super-block
Q8_BLOCK = 32          # values per Q8 activation block
Q4K_BYTES = 144
Q5K_BYTES = 176
Q6K_BYTES = 210

HIDDEN = 3584
FFN = 18944
KV_DIM = 4 * 128
VOCAB = 152064
PREFILL_TOKENS = 3314
N_LAYERS = 28


def seed(case: int, stream: int) -> int:
    return SEED_BASE + 100 * case + stream


def rng(case: int, stream: int, *extra: int) -> np.random.Generator:
    """PCG64 generator for one (workload case, stream[, layer, matrix]) input."""
    if extra:
        return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed(case, stream), *extra])))
    return np.random.Generator(np.random.PCG64(seed(case, stream)))


def _fp16_bytes(r: np.random.Generator, shape, lo: float, hi: float) -> np.ndarray:
    """fp16 values drawn uniform in [lo, hi] (f64 draw, round-to-nearest-even to fp16), as LE bytes."""
    v = r.uniform(lo, hi, size=shape).astype(np.float16)
    return v.astype("<f2").view(np.uint8).reshape(*shape, 2)


def q4k_weights(r: np.random.Generator, n_rows: int, k: int,
                d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Q4_K weight matrix as raw bytes, shape [n_rows, k/256, 144].

    d and dmin are fp16 drawn uniform in ``d_range``; the 12 packed scale/min
    bytes and the 128 quant bytes are uniform random bytes (the 6-bit packing
    maps 12 uniform bytes onto 16 uniform 6-bit fields, and a uniform byte holds
    two uniform 4-bit quants).
    """
    assert k % QK_K == 0
    nb = k // QK_K
    w = np.frombuffer(r.bytes(n_rows * nb * Q4K_BYTES), dtype=np.uint8).reshape(n_rows, nb, Q4K_BYTES).copy()
    w[..., 0:2] = _fp16_bytes(r, (n_rows, nb), *d_range)
    w[..., 2:4] = _fp16_bytes(r, (n_rows, nb), *d_range)
    return w


def q5k_weights(r: np.random.Generator, n_rows: int, k: int,
                d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Q5_K weight matrix as raw bytes, shape [n_rows, k/256, 176].

    As Q4_K: d and dmin fp16 uniform in ``d_range``; the 12 packed scale/min bytes, the
    32 high-bit bytes and the 128 low-nibble bytes are uniform random bytes (uniform
    5-bit quants).
    """
    assert k % QK_K == 0
    nb = k // QK_K
    w = np.frombuffer(r.bytes(n_rows * nb * Q5K_BYTES), dtype=np.uint8).reshape(n_rows, nb, Q5K_BYTES).copy()
    w[..., 0:2] = _fp16_bytes(r, (n_rows, nb), *d_range)
    w[..., 2:4] = _fp16_bytes(r, (n_rows, nb), *d_range)
    return w


# the 32-value block formats: bytes per block
B32_BYTES = {"q4_0": 18, "q4_1": 20, "q5_0": 22, "q5_1": 24, "q8_0": 34}


def b32_weights(r: np.random.Generator, n_rows: int, k: int, fmt: str,
                d_range=(1e-3, 1e-2), m_range=(-0.08, 0.0)) -> np.ndarray:
    """Weight matrix in a 32-value block format as raw bytes, shape [n_rows, k/32, B32_BYTES[fmt]].

    d is fp16 uniform in ``d_range``; Q4_1 / Q5_1 add an fp16 block offset m uniform in
    ``m_range`` (a block minimum, so at most 0); the high-bit words, nibbles and Q8_0's int8
    quants are uniform random bytes.
    """
    assert k % 32 == 0
    nb, bs = k // 32, B32_BYTES[fmt]
    w = np.frombuffer(r.bytes(n_rows * nb * bs), dtype=np.uint8).reshape(n_rows, nb, bs).copy()
    w[..., 0:2] = _fp16_bytes(r, (n_rows, nb), *d_range)
    if fmt in ("q4_1", "q5_1"):
        w[..., 2:4] = _fp16_bytes(r, (n_rows, nb), *m_range)
    return w


def q6k_weights(r: np.random.Generator, n_rows: int, k: int,
                scale_range=(-128, 127), d_range=(1e-3, 1e-2)) -> np.ndarray:
    """Q6_K weight matrix as raw bytes, shape [n_rows, k/256, 210].

    The 128 low-bit bytes and 64 high-bit bytes are uniform random bytes; the
    16 int8 sub-block scales are uniform integers in ``scale_range``
    (inclusive; by default the whole int8 range, as a quantizer that maps each
    super-block's largest sub-block scale to the end of the range produces:
    a quarter of them odd with magnitude above 64); d is fp16 drawn uniform in
    ``d_range``.
    """
    assert k % QK_K == 0
    nb = k // QK_K
    w = np.frombuffer(r.bytes(n_rows * nb * Q6K_BYTES), dtype=np.uint8).reshape(n_rows, nb, Q6K_BYTES).copy()
    sc = r.integers(scale_range[0], scale_range[1] + 1, size=(n_rows, nb, 16), dtype=np.int16).astype(np.int8)
    w[..., 192:208] = sc.view(np.uint8)
    w[..., 208:210] = _fp16_bytes(r, (n_rows, nb), *d_range)
    return w


def activations(r: np.random.Generator, m: int, k: int) -> np.ndarray:
    """f32 activations [m, k] drawn N(0, 1)."""
    return r.standard_normal((m, k), dtype=np.float32)


def outlier_channels(r: np.random.Generator, k: int, fraction: float = 0.01) -> np.ndarray:
    """Sorted channel indices (round(fraction * k) of them) from a seeded permutation."""
    n = int(round(fraction * k))
    return np.sort(r.permutation(k)[:n])


def swiglu_inputs(r: np.random.Generator, m: int, k: int):
    """Gate and up projections [m, k] f32 for the SwiGLU producer: N(0, 4^2) and N(0, 2^2)
    (the spread of the 7B FFN prefill's gate / up outputs), a few gate values pushed into the
    tails where exp saturates."""
    g = (4.0 * r.standard_normal((m, k))).astype(np.float32)
    u = (2.0 * r.standard_normal((m, k))).astype(np.float32)
    idx = r.integers(0, g.size, size=max(1, g.size // 1000))
    g.flat[idx] = r.choice(np.array([-120.0, -90.0, -87.5, -30.0, 30.0, 87.5, 90.0, 120.0], np.float32), idx.size)
    return g, u


def rms_weight(r: np.random.Generator, k: int) -> np.ndarray:
    """RMSNorm weight [k] drawn N(1, 0.1) in f32."""
    return (1.0 + 0.1 * r.standard_normal(k)).astype(np.float32)


# --------------------------------------------------------------------------------------------
# The five workloads.  Each returns plain numpy arrays; sizes are in the docstrings.
# --------------------------------------------------------------------------------------------

def tiny_q4k():
    """Tiny Q4_K GEMM: W 256 x 512 (Q4_K), X 8 x 512 N(0,1); Y is 8 x 256."""
    w = q4k_weights(rng(0, STREAM_W), 256, 512)
    x = activations(rng(0, STREAM_X), 8, 512)
    return {"w": w, "x": x, "fmt": "q4k"}


def qproj_prefill():
    """q_proj prefill: W 3584 x 3584 (Q4_K), X 512 x 3584 N(0,1) with 36 channels x20."""
    w = q4k_weights(rng(1, STREAM_W), HIDDEN, HIDDEN)
    x = activations(rng(1, STREAM_X), 512, HIDDEN)
    ch = outlier_channels(rng(1, STREAM_OUTLIERS), HIDDEN)
    x[:, ch] *= np.float32(20.0)
    return {"w": w, "x": x, "fmt": "q4k", "outlier_channels": ch}


def ffn_prefill(m: int = PREFILL_TOKENS):
    """7B FFN prefill: gate/up W 18944 x 3584 (Q4_K), down W 3584 x 18944 (Q6_K, int8 scales over the whole range).

    x_hidden [m, 3584] N(0,1) goes through the RMSNorm producer (weight N(1, 0.1), eps 1e-6)
    for gate and up; x_ffn [m, 18944] N(0,1) is the down projection's plain input.
    """
    return {
        "w_gate": q4k_weights(rng(2, STREAM_W, 0), FFN, HIDDEN),
        "w_up": q4k_weights(rng(2, STREAM_W, 1), FFN, HIDDEN),
        "w_down": q6k_weights(rng(2, STREAM_W, 2), HIDDEN, FFN),
        "x_hidden": activations(rng(2, STREAM_X, 0), m, HIDDEN),
        "x_ffn": activations(rng(2, STREAM_X, 1), m, FFN),
        "rms_w": rms_weight(rng(2, STREAM_RMS_W), HIDDEN),
        "eps": np.float32(1e-6),
    }


# matrices of one decoder layer: (name, rows N, reduction K)
LAYER_MATRICES = (("q", HIDDEN, HIDDEN), ("k", KV_DIM, HIDDEN), ("v", KV_DIM, HIDDEN),
                  ("o", HIDDEN, HIDDEN), ("gate", FFN, HIDDEN), ("up", FFN, HIDDEN),
                  ("down", HIDDEN, FFN))


def decode_layout(n_layers: int = N_LAYERS):
    """The decode sweep's matmul list: (layer, index, name, fmt, N, K).

    q, k, o, gate, up are Q4_K.  v and down are Q6_K in even layers and Q4_K in
    odd layers (14 of 28 layers carry a Q6_K attn_v, the q4_K_m mix).
    """
    out = []
    for layer in range(n_layers):
        for idx, (name, n, k) in enumerate(LAYER_MATRICES):
            fmt = "q6k" if (name in ("v", "down") and layer % 2 == 0) else "q4k"
            out.append((layer, idx, name, fmt, n, k))
    return out


def decode_matrix(layer: int, idx: int):
    """Weight bytes and the 1 x K activation for one matmul of the decode sweep."""
    _, _, name, fmt, n, k = next(e for e in decode_layout(layer + 1) if e[0] == layer and e[1] == idx)
    gen = q6k_weights if fmt == "q6k" else q4k_weights
    w = gen(rng(3, STREAM_W, layer, idx), n, k)
    x = activations(rng(3, STREAM_X, layer, idx), 1, k)
    return {"w": w, "x": x, "fmt": fmt, "name": name}


def q5k_vocab_weights():
    """Synthetic Q5_K weights of the LM-head shape (VOCAB x HIDDEN), for the Q5_K decode GEMV."""
    return q5k_weights(rng(4, STREAM_W, 5), VOCAB, HIDDEN)


def b32_vocab_weights(fmt: str):
    """Synthetic weights of the LM-head shape (VOCAB x HIDDEN) in a 32-value block format, for
    that format's decode GEMV (one seed stream per format)."""
    return b32_weights(rng(4, STREAM_W, 6 + list(B32_BYTES).index(fmt)), VOCAB, HIDDEN, fmt)


def lm_head_weights():
    """LM head weights: 152064 x 3584 Q6_K (int8 scales over the whole range), 447,068,160 bytes."""
    return q6k_weights(rng(4, STREAM_W), VOCAB, HIDDEN)


def ffn_swiglu_inputs(m: int = PREFILL_TOKENS):
    """The down projection's SwiGLU producer inputs at the 7B FFN prefill size: gate, up m x 18944."""
    return swiglu_inputs(rng(2, STREAM_SWIGLU), m, FFN)


def lm_head_x(m: int):
    """LM head activations: m x 3584 f32 N(0,1), m in {1, 16, 3314}."""
    return activations(rng(4, STREAM_X, m), m, HIDDEN)


def lm_head_case(m: int):
    """LM head: W 152064 x 3584 (Q6_K, int8 scales over the whole range), X m x 3584 N(0,1), m in {1, 16, 3314}."""
    return {"w": lm_head_weights(), "x": lm_head_x(m), "fmt": "q6k"}
