"""Pins for the oracle's block decoders (C1 Q4_K, C1' Q5_K, C2 Q6_K) and its fp16 decode.

What pins them, besides the oracle itself:
* numpy's float16 (an independent library routine) for every fp16 bit pattern;
* hand-built blocks whose decodes were worked out by hand (tests/golden);
* bijectivity of the quant-position maps (every (byte, nibble/bit) slot feeds exactly
  one element, every element is fed by exactly one slot);
* the 144 / 176 / 210 byte block sizes and the config value ranges;
* Q5_K's scale fields decoded against Q4_K's (the same 12 bytes, the same packing).
"""
import numpy as np
import pytest

import oracle
from quantized_q8_activation_quantize_gb300 import inputs
from tests import golden_blocks


def test_half_to_double_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("blk", golden_blocks.load(), ids=lambda b: b["name"])
def test_hand_built_blocks(blk):
    b = blk["bytes"]
    if blk["fmt"] in oracle.B32:
        assert b.size == oracle.B32[blk["fmt"]][0]
        d, m, q = oracle.b32_fields(b, blk["fmt"])
        assert d == blk["d"]
        for e, v in blk["q"].items():
            assert q[e] == v, f"q[{e}]"
        deq = oracle.dequantize(b.reshape(1, 1, -1), blk["fmt"])[0]
        for e, v in blk["value"].items():
            assert deq[e] == v, f"value[{e}]"
        return
    if blk["fmt"] in ("q4k", "q5k"):
        assert b.size == (144 if blk["fmt"] == "q4k" else 176)
        d, dmin, sc, mn, q = (oracle.q4k_fields if blk["fmt"] == "q4k" else oracle.q5k_fields)(b)
        assert d == blk["d"] and dmin == blk["dmin"]
        assert sc.tolist() == blk["sc"] and mn.tolist() == blk["m"]
    else:
        assert b.size == 210
        d, sc, q = oracle.q6k_fields(b)
        if "d" in blk:
            assert d == blk["d"]
        if "sc" in blk:
            assert sc.tolist() == blk["sc"]
    for e, v in blk["q"].items():
        assert q[e] == v, f"q[{e}]"
    deq = oracle.dequantize(b.reshape(1, 1, -1), blk["fmt"])[0]
    for e, v in blk["value"].items():
        assert deq[e] == v, f"value[{e}]"


def test_block_sizes():
    r = np.random.default_rng(0)
    assert inputs.q4k_weights(r, 3, 512).shape == (3, 2, 144)
    assert inputs.q5k_weights(r, 3, 512).shape == (3, 2, 176)
    assert inputs.q6k_weights(r, 3, 512).shape == (3, 2, 210)
    assert (inputs.Q4K_BYTES, inputs.Q5K_BYTES, inputs.Q6K_BYTES) == (144, 176, 210)
    # 4.5, 5.5 and 6.5625 bits per weight
    assert inputs.Q4K_BYTES * 8 / 256 == 4.5 and inputs.Q5K_BYTES * 8 / 256 == 5.5
    assert inputs.Q6K_BYTES * 8 / 256 == 6.5625


def test_q4k_quant_slots_are_a_bijection():
    # Set one nibble of qs to 1 at a time (all scales 1, d 1, dmin 0): exactly one element
    # must decode to 1, and over all 256 slots every element must be hit once.
    hit = np.zeros(256, int)
    base = np.zeros(144, np.uint8)
    base[0:2] = [0x00, 0x3C]                     # d = 1
    base[4:8] = 1                                 # sc0..3 = 1
    base[12:16] = 0x01                            # sc4..7 = 1, m4..7 = 0
    for byte in range(128):
        for nib in range(2):
            b = base.copy()
            b[16 + byte] = 1 << (4 * nib)
            _, _, sc, mn, q = oracle.q4k_fields(b)
            assert sc.tolist() == [1] * 8 and mn.tolist() == [0] * 8
            nz = np.flatnonzero(q)
            assert nz.size == 1 and q[nz[0]] == 1
            hit[nz[0]] += 1
            # each 32-element sub-block draws all its quants from one 32-byte run of qs
            assert nz[0] // 64 == byte // 32
    assert (hit == 1).all()


def test_q4k_scale_fields_are_a_bijection_of_the_96_bits():
    # Each of the 96 bits of the 12 scale bytes must land in exactly one of the 16 six-bit
    # fields (8 scales, 8 mins), each field bit being fed exactly once.
    seen = np.zeros((2, 8, 6), int)
    for bit in range(96):
        b = np.zeros(144, np.uint8)
        b[4 + bit // 8] = 1 << (bit % 8)
        _, _, sc, mn, _ = oracle.q4k_fields(b)
        vals = np.concatenate([sc, mn])
        nz = np.flatnonzero(vals)
        assert nz.size == 1
        v = vals[nz[0]]
        assert v & (v - 1) == 0 and v < 64
        seen[nz[0] // 8, nz[0] % 8, int(np.log2(v))] += 1
    assert (seen == 1).all()


def test_q6k_quant_slots_are_a_bijection():
    # low nibbles: one ql nibble at a time -> exactly one element moves from -32
    hit = np.zeros(256, int)
    for byte in range(128):
        for nib in range(2):
            b = np.zeros(210, np.uint8)
            b[192:208] = 1
            b[208:210] = [0x00, 0x3C]
            b[byte] = 1 << (4 * nib)
            _, sc, q = oracle.q6k_fields(b)
            nz = np.flatnonzero(q != -32)
            assert nz.size == 1 and q[nz[0]] == -31
            hit[nz[0]] += 1
    assert (hit == 1).all()
    # high bit pairs: one qh bit pair at a time -> exactly one element gets +16
    hit = np.zeros(256, int)
    for byte in range(64):
        for pair in range(4):
            b = np.zeros(210, np.uint8)
            b[128 + byte] = 1 << (2 * pair)
            _, _, q = oracle.q6k_fields(b)
            nz = np.flatnonzero(q != -32)
            assert nz.size == 1 and q[nz[0]] == -16
            hit[nz[0]] += 1
    assert (hit == 1).all()


def test_q6k_scale_per_16_elements():
    # one-hot scale s -> exactly elements 16s..16s+15 are non-zero
    for s in range(16):
        b = np.zeros(210, np.uint8)
        b[0:128] = 0x11                          # low nibbles 1 -> q = -31 everywhere
        b[192 + s] = 2
        b[208:210] = [0x00, 0x3C]
        deq = oracle.dequantize(b.reshape(1, 1, 210), "q6k")[0]
        nz = np.flatnonzero(deq)
        assert nz.tolist() == list(range(16 * s, 16 * s + 16))
        assert (deq[nz] == -62).all()


def test_generated_value_ranges():
    w = inputs.tiny_q4k()["w"]
    ds = np.array([[oracle.q4k_fields(w[n, b])[:2] for b in range(w.shape[1])] for n in range(w.shape[0])])
    assert ds.min() >= np.float16(1e-3) and ds.max() <= np.float16(1e-2)
    _, _, sc, mn, q = oracle.q4k_fields(w[0, 0])
    assert sc.max() < 64 and mn.max() < 64 and q.min() >= 0 and q.max() <= 15
    w6 = inputs.q6k_weights(inputs.rng(2, 0, 2), 4, 3584)
    for n in range(4):
        for b in range(w6.shape[1]):
            d, sc, q = oracle.q6k_fields(w6[n, b])
            assert 1e-3 * 0.999 <= d <= 1e-2 * 1.001
            assert sc.min() >= -128 and sc.max() <= 127 and q.min() >= -32 and q.max() <= 31
    # the default scale range is the whole int8 range: odd scales above 64 in magnitude occur
    sc_all = np.array([oracle.q6k_fields(w6[n, b])[1] for n in range(4) for b in range(w6.shape[1])])
    assert ((np.abs(sc_all.astype(int)) > 64) & (sc_all % 2 != 0)).any()



def test_q5k_quant_slots_are_a_bijection():
    # low nibbles: one qs nibble at a time (all scales 1, d 1, dmin 0) -> exactly one element
    # decodes to 1, every element once; high bits: one qh bit at a time -> exactly one
    # element decodes to 16, every element once
    base = np.zeros(176, np.uint8)
    base[0:2] = [0x00, 0x3C]
    base[4:8] = 1
    base[12:16] = 0x01
    for lo, n_slots, val in ((48, 256, 1), (16, 256, 16)):
        hit = np.zeros(256, int)
        for slot in range(n_slots):
            b = base.copy()
            if lo == 48:
                b[48 + slot // 2] = 1 << (4 * (slot % 2))
            else:
                b[16 + slot // 8] = 1 << (slot % 8)
            _, _, sc, mn, q = oracle.q5k_fields(b)
            assert sc.tolist() == [1] * 8 and mn.tolist() == [0] * 8
            nz = np.flatnonzero(q)
            assert nz.size == 1 and q[nz[0]] == val
            if lo == 16:
                # qh byte l feeds position l of every sub-block; bit j selects sub-block j
                assert nz[0] == 32 * (slot % 8) + slot // 8
            hit[nz[0]] += 1
        assert (hit == 1).all()


def test_q5k_scales_and_low_bits_match_q4k():
    # the same d, dmin, 12 scale bytes and 128 qs bytes decode to the same sc, m and low
    # four bits in both formats; Q5_K adds 16 * (its qh bit)
    r = np.random.default_rng(11)
    for _ in range(20):
        b5 = np.frombuffer(r.bytes(176), np.uint8).copy()
        b4 = np.concatenate([b5[0:16], b5[48:176]])
        d4, m4, sc4, mn4, q4 = oracle.q4k_fields(b4)
        d5, m5, sc5, mn5, q5 = oracle.q5k_fields(b5)
        assert (d4, m4) == (d5, m5) and np.array_equal(sc4, sc5) and np.array_equal(mn4, mn5)
        assert np.array_equal(q5 % 16, q4) and q5.max() <= 31
        qh = np.unpackbits(b5[16:48].reshape(32, 1), axis=1, bitorder="little")   # [l][j]
        assert np.array_equal(q5 // 16, qh.T.reshape(256))


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q5_0", "q5_1", "q8_0"])
def test_b32_quant_slots_are_a_bijection(fmt):
    # with d = 1 and m = 0, setting one quant bit-field slot at a time moves exactly one
    # element away from the all-zero block's integer, and every element is moved once
    nbytes = oracle.B32[fmt][0]
    base = np.zeros(nbytes, np.uint8)
    base[0:2] = [0x00, 0x3C]
    _, _, q0 = oracle.b32_fields(base, fmt)
    if fmt == "q8_0":
        slots = [(2 + l, 1) for l in range(32)]
    else:
        qs = nbytes - 16
        slots = [(qs + byte, 1 << (4 * nib)) for byte in range(16) for nib in range(2)]
        if fmt in ("q5_0", "q5_1"):
            qh = qs - 4
            slots += [(qh + bit // 8, 1 << (bit % 8)) for bit in range(32)]
    hit = np.zeros(32, int)
    for pos, val in slots:
        b = base.copy()
        b[pos] |= val
        _, _, q = oracle.b32_fields(b, fmt)
        nz = np.flatnonzero(q != q0)
        assert nz.size == 1, (pos, val, nz)
        hit[nz[0]] += 1
    assert (hit == (2 if fmt in ("q5_0", "q5_1") else 1)).all()   # Q5: a nibble slot and a bit slot each


@pytest.mark.parametrize("fmt", ["q4_0", "q4_1", "q5_0", "q5_1", "q8_0"])
def test_b32_generated_ranges(fmt):
    w = inputs.b32_weights(np.random.default_rng(3), 5, 256, fmt)
    assert w.shape == (5, 8, inputs.B32_BYTES[fmt])
    lo = {"q4_0": -8, "q4_1": 0, "q5_0": -16, "q5_1": 0, "q8_0": -128}[fmt]
    hi = {"q4_0": 7, "q4_1": 15, "q5_0": 15, "q5_1": 31, "q8_0": 127}[fmt]
    for n in range(5):
        for b in range(8):
            d, m, q = oracle.b32_fields(w[n, b], fmt)
            assert 1e-3 * 0.999 <= d <= 1e-2 * 1.001
            assert (m == 0.0) if fmt in ("q4_0", "q5_0", "q8_0") else (-0.08 * 1.001 <= m <= 0.0)
            assert q.min() >= lo and q.max() <= hi
