"""Pins of the oracle's Q2_K / Q3_K / q8_1 code (no GPU).

The pages name the formats (page spark_model/layers/moe_v41.rs: gate and up
in Q2_K, down in Q3_K, activation in q8_1) but print no layout; the oracle
takes the public GGUF layouts. Each test below builds blocks byte by byte with
patterns whose weights have a closed form, so a wrong byte, shift, nibble or
sign in the decoder fails one of them.
"""
import numpy as np
import pytest

import oracle
from moe_decode_quantized_gb300 import synth

F16_ONE, F16_HALF = 0x3C00, 0x3800


def _q2k(scales, qs, d=F16_ONE, dmin=F16_HALF):
    b = np.zeros(84, np.uint8)
    b[0:16] = scales
    b[16:80] = qs
    b[80], b[81] = d & 0xFF, d >> 8
    b[82], b[83] = dmin & 0xFF, dmin >> 8
    return b


def test_q2k_quant_index_pattern_lane():
    # scale nibble of sub-block s = s % 16, min nibble = 15 - s % 16
    scales = np.array([(s % 16) | ((15 - s % 16) << 4) for s in range(16)], np.uint8)
    # every qs byte i holds the value (i % 4) in all four 2-bit fields: then
    # weight j must read q = j % 4 (its byte index is congruent to j mod 4)
    qs = np.array([(i % 4) * 0x55 for i in range(64)], np.uint8)
    w = oracle.dequant_q2k(_q2k(scales, qs))[0]
    for j in range(256):
        s = j // 16
        assert w[j] == 1.0 * s * (j % 4) - 0.5 * (15 - s), j


def test_q2k_quant_shift_pattern():
    # byte 0xE4 = fields (0, 1, 2, 3) from the low bits: weight j reads field
    # (j % 128) // 32, i.e. its quant is its 32-weight group inside the half
    scales = np.full(16, 0x0F | (3 << 4), np.uint8)     # scale 15, min 3
    qs = np.full(64, 0xE4, np.uint8)
    w = oracle.dequant_q2k(_q2k(scales, qs))[0]
    for j in range(256):
        assert w[j] == 15.0 * ((j % 128) // 32) - 0.5 * 3, j


def test_q2k_half_pattern_and_factors():
    # bytes 0..31 all zero, 32..63 all 0xFF: weights 0..127 read 0, 128..255 read 3
    scales = np.full(16, 0x21, np.uint8)                # scale 1, min 2
    qs = np.concatenate([np.zeros(32, np.uint8), np.full(32, 0xFF, np.uint8)])
    d, dmin = 0x4000, 0x3400                           # 2.0, 0.25
    w = oracle.dequant_q2k(_q2k(scales, qs, d, dmin))[0]
    for j in range(256):
        q = 3 if j >= 128 else 0
        assert w[j] == 2.0 * 1 * q - 0.25 * 2, j


def test_q2k_zero_block_is_zero():
    assert not oracle.dequant_q2k(np.zeros(84, np.uint8)).any()


def _q3k(hmask, qs, sc, d=F16_ONE):
    b = np.zeros(110, np.uint8)
    b[0:32] = hmask
    b[32:96] = qs
    b[96:108] = sc
    b[108], b[109] = d & 0xFF, d >> 8
    return b


def test_q3k_closed_form():
    # scales: bytes 0..7 = 0x21 -> low 4 bits 1 (scales 0..7) and 2 (scales
    # 8..15); bytes 8..11 = 0xE4 -> high 2 bits of scale i = i // 4; with the
    # +32 offset: scale = [-31, -15, 2, 18][i // 4]
    sc = np.array([0x21] * 8 + [0xE4] * 4, np.uint8)
    # hmask bytes 0xF0: high bit set for weights j >= 128 (bit j // 32 >= 4)
    hmask = np.full(32, 0xF0, np.uint8)
    # qs bytes 0x1B: field g (bits 2g) = 3 - g
    qs = np.full(64, 0x1B, np.uint8)
    w = oracle.dequant_q3k(_q3k(hmask, qs, sc))[0]
    for j in range(256):
        g = (j % 128) // 32
        q = (3 - g) - (0 if j >= 128 else 4)
        scale = [-31, -15, 2, 18][(j // 16) // 4]
        assert w[j] == 1.0 * scale * q, j


def test_q3k_hmask_bit_per_group():
    # hmask byte l = 1 << (l % 8): weight j has its high bit iff j // 32 == (j % 32) % 8
    hmask = np.array([1 << (l % 8) for l in range(32)], np.uint8)
    qs = np.zeros(64, np.uint8)                       # low bits all 0
    sc = np.array([0x11] * 8 + [0xAA] * 4, np.uint8)  # low4 1, high2 2 -> 33 - 32 = 1
    w = oracle.dequant_q3k(_q3k(hmask, qs, sc, 0x4000))[0]
    for j in range(256):
        hb = (j // 32) == ((j % 32) % 8)
        assert w[j] == 2.0 * 1 * (0 if hb else -4), j


def _int_form_q2k_dot(blk, xq8_blocks):
    """Integer form: per 32-block, d8 * (d * sum_s sc_s * sum q*q8 - dmin * sum_s m_s * sum q8)."""
    sc = blk[0:16]
    qs = blk[16:80]
    d = np.array([int(blk[80]) | (int(blk[81]) << 8)], np.uint16).view(np.float16)[0]
    dmin = np.array([int(blk[82]) | (int(blk[83]) << 8)], np.uint16).view(np.float16)[0]
    q = np.zeros(256, np.int64)
    for j in range(256):
        q[j] = (int(qs[32 * (j // 128) + j % 32]) >> (2 * ((j % 128) // 32))) & 3
    total = 0.0
    for b in range(8):
        xb = xq8_blocks[b]
        d8 = float(np.array([int(xb[0]) | (int(xb[1]) << 8)], np.uint16).view(np.float16)[0])
        q8 = xb[4:36].view(np.int8).astype(np.int64)
        main = 0
        mins = 0
        for half in range(2):
            s = 2 * b + half
            seg = slice(16 * half, 16 * half + 16)
            main += int(sc[s] & 15) * int(np.dot(q[32 * b:32 * b + 32][seg], q8[seg]))
            mins += int(sc[s] >> 4) * int(q8[seg].sum())
        total += d8 * (float(d) * main - float(dmin) * mins)
    return total


def test_q2k_dot_integer_form_equals_dequant_form():
    rng = np.random.default_rng(4)
    blocks = synth.q2k_blocks(synth.tensor_key(7, 0, synth.T_GATE, 0), 6)
    for i in range(blocks.shape[0]):
        x = (rng.standard_normal(256) * 1.3).astype(np.float32)
        xq = oracle.quant_q8_1(x)
        xv = oracle.dequant_q8_1(xq).ravel()
        w = oracle.dequant_q2k(blocks[i])[0]
        assert np.isclose(np.dot(w, xv), _int_form_q2k_dot(blocks[i], xq), rtol=1e-12, atol=1e-12)


def test_one_hot_activation_returns_a_column():
    blocks = synth.q3k_blocks(synth.tensor_key(7, 0, synth.T_DOWN, 1), 1)
    w = oracle.dequant_q3k(blocks[0])[0]
    for j in (0, 37, 128, 255):
        x = np.zeros(256, np.float32)
        x[j] = 1.0
        xv = oracle.dequant_q8_1(oracle.quant_q8_1(x)).ravel()
        # the single nonzero quant is 127 at scale f16(1 / 127)
        one = float(np.float16(np.float32(1.0) / np.float32(127.0))) * 127
        assert xv[j] == one and np.count_nonzero(xv) == 1
        assert np.dot(w, xv) == w[j] * one


# ------------------------------------------------------------------ q8_1

def test_q8_1_layout_and_round_trip_bound():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal(32 * 64) * rng.uniform(0.01, 10, 2048)).astype(np.float32)
    blocks = oracle.quant_q8_1(x)
    for b in range(64):
        xb = x[32 * b:32 * b + 32]
        amax = np.float32(np.abs(xb).max())
        d = np.float32(amax / np.float32(127.0))
        q = blocks[b, 4:].view(np.int8).astype(np.int64)
        # the stored scale is f16(d), the stored sum f16(d * sum q)
        assert int(blocks[b, 0]) | (int(blocks[b, 1]) << 8) == np.float16(d).view(np.uint16)
        s = np.float32(d * np.float32(q.sum()))
        assert int(blocks[b, 2]) | (int(blocks[b, 3]) << 8) == np.float16(s).view(np.uint16)
        # |x - d q| <= d / 2 elementwise (q = round(x / d)), the max maps to +-127
        assert np.all(np.abs(xb.astype(np.float64) - float(d) * q) <= float(d) * 0.5 * (1 + 1e-6))
        i = int(np.argmax(np.abs(xb)))
        assert abs(q[i]) == 127 and np.sign(q[i]) == np.sign(xb[i])


def test_q8_1_zero_block_and_half_away_rounding():
    z = oracle.quant_q8_1(np.zeros(32, np.float32))
    assert not z.any()
    # amax 127 -> d = 1: x / d = k + 0.5 must round away from zero
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1], x[2], x[3], x[4] = 2.5, -2.5, 0.5, -0.5
    q = oracle.quant_q8_1(x)[0, 4:].view(np.int8)
    assert list(q[:5]) == [127, 3, -3, 1, -1]


def test_quantisers_reproduce_their_input_within_one_step():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal(256 * 4) * 0.02).astype(np.float32)
    w2 = oracle.dequant_q2k(oracle.quantize_q2k(x)).ravel()
    w3 = oracle.dequant_q3k(oracle.quantize_q3k(x)).ravel()
    # the codes are input-making only; a coarse bound is enough
    assert np.abs(w2 - x).max() < 0.03
    assert np.abs(w3 - x).max() < 0.03
    assert np.corrcoef(w2, x)[0, 1] > 0.9 and np.corrcoef(w3, x)[0, 1] > 0.9
