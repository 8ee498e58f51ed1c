"""Pins for the oracle's binary16 conversions and Q4_K / Q5_K / Q6_K block decoders.

Pinned against: numpy's binary16 conversions (a library routine, exhaustive or
dense samples), hand-worked single blocks, and round trips through the
independent encoders in kquant_pack.py.
"""
import numpy as np
import pytest

import oracle
from tests.kquant_pack import pack_q4k, pack_q5k, pack_q6k, q4k_expected, q5k_expected, q6k_expected


def test_f16_decode_exhaustive_matches_numpy():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.f16_to_f64(h)
    ref = h.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _f32_to_f16_ref(f):
    with np.errstate(over="ignore"):
        return f.astype(np.float16).view(np.uint16)


def test_f32_to_f16_specials_and_ties():
    vals = [0.0, -0.0, 1.0, -1.0, 65504.0, 65519.996, 65520.0, 65536.0, 1e9, -1e9,
            np.inf, -np.inf, 2.0 ** -14, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 * 1.0000001,
            2.0 ** -26, 3 * 2.0 ** -25, 1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11,
            2048.0 + 1.0, 2048.0 + 3.0, 6.1e-5, 5.96e-8, 1.0e-40]
    f = np.array(vals, np.float32)
    assert np.array_equal(oracle.f32_to_f16(f), _f32_to_f16_ref(f))
    nanbits = oracle.f32_to_f16(np.array([np.nan], np.float32))
    assert np.isnan(nanbits.view(np.float16)[0])


def test_f32_to_f16_dense_random_bit_patterns():
    rng = np.random.default_rng(1234)
    bits = rng.integers(0, 2 ** 32, size=1 << 22, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    got = oracle.f32_to_f16(f)
    ref = _f32_to_f16_ref(f)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(got[nan].view(np.float16)))


def test_f32_to_f16_all_values_near_half_range():
    # every binary32 in [2^-26, 2^17): all binary16 exponents, subnormal and
    # overflow boundaries, every tie, sampled with stride 7 (~13M values)
    lo = np.array(2.0 ** -26, np.float32).view(np.uint32)
    hi = np.array(2.0 ** 17, np.float32).view(np.uint32)
    bits = np.arange(lo, hi, 7, dtype=np.uint32)
    f = bits.view(np.float32)
    assert np.array_equal(oracle.f32_to_f16(f), _f32_to_f16_ref(f))
    assert np.array_equal(oracle.f32_to_f16(-f), _f32_to_f16_ref(-f))


# ------------------------------------------------------------------- Q4_K
def test_q4k_hand_worked_block():
    # d = 0.5, dmin = 0.25, sub-block 0 scale 3 min 1, weight 0 code 5:
    # weight 0 = 0.5*3*5 - 0.25*1 = 7.25; the rest of sub-block 0 has code 0
    # (-0.25); sub-blocks 1..7 have scale = min = 0 (0.0).
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [0x00, 0x38]      # 0x3800 = 0.5
    blk[2:4] = [0x00, 0x34]      # 0x3400 = 0.25
    blk[4 + 0] = 3               # scale of sub-block 0
    blk[4 + 4] = 1               # min of sub-block 0
    blk[16 + 0] = 0x05           # low nibble of code byte 0 -> weight 0
    w = oracle.q4k_block(blk)
    assert w[0] == 7.25
    assert np.all(w[1:32] == -0.25)
    assert np.all(w[32:] == 0.0)


def test_q4k_top_bits_of_low_scales_feed_sub_block_4():
    # packed byte 0 = 0x43: sub-block 0 scale keeps 3 (low six bits); its top
    # two bits (01) become bits 4-5 of sub-block 4's scale -> 16.
    blk = np.zeros(144, np.uint8)
    blk[0:2] = [0x00, 0x3C]      # d = 1.0
    blk[4 + 0] = 0x43
    blk[16:144] = 0x11           # every code = 1
    w = oracle.q4k_block(blk)
    assert oracle.q4k_scale_min(blk[4:16], 0) == (3, 0)
    assert oracle.q4k_scale_min(blk[4:16], 4) == (16, 0)
    assert np.all(w[0:32] == 3.0)
    assert np.all(w[128:160] == 16.0)
    assert np.all(w[32:128] == 0.0) and np.all(w[160:] == 0.0)


@pytest.mark.parametrize("j", range(8))
def test_q4k_one_hot_scale_selects_sub_block(j):
    sc = [0] * 8
    sc[j] = 1
    blk = pack_q4k(1.0, 0.0, sc, [0] * 8, [1] * 256)
    w = oracle.q4k_block(blk)
    ref = np.zeros(256, np.float32)
    ref[32 * j:32 * j + 32] = 1.0
    assert np.array_equal(w, ref)


def test_q4k_one_hot_code_positions():
    for i in range(256):
        q = [0] * 256
        q[i] = 15
        blk = pack_q4k(1.0, 0.0, [1] * 8, [0] * 8, q)
        w = oracle.q4k_block(blk)
        assert w[i] == 15.0 and np.count_nonzero(w) == 1, i


def test_q4k_encoder_round_trip_random_fields():
    rng = np.random.default_rng(7)
    for _ in range(300):
        d = float(rng.uniform(1e-4, 2.0))
        dmin = float(rng.uniform(0.0, 1.0))
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        q = rng.integers(0, 16, 256)
        blk = pack_q4k(d, dmin, sc, mn, q)
        assert np.array_equal(oracle.q4k_block(blk), q4k_expected(d, dmin, sc, mn, q))


def test_q4k_extreme_and_subnormal_halves():
    # largest finite half d and a subnormal dmin: still an exact fp64 value
    # rounded once
    sc = [63] * 8
    mn = [63] * 8
    q = list(range(16)) * 16
    for d, dmin in [(65504.0, 2.0 ** -24), (2.0 ** -24, 65504.0), (6.0e-5, 3.0e-7)]:
        blk = pack_q4k(d, dmin, sc, mn, q)
        assert np.array_equal(oracle.q4k_block(blk), q4k_expected(d, dmin, sc, mn, q))


def test_q4k_zero_scales_give_zero():
    rng = np.random.default_rng(3)
    blk = rng.integers(0, 256, 144).astype(np.uint8)
    blk[0:4] = 0                 # d = dmin = +0
    assert np.all(oracle.q4k_block(blk) == 0.0)


# ------------------------------------------------------------------- Q5_K
def test_q5k_hand_worked_block():
    # d = 0.5, dmin = 0.25; sub-block 0: scale 3, min 1; sub-block 1: scale 2;
    # sub-block 2: scale 1.
    #   weight 0:  low nibble 5 of code byte 0, fifth bit (qh[0] bit 0) -> q 21:
    #              0.5*3*21 - 0.25 = 31.25
    #   weight 1:  fifth bit only (qh[1] bit 0) -> q 16: 24 - 0.25 = 23.75
    #   weight 32: high nibble 7 of code byte 0, qh[0] bit 1 -> q 23: 0.5*2*23 = 23
    #   weight 67: chunk 1, l = 3: qh[3] bit 2 -> q 16: 0.5*1*16 = 8
    # the rest of sub-block 0 is -0.25, everything else 0.
    blk = np.zeros(176, np.uint8)
    blk[0:2] = [0x00, 0x38]      # d = 0.5
    blk[2:4] = [0x00, 0x34]      # dmin = 0.25
    blk[4 + 0] = 3
    blk[4 + 1] = 2
    blk[4 + 2] = 1
    blk[4 + 4] = 1
    blk[16 + 0] = 0b11
    blk[16 + 1] = 0b01
    blk[16 + 3] = 0b100
    blk[48 + 0] = 0x75
    w = oracle.q5k_block(blk)
    ref = np.zeros(256, np.float32)
    ref[0:32] = -0.25
    ref[0], ref[1], ref[32], ref[67] = 31.25, 23.75, 23.0, 8.0
    assert np.array_equal(w, ref)


def test_q5k_without_fifth_bits_is_q4k():
    # a Q5_K block whose qh is zero decodes as the Q4_K block with the same
    # header and code bytes; with every fifth bit set each weight gains 16*d*sc
    rng = np.random.default_rng(21)
    for _ in range(50):
        b4 = rng.integers(0, 256, 144).astype(np.uint8)
        b4[0:2] = np.array([np.float16(rng.uniform(1e-3, 1.0))]).view(np.uint8)
        b4[2:4] = np.array([np.float16(rng.uniform(0.0, 1.0))]).view(np.uint8)
        b5 = np.concatenate([b4[:16], np.zeros(32, np.uint8), b4[16:]])
        assert np.array_equal(oracle.q5k_block(b5), oracle.q4k_block(b4))
        b5[16:48] = 0xFF
        d = float(b4[0:2].view(np.float16)[0])
        sc = [oracle.q4k_scale_min(b4[4:16], j)[0] for j in range(8)]
        # d*sc*(q + 16) - dmin*m, exact in fp64 and rounded once
        dmin = float(b4[2:4].view(np.float16)[0])
        mn = [oracle.q4k_scale_min(b4[4:16], j)[1] for j in range(8)]
        qs = b4[16:144]
        low = [(int(qs[32 * (i // 64) + i % 32]) >> (4 * ((i % 64) >= 32))) & 15 for i in range(256)]
        exact = np.array([d * sc[i // 32] * (low[i] + 16) - dmin * mn[i // 32] for i in range(256)])
        assert np.array_equal(oracle.q5k_block(b5), exact.astype(np.float32))


def test_q5k_one_hot_fifth_bit_positions():
    for i in range(256):
        q = [0] * 256
        q[i] = 16
        blk = pack_q5k(1.0, 0.0, [1] * 8, [0] * 8, q)
        w = oracle.q5k_block(blk)
        assert w[i] == 16.0 and np.count_nonzero(w) == 1, i


@pytest.mark.parametrize("j", range(8))
def test_q5k_one_hot_scale_selects_sub_block(j):
    sc = [0] * 8
    sc[j] = 1
    blk = pack_q5k(1.0, 0.0, sc, [0] * 8, [31] * 256)
    ref = np.zeros(256, np.float32)
    ref[32 * j:32 * j + 32] = 31.0
    assert np.array_equal(oracle.q5k_block(blk), ref)


def test_q5k_encoder_round_trip_random_fields():
    rng = np.random.default_rng(13)
    for _ in range(300):
        d = float(rng.uniform(1e-4, 2.0))
        dmin = float(rng.uniform(0.0, 1.0))
        sc = rng.integers(0, 64, 8)
        mn = rng.integers(0, 64, 8)
        q = rng.integers(0, 32, 256)
        blk = pack_q5k(d, dmin, sc, mn, q)
        assert np.array_equal(oracle.q5k_block(blk), q5k_expected(d, dmin, sc, mn, q))
    for d, dmin in [(65504.0, 2.0 ** -24), (2.0 ** -24, 65504.0)]:
        sc, mn, q = [63] * 8, [63] * 8, list(range(32)) * 8
        blk = pack_q5k(d, dmin, sc, mn, q)
        assert np.array_equal(oracle.q5k_block(blk), q5k_expected(d, dmin, sc, mn, q))


# ------------------------------------------------------------------- Q6_K
def test_q6k_hand_worked_block():
    # d = 1, scale[0] = 2, low nibble 1 and high bits 2 for weight 0 -> q = 33,
    # w = 2*(33-32) = 2; other sub-block-0 weights have q = 0 -> 2*(-32) = -64.
    blk = np.zeros(210, np.uint8)
    blk[208:210] = [0x00, 0x3C]
    blk[192] = 2
    blk[0] = 0x01
    blk[128] = 0x02
    w = oracle.q6k_block(blk)
    assert w[0] == 2.0
    assert np.all(w[1:16] == -64.0)
    assert np.all(w[16:] == 0.0)


def test_q6k_group_positions():
    # the four 2-bit fields of qh[l] are the high bits of weights l, l+32,
    # l+64, l+96; the ql nibbles: low of ql[l] -> l, low of ql[l+32] -> l+32,
    # high of ql[l] -> l+64, high of ql[l+32] -> l+96 (first half).
    blk = np.zeros(210, np.uint8)
    blk[208:210] = [0x00, 0x3C]
    blk[192:208] = 1
    blk[128 + 5] = 0b11_10_01_00   # fields 0,1,2,3 for weights 5, 37, 69, 101
    blk[5] = 0x00
    blk[37] = 0x00
    w = oracle.q6k_block(blk)
    assert w[5] == 0 - 32 and w[37] == 16 - 32 and w[69] == 32 - 32 and w[101] == 48 - 32


def test_q6k_one_hot_code_positions():
    for i in range(256):
        q = [32] * 256
        q[i] = 63
        blk = pack_q6k(1.0, [1] * 16, q)
        w = oracle.q6k_block(blk)
        assert w[i] == 31.0 and np.count_nonzero(w) == 1, i


@pytest.mark.parametrize("s", range(16))
def test_q6k_one_hot_scale_selects_sub_block(s):
    sc = [0] * 16
    sc[s] = -3
    blk = pack_q6k(1.0, sc, [33] * 256)
    w = oracle.q6k_block(blk)
    ref = np.zeros(256, np.float32)
    ref[16 * s:16 * s + 16] = -3.0
    assert np.array_equal(w, ref)


def test_q6k_encoder_round_trip_random_fields():
    rng = np.random.default_rng(11)
    for _ in range(300):
        d = float(rng.uniform(1e-4, 4.0))
        sc = rng.integers(-128, 128, 16)
        q = rng.integers(0, 64, 256)
        blk = pack_q6k(d, sc, q)
        assert np.array_equal(oracle.q6k_block(blk), q6k_expected(d, sc, q))


def test_dequantize_matrix_is_blockwise():
    import synth
    W = synth.q6k_matrix(3, 512, seed=5)
    full = oracle.dequantize("q6_k", W, 3, 512)
    for r in range(3):
        for b in range(2):
            blk = W[r, b * 210:(b + 1) * 210]
            assert np.array_equal(full[r, b * 256:(b + 1) * 256], oracle.q6k_block(blk))
    W4 = synth.q4k_matrix(2, 768, seed=6)
    full4 = oracle.dequantize("q4_k", W4, 2, 768)
    for r in range(2):
        for b in range(3):
            blk = W4[r, b * 144:(b + 1) * 144]
            assert np.array_equal(full4[r, b * 256:(b + 1) * 256], oracle.q4k_block(blk))
    W5 = synth.q5k_matrix(2, 512, seed=7)
    full5 = oracle.dequantize("q5_k", W5, 2, 512)
    for r in range(2):
        for b in range(2):
            blk = W5[r, b * 176:(b + 1) * 176]
            assert np.array_equal(full5[r, b * 256:(b + 1) * 256], oracle.q5k_block(blk))
