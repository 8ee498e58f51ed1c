"""Pins for the oracle's binary16 conversions and Q4_K / Q6_K block decoders.

Pinned against: numpy's binary16 conversions (a library routine, exhaustive or
dense samples), hand-worked single blocks, and round trips through the
independent encoders in kquant_pack.py.
"""
import numpy as np
import pytest

import oracle
from tests.kquant_pack import pack_q4k, pack_q6k, q4k_expected, q6k_expected


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
