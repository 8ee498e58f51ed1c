"""Independent block ENCODERS used to pin the oracle's decoders.

These pack field values (scales, mins, codes, d) into Q4_K / Q5_K / Q6_K super-block
bytes.  They are the inverse map of the layout, written from its description
(field lists in the Muser book Ch 19 §19.3; ggml/GGUF super-block conventions
for the bit positions), so a decoder that reads a wrong bit, byte or nibble
fails the round trip.  Test-only helpers.
"""
import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array(v, dtype=np.float16).view(np.uint16))


def pack_q4k(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    """sc, mn: 8 ints in 0..63 (per 32-weight sub-block); q: 256 ints in 0..15."""
    sc = [int(v) for v in sc]
    mn = [int(v) for v in mn]
    q = [int(v) for v in q]
    assert len(sc) == 8 and len(mn) == 8 and len(q) == 256
    assert all(0 <= v < 64 for v in sc + mn) and all(0 <= v < 16 for v in q)
    blk = np.zeros(144, np.uint8)
    blk[0:2] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    blk[2:4] = np.array([f16_bits(dmin)], np.uint16).view(np.uint8)
    s = [0] * 12
    for j in range(4):
        # sub-blocks 0..3: six bits in bytes j (scale) and j+4 (min)
        s[j] |= sc[j]
        s[j + 4] |= mn[j]
    for j in range(4, 8):
        # sub-blocks 4..7: low four bits in byte j+4 (scale low nibble, min high
        # nibble), top two bits parked in the spare top bits of bytes j-4 / j
        s[j + 4] |= (sc[j] & 0x0F) | ((mn[j] & 0x0F) << 4)
        s[j - 4] |= (sc[j] >> 4) << 6
        s[j] |= (mn[j] >> 4) << 6
    blk[4:16] = np.array(s, np.uint8)
    qs = [0] * 128
    for i in range(256):
        c, r = divmod(i, 64)
        if r < 32:
            qs[32 * c + r] |= q[i]
        else:
            qs[32 * c + (r - 32)] |= q[i] << 4
    blk[16:144] = np.array(qs, np.uint8)
    return blk


def q4k_expected(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    """The dequantised values from the fields: d*sc*q - dmin*min, rounded once."""
    d = float(np.float16(d))
    dmin = float(np.float16(dmin))
    out = np.empty(256, np.float64)
    for i in range(256):
        j = i // 32
        out[i] = d * sc[j] * q[i] - dmin * mn[j]
    return out.astype(np.float32)


def pack_q5k(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    """Q5_K (ggml layout): sc, mn as for Q4_K; q: 256 ints in 0..31.  Bytes: d,
    dmin, the Q4_K scale/min packing, 32 bytes of fifth bits, 128 code bytes."""
    q = [int(v) for v in q]
    assert len(q) == 256 and all(0 <= v < 32 for v in q)
    # the header and scale packing are Q4_K's; the low four code bits too
    q4 = pack_q4k(d, dmin, sc, mn, [v & 15 for v in q])
    blk = np.zeros(176, np.uint8)
    blk[0:16] = q4[0:16]
    blk[48:176] = q4[16:144]
    qh = [0] * 32
    for i in range(256):
        c, r = divmod(i, 64)
        half, l = divmod(r, 32)
        if q[i] >> 4:
            qh[l] |= 1 << (2 * c + half)
    blk[16:48] = np.array(qh, np.uint8)
    return blk


def q5k_expected(d: float, dmin: float, sc, mn, q) -> np.ndarray:
    return q4k_expected(d, dmin, sc, mn, q)


def pack_q6k(d: float, sc, q) -> np.ndarray:
    """sc: 16 ints in -128..127 (per 16-weight sub-block); q: 256 ints in 0..63."""
    sc = [int(v) for v in sc]
    q = [int(v) for v in q]
    assert len(sc) == 16 and len(q) == 256
    assert all(-128 <= v < 128 for v in sc) and all(0 <= v < 64 for v in q)
    ql = [0] * 128
    qh = [0] * 64
    for i in range(256):
        h, r = divmod(i, 128)
        g, l = divmod(r, 32)
        lo, top = q[i] & 0x0F, q[i] >> 4
        idx = 64 * h + 32 * (g & 1) + l
        ql[idx] |= lo << 4 if g >= 2 else lo
        qh[32 * h + l] |= top << (2 * g)
    blk = np.zeros(210, np.uint8)
    blk[0:128] = np.array(ql, np.uint8)
    blk[128:192] = np.array(qh, np.uint8)
    blk[192:208] = np.array(sc, np.int8).view(np.uint8)
    blk[208:210] = np.array([f16_bits(d)], np.uint16).view(np.uint8)
    return blk


def q6k_expected(d: float, sc, q) -> np.ndarray:
    d = float(np.float16(d))
    out = np.empty(256, np.float64)
    for i in range(256):
        out[i] = d * sc[i // 16] * (q[i] - 32)
    return out.astype(np.float32)
