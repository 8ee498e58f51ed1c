// mv1_core.cuh -- device pieces of the one-token (M = 1) dp4a matvec shared
// by the per-call kernel (mv1.cu) and the persistent stack kernel (mvs.cu):
// the per-thread input slice held as 24-bit fixed-point digits, its
// conversion, and the Q4_K / Q5_K / Q6_K dot products of weight rows against
// one slice (Muser book Ch 19 §19.3, §19.5-§19.6; the block layouts are the
// ggml super-blocks).
#pragma once

#include <type_traits>

#include "common.cuh"

namespace muser {
namespace {

// --------------------------------------------------- per-thread input slice
// The input slice is held as integers.  With one power of two 2^e per slice
// (max |x| * 2^e in [2^22, 2^23)), X = rint(x * 2^e) is a 24-bit two's
// complement integer, split into bytes X = D2*65536 + D1*256 + D0 (D0, D1
// unsigned, D2 signed), each digit packed four to a register in the byte
// order of the code words.  A code word masked to its nibbles (or rebuilt
// Q6_K codes) is four unsigned bytes; one dp4a per digit adds four
// code * digit products into an int32, so the per-digit sub-block sums are
// exact integers.  The roundings are X itself (at most 2^-23 of the slice's
// largest |x|) and the binary32 combination of the three digit sums.

// Exponent e of a slice with largest magnitude m (0 for m == 0): m * 2^e is
// in [2^21, 2^23 - 1.5], so rint(x * 2^e) is in [-2^23 + 1, 2^23 - 1] for
// every |x| <= m.  Reading the binade of m * (1 + 2^-23) moves the m whose
// significand is within two units of 2 to the next binade (one bit less
// precision for those slices, never an overflow).
__device__ __forceinline__ int slice_exponent(float m) {
    if (!(m > 0.0f)) return 0;
    const float mu = m * 1.00000012f;
    const int E = static_cast<int>((__float_as_uint(mu) >> 23) & 0xFFu) - 127;
    return min(22 - E, 126);
}
// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// Bytes 0, 1 and 2 (the digits) of four 24-bit integers, each packed in order.
__device__ __forceinline__ void pack_digits(int X0, int X1, int X2, int X3, uint32_t* w3) {
    const uint32_t a = static_cast<uint32_t>(X0), b = static_cast<uint32_t>(X1);
    const uint32_t c = static_cast<uint32_t>(X2), d = static_cast<uint32_t>(X3);
    const uint32_t p01 = __byte_perm(a, b, 0x5140u), p23 = __byte_perm(c, d, 0x5140u);
    w3[0] = __byte_perm(p01, p23, 0x5410u);
    w3[1] = __byte_perm(p01, p23, 0x7632u);
    w3[2] = __byte_perm(__byte_perm(a, b, 0x0062u), __byte_perm(c, d, 0x0062u), 0x5410u);
}

// Four-way byte dot products with int32 accumulation: unsigned codes times
// the unsigned low digits, and times the signed top digit.
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// D2*65536 + D1*256 + D0 from the three digit sums: T = D2*256 + D1 is an
// exact int32 for every code range here (|T| < 2^28); the rest in binary32.
__device__ __forceinline__ float combine3(int a0, int a1, int a2) {
    return fmaf(static_cast<float>(a2 * 256 + a1), 256.0f, static_cast<float>(a0));
}

// Small unsigned byte / 16 -> float through the 2^19 magic exponent: the
// float with bits 0x490000XX is 2^19 + XX/16, exactly.
__device__ __forceinline__ float byte_to_f16th(uint32_t word, uint32_t sel_with_magic) {
    return __uint_as_float(__byte_perm(word, 0x49000000u, sel_with_magic)) - 524288.0f;
}

// Q4_K slice (b, c): weights 64c + l of super-block b, l = 0..63.  Code byte
// 32c + 4t + i holds weight 64c + 4t + i in its low nibble (sub-block 2c) and
// 64c + 32 + 4t + i in its high nibble (sub-block 2c+1).
struct SliceQ4 {
    uint32_t lo[3][8];  // [digit][word t]: digits of X at weights 64c + 4t + i, byte i
    uint32_t hi[3][8];  // the same for weights 64c + 32 + 4t + i
    float s_lo, s_hi;   // sums of x over sub-blocks 2c and 2c+1 (unscaled)
    float inv;          // 2^-e
};

// Q6_K slice (b, c = 2h + j): weights 128h + 32g + 16j + l, g = 0..3,
// l = 0..15 (sub-blocks 8h + 2g + j); word i of a code field covers
// l = 4i..4i+3, or l = 4i-2..4i+1 (mod 16) when the block is rotated.
struct SliceQ6 {
    uint32_t x[4][3][4];  // [group g][digit][word i]
    int neg32[4][3];      // -32 * sum of digit k of X over sub-block 8h + 2g + j
    float inv;            // 2^-e
};

// rot: the thread's blocks start 2 bytes past a word boundary.  Their code
// fields are read as aligned words W0..W4 around the field; W1..W3 hold field
// bytes 2..13 and one byte permute folds W4 (bytes 14, 15) and W0 (bytes 0, 1)
// into the first word, so word i of the field holds bytes 4i-2..4i+1 (mod 16)
// and the slice's digit words are rotated the same way.
// ------------------------------------------------ slice conversion
// The consumer threads convert the slices in quarters: quarter k of slot s
// holds 16 of its 64 inputs (Q4_K and Q5_K: words 4(k&1)..4(k&1)+3 of the low half
// for k < 2, of the high half for k >= 2; Q6_K: group k).  The four quarters
// of a slot sit in four neighbouring lanes, which agree on the slot's
// exponent with two shuffles.  The digit words and the slot's scalars then
// overwrite the slot's inputs, and every thread loads the record of its own
// slot.  Record layouts (32-bit words):
//   Q4_K, Q5_K: lo[d][t] at 8d + t, hi[d][t] at 24 + 8d + t; inv, s_lo, s_hi at 48..50.
//   Q6_K: x[g][d][i] at 12g + 4d + i; neg32[g][d] at 48 + 3g + d; inv at 60.
// All 32 lanes of a warp call it (shuffles); a lane with !valid converts
// zeros and stores nothing.
template <int QT>
__device__ __forceinline__ void convert_quarter(uint8_t* slot, int k, bool valid, bool rot) {
    float v[16];
    const float* xs = reinterpret_cast<const float*>(slot) + 16 * k;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 f = valid ? lds_float4(xs + 4 * q) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[4 * q + 0] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    float m = 0.0f;
#pragma unroll
    for (int l = 0; l < 16; ++l) m = fmaxf(m, fabsf(v[l]));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    const int e = slice_exponent(m);
    const float p2e = pow2f(e);
    const float inv = pow2f(-e);
    uint32_t D[4][3];
#pragma unroll
    for (int i = 0; i < 4; ++i)
        pack_digits(__float2int_rn(v[4 * i] * p2e), __float2int_rn(v[4 * i + 1] * p2e),
                    __float2int_rn(v[4 * i + 2] * p2e), __float2int_rn(v[4 * i + 3] * p2e), D[i]);
    uint32_t* rec = reinterpret_cast<uint32_t*>(slot);
    if constexpr (QT != MUSER_Q6_K) {
        float sum = 0.0f;
#pragma unroll
        for (int l = 0; l < 16; ++l) sum += v[l];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);  // the half's sum (quarters 2j, 2j + 1)
        __syncwarp();
        if (valid) {
            const int base = (k >= 2 ? 24 : 0) + 4 * (k & 1);
#pragma unroll
            for (int d = 0; d < 3; ++d) sts_uint4(rec + base + 8 * d, make_uint4(D[0][d], D[1][d], D[2][d], D[3][d]));
            if (k == 0) {
                rec[48] = __float_as_uint(inv);
                rec[49] = __float_as_uint(sum);
            }
            if (k == 2) rec[50] = __float_as_uint(sum);
        }
    } else {
        int sums[3] = {0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sums[0] = dp4a_uu(D[i][0], 0x01010101u, sums[0]);
            sums[1] = dp4a_uu(D[i][1], 0x01010101u, sums[1]);
            sums[2] = dp4a_us(0x01010101u, D[i][2], sums[2]);
        }
        // a rotated word i holds bytes 4i - 2 .. 4i + 1 (mod 16) of the field
        const uint32_t rsel = rot ? 0x5432u : 0x7654u;
        __syncwarp();
        if (valid) {
#pragma unroll
            for (int d = 0; d < 3; ++d)
                sts_uint4(rec + 12 * k + 4 * d,
                          make_uint4(__byte_perm(D[3][d], D[0][d], rsel), __byte_perm(D[0][d], D[1][d], rsel),
                                     __byte_perm(D[1][d], D[2][d], rsel), __byte_perm(D[2][d], D[3][d], rsel)));
#pragma unroll
            for (int d = 0; d < 3; ++d) rec[48 + 3 * k + d] = static_cast<uint32_t>(-32 * sums[d]);
            if (k == 0) rec[60] = __float_as_uint(inv);
        }
    }
}

// One thread converts a whole Q4_K / Q5_K slot (its 64 inputs in order at xs)
// into its own slice: the arithmetic of convert_quarter's four quarters (the
// same exponent, digits and half sums, each half summed as two sequential
// 16-input sums) without the shared-memory record.
__device__ __forceinline__ void load_slice_q4(SliceQ4& s, const float* xs) {
    float v[64];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const float4 f = lds_float4(xs + 4 * q);
        v[4 * q + 0] = f.x;
        v[4 * q + 1] = f.y;
        v[4 * q + 2] = f.z;
        v[4 * q + 3] = f.w;
    }
    float m = 0.0f;
#pragma unroll
    for (int l = 0; l < 64; ++l) m = fmaxf(m, fabsf(v[l]));
    const int e = slice_exponent(m);
    const float p2e = pow2f(e);
    s.inv = pow2f(-e);
    float qs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float sum = 0.0f;
#pragma unroll
        for (int l = 0; l < 16; ++l) sum += v[16 * k + l];
        qs[k] = sum;
    }
    s.s_lo = qs[0] + qs[1];
    s.s_hi = qs[2] + qs[3];
#pragma unroll
    for (int t = 0; t < 16; ++t) {
        uint32_t D[3];
        pack_digits(__float2int_rn(v[4 * t] * p2e), __float2int_rn(v[4 * t + 1] * p2e),
                    __float2int_rn(v[4 * t + 2] * p2e), __float2int_rn(v[4 * t + 3] * p2e), D);
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            if (t < 8) s.lo[d][t] = D[d];
            else s.hi[d][t - 8] = D[d];
        }
    }
}

// One thread converts a whole Q6_K slot (four 16-input groups, group g at xs
// + 16g) into its own slice.
__device__ __forceinline__ void load_slice_q6(SliceQ6& s, const float* xs, bool rot) {
    float v[4][16];
    float m = 0.0f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = lds_float4(xs + 16 * g + 4 * q);
            v[g][4 * q + 0] = f.x;
            v[g][4 * q + 1] = f.y;
            v[g][4 * q + 2] = f.z;
            v[g][4 * q + 3] = f.w;
        }
#pragma unroll
        for (int l = 0; l < 16; ++l) m = fmaxf(m, fabsf(v[g][l]));
    }
    const int e = slice_exponent(m);
    const float p2e = pow2f(e);
    s.inv = pow2f(-e);
    // a rotated word i holds bytes 4i - 2 .. 4i + 1 (mod 16) of the field
    const uint32_t rsel = rot ? 0x5432u : 0x7654u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t D[4][3];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            pack_digits(__float2int_rn(v[g][4 * i] * p2e), __float2int_rn(v[g][4 * i + 1] * p2e),
                        __float2int_rn(v[g][4 * i + 2] * p2e), __float2int_rn(v[g][4 * i + 3] * p2e), D[i]);
        int sum[3] = {0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            sum[0] = dp4a_uu(D[i][0], 0x01010101u, sum[0]);
            sum[1] = dp4a_uu(D[i][1], 0x01010101u, sum[1]);
            sum[2] = dp4a_us(0x01010101u, D[i][2], sum[2]);
        }
#pragma unroll
        for (int k = 0; k < 3; ++k) {
            s.neg32[g][k] = -32 * sum[k];
#pragma unroll
            for (int i = 0; i < 4; ++i) s.x[g][k][i] = __byte_perm(D[(i + 3) & 3][k], D[i][k], rsel);
        }
    }
}

__device__ __forceinline__ void load_record(SliceQ4& s, const uint8_t* slot) {
    const uint32_t* rec = reinterpret_cast<const uint32_t*>(slot);
#pragma unroll
    for (int d = 0; d < 3; ++d)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 a = lds_uint4(rec + 8 * d + 4 * h), b = lds_uint4(rec + 24 + 8 * d + 4 * h);
            s.lo[d][4 * h + 0] = a.x; s.lo[d][4 * h + 1] = a.y; s.lo[d][4 * h + 2] = a.z; s.lo[d][4 * h + 3] = a.w;
            s.hi[d][4 * h + 0] = b.x; s.hi[d][4 * h + 1] = b.y; s.hi[d][4 * h + 2] = b.z; s.hi[d][4 * h + 3] = b.w;
        }
    const uint4 t = lds_uint4(rec + 48);
    s.inv = __uint_as_float(t.x);
    s.s_lo = __uint_as_float(t.y);
    s.s_hi = __uint_as_float(t.z);
}
__device__ __forceinline__ void load_record(SliceQ6& s, const uint8_t* slot) {
    const uint32_t* rec = reinterpret_cast<const uint32_t*>(slot);
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int d = 0; d < 3; ++d) {
            const uint4 a = lds_uint4(rec + 12 * g + 4 * d);
            s.x[g][d][0] = a.x; s.x[g][d][1] = a.y; s.x[g][d][2] = a.z; s.x[g][d][3] = a.w;
        }
#pragma unroll
    for (int q = 0; q < 3; ++q) {
        const uint4 a = lds_uint4(rec + 48 + 4 * q);
        const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) s.neg32[(4 * q + u) / 3][(4 * q + u) % 3] = static_cast<int>(w[u]);
    }
    s.inv = __uint_as_float(rec[60]);
}

// ------------------------------------------------ rows x one slice (dot)
// NR independent weight rows (two matrices, or two rows of one) against the
// same input slice, interleaved so each warp has several independent dp4a
// chains in flight.

// The packed six-bit scales and mins of a Q4_K / Q5_K header (words y, z, w
// after d, dmin): sub-blocks 0..3 are the low six bits of bytes y (scales)
// and z (mins); sub-blocks 4..7 take their low four bits from w and their top
// two bits from the top of y and z.  A slice c uses sub-blocks 2c and 2c+1,
// so one shift and two masks select its bytes for either half:
//   scales = ((y >> sh) & m1) | (w & m2),  mins = ((z >> sh) & m1) | ((w >> 4) & m2).
struct ScaleSel {
    uint32_t sh, m1, m2;
};
__device__ __forceinline__ ScaleSel scale_sel(int c) {
    return c < 2 ? ScaleSel{0u, 0x3F3F3F3Fu, 0u} : ScaleSel{2u, 0x30303030u, 0x0F0F0F0Fu};
}

// Q4_K: out[r] = sum over the slice's 64 weights of w * x, with
// w = d*sc_j*q - dmin*m_j (j = 2c, 2c+1).  Low nibbles are masked in place
// as the bytes q; high nibbles are masked in place too, as the bytes 16q,
// and their scale carries the 1/16.
template <int NR>
__device__ __forceinline__ void dot_q4(const SliceQ4& s, const uint8_t* const* blk, int c,
                                       uint32_t sel_lo, uint32_t sel_hi, float* out) {
    uint4 hd[NR];
    uint32_t W[NR][8];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        hd[r] = *reinterpret_cast<const uint4*>(blk[r]);
        const uint4 qa = *reinterpret_cast<const uint4*>(blk[r] + 16 + 32 * c);
        const uint4 qb = *reinterpret_cast<const uint4*>(blk[r] + 32 + 32 * c);
        W[r][0] = qa.x; W[r][1] = qa.y; W[r][2] = qa.z; W[r][3] = qa.w;
        W[r][4] = qb.x; W[r][5] = qb.y; W[r][6] = qb.z; W[r][7] = qb.w;
    }
    int acc[NR][6];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int k = 0; k < 6; ++k) acc[r][k] = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t ql = W[r][t] & 0x0F0F0F0Fu;
            const uint32_t qh = W[r][t] & 0xF0F0F0F0u;
            acc[r][0] = dp4a_uu(ql, s.lo[0][t], acc[r][0]);
            acc[r][1] = dp4a_uu(ql, s.lo[1][t], acc[r][1]);
            acc[r][2] = dp4a_us(ql, s.lo[2][t], acc[r][2]);
            acc[r][3] = dp4a_uu(qh, s.hi[0][t], acc[r][3]);
            acc[r][4] = dp4a_uu(qh, s.hi[1][t], acc[r][4]);
            acc[r][5] = dp4a_us(qh, s.hi[2][t], acc[r][5]);
        }
    }
    const ScaleSel k = scale_sel(c);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        // sum(q * X) over sub-block 2c, and 16 * sum(q * X) over sub-block 2c+1
        const float flo = combine3(acc[r][0], acc[r][1], acc[r][2]);
        const float fhi = combine3(acc[r][3], acc[r][4], acc[r][5]);
        // six-bit scales/mins of sub-blocks 0..3 (low bits) and 4..7 (split)
        const uint32_t scw = ((hd[r].y >> k.sh) & k.m1) | (hd[r].w & k.m2);
        const uint32_t mnw = ((hd[r].z >> k.sh) & k.m1) | ((hd[r].w >> 4) & k.m2);
        const float sc_lo = byte_to_f(scw, sel_lo);
        const float sc_hi = byte_to_f16th(scw, sel_hi);  // sc / 16
        const float2 mins = make_float2(byte_to_f(mnw, sel_lo), byte_to_f(mnw, sel_hi));
        const float d = h2f(hd[r].x), dmin = h2f(hd[r].x >> 16);
        const float dot = fmaf(sc_lo, flo, sc_hi * fhi);
        const float msum = fmaf(mins.x, s.s_lo, mins.y * s.s_hi);
        out[r] = fmaf(d * s.inv, dot, -(dmin * msum));
    }
}

// Q5_K (Ch 4 §4.4's third k-quant; ggml layout): Q4_K's header and code
// nibbles (code bytes at 48 + 32c) plus a fifth code bit, bit 2c (low half) or
// 2c + 1 (high half) of qh[l] at byte 16 + l.  One rotation brings that bit of
// every qh byte to bit 4, where it joins the nibble, so both halves' codes are
// bytes q = 0..31 and both scales apply unscaled.
template <int NR>
__device__ __forceinline__ void dot_q5(const SliceQ4& s, const uint8_t* const* blk, int c,
                                       uint32_t sel_lo, uint32_t sel_hi, float* out) {
    const int rot_lo = (4 - 2 * c) & 31, rot_hi = (3 - 2 * c) & 31;
    uint4 hd[NR];
    uint32_t W[NR][8], Hb[NR][8];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        hd[r] = *reinterpret_cast<const uint4*>(blk[r]);
        const uint4 ha = *reinterpret_cast<const uint4*>(blk[r] + 16);
        const uint4 hb = *reinterpret_cast<const uint4*>(blk[r] + 32);
        const uint4 qa = *reinterpret_cast<const uint4*>(blk[r] + 48 + 32 * c);
        const uint4 qb = *reinterpret_cast<const uint4*>(blk[r] + 64 + 32 * c);
        W[r][0] = qa.x; W[r][1] = qa.y; W[r][2] = qa.z; W[r][3] = qa.w;
        W[r][4] = qb.x; W[r][5] = qb.y; W[r][6] = qb.z; W[r][7] = qb.w;
        Hb[r][0] = ha.x; Hb[r][1] = ha.y; Hb[r][2] = ha.z; Hb[r][3] = ha.w;
        Hb[r][4] = hb.x; Hb[r][5] = hb.y; Hb[r][6] = hb.z; Hb[r][7] = hb.w;
    }
    int acc[NR][6];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int k = 0; k < 6; ++k) acc[r][k] = 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t h = Hb[r][t];
            const uint32_t ql = (W[r][t] & 0x0F0F0F0Fu) | (__funnelshift_l(h, h, rot_lo) & 0x10101010u);
            const uint32_t qh = ((W[r][t] >> 4) & 0x0F0F0F0Fu) | (__funnelshift_l(h, h, rot_hi) & 0x10101010u);
            acc[r][0] = dp4a_uu(ql, s.lo[0][t], acc[r][0]);
            acc[r][1] = dp4a_uu(ql, s.lo[1][t], acc[r][1]);
            acc[r][2] = dp4a_us(ql, s.lo[2][t], acc[r][2]);
            acc[r][3] = dp4a_uu(qh, s.hi[0][t], acc[r][3]);
            acc[r][4] = dp4a_uu(qh, s.hi[1][t], acc[r][4]);
            acc[r][5] = dp4a_us(qh, s.hi[2][t], acc[r][5]);
        }
    }
    const ScaleSel k = scale_sel(c);
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float flo = combine3(acc[r][0], acc[r][1], acc[r][2]);
        const float fhi = combine3(acc[r][3], acc[r][4], acc[r][5]);
        const uint32_t scw = ((hd[r].y >> k.sh) & k.m1) | (hd[r].w & k.m2);
        const uint32_t mnw = ((hd[r].z >> k.sh) & k.m1) | ((hd[r].w >> 4) & k.m2);
        const float d = h2f(hd[r].x), dmin = h2f(hd[r].x >> 16);
        const float dot = fmaf(byte_to_f(scw, sel_lo), flo, byte_to_f(scw, sel_hi) * fhi);
        const float msum = fmaf(byte_to_f(mnw, sel_lo), s.s_lo, byte_to_f(mnw, sel_hi) * s.s_hi);
        out[r] = fmaf(d * s.inv, dot, -(dmin * msum));
    }
}

// Code-field loads.  kAlign: the field is 4-byte aligned.  kRotated: the
// field sits 2 bytes past a word boundary and the thread's input slice is
// rotated to match (convert_quarter): word 0 = (bytes 14,15,0,1), words 1..3 =
// the aligned words W1..W3 from p - 2.  kRealign: 2 bytes past a boundary,
// words realigned by byte permutes (rows whose alignment alternates).
constexpr int kAlign = 0, kRotated = 1, kRealign = 2;

template <int kMode>
__device__ __forceinline__ void lds_field(const uint8_t* p, uint32_t* w4) {
    if constexpr (kMode == kAlign) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = w[i];
    } else if constexpr (kMode == kRotated) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
        w4[0] = __byte_perm(w[4], w[0], 0x7610u);
        w4[1] = w[1];
        w4[2] = w[2];
        w4[3] = w[3];
    } else {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
        uint32_t a[5];
#pragma unroll
        for (int i = 0; i < 5; ++i) a[i] = w[i];
#pragma unroll
        for (int i = 0; i < 4; ++i) w4[i] = __byte_perm(a[i], a[i + 1], 0x5432u);
    }
}
// 8 bytes (two words) at shared address p, aligned as above.
template <bool kAligned>
__device__ __forceinline__ uint2 lds_w2(const uint8_t* p) {
    if constexpr (kAligned) {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p);
        return make_uint2(w[0], w[1]);
    } else {
        const uint32_t* w = reinterpret_cast<const uint32_t*>(p - 2);
        const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
        return make_uint2(__byte_perm(w0, w1, 0x5432u), __byte_perm(w1, w2, 0x5432u));
    }
}

// Q6_K: out[r] = sum over the slice of d*sc_s*(q-32) * x.  The six-bit codes
// are rebuilt four to a word as the bytes q; the -32 offset enters as each
// digit accumulator's start, -32 * (sum of that digit).  With rows of a
// multiple of 4 bytes, even blocks start 4-byte aligned in the stage and odd
// ones 2 bytes past a boundary (210-byte blocks).
template <int NR, int kMode>
__device__ __forceinline__ void dot_q6(const SliceQ6& s, const uint8_t* const* blk, int c,
                                       uint32_t sel_sc, float* out) {
    const int h = c >> 1, j = c & 1;
    int acc[NR][4][3];
#pragma unroll
    for (int r = 0; r < NR; ++r)
#pragma unroll
        for (int g = 0; g < 4; ++g)
#pragma unroll
            for (int k = 0; k < 3; ++k) acc[r][g][k] = s.neg32[g][k];
    uint32_t A[NR][4], B[NR][4], H[NR][4];
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        lds_field<kMode>(blk[r] + 64 * h + 16 * j, A[r]);
        lds_field<kMode>(blk[r] + 64 * h + 32 + 16 * j, B[r]);
        lds_field<kMode>(blk[r] + 128 + 32 * h + 16 * j, H[r]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int r = 0; r < NR; ++r) {
            const uint32_t a = A[r][i], bq = B[r][i], hq = H[r][i];
            uint32_t Q[4];
            Q[0] = (a & 0x0F0F0F0Fu) | ((hq & 0x03030303u) << 4);
            Q[1] = (bq & 0x0F0F0F0Fu) | ((hq & 0x0C0C0C0Cu) << 2);
            Q[2] = ((a >> 4) & 0x0F0F0F0Fu) | (hq & 0x30303030u);
            Q[3] = ((bq >> 4) & 0x0F0F0F0Fu) | ((hq >> 2) & 0x30303030u);
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                acc[r][g][0] = dp4a_uu(Q[g], s.x[g][0][i], acc[r][g][0]);
                acc[r][g][1] = dp4a_uu(Q[g], s.x[g][1][i], acc[r][g][1]);
                acc[r][g][2] = dp4a_us(Q[g], s.x[g][2][i], acc[r][g][2]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const uint2 sc8 = lds_w2<kMode == kAlign>(blk[r] + 192 + 8 * h);
        const uint32_t dbits = *reinterpret_cast<const uint16_t*>(blk[r] + 208);
        // int8 scales of sub-blocks 8h + 2g + j, byte g of sc4
        const uint32_t sc4 = __byte_perm(sc8.x, sc8.y, sel_sc);
        // Per digit k, sum over the four sub-blocks of scale * sum((q - 32) * D_k):
        // |sum((q - 32) * D_k)| <= 16 * 32 * 255 < 2^17 and |scale| <= 128, so
        // the four products and their sum stay below 2^26, exact in int32.
        int T[3] = {0, 0, 0};
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int scg = static_cast<int8_t>((sc4 >> (8 * g)) & 0xFFu);
#pragma unroll
            for (int k = 0; k < 3; ++k) T[k] += scg * acc[r][g][k];
        }
        const float sum = fmaf(static_cast<float>(T[2]), 65536.0f,
                               fmaf(static_cast<float>(T[1]), 256.0f, static_cast<float>(T[0])));
        out[r] = (h2f(dbits) * s.inv) * sum;
    }
}

// ---------------------------------------------------------- input slots
// Row-group thread idx owns slice (b, c).  Q6_K with an even number of
// super-blocks per row: the first half of a row group's slices take the even
// super-blocks, the second half (from thread HP) the odd ones, so whole warps
// share one block alignment (even blocks start 4-byte aligned in the stage,
// odd ones 2 bytes past a boundary); threads in the padding idle.  Returns
// whether idx owns a slice.
__device__ __forceinline__ bool slice_of(int idx, int nbc, bool parity_split, int HP, int& b, int& c) {
    if (parity_split) {
        const bool odd = idx >= HP;
        const int i2 = odd ? idx - HP : idx;
        b = 2 * (i2 >> 2) + (odd ? 1 : 0);
        c = i2 & 3;
        return i2 < nbc / 2;
    }
    b = idx >> 2;
    c = idx & 3;
    return idx < nbc;
}
// The consumer warps copy x into shared memory with coalesced float4 loads,
// each slice's 64 inputs into a slot of its own (slot idx at idx * kXSlot
// bytes; Q6_K groups g at 64g).  The 16-byte pad makes a quarter warp's float4
// reads of consecutive slots fall in distinct banks.  (Read straight from
// global memory, every warp-wide load of a slice touched 32 lines.)
constexpr int kXSlot = 272;
// Byte offset in the slots of x's float4 number i.
__device__ __forceinline__ int xslot_offset(int i, bool q4, bool parity_split, int HP) {
    if (q4) return (i >> 4) * kXSlot + (i & 15) * 16;  // slot 4b + c, chunk q
    const int b = i >> 6, f = (i & 63) * 4;              // float f of super-block b
    const int h = f >> 7, g = (f >> 5) & 3, j = (f >> 4) & 1, l4 = (f >> 2) & 3;
    const int c = 2 * h + j;
    const int idx = parity_split ? ((b & 1) ? HP : 0) + 4 * (b >> 1) + c : 4 * b + c;
    return idx * kXSlot + 64 * g + 16 * l4;
}

// Sum of v over the first nwarps warps of the block (all of them call it):
// warp trees, then every thread adds the warp sums in warp order, so every
// thread gets the same value.  red needs nwarps floats; named barrier 1.
__device__ __forceinline__ float warps_sum(float v, float* red, int nwarps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    named_barrier_sync(1, nwarps * 32);
    float t = 0.0f;
    for (int w = 0; w < nwarps; ++w) t += red[w];
    named_barrier_sync(1, nwarps * 32);
    return t;
}

}  // namespace
}  // namespace muser
