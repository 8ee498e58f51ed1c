// mv1.cu -- one-token (M = 1) quantized matvec over Q4_K / Q5_K / Q6_K super-blocks,
// the decode projection of the Muser book (Ch 19 §19.1 operation 1, §19.3,
// §19.5), re-designed for sm_103a:
//
//  * Each CTA owns a contiguous range of output rows (balanced over the SMs)
//    and streams those rows' bytes HBM -> shared memory with 1-D TMA bulk
//    copies (cp.async.bulk + mbarrier), NS stages of about 32 KB (64 KB for
//    Q6_K and for rows one row group spans) deep.  Q6_K's 210-byte
//    blocks are only 2-byte aligned, so staging whole row spans is what keeps
//    the global traffic in 16-byte-aligned bulk transfers.
//  * Each thread owns a fixed 64-weight slice (super-block b, chunk c) of the
//    input vector for the whole kernel and keeps it in registers, held as
//    the three bytes of a 24-bit fixed-point copy (one power of two per
//    slice).  Codes are masked in place, four to a 32-bit word, and dp4a
//    adds four code * digit products per instruction into exact int32
//    per-digit sub-block sums.  Q4_K/Q5_K scales are applied once per
//    sub-block; Q6_K's int8 scales are folded into the integer digit sums.
//  * Per stage, the slice partials of every row land in shared memory and
//    one warp per row adds them in a fixed order (deterministic results).
//  * Epilogues: store y; scale and soft-cap logits (the LM head, Ch 10
//    Figure 10.1 box 15); SiLU-gate two matrices (gate/up, Ch 10 §10.3 (d));
//    or write `projected` and let the last CTA to finish run the dual-eps
//    tail of Ch 19 §19.4 (atomic ticket, no spinning).
#include <algorithm>
#include <cstdio>
#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace muser {

// Device status word of this library's bounded waits (see read_device_status).
__device__ unsigned g_device_status = 0u;

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
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        // sum(q * X) over sub-block 2c, and 16 * sum(q * X) over sub-block 2c+1
        const float flo = combine3(acc[r][0], acc[r][1], acc[r][2]);
        const float fhi = combine3(acc[r][3], acc[r][4], acc[r][5]);
        // six-bit scales/mins of sub-blocks 0..3 (low bits) and 4..7 (split)
        const uint32_t scw = (c < 2) ? (hd[r].y & 0x3F3F3F3Fu)
                                     : ((hd[r].w & 0x0F0F0F0Fu) | ((hd[r].y >> 2) & 0x30303030u));
        const uint32_t mnw = (c < 2) ? (hd[r].z & 0x3F3F3F3Fu)
                                     : (((hd[r].w >> 4) & 0x0F0F0F0Fu) | ((hd[r].z >> 2) & 0x30303030u));
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
#pragma unroll
    for (int r = 0; r < NR; ++r) {
        const float flo = combine3(acc[r][0], acc[r][1], acc[r][2]);
        const float fhi = combine3(acc[r][3], acc[r][4], acc[r][5]);
        const uint32_t scw = (c < 2) ? (hd[r].y & 0x3F3F3F3Fu)
                                     : ((hd[r].w & 0x0F0F0F0Fu) | ((hd[r].y >> 2) & 0x30303030u));
        const uint32_t mnw = (c < 2) ? (hd[r].z & 0x3F3F3F3Fu)
                                     : (((hd[r].w >> 4) & 0x0F0F0F0Fu) | ((hd[r].z >> 2) & 0x30303030u));
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

// -------------------------------------------------------------- the kernel
// Warp roles: warps 0..nconsumer-1 compute (each thread one input slice and a
// row group); the next warp issues the bulk copies; the last two reduce the
// partials of alternate stages per row and write the outputs (epilogue).
// Stage buffer s has a "full" mbarrier (producer arrival + TMA
// transaction bytes) and an "empty" mbarrier (one arrival per consumer warp
// once it has read the stage and stored its partials).  No block-wide barrier
// runs per stage.
// XS: where x comes from.  kXMemory: x is p.x.  kXTail: x is the next-norm
// output of the previous layer's dual-eps tail (Ch 19 §19.4), computed here
// by every block from p.x (= projected), p.resid, p.w1, p.w2: block 0 writes
// the updated residual (and x to p.out when that is set).
template <int QT, int NMAT, int EPI, int XS>
__global__ void __launch_bounds__(512, 1) mv1_kernel(const Mv1Args p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kBlk = kBlockBytes<QT>;
    const int nsb = p.nsb;
    const int nbc = nsb * 4;
    const int G = p.G, RS = p.RS, NS = p.ns;
    const int ncw = p.nconsumer_warps;
    const uint32_t rowbytes = static_cast<uint32_t>(nsb) * kBlk;
    const int64_t r0 = p.rows * blockIdx.x / gridDim.x;
    const int64_t r1 = p.rows * (blockIdx.x + 1) / gridDim.x;
    const int nloc = static_cast<int>(r1 - r0);
    const int nstages = (nloc + RS - 1) / RS;

    // shared layout: barriers [full 8][empty 8][pfull 16][reduced 16][xissued][xready] |
    // red 64 | flag | partial slots (2*NS) | stage buffers (NS).  The input
    // slots overlay the partial slots and, when larger, the first p.rot stage
    // buffers, until every consumer holds its slice; stage k therefore uses
    // buffer (k + rot) % NS, so that the first NS - rot stages can be
    // requested before the slots are free.
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 8;
    uint64_t* pfull = full + 16;
    uint64_t* reduced = full + 32;
    uint64_t* xissued = full + 48;  // every consumer warp has issued its loads of x
    uint64_t* xready = full + 49;   // every consumer warp holds its slice
    float* red = reinterpret_cast<float*>(smem + 512);
    int* flag = reinterpret_cast<int*>(smem + 512 + 64 * 4);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    uint8_t* xslots = smem + p.x_off;
    const bool parity_split = (QT == MUSER_Q6_K) && (nsb % 2 == 0);
    uint8_t* stage_base = smem + p.stage_off;
    const uint32_t stage_bytes = p.stage_bytes;  // per matrix
    const int part_stride = NMAT * RS * nbc;
    int L = 32;
    while (L > 1 && L * RS * NMAT > 32) L >>= 1;

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int NP = 2 * NS;  // partial slots

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], static_cast<uint32_t>(ncw));
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(&pfull[i], static_cast<uint32_t>(ncw));
            mbar_init(&reduced[i], 1);
        }
        mbar_init(xissued, static_cast<uint32_t>(ncw));
        mbar_init(xready, static_cast<uint32_t>(ncw));
        fence_mbar_init();
    }
    __syncthreads();

    bool ok = true;
    if (warp == ncw) {
        // ---------------------------------------------------------- TMA warp
        // Bulk copies of stage k (all matrices) into buffer buf = k % NS.
        // Each weight byte is read once per call: evict-first in L2.
        const uint64_t wpol = l2_policy_evict_first();
        auto issue = [&](int k, int buf) {
            const int64_t lr0 = static_cast<int64_t>(k) * RS;
            const int64_t lr1 = min(static_cast<int64_t>(nloc), lr0 + RS);
            if (QT == MUSER_Q4_K && NMAT == 1 && EPI == kEpiStore && p.nseg > 0) {
                // Rows of several matrices (rows are whole 16-byte units): one
                // copy per segment the stage touches, back to back in the buffer.
                const int64_t v0 = r0 + lr0, v1 = r0 + lr1;
                uint8_t* dst = stage_base + static_cast<size_t>(buf) * NMAT * stage_bytes;
                mbar_arrive_expect_tx(&full[buf], static_cast<uint32_t>((v1 - v0) * rowbytes));
                for (int sg = 0; sg < p.nseg; ++sg) {
                    const int64_t a0 = max(v0, p.seg0[sg]), a1 = min(v1, p.seg0[sg + 1]);
                    if (a1 > a0)
                        tma_load_1d_hint(dst + (a0 - v0) * rowbytes, p.segW[sg] + (a0 - p.seg0[sg]) * rowbytes,
                                         static_cast<uint32_t>((a1 - a0) * rowbytes), &full[buf], wpol);
                }
                return;
            }
            uint32_t total = 0;
            uint32_t sizes[NMAT];
            const uint8_t* srcs[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const uint8_t* start = p.W[m] + (r0 + lr0) * rowbytes;
                const uint8_t* end = p.W[m] + (r0 + lr1) * rowbytes;
                const uint8_t* matend = p.W[m] + p.rows * rowbytes;
                const uint8_t* s16 = reinterpret_cast<const uint8_t*>(
                    reinterpret_cast<uintptr_t>(start) & ~static_cast<uintptr_t>(15));
                uintptr_t e16 = (reinterpret_cast<uintptr_t>(end) + 15) & ~static_cast<uintptr_t>(15);
                const uintptr_t mend16 = reinterpret_cast<uintptr_t>(matend) & ~static_cast<uintptr_t>(15);
                if (e16 > mend16) e16 = mend16;  // never read past the matrix
                uint8_t* dst = stage_base + (static_cast<size_t>(buf) * NMAT + m) * stage_bytes;
                // bytes in [e16, end) (only at the matrix end) are copied by hand
                for (const uint8_t* q = reinterpret_cast<const uint8_t*>(e16); q < end; ++q)
                    dst[q - s16] = static_cast<uint8_t>(ldg_u8(q));
                sizes[m] = static_cast<uint32_t>(e16 - reinterpret_cast<uintptr_t>(s16));
                srcs[m] = s16;
                total += sizes[m];
            }
            mbar_arrive_expect_tx(&full[buf], total);
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                if (sizes[m] == 0) continue;
                uint8_t* dst = stage_base + (static_cast<size_t>(buf) * NMAT + m) * stage_bytes;
                tma_load_1d_hint(dst, srcs[m], sizes[m], &full[buf], wpol);
            }
        };
        // The weights do not depend on the previous kernel: the stages whose
        // buffers lie below the input slots are requested at once, so the
        // stream overlaps the previous kernel's tail and the slice set-up.
        // Requests queue in order: only p.lead stages go ahead of the loads
        // of x, the rest of the free buffers follow them.
        const int nfirst = min(NS, nstages);
        const int rot = p.rot;
        const int early = min(NS - rot, nfirst);
        const int lead = min(p.lead, early);
        if (lane == 0)
            for (int k = 0; k < lead; ++k) issue(k, k + rot);
        __syncwarp();
        pdl_launch_dependents();
        ok = mbar_wait_bounded(xissued, 0, &g_device_status, kDevStatusWaitTimeout);
        if (ok && lane == 0)
            for (int k = lead; k < early; ++k) issue(k, k + rot);
        __syncwarp();
        // The rest of the first NS stages once the slots are free again.
        if (ok) ok = mbar_wait_bounded(xready, 0, &g_device_status, kDevStatusWaitTimeout);
        if (ok && lane == 0)
            for (int k = early; k < nfirst; ++k) issue(k, k + rot - NS);
        __syncwarp();
        // Buffer k % NS is free once every consumer warp has read stage k;
        // the partial slot of stage k + NS once stage k - NS is reduced.
        // Ring positions advance by counters.
        int ebuf = rot, elap = 0, rslot = NS;
        uint32_t ephase = 0, rphase = 0;
        for (int k = 0; k + NS < nstages && ok; ++k) {
            ok = mbar_wait_bounded(&empty[ebuf], ephase, &g_device_status, kDevStatusWaitTimeout);
            const int kp = k + NS;
            if (ok && kp >= NP)
                ok = mbar_wait_bounded(&reduced[rslot], rphase, &g_device_status, kDevStatusWaitTimeout);
            if (ok && lane == 0) issue(kp, ebuf);
            __syncwarp();
            if (++ebuf == NS) ebuf = 0;
            if (++elap == NS) {
                elap = 0;
                ephase ^= 1u;
            }
            if (++rslot == NP) rslot = 0;
            if (kp >= NP && rslot == 0) rphase ^= 1u;
        }
    } else if (warp > ncw) {
        // ----------------------------------------------------- reducer warps
        // Two warps take alternate stages (the 2*NS partial slots alternate
        // with them, so each slot has one reducer).
        pdl_launch_dependents();
        pdl_wait();  // outputs of the previous kernel are complete before ours are written
        const int n4 = nbc / 4;
        int slot = warp - ncw - 1;  // k % NP (NP is even)
        uint32_t sphase = 0;        // (k / NP) & 1
        float tss = 0.0f;           // tail: sum of this warp's projected^2
        for (int k = warp - ncw - 1; k < nstages; k += 2) {
            if (ok) ok = mbar_wait_bounded(&pfull[slot], sphase, &g_device_status, kDevStatusWaitTimeout);
            if (!ok) break;
            const int64_t lr0 = static_cast<int64_t>(k) * RS;
            const int rows_here = static_cast<int>(min(static_cast<int64_t>(RS), nloc - lr0));
            const float* pk = part + slot * part_stride;
            // Output o = rs*NMAT + m owns lanes [o*L, o*L + L); each lane adds
            // a fixed strided set of float4 partials (loads issued first), then
            // a shuffle tree inside the lane group finishes the sum.
            for (int o0 = 0; o0 < rows_here * NMAT; o0 += 32 / L) {
                const int o = o0 + lane / L;
                const int sub = lane % L;
                const int rs = o / NMAT, m = o % NMAT;
                float acc = 0.0f;
                if (rs < rows_here) {
                    const float4* pr = reinterpret_cast<const float4*>(pk + (m * RS + rs) * nbc);
                    for (int j0 = sub; j0 < n4; j0 += 8 * L) {
                        float4 q[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) {
                            const int j = j0 + u * L;
                            q[u] = j < n4 ? pr[j] : make_float4(0.f, 0.f, 0.f, 0.f);
                        }
#pragma unroll
                        for (int u = 0; u < 8; ++u) acc += (q[u].x + q[u].y) + (q[u].z + q[u].w);
                    }
                }
                for (int off = L / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                float other = 0.0f;
                if constexpr (NMAT == 2) other = __shfl_down_sync(0xffffffffu, acc, L);
                if (sub == 0 && rs < rows_here && m == 0) {
                    const int64_t row = r0 + lr0 + rs;
                    if constexpr (EPI == kEpiSiluMul) {
                        p.y0[row] = silu_mul_f(acc, other);
                    } else if constexpr (EPI == kEpiSoftcap) {
                        p.y0[row] = softcap_f(acc, p.scale, p.cap);
                    } else if (QT == MUSER_Q4_K && NMAT == 1 && EPI == kEpiStore && p.nseg > 0) {
                        int sg = 0;
                        while (sg + 1 < p.nseg && row >= p.seg0[sg + 1]) ++sg;
                        p.segY[sg][row - p.seg0[sg]] = acc;
                    } else {
                        p.y0[row] = acc;
                        if constexpr (NMAT == 2) p.y1[row] = other;
                    }
                    if constexpr (EPI == kEpiTail) {
                        tss = fmaf(acc, acc, tss);
                        __threadfence();
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&reduced[slot]);
            slot += 2;
            if (slot >= NP) {
                slot -= NP;
                sphase ^= 1u;
            }
        }
        if constexpr (EPI == kEpiTail) {
            tss = warp_sum(tss);
            if (lane == 0) red[40 + warp - ncw - 1] = tss;
        }
    } else {
        // Thread -> (row group g, slice (b, c) of slice_of); a row group spans
        // p.TG threads.
        const int g = tid / p.TG;
        const int idx = tid - g * p.TG;
        int b, c;
        bool active = slice_of(idx, nbc, parity_split, p.HP, b, c) && g < G;
        if (!active) b = c = 0;
        const int bc = b * 4 + c;  // partial slot of this slice
        pdl_launch_dependents();
        using Slice = typename std::conditional<QT != MUSER_Q6_K, SliceQ4, SliceQ6>::type;
        Slice sl;
        // Every block reads all of x: block b starts its loads at float4 number
        // b * n4 / grid (then wraps), so the blocks do not all ask for the
        // same lines of L2 at the same time.
        const int n4 = nbc * 16, nthr = ncw * 32;
        const int x0 = static_cast<int>((static_cast<int64_t>(blockIdx.x) * n4) / gridDim.x);
        auto xi = [&](int j) { return j + x0 < n4 ? j + x0 : j + x0 - n4; };
        if constexpr (XS == kXTail) {
            // The tail of the previous layer, at most 4 float4 of each vector
            // per thread (the launcher checks), in registers.  The norm
            // weights do not depend on the previous kernel.
            const float n = static_cast<float>(nbc * 64);
            const float4* p4 = reinterpret_cast<const float4*>(p.x);
            const float4* r4 = reinterpret_cast<const float4*>(p.resid);
            const float4* a4 = reinterpret_cast<const float4*>(p.w1);
            const float4* b4 = reinterpret_cast<const float4*>(p.w2);
            float4 pv[4], rv[4], av[4], bv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = tid + u * nthr;
                if (j < n4) {
                    av[u] = __ldg(a4 + xi(j));
                    bv[u] = __ldg(b4 + xi(j));
                }
            }
            pdl_wait();  // projected and the residual are the previous kernels' outputs
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = tid + u * nthr;
                if (j < n4) {
                    pv[u] = __ldcg(p4 + xi(j));
                    rv[u] = __ldcg(r4 + xi(j));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(xissued);
            float ss = 0.0f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (tid + u * nthr < n4) {
                    ss = fmaf(pv[u].x, pv[u].x, ss);
                    ss = fmaf(pv[u].y, pv[u].y, ss);
                    ss = fmaf(pv[u].z, pv[u].z, ss);
                    ss = fmaf(pv[u].w, pv[u].w, ss);
                }
            ss = warps_sum(ss, red, ncw);
            const float inv1 = 1.0f / sqrtf(ss / n + p.eps1);
            float sh = 0.0f;
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (tid + u * nthr < n4) {
                    float4 h;
                    h.x = fmaf(pv[u].x * inv1, av[u].x, rv[u].x);
                    h.y = fmaf(pv[u].y * inv1, av[u].y, rv[u].y);
                    h.z = fmaf(pv[u].z * inv1, av[u].z, rv[u].z);
                    h.w = fmaf(pv[u].w * inv1, av[u].w, rv[u].w);
                    sh = fmaf(h.x, h.x, sh);
                    sh = fmaf(h.y, h.y, sh);
                    sh = fmaf(h.z, h.z, sh);
                    sh = fmaf(h.w, h.w, sh);
                    rv[u] = h;
                }
            sh = warps_sum(sh, red, ncw);
            const float inv2 = 1.0f / sqrtf(sh / n + p.eps2);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = tid + u * nthr;
                if (j < n4) {
                    const int i = xi(j);
                    const float4 xv = make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y,
                                                  (rv[u].z * inv2) * bv[u].z, (rv[u].w * inv2) * bv[u].w);
                    sts_float4(xslots + xslot_offset(i, QT != MUSER_Q6_K, parity_split, p.HP), xv);
                    if (blockIdx.x == 0) {
                        reinterpret_cast<float4*>(p.resid)[i] = rv[u];
                        if (p.out) reinterpret_cast<float4*>(p.out)[i] = xv;
                    }
                }
            }
        } else {
            // All of a thread's copies (at most 16: x holds 16 float4 per slice
            // and there are at least as many consumer threads as slices) are
            // in flight before the copy warp queues more weight requests.
            // 16-byte asynchronous copies straight into the slots.
            pdl_wait();  // x is the previous kernel's output
            const float4* x4 = reinterpret_cast<const float4*>(p.x);
#pragma unroll
            for (int u = 0; u < 16; ++u)
                if (tid + u * nthr < n4) {
                    const int i = xi(tid + u * nthr);
                    cp_async16(xslots + xslot_offset(i, QT != MUSER_Q6_K, parity_split, p.HP), x4 + i);
                }
            cp_async_commit();
            __syncwarp();
            if (lane == 0) mbar_arrive(xissued);
            cp_async_wait_all();
        }
        named_barrier_sync(1, ncw * 32);  // the consumer warps only
        if (QT != MUSER_Q6_K || G > 1) {
            // Every slot converted once, a quarter per thread (the row groups
            // share the slots), then each thread loads its own slot's record.
            for (int q0 = 0; q0 < 4 * p.TG; q0 += nthr) {
                const int q = q0 + tid, sq = q >> 2;
                int bq = 0, cq = 0;
                const bool valid = q < 4 * p.TG && slice_of(sq, nbc, parity_split, p.HP, bq, cq);
                convert_quarter<QT>(xslots + (valid ? sq : 0) * kXSlot, q & 3, valid, parity_split && (bq & 1));
            }
            named_barrier_sync(1, ncw * 32);
            if (active) load_record(sl, xslots + idx * kXSlot);
        } else if constexpr (QT == MUSER_Q6_K) {
            // one row group: each slot has one thread, which converts it
            if (active) load_slice_q6(sl, reinterpret_cast<const float*>(xslots + idx * kXSlot), parity_split && (b & 1));
        }
        // the slots' generic writes come before the bulk copies that reuse
        // the overlaid stage buffers
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(xready);
        // the slots overlay the partial slots: every slice is read first
        ok = mbar_wait_bounded(xready, 0, &g_device_status, kDevStatusWaitTimeout);
        const uint32_t sel_lo = 0x7540u | static_cast<uint32_t>(2 * (c & 1));
        const uint32_t sel_hi = 0x7540u | static_cast<uint32_t>(2 * (c & 1) + 1);
        const uint32_t jq = static_cast<uint32_t>(c & 1);
        const uint32_t sel_sc = jq | ((jq + 2) << 4) | ((jq + 4) << 8) | ((jq + 6) << 12);
        const uint32_t slice_off = static_cast<uint32_t>(b) * kBlk;

        // One stage's rows for this thread; kAl selects the Q6_K load path.
        auto stage = [&](auto al_tag, const uint8_t* const* sb, int rows_here, float* pk) {
            constexpr bool kAl = decltype(al_tag)::value;
            auto dots = [&](auto nr_tag, const uint8_t* const* blk, float* out) {
                constexpr int NR = decltype(nr_tag)::value;
                if constexpr (QT == MUSER_Q4_K) dot_q4<NR>(sl, blk, c, sel_lo, sel_hi, out);
                else if constexpr (QT == MUSER_Q5_K) dot_q5<NR>(sl, blk, c, sel_lo, sel_hi, out);
                else dot_q6<NR, kAl ? kAlign : kRotated>(sl, blk, c, sel_sc, out);
            };
            using One = std::integral_constant<int, 1>;
            using Two = std::integral_constant<int, 2>;
            if constexpr (NMAT == 2) {
                // the gate and up rows of row rs, interleaved
                for (int rs = g; rs < rows_here; rs += G) {
                    const uint8_t* blk[2] = {sb[0] + rs * rowbytes, sb[1] + rs * rowbytes};
                    float v[2];
                    dots(Two{}, blk, v);
                    pk[rs * nbc + bc] = v[0];
                    pk[(RS + rs) * nbc + bc] = v[1];
                }
            } else {
                // rows rs and rs + G, interleaved
                for (int rs = g; rs < rows_here; rs += 2 * G) {
                    const uint8_t* blk[2] = {sb[0] + rs * rowbytes, sb[0] + (rs + G) * rowbytes};
                    float v[2];
                    if (rs + G < rows_here) {
                        dots(Two{}, blk, v);
                        pk[rs * nbc + bc] = v[0];
                        pk[(rs + G) * nbc + bc] = v[1];
                    } else {
                        dots(One{}, blk, v);
                        pk[rs * nbc + bc] = v[0];
                    }
                }
            }
        };
        // Q6_K rows whose byte length is not a multiple of 4: alignment
        // alternates by row, so each row picks its path (one row at a time).
        auto stage_any = [&](const uint8_t* const* sb, int rows_here, float* pk) {
            for (int m = 0; m < NMAT; ++m)
                for (int rs = g; rs < rows_here; rs += G) {
                    const uint8_t* blk[1] = {sb[m] + rs * rowbytes};
                    float v[1];
                    if constexpr (QT == MUSER_Q4_K) {
                        dot_q4<1>(sl, blk, c, sel_lo, sel_hi, v);
                    } else if constexpr (QT == MUSER_Q5_K) {
                        dot_q5<1>(sl, blk, c, sel_lo, sel_hi, v);
                    } else {
                        if ((reinterpret_cast<uintptr_t>(blk[0]) & 2) == 0) dot_q6<1, kAlign>(sl, blk, c, sel_sc, v);
                        else dot_q6<1, kRealign>(sl, blk, c, sel_sc, v);
                    }
                    pk[(m * RS + rs) * nbc + bc] = v[0];
                }
        };
        const bool rows4 = (rowbytes & 3u) == 0;
        const bool aligned = (b % 2 == 0);
        // Ring positions advance by counters (no division per stage).  A
        // stage's copy starts at the 16-byte boundary below its first row, so
        // the rows sit `delta` bytes into the buffer; delta advances by
        // RS * rowbytes mod 16 per stage.
        int buf = p.rot, lap = 0, slot = 0, rows_left = nloc;
        uint32_t phase = 0;
        uint32_t delta[NMAT];
        const uint8_t* sbase[NMAT];
        const uint32_t dstep = (static_cast<uint32_t>(RS) * rowbytes) & 15u;
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
            delta[m] = static_cast<uint32_t>((reinterpret_cast<uintptr_t>(p.W[m]) +
                                              static_cast<uint64_t>(r0) * rowbytes) & 15u);
            sbase[m] = stage_base + m * stage_bytes + slice_off;
        }
        const uint32_t buf_stride = NMAT * stage_bytes;
        for (int k = 0; k < nstages; ++k) {
            const int rows_here = min(RS, rows_left);
            if (ok) ok = mbar_wait_bounded(&full[buf], phase, &g_device_status, kDevStatusWaitTimeout);
            float* pk = part + slot * part_stride;
            if (active && ok) {
                const uint8_t* sb[NMAT];
#pragma unroll
                for (int m = 0; m < NMAT; ++m) sb[m] = sbase[m] + buf * buf_stride + delta[m];
                if (QT == MUSER_Q6_K && !rows4) stage_any(sb, rows_here, pk);
                else if (QT != MUSER_Q6_K || aligned) stage(std::true_type{}, sb, rows_here, pk);
                else stage(std::false_type{}, sb, rows_here, pk);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[buf]);
                mbar_arrive(&pfull[slot]);
            }
#pragma unroll
            for (int m = 0; m < NMAT; ++m) delta[m] = (delta[m] + dstep) & 15u;
            rows_left -= RS;
            if (++buf == NS) buf = 0;
            if (++lap == NS) {
                lap = 0;
                phase ^= 1u;
            }
            if (++slot == NP) slot = 0;
        }
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        // A bounded wait gave up (status word set).  Give the copies still in
        // flight a bounded chance to land before the block's shared memory is
        // released, then leave without writing the tail.
        if (tid == 0) {
            for (int k = max(0, nstages - NS); k < nstages; ++k)
                (void)mbar_wait_bounded(&full[(k + p.rot) % NS], static_cast<uint32_t>((k / NS) & 1),
                                        &g_device_status, kDevStatusTxTimeout, 200000000ull);
        }
        return;
    }

    if constexpr (EPI == kEpiTail) {
        // Last CTA to finish runs the dual-eps tail over the whole row.  With
        // p.tail_part, every CTA first leaves the sum of its rows' squares
        // there (its two reducers' sums, in order).
        if (tid == 0) {
            if (p.tail_part) p.tail_part[blockIdx.x] = red[40] + red[41];
            __threadfence();
            const unsigned t = atomicAdd(p.ticket, 1u);
            *flag = (t == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (*flag) {
            __threadfence();
            const int n = static_cast<int>(p.rows);
            if (p.tail_part && (n >> 2) <= 4 * static_cast<int>(blockDim.x))
                block_dual_tail_row_parts(p.resid, p.y0, p.out, p.w1, p.w2, n, p.eps1, p.eps2, p.tail_part,
                                          static_cast<int>(gridDim.x), red);
            else
                block_dual_tail_row(p.resid, p.y0, p.out, p.w1, p.w2, n, p.eps1, p.eps2, red);
            // leave the scratch zeroed for the next call (the partials were
            // read before the tail's block-wide sums)
            if (p.tail_part)
                for (int i = tid; i < static_cast<int>(gridDim.x); i += blockDim.x) p.tail_part[i] = 0.0f;
            if (tid == 0) *p.ticket = 0u;
        }
    }
}

}  // namespace

unsigned* device_status_word() {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
    return static_cast<unsigned*>(ptr);
}

unsigned read_device_status(bool reset) {
    unsigned v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(v));
    if (e != cudaSuccess) return 0xFFFFFFFFu;
    if (reset) {
        const unsigned z = 0;
        cudaMemcpyToSymbol(g_device_status, &z, sizeof(z));
    }
    return v;
}

// ------------------------------------------------------------------ launch
constexpr int kMaxConsumerThreads = 416;  // + the TMA warp and two reducer warps = 512 threads

bool mv1_supported(int qtype, int64_t cols) {
    (void)qtype;
    const int64_t nbc = (cols / kQK) * 4;
    return cols % kQK == 0 && nbc >= 1 && nbc <= kMaxConsumerThreads;
}

// Consumer geometry of a row of `cols` inputs: threads per row group (TG),
// the odd-half start (HP), row groups (G) and consumer warps.
struct Mv1Geom {
    int TG, HP, G, ncw;
};
static Mv1Geom mv1_geom(int qtype, int nsb) {
    const int nbc = nsb * 4;
    Mv1Geom g{nbc, nbc / 2, 1, 1};
    if (qtype == MUSER_Q6_K && nsb % 2 == 0) {
        const int hp = (nbc / 2 + 31) / 32 * 32;
        if (2 * hp <= kMaxConsumerThreads) {
            g.HP = hp;
            g.TG = 2 * hp;
        }
    }
    g.G = std::max(1, kMaxConsumerThreads / g.TG);
    g.ncw = (g.TG * g.G + 31) / 32;
    return g;
}

bool mv1_tail_prologue_supported(int qtype, int64_t cols) {
    if (!mv1_supported(qtype, cols)) return false;
    const int nsb = static_cast<int>(cols / kQK);
    // the tail keeps at most 4 float4 of each vector per consumer thread
    return nsb * 4 * 16 <= 4 * 32 * mv1_geom(qtype, nsb).ncw;
}

template <int QT, int NMAT, int EPI, int XS>
static int launch_mv1_t(Mv1Args a, cudaStream_t stream) {
    constexpr int kBlk = kBlockBytes<QT>;
    const int nbc = a.nsb * 4;
    const int64_t rowbytes = static_cast<int64_t>(a.nsb) * kBlk;
    const int sms = sm_count();
    if (sms <= 0) return set_error(MUSER_ERR_CUDA, "mv1: cannot query the SM count");
    const int grid = static_cast<int>(std::min<int64_t>(sms, a.rows));
    if (EPI == kEpiTail && grid > kMv1TailParts) a.tail_part = nullptr;
    // Q6_K rows of an even number of super-blocks split their slices by block
    // parity; each half is padded to whole warps when that still fits.
    const Mv1Geom geo = mv1_geom(QT, a.nsb);
    a.TG = geo.TG;
    a.HP = geo.HP;
    a.G = geo.G;
    a.nconsumer_warps = geo.ncw;
    if (a.nseg > 0) {
        if (QT != MUSER_Q4_K || NMAT != 1 || EPI != kEpiStore || a.nseg > kMv1MaxSeg || a.seg0[0] != 0 ||
            a.seg0[a.nseg] != a.rows)
            return set_error(MUSER_ERR_UNSUPPORTED, "mv1: row segments need one 16-byte-row matrix, store epilogue");
        a.W[0] = a.W[1] = a.segW[0];
    }
    if (XS == kXTail && !(nbc * 16 <= 4 * 32 * geo.ncw))
        return set_error(MUSER_ERR_UNSUPPORTED, "mv1: %d inputs exceed the fused tail's registers", nbc * 64);
    const int threads = (a.nconsumer_warps + 3) * 32;
    // Rows per stage: a multiple of G, the stage near 32 KB over all matrices,
    // or near 64 KB for Q6_K and for rows that one row group spans.  There
    // each thread has more work per stage and the per-stage cost (barrier
    // waits, ring bookkeeping, one bulk copy) weighs more: on GB300 the
    // larger stages took a 202,048 x 6,656 Q6_K matvec from 202 to 174 us and
    // the 52-layer stack from 53.2 to 51.0 us per layer.  Gate/up (four row
    // groups, two matrices) ran slower with them.
    const bool big = QT == MUSER_Q6_K || geo.G == 1;
    const int64_t per_row = rowbytes * NMAT;
    const int64_t unit = static_cast<int64_t>(a.G) * (NMAT == 1 ? 2 : 1);  // one matrix: rows go in pairs
    int64_t rs = std::max<int64_t>(1, (big ? 64 * 1024 : 32 * 1024) / (per_row * unit)) * unit;
    const int64_t rows_per_cta = (a.rows + grid - 1) / grid;
    rs = std::min<int64_t>(rs, ((rows_per_cta + unit - 1) / unit) * unit);
    a.RS = static_cast<int>(rs);
    a.stage_bytes = static_cast<uint32_t>(((rs * rowbytes + 32) + 127) / 128 * 128);
    const int head = 512 + 64 * 4 + 64;  // barriers, red, flag
    a.part_off = (head + 127) / 128 * 128;
    const int64_t budget = max_smem_optin();
    const int64_t per_stage = static_cast<int64_t>(a.stage_bytes) * NMAT;
    const int64_t part_per_stage = static_cast<int64_t>(NMAT) * a.RS * nbc * 4;
    int ns = static_cast<int>((budget - a.part_off - 256) / (per_stage + 2 * part_per_stage));
    ns = std::min(ns, 8);
    if (ns < 2)
        return set_error(MUSER_ERR_UNSUPPORTED, "mv1: shape needs %lld B of shared memory per stage",
                         (long long)per_stage);
    a.ns = ns;
    a.stage_off = static_cast<int>((a.part_off + 2 * ns * part_per_stage + 127) / 128 * 128);
    const size_t smem = static_cast<size_t>(a.stage_off + ns * per_stage);
    // input slots over the partial slots and, when larger, the first stage
    // buffers; the other buffers take the first weight copies
    const int64_t xbytes = (static_cast<int64_t>(a.TG) * kXSlot + 127) / 128 * 128;
    if (a.part_off + xbytes > static_cast<int64_t>(smem))
        return set_error(MUSER_ERR_UNSUPPORTED, "mv1: input slots (%lld B) exceed the stage buffers",
                         (long long)xbytes);
    a.x_off = a.part_off;
    const int64_t over = a.part_off + xbytes - a.stage_off;
    a.rot = over > 0 ? static_cast<int>((over + per_stage - 1) / per_stage) : 0;
    a.lead = big ? 1 : 2;
    auto kern = mv1_kernel<QT, NMAT, EPI, XS>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "mv1: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "mv1: cudaLaunchKernelEx");
    return check_launch("mv1_kernel");
}

int launch_mv1(int qtype, int nmat, int epi, const Mv1Args& a, cudaStream_t s, int xs) {
    if (xs == kXTail) {
        if (qtype == MUSER_Q4_K && nmat == 2 && epi == kEpiSiluMul)
            return launch_mv1_t<MUSER_Q4_K, 2, kEpiSiluMul, kXTail>(a, s);
        if (qtype == MUSER_Q4_K && nmat == 1 && epi == kEpiStore)
            return launch_mv1_t<MUSER_Q4_K, 1, kEpiStore, kXTail>(a, s);
        if (qtype == MUSER_Q6_K && nmat == 2 && epi == kEpiSiluMul)
            return launch_mv1_t<MUSER_Q6_K, 2, kEpiSiluMul, kXTail>(a, s);
    } else if (qtype == MUSER_Q4_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q4_K, 1, kEpiStore, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q4_K, 1, kEpiTail, kXMemory>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q4_K, 2, kEpiSiluMul, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiSoftcap) return launch_mv1_t<MUSER_Q4_K, 1, kEpiSoftcap, kXMemory>(a, s);
    } else if (qtype == MUSER_Q5_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q5_K, 1, kEpiStore, kXMemory>(a, s);
    } else if (qtype == MUSER_Q6_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q6_K, 1, kEpiStore, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q6_K, 1, kEpiTail, kXMemory>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q6_K, 2, kEpiSiluMul, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiSoftcap) return launch_mv1_t<MUSER_Q6_K, 1, kEpiSoftcap, kXMemory>(a, s);
    }
    return set_error(MUSER_ERR_UNSUPPORTED, "mv1: no kernel for qtype %d nmat %d epilogue %d", qtype, nmat, epi);
}

}  // namespace muser
