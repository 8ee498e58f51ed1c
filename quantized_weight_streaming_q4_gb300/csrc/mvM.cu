// mvM.cu -- quantized matvec for M = 1..16 activation rows (the speculative
// verify shape of the Muser book, Ch 10 §10.1, MAX_DFLASH_BLOCK = 16), on CUDA
// cores.
//
// Each thread dequantises 32 weights of one sub-block slot for two weight rows
// to exact binary32 values (the same values muser_dequantize produces), then
// multiplies them against an input tile held transposed in shared memory,
// M values per weight through packed fma.rn.f32x2.  The input tile of the
// next super-block is fetched while the current one is used.  Slot partials
// of a row are added by a fixed shuffle tree.
#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace muser {

namespace {

constexpr int kThreadsM = 256;

// 16 bytes at a 2-byte-aligned global address.
__device__ __forceinline__ uint4 ldg16_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint8_t* w = reinterpret_cast<const uint8_t*>(a & ~static_cast<uintptr_t>(3));
    const bool mis = (a & 2) != 0;
    const uint32_t sel = mis ? 0x5432u : 0x3210u;
    const uint32_t w0 = ldg_u32(w), w1 = ldg_u32(w + 4), w2 = ldg_u32(w + 8), w3 = ldg_u32(w + 12);
    const uint32_t w4 = mis ? ldg_u32(w + 16) : 0u;
    return make_uint4(__byte_perm(w0, w1, sel), __byte_perm(w1, w2, sel), __byte_perm(w2, w3, sel),
                      __byte_perm(w3, w4, sel));
}

// The 32 weights of sub-block slot j8 of one super-block, exact binary32.
// Q4_K: slot j8 = sub-block j8 (weights 32*j8 + l).
__device__ __forceinline__ void decode_slot_q4(const uint8_t* blk, int j8, float w[32]) {
    const uint4 hd = ldg_stream16(blk);
    const int c = j8 >> 1;
    const uint4 qa = ldg_stream16(blk + 16 + 32 * c);
    const uint4 qb = ldg_stream16(blk + 32 + 32 * c);
    const uint32_t s0 = hd.y, s1 = hd.z, s2 = hd.w;
    uint32_t sc, mn;
    if (j8 < 4) {
        sc = (s0 >> (8 * j8)) & 63u;
        mn = (s1 >> (8 * j8)) & 63u;
    } else {
        const int jj = j8 - 4;
        sc = ((s2 >> (8 * jj)) & 0x0Fu) | (((s0 >> (8 * jj + 6)) & 3u) << 4);
        mn = ((s2 >> (8 * jj + 4)) & 0x0Fu) | (((s1 >> (8 * jj + 6)) & 3u) << 4);
    }
    const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
    const float dsc = __fmul_rn(d, static_cast<float>(sc));   // exact (<= 17 bits)
    const float ndm = -__fmul_rn(dmin, static_cast<float>(mn));
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const int sh = (j8 & 1) ? 4 : 0;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q4 = (words[t] >> sh) & 0x0F0F0F0Fu;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float q = byte_to_f(q4, 0x7540u | e);
            w[4 * t + e] = __fmaf_rn(dsc, q, ndm);  // d*sc*q - dmin*m, one rounding
        }
    }
}

// Q5_K: slot j8 = sub-block j8, as Q4_K, with the codes at byte 48 and the
// fifth code bit of weight l at bit 2*(j8 >> 1) + (j8 & 1) of qh[l] (byte 16 + l).
__device__ __forceinline__ void decode_slot_q5(const uint8_t* blk, int j8, float w[32]) {
    const uint4 hd = ldg_stream16(blk);
    const int c = j8 >> 1;
    const uint4 ha = ldg_stream16(blk + 16);
    const uint4 hb = ldg_stream16(blk + 32);
    const uint4 qa = ldg_stream16(blk + 48 + 32 * c);
    const uint4 qb = ldg_stream16(blk + 64 + 32 * c);
    const uint32_t s0 = hd.y, s1 = hd.z, s2 = hd.w;
    uint32_t sc, mn;
    if (j8 < 4) {
        sc = (s0 >> (8 * j8)) & 63u;
        mn = (s1 >> (8 * j8)) & 63u;
    } else {
        const int jj = j8 - 4;
        sc = ((s2 >> (8 * jj)) & 0x0Fu) | (((s0 >> (8 * jj + 6)) & 3u) << 4);
        mn = ((s2 >> (8 * jj + 4)) & 0x0Fu) | (((s1 >> (8 * jj + 6)) & 3u) << 4);
    }
    const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
    const float dsc = __fmul_rn(d, static_cast<float>(sc));   // exact (<= 17 bits)
    const float ndm = -__fmul_rn(dmin, static_cast<float>(mn));
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t hbits[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
    const int sh = (j8 & 1) ? 4 : 0;
    const int hsh = 2 * c + (j8 & 1);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q5 = ((words[t] >> sh) & 0x0F0F0F0Fu) | (((hbits[t] >> hsh) & 0x01010101u) << 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float q = byte_to_f(q5, 0x7540u | e);
            w[4 * t + e] = __fmaf_rn(dsc, q, ndm);  // d*sc*q - dmin*m, one rounding
        }
    }
}

// Q6_K: slot j8 = (h, g) = (j8 >> 2, j8 & 3): weights 128h + 32g + l.
__device__ __forceinline__ void decode_slot_q6(const uint8_t* blk, int j8, float w[32]) {
    const int h = j8 >> 2, g = j8 & 3;
    const uint8_t* ql = blk + 64 * h + 32 * (g & 1);
    const uint4 L0 = ldg16_a2(ql), L1 = ldg16_a2(ql + 16);
    const uint4 H0 = ldg16_a2(blk + 128 + 32 * h), H1 = ldg16_a2(blk + 128 + 32 * h + 16);
    const uint32_t scb = ldg_u16(blk + 192 + 8 * h + 2 * g);  // scales of 8h+2g, 8h+2g+1
    const float d = h2f(ldg_u16(blk + 208));
    const float dsc0 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(scb & 0xFFu)));
    const float dsc1 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(scb >> 8)));
    const uint32_t lw[8] = {L0.x, L0.y, L0.z, L0.w, L1.x, L1.y, L1.z, L1.w};
    const uint32_t hw[8] = {H0.x, H0.y, H0.z, H0.w, H1.x, H1.y, H1.z, H1.w};
    const int lsh = (g & 2) ? 4 : 0;
    const int hsh = 2 * g;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q4 = ((lw[t] >> lsh) & 0x0F0F0F0Fu) | (((hw[t] >> hsh) & 0x03030303u) << 4);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float q = byte_to_f(q4, 0x7540u | e) - 32.0f;
            w[4 * t + e] = __fmul_rn(t < 4 ? dsc0 : dsc1, q);  // d*sc*(q-32), one rounding
        }
    }
}

// x tile of one super-block: xs[quad][p][4] (MB >= 4) or xs[0][p][2] (MB == 2),
// p = 32*j + ((k % 32) ^ j) for k = 32*j + l -- the xor spreads the eight slots'
// reads over distinct bank groups.
template <int MB>
struct Tile {
    static constexpr int kW = MB >= 4 ? 4 : 2;  // floats per (quad, p)
    static constexpr int kQ = MB / kW;
    static constexpr int kFloats = kQ * kQK * kW;
};

__device__ __forceinline__ int swz(int k) { return (k & ~31) | ((k & 31) ^ (k >> 5)); }

template <int MB>
__device__ __forceinline__ void load_tile(float* xs, const float* x, int M, int64_t K, int b) {
    using T = Tile<MB>;
    const int k = threadIdx.x;  // 256 threads, one input position each
    const int p = swz(k);
#pragma unroll
    for (int q = 0; q < T::kQ; ++q) {
        float v[T::kW];
#pragma unroll
        for (int e = 0; e < T::kW; ++e) {
            const int m = q * T::kW + e;
            v[e] = (m < M) ? __ldg(x + static_cast<int64_t>(m) * K + static_cast<int64_t>(b) * kQK + k) : 0.0f;
        }
        float* dst = xs + (q * kQK + p) * T::kW;
        if constexpr (T::kW == 4) *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        else *reinterpret_cast<float2*>(dst) = make_float2(v[0], v[1]);
    }
}

template <int QT, int NMAT, int MB, int EPI>
__global__ void __launch_bounds__(kThreadsM) mvM_kernel(const MvMArgs p) {
    using T = Tile<MB>;
    constexpr int kBlk = kBlockBytes<QT>;
    constexpr int kRowsPerCta = (NMAT == 1) ? 64 : 32;
    __shared__ __align__(16) float xs[2][T::kFloats];

    const int tid = threadIdx.x;
    const int rp = tid >> 3, j8 = tid & 7;
    const int nsb = p.nsb;
    const int64_t K = static_cast<int64_t>(nsb) * kQK;
    const int64_t rowbytes = static_cast<int64_t>(nsb) * kBlk;
    const int64_t row_base = static_cast<int64_t>(blockIdx.x) * kRowsPerCta;

    // the thread's two weight rows: (matrix, row)
    int mat[2];
    int64_t row[2];
    if constexpr (NMAT == 1) {
        mat[0] = mat[1] = 0;
        row[0] = row_base + 2 * rp;
        row[1] = row_base + 2 * rp + 1;
    } else {
        mat[0] = 0;
        mat[1] = 1;
        row[0] = row[1] = row_base + rp;
    }
    const bool valid[2] = {row[0] < p.rows, row[1] < p.rows};

    float2 acc[2][MB / 2];
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int q = 0; q < MB / 2; ++q) acc[r][q] = make_float2(0.0f, 0.0f);

    load_tile<MB>(xs[0], p.x, p.M, K, 0);
    __syncthreads();
    for (int b = 0; b < nsb; ++b) {
        const float* cur = xs[b & 1];
        if (b + 1 < nsb) load_tile<MB>(xs[(b + 1) & 1], p.x, p.M, K, b + 1);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if (!valid[r]) continue;
            const uint8_t* blk = p.W[mat[r]] + row[r] * rowbytes + static_cast<int64_t>(b) * kBlk;
            float w[32];
            if constexpr (QT == MUSER_Q4_K) decode_slot_q4(blk, j8, w);
            else if constexpr (QT == MUSER_Q5_K) decode_slot_q5(blk, j8, w);
            else decode_slot_q6(blk, j8, w);
#pragma unroll
            for (int l = 0; l < 32; ++l) {
                const int pidx = 32 * j8 + (l ^ j8);
                const float2 ww = make_float2(w[l], w[l]);
#pragma unroll
                for (int q = 0; q < T::kQ; ++q) {
                    const float* src = cur + (q * kQK + pidx) * T::kW;
                    if constexpr (T::kW == 4) {
                        const float4 xv = *reinterpret_cast<const float4*>(src);
                        acc[r][2 * q] = __ffma2_rn(ww, make_float2(xv.x, xv.y), acc[r][2 * q]);
                        acc[r][2 * q + 1] = __ffma2_rn(ww, make_float2(xv.z, xv.w), acc[r][2 * q + 1]);
                    } else {
                        const float2 xv = *reinterpret_cast<const float2*>(src);
                        acc[r][q] = __ffma2_rn(ww, xv, acc[r][q]);
                    }
                }
            }
        }
        __syncthreads();
    }

    // add the eight slots of each row (lanes j8 = 0..7 are consecutive)
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int q = 0; q < MB / 2; ++q) {
            float2 v = acc[r][q];
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
                v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
                v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
            }
            acc[r][q] = v;
        }
    if (j8 != 0) return;
#pragma unroll
    for (int q = 0; q < MB / 2; ++q) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int m = 2 * q + e;
            if (m >= p.M) continue;
            const float v0 = e ? acc[0][q].y : acc[0][q].x;
            const float v1 = e ? acc[1][q].y : acc[1][q].x;
            if constexpr (EPI == kEpiSiluMul) {
                if (valid[0]) p.y0[static_cast<int64_t>(m) * p.rows + row[0]] = silu_mul_f(v0, v1);
            } else if constexpr (NMAT == 2) {
                if (valid[0]) {
                    p.y0[static_cast<int64_t>(m) * p.rows + row[0]] = v0;
                    p.y1[static_cast<int64_t>(m) * p.rows + row[1]] = v1;
                }
            } else {
                if (valid[0]) p.y0[static_cast<int64_t>(m) * p.rows + row[0]] = v0;
                if (valid[1]) p.y0[static_cast<int64_t>(m) * p.rows + row[1]] = v1;
            }
        }
    }
}

template <int QT, int NMAT, int EPI>
int launch_mb(const MvMArgs& a, cudaStream_t s) {
    const int rows_per_cta = (NMAT == 1) ? 64 : 32;
    const int grid = static_cast<int>((a.rows + rows_per_cta - 1) / rows_per_cta);
    if (a.M <= 2) mvM_kernel<QT, NMAT, 2, EPI><<<grid, kThreadsM, 0, s>>>(a);
    else if (a.M <= 4) mvM_kernel<QT, NMAT, 4, EPI><<<grid, kThreadsM, 0, s>>>(a);
    else if (a.M <= 8) mvM_kernel<QT, NMAT, 8, EPI><<<grid, kThreadsM, 0, s>>>(a);
    else mvM_kernel<QT, NMAT, 16, EPI><<<grid, kThreadsM, 0, s>>>(a);
    return check_launch("mvM_kernel");
}

}  // namespace

int launch_mvM(int qtype, int nmat, int epi, const MvMArgs& a, cudaStream_t s) {
    if (a.M < 1 || a.M > MUSER_MAX_M)
        return set_error(MUSER_ERR_INVALID_ARG, "M = %d outside 1..%d", a.M, MUSER_MAX_M);
    if (qtype == MUSER_Q4_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mb<MUSER_Q4_K, 1, kEpiStore>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mb<MUSER_Q4_K, 2, kEpiSiluMul>(a, s);
        if (nmat == 2 && epi == kEpiStore) return launch_mb<MUSER_Q4_K, 2, kEpiStore>(a, s);
    } else if (qtype == MUSER_Q5_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mb<MUSER_Q5_K, 1, kEpiStore>(a, s);
    } else if (qtype == MUSER_Q6_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mb<MUSER_Q6_K, 1, kEpiStore>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mb<MUSER_Q6_K, 2, kEpiSiluMul>(a, s);
        if (nmat == 2 && epi == kEpiStore) return launch_mb<MUSER_Q6_K, 2, kEpiStore>(a, s);
    }
    return set_error(MUSER_ERR_UNSUPPORTED, "mvM: no kernel for qtype %d nmat %d epilogue %d",
                     qtype, nmat, epi);
}

}  // namespace muser
