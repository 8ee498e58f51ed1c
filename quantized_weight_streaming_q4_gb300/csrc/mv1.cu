// mv1.cu -- one-token (M = 1) quantized matvec over Q4_K / Q6_K super-blocks,
// the decode projection of the Muser book (Ch 19 §19.1 operation 1, §19.3,
// §19.5), re-designed for sm_103a:
//
//  * Each CTA owns a contiguous range of output rows (balanced over the SMs)
//    and streams those rows' bytes HBM -> shared memory with 1-D TMA bulk
//    copies (cp.async.bulk + mbarrier), NS stages deep.  Q6_K's 210-byte
//    blocks are only 2-byte aligned, so staging whole row spans is what keeps
//    the global traffic in 16-byte-aligned bulk transfers.
//  * Each thread owns a fixed 64-weight slice (super-block b, chunk c) of the
//    input vector for the whole kernel and keeps it in registers, pre-scaled
//    by powers of two so that a 4- or 6-bit code masked in place inside its
//    32-bit word -- a subnormal float equal to code * 2^(p-149) -- times the
//    scaled input is exactly code * x * 2^-96.  One AND per weight turns a
//    code into an exact float operand; products go through packed
//    fma.rn.f32x2.  Scales are applied once per sub-block.
//  * Per stage, the slice partials of every row land in shared memory and
//    one warp per row adds them in a fixed order (deterministic results).
//  * Epilogues: store y; SiLU-gate two matrices (gate/up, Ch 10 §10.3 (d));
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

constexpr float kTwo96 = 79228162514264337593543950336.0f;  // 2^96

// ------------------------------------------------------ shared-memory reads
// 16 bytes at a 2-byte-aligned shared address (five word loads, byte permute).
__device__ __forceinline__ uint4 lds16_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
    const uint32_t sel = (a & 2) ? 0x5432u : 0x3210u;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2], w3 = w[3], w4 = w[4];
    return make_uint4(__byte_perm(w0, w1, sel), __byte_perm(w1, w2, sel), __byte_perm(w2, w3, sel),
                      __byte_perm(w3, w4, sel));
}
__device__ __forceinline__ uint2 lds8_a2(const uint8_t* p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* w = reinterpret_cast<const uint32_t*>(a & ~static_cast<uintptr_t>(3));
    const uint32_t sel = (a & 2) ? 0x5432u : 0x3210u;
    const uint32_t w0 = w[0], w1 = w[1], w2 = w[2];
    return make_uint2(__byte_perm(w0, w1, sel), __byte_perm(w1, w2, sel));
}

// --------------------------------------------------- per-thread input slice
// Q4_K slice (b, c): weights 64c + l of super-block b, l = 0..63.  Code byte
// 32c + 4t + j holds weight 64c + 4t + j (low nibble) and 64c + 32 + 4t + j
// (high nibble).  Inside the 32-bit word t the nibbles are used at bit
// positions lo: 0, 8, 16, 12 and hi: 4, 12, 8, 16 (bytes 0..3; the top three
// nibbles after a 12-bit shift), so the slice stores x * 2^(53 - p).
struct SliceQ4 {
    float xr[64];
    float s_lo, s_hi;  // sums of x over sub-blocks 2c and 2c+1 (unscaled)
};

__device__ __forceinline__ void load_slice_q4(SliceQ4& s, const float* x, int b, int c) {
    const float* xb = x + b * kQK + 64 * c;
    float slo = 0.0f, shi = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const float4 lo = __ldg(reinterpret_cast<const float4*>(xb + 4 * t));
        const float4 hi = __ldg(reinterpret_cast<const float4*>(xb + 32 + 4 * t));
        s.xr[8 * t + 0] = lo.x * 0x1p53f;
        s.xr[8 * t + 1] = lo.y * 0x1p45f;
        s.xr[8 * t + 2] = lo.z * 0x1p37f;
        s.xr[8 * t + 3] = lo.w * 0x1p41f;
        s.xr[8 * t + 4] = hi.x * 0x1p49f;
        s.xr[8 * t + 5] = hi.y * 0x1p41f;
        s.xr[8 * t + 6] = hi.z * 0x1p45f;
        s.xr[8 * t + 7] = hi.w * 0x1p37f;
        slo += (lo.x + lo.y) + (lo.z + lo.w);
        shi += (hi.x + hi.y) + (hi.z + hi.w);
    }
    s.s_lo = slo;
    s.s_hi = shi;
}

// Q6_K slice (b, c = 2h + j): weights 128h + 32g + 16j + l, g = 0..3,
// l = 0..15 (sub-blocks 8h + 2g + j).  Six-bit codes are rebuilt four to a
// word (bytes at bit 0, 8, 16 and, after a 16-bit shift, 8), so the slice
// stores x * 2^(53 - p) with p = 0, 8, 16, 8.
struct SliceQ6 {
    float xr[64];      // [(i*4 + g)*4 + jj] for l = 4i + jj
    float s_neg32[4];  // -32 * sum of x over sub-block 8h + 2g + j
};

__device__ __forceinline__ void load_slice_q6(SliceQ6& s, const float* x, int b, int c) {
    const int h = c >> 1, j = c & 1;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const float* xg = x + b * kQK + 128 * h + 32 * g + 16 * j;
        float sum = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = __ldg(reinterpret_cast<const float4*>(xg + 4 * i));
            s.xr[(i * 4 + g) * 4 + 0] = v.x * 0x1p53f;
            s.xr[(i * 4 + g) * 4 + 1] = v.y * 0x1p45f;
            s.xr[(i * 4 + g) * 4 + 2] = v.z * 0x1p37f;
            s.xr[(i * 4 + g) * 4 + 3] = v.w * 0x1p45f;
            sum += (v.x + v.y) + (v.z + v.w);
        }
        s.s_neg32[g] = -32.0f * sum;
    }
}

// ------------------------------------------------ one row x one slice (dot)
// Q4_K: sum over the slice's 64 weights of w * x, with
// w = d*sc_j*q - dmin*m_j (j = 2c, 2c+1).
__device__ __forceinline__ float dot_q4(const SliceQ4& s, const uint8_t* blk, int c,
                                        uint32_t sel_lo, uint32_t sel_hi) {
    const uint4 hd = *reinterpret_cast<const uint4*>(blk);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    float2 A = make_float2(0.0f, 0.0f), B = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t w = words[t];
        const uint32_t v = w >> 12;
        A = __ffma2_rn(make_float2(bits_f(w & 0xFu), bits_f(w & 0xF00u)),
                       make_float2(s.xr[8 * t + 0], s.xr[8 * t + 1]), A);
        A = __ffma2_rn(make_float2(bits_f(w & 0xF0000u), bits_f(v & 0xF000u)),
                       make_float2(s.xr[8 * t + 2], s.xr[8 * t + 3]), A);
        B = __ffma2_rn(make_float2(bits_f(w & 0xF0u), bits_f(w & 0xF000u)),
                       make_float2(s.xr[8 * t + 4], s.xr[8 * t + 5]), B);
        B = __ffma2_rn(make_float2(bits_f(v & 0xF00u), bits_f(v & 0xF0000u)),
                       make_float2(s.xr[8 * t + 6], s.xr[8 * t + 7]), B);
    }
    // six-bit scales/mins of sub-blocks 0..3 (low bits) and 4..7 (split)
    const uint32_t scw = (c < 2) ? (hd.y & 0x3F3F3F3Fu)
                                 : ((hd.w & 0x0F0F0F0Fu) | ((hd.y >> 2) & 0x30303030u));
    const uint32_t mnw = (c < 2) ? (hd.z & 0x3F3F3F3Fu)
                                 : (((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u));
    const float2 scm_lo = make_float2(byte_to_f(scw, sel_lo), byte_to_f(mnw, sel_lo));
    const float2 scm_hi = make_float2(byte_to_f(scw, sel_hi), byte_to_f(mnw, sel_hi));
    const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
    float2 T = __fmul2_rn(scm_lo, make_float2(A.x + A.y, s.s_lo));
    T = __ffma2_rn(scm_hi, make_float2(B.x + B.y, s.s_hi), T);
    return fmaf(d * kTwo96, T.x, -(dmin * T.y));
}

// Q6_K: sum over the slice of d*sc_s*(q-32) * x.
__device__ __forceinline__ float dot_q6(const SliceQ6& s, const uint8_t* blk, int c,
                                        uint32_t sel_sc) {
    const int h = c >> 1, j = c & 1;
    const uint4 ql0 = lds16_a2(blk + 64 * h + 16 * j);
    const uint4 ql1 = lds16_a2(blk + 64 * h + 32 + 16 * j);
    const uint4 qh = lds16_a2(blk + 128 + 32 * h + 16 * j);
    const uint2 sc8 = lds8_a2(blk + 192 + 8 * h);
    const uint32_t dbits = *reinterpret_cast<const uint16_t*>(blk + 208);
    const uint32_t A4[4] = {ql0.x, ql0.y, ql0.z, ql0.w};
    const uint32_t B4[4] = {ql1.x, ql1.y, ql1.z, ql1.w};
    const uint32_t H4[4] = {qh.x, qh.y, qh.z, qh.w};
    float2 acc[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) acc[g] = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t A = A4[i], B = B4[i], H = H4[i];
        uint32_t Q[4];
        Q[0] = (A & 0x0F0F0F0Fu) | ((H & 0x03030303u) << 4);
        Q[1] = (B & 0x0F0F0F0Fu) | ((H & 0x0C0C0C0Cu) << 2);
        Q[2] = ((A >> 4) & 0x0F0F0F0Fu) | (H & 0x30303030u);
        Q[3] = ((B >> 4) & 0x0F0F0F0Fu) | ((H >> 2) & 0x30303030u);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const float* xq = &s.xr[(i * 4 + g) * 4];
            acc[g] = __ffma2_rn(make_float2(bits_f(Q[g] & 0x3Fu), bits_f(Q[g] & 0x3F00u)),
                                make_float2(xq[0], xq[1]), acc[g]);
            acc[g] = __ffma2_rn(make_float2(bits_f(Q[g] & 0x3F0000u), bits_f((Q[g] >> 16) & 0x3F00u)),
                                make_float2(xq[2], xq[3]), acc[g]);
        }
    }
    // int8 scales of sub-blocks 8h + 2g + j -> floats (offset-binary via 2^23 magic)
    const uint32_t sc4 = __byte_perm(sc8.x, sc8.y, sel_sc) ^ 0x80808080u;
    float sum = 0.0f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const float scg = byte_to_f(sc4, 0x7540u | g) - 128.0f;
        const float tg = fmaf(acc[g].x + acc[g].y, kTwo96, s.s_neg32[g]);
        sum = fmaf(scg, tg, sum);
    }
    return h2f(dbits) * sum;
}

// -------------------------------------------------------------- the kernel
template <int QT, int NMAT, int EPI>
__global__ void __launch_bounds__(512, 1) mv1_kernel(const Mv1Args p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int kBlk = (QT == MUSER_Q4_K) ? kQ4KBytes : kQ6KBytes;
    const int nsb = p.nsb;
    const int nbc = nsb * 4;
    const int G = p.G, RS = p.RS, NS = p.ns;
    const int64_t rowbytes = static_cast<int64_t>(nsb) * kBlk;
    const int64_t r0 = p.rows * blockIdx.x / gridDim.x;
    const int64_t r1 = p.rows * (blockIdx.x + 1) / gridDim.x;
    const int nloc = static_cast<int>(r1 - r0);
    const int nstages = (nloc + RS - 1) / RS;

    // shared layout: [bars NS x 8 B][red 64 floats][flag][partials 2*NMAT*RS*nbc][stages]
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
    float* red = reinterpret_cast<float*>(smem + 8 * 16);
    int* flag = reinterpret_cast<int*>(smem + 8 * 16 + 64 * 4);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    uint8_t* stage_base = smem + p.stage_off;
    const uint32_t stage_bytes = p.stage_bytes;  // per matrix

    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int g = tid / nbc;
    const int bc = tid - g * nbc;
    const int b = bc >> 2, c = bc & 3;
    const bool active = g < G;

    // Issue the bulk copies of stage k (all matrices) into buffer k % NS.
    auto issue = [&](int k) {
        const int buf = k % NS;
        const int64_t lr0 = static_cast<int64_t>(k) * RS;
        const int64_t lr1 = min(static_cast<int64_t>(nloc), lr0 + RS);
        uint32_t total = 0;
        uint32_t sizes[NMAT];
        const uint8_t* srcs[NMAT];
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
        mbar_arrive_expect_tx(&bars[buf], total);
        for (int m = 0; m < NMAT; ++m) {
            if (sizes[m] == 0) continue;
            uint8_t* dst = stage_base + (static_cast<size_t>(buf) * NMAT + m) * stage_bytes;
            tma_load_1d(dst, srcs[m], sizes[m], &bars[buf]);
        }
    };

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        for (int k = 0; k < min(NS, nstages); ++k) issue(k);
    }

    // This thread's input slice, in registers for the whole kernel.
    using Slice = typename std::conditional<QT == MUSER_Q4_K, SliceQ4, SliceQ6>::type;
    Slice sl;
    if (active) {
        if constexpr (QT == MUSER_Q4_K) load_slice_q4(sl, p.x, b, c);
        else load_slice_q6(sl, p.x, b, c);
    }
    const uint32_t sel_lo = 0x7540u | static_cast<uint32_t>(2 * (c & 1));
    const uint32_t sel_hi = 0x7540u | static_cast<uint32_t>(2 * (c & 1) + 1);
    const uint32_t jq = static_cast<uint32_t>(c & 1);
    const uint32_t sel_sc = jq | ((jq + 2) << 4) | ((jq + 4) << 8) | ((jq + 6) << 12);
    __syncthreads();  // hand-copied stage tails (matrix end) are visible

    bool ok = true;
    const int part_stride = NMAT * RS * nbc;
    for (int k = 0; k < nstages; ++k) {
        const int buf = k % NS;
        const int64_t lr0 = static_cast<int64_t>(k) * RS;
        const int rows_here = static_cast<int>(min(static_cast<int64_t>(RS), nloc - lr0));
        if (ok) ok = mbar_wait_bounded(&bars[buf], static_cast<uint32_t>((k / NS) & 1),
                                       &g_device_status, kDevStatusWaitTimeout);
        float* pk = part + (k & 1) * part_stride;
        if (active && ok) {
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const uint8_t* sbuf = stage_base + (static_cast<size_t>(buf) * NMAT + m) * stage_bytes;
                const uint8_t* start = p.W[m] + (r0 + lr0) * rowbytes;
                const int delta = static_cast<int>(reinterpret_cast<uintptr_t>(start) & 15);
                for (int rs = g; rs < rows_here; rs += G) {
                    const uint8_t* blk = sbuf + delta + rs * rowbytes + static_cast<int64_t>(b) * kBlk;
                    float v;
                    if constexpr (QT == MUSER_Q4_K) v = dot_q4(sl, blk, c, sel_lo, sel_hi);
                    else v = dot_q6(sl, blk, c, sel_sc);
                    pk[(m * RS + rs) * nbc + bc] = v;
                }
            }
        }
        ok = __syncthreads_and(ok);  // stage k consumed; partials of stage k complete
        if (tid == 0 && ok && k + NS < nstages) {
            fence_proxy_async_smem();
            issue(k + NS);
        }
        // One warp per row adds the slice partials in a fixed order.
        for (int rs = warp; rs < rows_here; rs += nwarps) {
            float v[NMAT];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                const float* pr = pk + (m * RS + rs) * nbc;
                float s = 0.0f;
                for (int i = lane; i < nbc; i += 32) s += pr[i];
                v[m] = warp_sum(s);
            }
            if (lane == 0) {
                const int64_t row = r0 + lr0 + rs;
                if constexpr (EPI == kEpiSiluMul) {
                    p.y0[row] = silu_mul_f(v[0], v[NMAT - 1]);
                } else {
                    p.y0[row] = v[0];
                    if constexpr (NMAT == 2) p.y1[row] = v[NMAT - 1];
                }
                if constexpr (EPI == kEpiTail) __threadfence();
            }
        }
    }
    if (!ok) {
        // A bounded wait gave up (status word set).  Give the copies still in
        // flight a bounded chance to land before the block's shared memory is
        // released, then leave without writing the tail.
        if (tid == 0) {
            for (int k = max(0, nstages - NS); k < nstages; ++k)
                (void)mbar_wait_bounded(&bars[k % NS], static_cast<uint32_t>((k / NS) & 1),
                                        &g_device_status, kDevStatusTxTimeout, 1u << 20);
        }
        return;
    }

    if constexpr (EPI == kEpiTail) {
        // Last CTA to finish runs the dual-eps tail over the whole row.
        __syncthreads();
        if (tid == 0) {
            __threadfence();
            const unsigned t = atomicAdd(p.ticket, 1u);
            *flag = (t == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (*flag) {
            __threadfence();
            block_dual_tail_row(p.resid, p.y0, p.out, p.w1, p.w2, static_cast<int>(p.rows), p.eps1,
                                p.eps2, red);
            if (tid == 0) *p.ticket = 0u;  // leave the scratch zeroed for the next call
        }
    }
}

}  // namespace

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
bool mv1_supported(int qtype, int64_t cols) {
    (void)qtype;
    const int64_t nbc = (cols / kQK) * 4;
    return cols % kQK == 0 && nbc >= 1 && nbc <= 512;
}

template <int QT, int NMAT, int EPI>
static int launch_mv1_t(Mv1Args a, cudaStream_t stream) {
    constexpr int kBlk = (QT == MUSER_Q4_K) ? kQ4KBytes : kQ6KBytes;
    const int nbc = a.nsb * 4;
    const int64_t rowbytes = static_cast<int64_t>(a.nsb) * kBlk;
    const int sms = sm_count();
    int grid = static_cast<int>(std::min<int64_t>(sms, a.rows));
    a.G = std::max(1, 512 / nbc);
    const int threads = ((nbc * a.G + 31) / 32) * 32;
    // rows per stage: a multiple of G, stage near 32 KB over all matrices
    const int64_t per_row = rowbytes * NMAT;
    int64_t rs = std::max<int64_t>(1, (32 * 1024) / (per_row * a.G)) * a.G;
    const int64_t rows_per_cta = (a.rows + grid - 1) / grid;
    rs = std::min<int64_t>(rs, ((rows_per_cta + a.G - 1) / a.G) * a.G);
    a.RS = static_cast<int>(rs);
    a.stage_bytes = static_cast<uint32_t>(((rs * rowbytes + 32) + 127) / 128 * 128);
    const int head = 8 * 16 + 64 * 4 + 64;  // bars, red, flag
    a.part_off = (head + 127) / 128 * 128;
    const int64_t part_bytes = static_cast<int64_t>(2) * NMAT * a.RS * nbc * 4;
    a.stage_off = static_cast<int>((a.part_off + part_bytes + 127) / 128 * 128);
    const int64_t budget = max_smem_optin();
    const int64_t per_stage = static_cast<int64_t>(a.stage_bytes) * NMAT;
    int ns = static_cast<int>((budget - a.stage_off) / per_stage);
    ns = std::min(ns, 8);
    if (ns < 2) return set_error(MUSER_ERR_UNSUPPORTED, "mv1: shape needs %lld B of shared memory per stage", (long long)per_stage);
    a.ns = ns;
    const size_t smem = static_cast<size_t>(a.stage_off + ns * per_stage);
    auto kern = mv1_kernel<QT, NMAT, EPI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return cuda_fail(e, "mv1: cudaFuncSetAttribute");
    kern<<<grid, threads, smem, stream>>>(a);
    return check_launch("mv1_kernel");
}

int launch_mv1(int qtype, int nmat, int epi, const Mv1Args& a, cudaStream_t s) {
    if (qtype == MUSER_Q4_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q4_K, 1, kEpiStore>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q4_K, 1, kEpiTail>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q4_K, 2, kEpiSiluMul>(a, s);
    } else if (qtype == MUSER_Q6_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q6_K, 1, kEpiStore>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q6_K, 1, kEpiTail>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q6_K, 2, kEpiSiluMul>(a, s);
    }
    return set_error(MUSER_ERR_UNSUPPORTED, "mv1: no kernel for qtype %d nmat %d epilogue %d", qtype, nmat, epi);
}

}  // namespace muser
