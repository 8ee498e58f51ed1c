// mvt.cu -- the one-token k-quant matvec of Ch 19 §19.1 (operation 1) and
// §19.5-§19.6 on the fifth-generation tensor cores (tcgen05), for GB300.
//
// What it computes: y[r] = sum_k w[r,k] * x[k] with w the Q4_K or Q6_K
// weight of Ch 19 §19.3, then the epilogue: store, silu(gate) * up
// (Ch 10 Figure 10.1 box 11), or the dual-eps tail of Ch 19 §19.4.
//
// How:
//  * Dequantisation is packed.  A 4-bit (or rebuilt 6-bit) code is OR-ed
//    into the mantissa of the binary16 1024.0, giving 1024 + q exactly, two
//    codes per 32-bit register.  One fma.rn.f16x2 per pair then makes the
//    integer sc*q (Q4_K) or sc*(q-32) (Q6_K), exact in binary16 (|.| <= 1024).
//  * Those integers are the A operand of tcgen05.mma kind::f16, written to
//    tensor memory (one TMEM lane per weight row, two values per column).
//  * x is the B operand, split into two binary16 parts,
//    x * 2^-e = hi + lo * 2^-11, with e a power-of-two scale chosen so that
//    max|x| * 2^-e < 2^15.  Each product is exact in the binary32
//    accumulator.  The two D columns are combined as (hi + lo/2048) * 2^e.
//  * One MMA chain covers one super-block (16 MMAs of K = 16).  Each
//    super-block's D is read back and scaled by its d (and, for Q4_K, the
//    min term dmin * sum_j m_j * sum(x over sub-block j) is subtracted), so
//    the per-block scales never enter the tensor core.
//  * The K order inside a super-block follows the order the codes come out
//    of the registers.  x is permuted to match when the B operand is built.
//
// Work split: (row tile, super-block) units are spread evenly over the
// grid.  A tile is 128 TMEM lanes: 128 rows of one matrix, or 64 rows of gate
// and the same 64 rows of up.  A tile whose units fall in several CTAs is
// summed from `part` in a fixed order by the last CTA to finish it (atomic
// ticket), so results do not depend on timing.
//
// Weights arrive by 2-D tensor copies: one box of (super-block bytes x tile
// rows) per matrix and unit.  Q6_K rows of 78 super-blocks are 2-byte
// aligned, so a tile takes rows of one residue class modulo P (P * row bytes
// = 0 mod 16): the class is a 2-D array with a 16-byte multiple row stride,
// every lane of a unit sees the same misalignment, and the box starts at the
// 16-byte boundary below the block (240-byte box rows).  The shared-memory
// loads are then 16-byte loads realigned by compile-time shifts.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "kernels.cuh"

namespace muser {
namespace {

// ------------------------------------------------------------ constants
constexpr int kDeqWarps = 8;                  // warps 0-7: dequantisation, two per TMEM lane quadrant
constexpr int kTmaWarp = kDeqWarps;           // warp 8: bulk copies
constexpr int kMmaWarp = kDeqWarps + 1;       // warp 9: TMEM allocation, MMA issue
constexpr int kRbWarp0 = kDeqWarps + 2;       // warps 10-13: D readback and epilogue, one per quadrant
constexpr int kBldWarp0 = kDeqWarps + 6;      // warps 14-15 (several rows of x): per-unit B operand
constexpr int kNB = 3;                        // B slabs in shared memory (several rows of x)
constexpr int kNA = 3;                        // A stages in TMEM (128 columns each)
constexpr int kND = 3;                        // D buffers in TMEM (16 columns, 32 for several rows)
// One MMA commit per unit releases its A stage and B slab and publishes its
// D buffer (a commit drains the MMA pipe, so there is only one), which needs
// the three per-unit rings to have the same length.
static_assert(kNA == kND && kNB == kND, "per-unit rings share one completion barrier");
// Threads of a CTA: one row of x, or several (two more warps build B).
__host__ __device__ constexpr int mvt_threads(bool multi) { return (kDeqWarps + (multi ? 8 : 6)) * 32; }
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kDCol0 = kNA * 128;        // first D column
constexpr int kMaxStages = 12;
// Several rows of x: one super-block's B image, as the builders leave it in
// shared memory: the 16 KB slab, then 8 sub-block sums of x per row (Q4_K)
// and the 16 rows' scales 2^e.
constexpr uint32_t kSlabBytes = 16384;
constexpr uint32_t kXrBytes = (16 * 8 + 16) * 4;
constexpr uint32_t kBImg = kSlabBytes + kXrBytes;
constexpr uint32_t kMagic2 = 0x64006400u;     // binary16 1024.0 in both halves

// ------------------------------------------------------- tcgen05 helpers
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 columns from this warp's lane quadrant, one column per register.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}
__device__ __forceinline__ void tmem_ld2(uint32_t taddr, uint32_t& a, uint32_t& b) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(a), "=r"(b) : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* v) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
        "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]),
          "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]),
          "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]),
          "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr)
        : "memory");
}

// Shared-memory matrix descriptor, no swizzle: start, leading (K-direction
// core-matrix) byte offset, stride (N-direction 8-row group) byte offset.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
// Instruction descriptor: D binary32, A and B binary16, both K-major,
// M = 128, N = 16 (one row of x) or 32 (up to 16 rows, hi and lo each).
constexpr uint32_t idesc_n(uint32_t n) { return (1u << 4) | ((n >> 3) << 17) | ((128u >> 4) << 24); }

// One super-block's MMA chain: 16 MMAs of K = 16 into D (the first one
// overwrites, the rest accumulate), A columns a_tmem + 8j, B descriptors
// b_desc + j * b_step.  One asm block, so the predicates and the operand
// advances cost one instruction each.
__device__ __forceinline__ void mma_chain16(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint64_t b_step) {
    asm volatile(
        "{\n\t.reg .pred pf, pt;\n\t.reg .b32 ra;\n\t.reg .b64 rd;\n\t"
        "setp.ne.b32 pf, %0, %0;\n\tsetp.eq.b32 pt, %0, %0;\n\t"
        "mov.b32 ra, %1;\n\tmov.b64 rd, %2;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pf;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "add.u32 ra, ra, 8;\n\tadd.u64 rd, rd, %4;\n\ttcgen05.mma.cta_group::1.kind::f16 [%0], [ra], rd, %3, pt;\n\t"
        "}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "l"(b_step)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// fma.rn.f16x2 on raw register pairs.
__device__ __forceinline__ uint32_t hfma2u(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// Both halves = the binary16 value of f (f exactly representable): one
// packed conversion.
__device__ __forceinline__ uint32_t h2rep(float f) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(f));
    return r;
}

// Shared-memory loads through the shared window (the pointers are generic).
__device__ __forceinline__ uint4 lds128(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ float4 lds_f4(const void* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(smem_u32(p)));
    return v;
}

// 2-D tensor copy of one box at (x bytes, y rows) into shared memory; the
// completed bytes are counted on `bar`.  x is a multiple of 16.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}
// The same with an L2 cache policy (the weight stream: evict-first).
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar,
                                                 uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// ------------------------------------------------------ Q4_K (144-byte block)
// Scale and min (6 bits each) of sub-block j from the packed bytes s[0..11],
// held as words s0 = s[0..3], s1 = s[4..7], s2 = s[8..11] (Ch 19 §19.3).
__device__ __forceinline__ void q4k_scale_min(uint32_t s0, uint32_t s1, uint32_t s2, int j, uint32_t& sc,
                                              uint32_t& m) {
    if (j < 4) {
        sc = (s0 >> (8 * j)) & 63u;
        m = (s1 >> (8 * j)) & 63u;
    } else {
        const int b = 8 * (j - 4);
        sc = ((s2 >> b) & 15u) | (((s0 >> b) >> 6 & 3u) << 4);
        m = ((s2 >> (b + 4)) & 15u) | (((s1 >> b) >> 6 & 3u) << 4);
    }
}

// Column order of a Q4_K super-block (128 TMEM columns, two K slots each):
// column 32c + 4t + j of chunk c (64 weights), code word t (bytes 4t..4t+3):
//   j = 0: weights 64c + 4t + {0, 2}     (low nibbles, sub-block 2c)
//   j = 1: weights 64c + 4t + {1, 3}
//   j = 2: weights 64c + 32 + 4t + {0, 2} (high nibbles, sub-block 2c + 1)
//   j = 3: weights 64c + 32 + 4t + {1, 3}

// Chunks 2hf and 2hf + 1 of the row's block at `blk` (16-byte aligned) into
// TMEM columns [col0 + 64hf, +64) of this warp's lanes.
__device__ __forceinline__ void q4k_dequant_half(const uint8_t* blk, int hf, uint32_t taddr) {
    const uint4 hd = lds128(blk);
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * hf + cc;
        const uint4 qa = lds128(blk + 16 + 32 * c);
        const uint4 qb = lds128(blk + 32 + 32 * c);
        const uint32_t P[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        uint32_t scA, scB, mu_;
        q4k_scale_min(hd.y, hd.z, hd.w, 2 * c, scA, mu_);
        q4k_scale_min(hd.y, hd.z, hd.w, 2 * c + 1, scB, mu_);
        const uint32_t kA = h2rep(static_cast<float>(scA)), cA = h2rep(-1024.0f * static_cast<float>(scA));
        const uint32_t kB = h2rep(static_cast<float>(scB) * 0.0625f), cB = h2rep(-64.0f * static_cast<float>(scB));
        uint32_t o[32];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t p = P[t], p8 = p >> 8;
            o[4 * t + 0] = hfma2u((p & 0x000F000Fu) | kMagic2, kA, cA);
            o[4 * t + 1] = hfma2u((p8 & 0x000F000Fu) | kMagic2, kA, cA);
            o[4 * t + 2] = hfma2u((p & 0x00F000F0u) | kMagic2, kB, cB);
            o[4 * t + 3] = hfma2u((p8 & 0x00F000F0u) | kMagic2, kB, cB);
        }
        tmem_st32(taddr + 32u * c, o);
    }
}

// d * 2^e scale and the min term of a Q4_K block for the readback.
__device__ __forceinline__ void q4k_block_scales(const uint8_t* blk, const float* X, float& d, float& minterm) {
    const uint4 hd = lds128(blk);
    d = h2f(hd.x);
    const float dmin = h2f(hd.x >> 16);
    float s = 0.0f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        uint32_t sc, m;
        q4k_scale_min(hd.y, hd.z, hd.w, j, sc, m);
        s = fmaf(static_cast<float>(m), X[j], s);
    }
    minterm = dmin * s;
}

// d, dmin and the eight 6-bit mins of a Q4_K block, one min per byte
// (sub-blocks 0-3 in m03, 4-7 in m47), for several rows of x.
__device__ __forceinline__ void q4k_block_dmins(const uint8_t* blk, float& d, float& dmin, uint32_t& m03,
                                                uint32_t& m47) {
    const uint4 hd = lds128(blk);
    d = h2f(hd.x);
    dmin = h2f(hd.x >> 16);
    m03 = hd.z & 0x3F3F3F3Fu;
    m47 = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
}

// ------------------------------------------------------ Q6_K (210-byte block)
// Column order of a Q6_K super-block: column 64h + 8i + jj, code word i
// (bytes 4i..4i+3 of the half's ql groups), jj = 2g + b:
//   weights 128h + 32g + 4i + b + {0, 2}    (g = 0..3, b = 0, 1)
// Group g takes the low (g < 2) or high (g >= 2) nibble of ql[64h + 32(g&1) + l]
// and qh[32h + l] bits 2g, 2g+1 (Ch 19 §19.3).

// Loads 16-byte blocks [B0, B1] of the row buffer into w[].
template <int B0, int B1>
__device__ __forceinline__ void load_blocks(const uint8_t* rb, uint32_t* w) {
#pragma unroll
    for (int b = B0; b <= B1; ++b) {
        const uint4 v = lds128(rb + 16 * b);
        w[4 * (b - B0)] = v.x;
        w[4 * (b - B0) + 1] = v.y;
        w[4 * (b - B0) + 2] = v.z;
        w[4 * (b - B0) + 3] = v.w;
    }
}

// The products sc * (q - 32) below are exact in binary16, and the constant
// -1056 * sc finite, for |sc| <= 62 (the book's workloads draw the scales on
// [-32, 31]); `bad` is set non-zero when one of the half's eight scales is
// outside that range.
// Half H of the row's block starting `delta` bytes into the 16-byte aligned
// row buffer `rb` (delta even, 0..14, the same for every lane of a unit),
// into TMEM columns [64H, +64) of this warp's lanes (taddr is the A stage's
// first column).  Sets d (the block's scale) for H == 0.  The fields' 16-byte
// blocks are loaded at fixed offsets; a uniform switch moves the words by
// delta / 4 and a uniform funnel shift handles the 2-byte remainder, so one
// code body serves every misalignment and both halves.
__device__ __forceinline__ void q6k_dequant_half(const uint8_t* rb, int H, int delta, uint32_t taddr, float& d,
                                                 uint32_t& bad) {
    uint32_t wl[20], wh[12], ws[12];
    load_blocks<0, 4>(rb + 64 * H, wl);         // ql: bytes 64H .. 64H + 79
    load_blocks<0, 2>(rb + 128 + 32 * H, wh);   // qh: bytes 128 + 32H .. + 47
    load_blocks<12, 14>(rb, ws);                // scales and d: bytes 192 .. 239
    uint32_t l[17], h[9], s[7];                 // words from delta (before the 2-byte shift)
    auto take = [&](int k) {
#pragma unroll
        for (int i = 0; i < 17; ++i) l[i] = wl[i + k];
#pragma unroll
        for (int i = 0; i < 9; ++i) h[i] = wh[i + k];
#pragma unroll
        for (int i = 0; i < 7; ++i) s[i] = ws[i + k];  // s[0..3] scales, s[4..5] d
    };
    switch (delta >> 2) {
        case 0: take(0); break;
        case 1: take(1); break;
        case 2: take(2); break;
        default: take(3); break;
    }
    if (delta & 2) {
#pragma unroll
        for (int i = 0; i < 16; ++i) l[i] = __funnelshift_r(l[i], l[i + 1], 16);
#pragma unroll
        for (int i = 0; i < 8; ++i) h[i] = __funnelshift_r(h[i], h[i + 1], 16);
#pragma unroll
        for (int i = 0; i < 6; ++i) s[i] = __funnelshift_r(s[i], s[i + 1], 16);
    }
    if (H == 0) d = h2f(s[4]);
    const uint32_t S0 = H ? s[2] : s[0], S1 = H ? s[3] : s[1];  // sc[8H .. 8H + 7]
    bad = __vcmpgtu4(__vabsss4(S0), 0x3E3E3E3Eu) | __vcmpgtu4(__vabsss4(S1), 0x3E3E3E3Eu);
#pragma unroll
    for (int ci = 0; ci < 2; ++ci) {
        // words i = 4ci..4ci+3 use the scales sc[8H + 2g + ci], g = 0..3
        uint32_t k[4], cst[4];
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int idx = 2 * g + ci;
            const uint32_t sw = idx < 4 ? S0 : S1;
            const float sc = static_cast<float>(static_cast<int8_t>((sw >> (8 * (idx & 3))) & 0xFFu));
            k[g] = h2rep(g < 2 ? sc : sc * 0.0625f);
            cst[g] = h2rep(g < 2 ? -1056.0f * sc : -96.0f * sc);
        }
        uint32_t o[32];
#pragma unroll
        for (int ii = 0; ii < 4; ++ii) {
            const int i = 4 * ci + ii;
            const uint32_t w0 = l[i];       // ql[64H + l], l = 4i..4i+3
            const uint32_t w1 = l[8 + i];   // ql[64H + 32 + l]
            const uint32_t hq = h[i];       // qh[32H + l]
            const uint32_t w0s = w0 >> 8, w1s = w1 >> 8;
            const uint32_t s4 = hq << 4, s4r = hq >> 4, s2 = hq << 2, s6r = hq >> 6;
            // g = 0, 1: 1024 + q; g = 2, 3: 1024 + 16 q (the scale carries 1/16)
            o[8 * ii + 0] = hfma2u((w0 & 0x000F000Fu) | (s4 & 0x00300030u) | kMagic2, k[0], cst[0]);
            o[8 * ii + 1] = hfma2u((w0s & 0x000F000Fu) | (s4r & 0x00300030u) | kMagic2, k[0], cst[0]);
            o[8 * ii + 2] = hfma2u((w1 & 0x000F000Fu) | (s2 & 0x00300030u) | kMagic2, k[1], cst[1]);
            o[8 * ii + 3] = hfma2u((w1s & 0x000F000Fu) | (s6r & 0x00300030u) | kMagic2, k[1], cst[1]);
            o[8 * ii + 4] = hfma2u((w0 & 0x00F000F0u) | (s4 & 0x03000300u) | kMagic2, k[2], cst[2]);
            o[8 * ii + 5] = hfma2u((w0s & 0x00F000F0u) | (s4r & 0x03000300u) | kMagic2, k[2], cst[2]);
            o[8 * ii + 6] = hfma2u((w1 & 0x00F000F0u) | (s2 & 0x03000300u) | kMagic2, k[3], cst[3]);
            o[8 * ii + 7] = hfma2u((w1s & 0x00F000F0u) | (s6r & 0x03000300u) | kMagic2, k[3], cst[3]);
        }
        tmem_st32(taddr + 64u * H + 32u * ci, o);
    }
}

// ---------------------------------------------------------------- kernel
__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
constexpr int kBarReadback = 1;  // the four readback warps (128 threads)
constexpr int kBarBuild = 2;     // one row of x: every warp but the bulk-copy warp

// Super-block of the k-th unit of a tile.  Q6_K visits a tile's blocks in
// (sb mod 8, sb / 8) order: the block's misalignment in shared memory
// depends only on sb mod 8, so one realignment code path serves runs of
// consecutive units.  Q4_K blocks are aligned and keep their order.
template <int QT>
__device__ __forceinline__ int unit_sb(int k, int nsb) {
    if constexpr (QT == MUSER_Q4_K) {
        return k;
    } else {
        int start = 0;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
            const int cnt = (nsb - r + 7) >> 3;  // blocks sb = r mod 8 below nsb
            if (k < start + cnt) return r + 8 * (k - start);
            start += cnt;
        }
        return 0;
    }
}

// Walks a CTA's units in order without divisions: tile t, position k in the
// tile, and the super-block sb visited at that position (see unit_sb).
template <int QT>
struct UnitIter {
    int t, k, sb, nsb;
    __device__ __forceinline__ UnitIter(int64_t u, int nsb_) : nsb(nsb_) {
        t = static_cast<int>(u / nsb_);
        k = static_cast<int>(u - static_cast<int64_t>(t) * nsb_);
        sb = unit_sb<QT>(k, nsb_);
    }
    __device__ __forceinline__ void next() {
        if (++k == nsb) {
            k = 0;
            ++t;
            sb = 0;
        } else if constexpr (QT == MUSER_Q4_K) {
            sb = k;
        } else {
            sb += 8;  // next block of the same residue, or the first of the next residue
            if (sb >= nsb) sb = (sb & 7) + 1;
        }
    }
};

// Slot and phase bit of a ring of barriers, advanced once per unit.
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void next(int n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// CTA that owns unit u when U units are split evenly over G CTAs.
__device__ __forceinline__ int cta_of(int64_t u, int64_t U, int64_t G) {
    return static_cast<int>(((u + 1) * G - 1) / U);
}

struct TileMap {
    int P, nmat;
    // Row and matrix of TMEM lane l in tile t.
    __device__ __forceinline__ int64_t row(int t, int l, int& mat) const {
        if (nmat == 2) {
            mat = l >> 6;
            return static_cast<int64_t>(t) * 64 + (l & 63);
        }
        mat = 0;
        return static_cast<int64_t>(t / P) * 128 * P + static_cast<int64_t>(l) * P + (t % P);
    }
};

// Splits a pair of scaled values (|a| < 2^15) into binary16 hi and lo with
// a = hi + lo * 2^-11: hi is a rounded to a multiple of 16 (the 1.5 * 2^27
// add/subtract rounds at that grid), exact in binary16; lo = (a - hi) * 2^11,
// |lo| <= 2^14, rounded once.  The error is at most 2^-8 in units of a, that
// is 2^-22 of the block maximum.
__device__ __forceinline__ void pack_hl(float2 a, uint32_t& hi, uint32_t& lo) {
    const float2 c = make_float2(201326592.0f, 201326592.0f);
    const float2 h = __fadd2_rn(__fadd2_rn(a, c), make_float2(-c.x, -c.y));
    const float2 r = __fmul2_rn(__fadd2_rn(a, make_float2(-h.x, -h.y)), make_float2(2048.0f, 2048.0f));
    const __half2 hh = __float22half2_rn(h), hl = __float22half2_rn(r);
    hi = *reinterpret_cast<const uint32_t*>(&hh);
    lo = *reinterpret_cast<const uint32_t*>(&hl);
}
__device__ __forceinline__ void pack_hl(float a, float b, uint32_t& hi, uint32_t& lo) {
    pack_hl(make_float2(a, b), hi, lo);
}
// Exponent E with max|x| < 2^E, kept in a range where both 2^(15-E) and
// 2^(E-15) are finite normal floats.
__device__ __forceinline__ int scale_exp(float mx) {
    int E = 0;
    if (mx > 0.0f) (void)frexpf(mx, &E);
    return min(max(E, -100), 120);
}

// One row of x for one super-block, by one warp: binary16 hi/lo words of the
// block's 128 columns (four per lane for Q4_K: words hi[0..3], lo[0..3] of
// chunk 8c + t; eight for Q6_K lanes 0-15: chunks 16h + 2i and + 1), the
// block's power-of-two scale 2^e (max|x| * 2^-e < 2^15) and, for Q4_K, the
// sub-block sums of x (valid in lanes t == 0: sub-blocks 2c and 2c + 1).
template <int QT>
struct BlockX {
    uint4 hi0, lo0, hi1, lo1;
    float esc, sa, sb;
};
// The lane's x values of a block: Q4_K v[0] = x[64c + 4t ..], v[1] = x[64c +
// 32 + 4t ..]; Q6_K v[g] = x[128h + 32g + 4i ..] (g = 0..3).  Read through L2:
// x may be the output of the kernel this one waits for.
template <int QT>
__device__ __forceinline__ void block_x_load(const float* xb, int lane, float4* v) {
    if constexpr (QT == MUSER_Q4_K) {
        const int c = lane >> 3, t = lane & 7;
        v[0] = __ldcg(reinterpret_cast<const float4*>(xb + 64 * c + 4 * t));
        v[1] = __ldcg(reinterpret_cast<const float4*>(xb + 64 * c + 32 + 4 * t));
    } else {
        const int item = lane & 15, h = item >> 3, i = item & 7;
#pragma unroll
        for (int g = 0; g < 4; ++g) v[g] = __ldcg(reinterpret_cast<const float4*>(xb + 128 * h + 32 * g + 4 * i));
    }
}
template <int QT>
__device__ __forceinline__ BlockX<QT> block_x(const float4* pv, int lane) {
    BlockX<QT> r;
    if constexpr (QT == MUSER_Q4_K) {
        const float4 xa = pv[0];
        const float4 xc = pv[1];
        float mx = fmaxf(fmaxf(fmaxf(fabsf(xa.x), fabsf(xa.y)), fmaxf(fabsf(xa.z), fabsf(xa.w))),
                         fmaxf(fmaxf(fabsf(xc.x), fabsf(xc.y)), fmaxf(fabsf(xc.z), fabsf(xc.w))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int E = scale_exp(mx);
        const float dn = ldexpf(1.0f, 15 - E);
        pack_hl(xa.x * dn, xa.z * dn, r.hi0.x, r.lo0.x);
        pack_hl(xa.y * dn, xa.w * dn, r.hi0.y, r.lo0.y);
        pack_hl(xc.x * dn, xc.z * dn, r.hi0.z, r.lo0.z);
        pack_hl(xc.y * dn, xc.w * dn, r.hi0.w, r.lo0.w);
        float sa = (xa.x + xa.y) + (xa.z + xa.w), sc = (xc.x + xc.y) + (xc.z + xc.w);
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
            sa += __shfl_xor_sync(0xffffffffu, sa, o);
            sc += __shfl_xor_sync(0xffffffffu, sc, o);
        }
        r.sa = sa;
        r.sb = sc;
        r.esc = ldexpf(1.0f, E - 15);
    } else {
        const float4* v = pv;
        float mx = 0.0f;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[g].x), fabsf(v[g].y)), fmaxf(fabsf(v[g].z), fabsf(v[g].w))));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const int E = scale_exp(mx);
        const float dn = ldexpf(1.0f, 15 - E);
        pack_hl(v[0].x * dn, v[0].z * dn, r.hi0.x, r.lo0.x);
        pack_hl(v[0].y * dn, v[0].w * dn, r.hi0.y, r.lo0.y);
        pack_hl(v[1].x * dn, v[1].z * dn, r.hi0.z, r.lo0.z);
        pack_hl(v[1].y * dn, v[1].w * dn, r.hi0.w, r.lo0.w);
        pack_hl(v[2].x * dn, v[2].z * dn, r.hi1.x, r.lo1.x);
        pack_hl(v[2].y * dn, v[2].w * dn, r.hi1.y, r.lo1.y);
        pack_hl(v[3].x * dn, v[3].z * dn, r.hi1.z, r.lo1.z);
        pack_hl(v[3].y * dn, v[3].w * dn, r.hi1.w, r.lo1.w);
        r.sa = r.sb = 0.0f;
        r.esc = ldexpf(1.0f, E - 15);
    }
    return r;
}

// Several rows of x: lane (m, q) of a builder warp converts a quarter of
// row m's block (64 values) straight into the B slab.  The quarter is the
// set of 16-byte x chunks j with j = q mod 4, which keeps the shared-memory
// reads of a warp at most 2-way conflicted; the row's block maximum and the
// Q4_K sub-block sums need only the 4 lanes of the row.  Returns 2^e, the
// row's block scale; the sums of sub-blocks 0..7 are valid in lane q == 0.
// store == false: the lanes only take part in the shuffles.
template <int QT>
__device__ __forceinline__ float build_row_quarter(const float* xrow, int q, uint8_t* slab, uint32_t rowoff,
                                                   float* xsum8, bool store_slab = true) {
    float4 v[16];
    if constexpr (QT == MUSER_Q4_K) {
        // B chunk 8c + t (t = q, q + 4): x chunks 16c + t and 16c + 8 + t
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int t = q + 4 * h;
                v[4 * c + 2 * h] = lds_f4(xrow + 64 * c + 4 * t);
                v[4 * c + 2 * h + 1] = lds_f4(xrow + 64 * c + 32 + 4 * t);
            }
    } else {
        // item (h, i), i = q + 4e: x chunks 32h + 8g + i, g = 0..3
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int g = 0; g < 4; ++g)
                    v[8 * h + 4 * e + g] = lds_f4(xrow + 128 * h + 32 * g + 4 * (q + 4 * e));
    }
    float mx = 0.0f;
#pragma unroll
    for (int k = 0; k < 16; ++k)
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v[k].x), fabsf(v[k].y)), fmaxf(fabsf(v[k].z), fabsf(v[k].w))));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const int E = scale_exp(mx);
    const float dn = ldexpf(1.0f, 15 - E);
    auto store = [&](int chunk, const float4& a, const float4& b) {
        // columns (a.x,a.z) (a.y,a.w) (b.x,b.z) (b.y,b.w) of the chunk
        uint4 hi, lo;
        const float2 d2 = make_float2(dn, dn);
        pack_hl(__fmul2_rn(make_float2(a.x, a.z), d2), hi.x, lo.x);
        pack_hl(__fmul2_rn(make_float2(a.y, a.w), d2), hi.y, lo.y);
        pack_hl(__fmul2_rn(make_float2(b.x, b.z), d2), hi.z, lo.z);
        pack_hl(__fmul2_rn(make_float2(b.y, b.w), d2), hi.w, lo.w);
        if (!store_slab) return;
        uint8_t* ch = slab + chunk * 512 + rowoff;
        *reinterpret_cast<uint4*>(ch) = hi;
        *reinterpret_cast<uint4*>(ch + 16) = lo;
    };
    if constexpr (QT == MUSER_Q4_K) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            float sa = 0.0f, sb = 0.0f;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const float4 a = v[4 * c + 2 * h], b = v[4 * c + 2 * h + 1];
                store(8 * c + q + 4 * h, a, b);
                sa += (a.x + a.y) + (a.z + a.w);
                sb += (b.x + b.y) + (b.z + b.w);
            }
            sa += __shfl_xor_sync(0xffffffffu, sa, 1);
            sa += __shfl_xor_sync(0xffffffffu, sa, 2);
            sb += __shfl_xor_sync(0xffffffffu, sb, 1);
            sb += __shfl_xor_sync(0xffffffffu, sb, 2);
            xsum8[2 * c] = sa;
            xsum8[2 * c + 1] = sb;
        }
    } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = q + 4 * e;
                store(16 * h + 2 * i, v[8 * h + 4 * e], v[8 * h + 4 * e + 1]);
                store(16 * h + 2 * i + 1, v[8 * h + 4 * e + 2], v[8 * h + 4 * e + 3]);
            }
    }
    return ldexpf(1.0f, E - 15);
}

template <int QT, int EPI, bool MULTI>
__global__ void __launch_bounds__(mvt_threads(MULTI), 1)
    mvt_kernel(const MvtArgs p, const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
               const __grid_constant__ CUtensorMap mapx, const __grid_constant__ CUtensorMap map2,
               const __grid_constant__ CUtensorMap map3) {
    constexpr int NMAT = (EPI == kEpiSiluMul) ? 2 : 1;
    constexpr int kBlk = (QT == MUSER_Q4_K) ? kQ4KBytes : kQ6KBytes;
    constexpr int RS = (QT == MUSER_Q4_K) ? 144 : 240;  // row slot of a stage (odd multiple of 16 B)
    constexpr uint32_t kStage = 128u * RS;
    constexpr int kThr = mvt_threads(MULTI);
    constexpr uint32_t kXSlot = 8 * 256 * 4;             // eight rows of x for one block
    constexpr int MB = MULTI ? 16 : 1;                   // rows of x a lane accumulates
    constexpr uint32_t kDCols = MULTI ? 32u : 16u;       // D columns per buffer
    constexpr uint32_t kIdesc = idesc_n(kDCols);
    constexpr uint32_t kSlab = 16384;                    // B slab of one unit (several rows of x)
    constexpr int kXr = MB * 8 + MB;                     // per-unit x sums (Q4_K) and scales, floats
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nsb = p.nsb;
    const int M = MULTI ? p.M : 1;
    const int64_t rowbytes = static_cast<int64_t>(nsb) * kBlk;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NS = p.ns;
    const int64_t U = static_cast<int64_t>(p.ntiles) * nsb, G = gridDim.x;
    // Even split of the units (tiles may straddle CTAs), or whole tiles.
    int64_t u0 = U * blockIdx.x / G, u1 = U * (blockIdx.x + 1) / G;
    if (p.tiles_per_cta > 0) {
        u0 = std::min<int64_t>(U, static_cast<int64_t>(blockIdx.x) * p.tiles_per_cta * nsb);
        u1 = std::min<int64_t>(U, u0 + static_cast<int64_t>(p.tiles_per_cta) * nsb);
    }
    const int nunits = static_cast<int>(u1 - u0);
    const TileMap tm{p.P, NMAT};

    // shared memory: barriers | TMEM address, flags | red | scale ring | xch |
    // x scales and sums | B operand | weight stages
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    uint64_t* afull = empty + kMaxStages;
    uint64_t* dfull = afull + kNA;   // MMA of the slot's unit done: A stage and B slab free, D ready
    uint64_t* dempty = dfull + kND;
    uint64_t* sfull = dempty + kND;
    uint64_t* bfull = sfull + kND;
    uint64_t* xfull = bfull + kNB;   // [2 builder warps][kNB]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 448);
    int* flags = reinterpret_cast<int*>(smem + 464);       // [0] run the tail, [1] tile ticket won
    float* red = reinterpret_cast<float*>(smem + 512);     // 64 floats
    float4* scr = reinterpret_cast<float4*>(smem + 1280);  // [kND][128] block scales per lane
    float* xch = reinterpret_cast<float*>(smem + p.xch_off);  // [MB][128] tile values
    // one row of x: esc[nsb] 2^e per block, X[nsb * 8] sub-block sums;
    // several rows: a ring [kND][kXr] of X[m][8] and esc[m] per unit
    float* esc = reinterpret_cast<float*>(smem + p.x_off);
    float* X = esc + ((nsb + 3) & ~3);
    float* xr = reinterpret_cast<float*>(smem + p.x_off);
    uint8_t* B = smem + p.b_off;
    uint8_t* xring = B + kNB * kSlab;  // several rows: [2 builder warps][kNB] slots of 8 rows of x
    uint8_t* stages = smem + p.stage_off;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kDeqWarps);
        }
        for (int i = 0; i < kNA; ++i) {
            mbar_init(&afull[i], kDeqWarps);
        }
        for (int i = 0; i < kND; ++i) {
            mbar_init(&dfull[i], 1);
            mbar_init(&dempty[i], 4);
            mbar_init(&sfull[i], MULTI ? 6 : 4);  // dequant warps of half 0 (+ the builders)
        }
        for (int i = 0; i < kNB; ++i) {
            mbar_init(&bfull[i], 2);
            mbar_init(&xfull[i], 1);
            mbar_init(&xfull[kNB + i], 1);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_launch_dependents();
    bool ok = true;

    if (warp == kTmaWarp) {
        // ------------------------------------------------ bulk-copy warp
        // Weights do not depend on the previous kernel: no PDL wait here.
        // Each weight byte is read once per call: evict-first in L2.
        const uint64_t wpol = l2_policy_evict_first();
        UnitIter<QT> it(u0, nsb);
        Ring rs;
        for (int i = 0; i < nunits && ok; ++i, it.next(), rs.next(NS)) {
            const int s = rs.slot;
            if (i >= NS) ok = mbar_wait_bounded(&empty[s], rs.phase ^ 1u, p.status, kDevStatusWaitTimeout);
            if (!ok) break;
            const int t = it.t, sb = it.sb;
            uint8_t* dst = stages + static_cast<size_t>(s) * kStage;
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], kStage);
                if constexpr (NMAT == 2) {
                    // gate rows to lanes 0..63, up rows to lanes 64..127
                    tma_load_2d_hint(dst, &map0, sb * kBlk, t * 64, &full[s], wpol);
                    tma_load_2d_hint(dst + 64 * RS, &map1, sb * kBlk, t * 64, &full[s], wpol);
                } else if constexpr (QT == MUSER_Q4_K) {
                    if (p.nseg > 0) {
                        // a group: the segment's own map, its own tile rows
                        int sg = 0;
                        while (sg + 1 < p.nseg && t >= p.seg_t0[sg + 1]) ++sg;
                        const CUtensorMap* mp = sg == 0 ? &map0 : sg == 1 ? &map1 : sg == 2 ? &map2 : &map3;
                        tma_load_2d_hint(dst, mp, sb * kBlk, (t - p.seg_t0[sg]) * 128, &full[s], wpol);
                    } else {
                        tma_load_2d_hint(dst, &map0, sb * kBlk, t * 128, &full[s], wpol);
                    }
                } else {
                    // class t % P of block t / P: box from the 16-byte boundary below the block
                    const int64_t off = static_cast<int64_t>(t % p.P) * rowbytes + static_cast<int64_t>(sb) * kBlk;
                    tma_load_2d_hint(dst, &map0, static_cast<int>(off & ~static_cast<int64_t>(15)), (t / p.P) * 128,
                                     &full[s], wpol);
                }
            }
            __syncwarp();
        }
    } else {
        // x is the previous kernel's output, and outputs are written after
        // it.  With several rows of x the dequantisation and MMA warps read
        // neither (weights, shared and tensor memory only): they fill the A
        // stages while the previous kernel finishes.
        if (!MULTI || !(warp == kMmaWarp || warp < kDeqWarps)) pdl_wait();
        if constexpr (!MULTI) {
            // ---------- one row of x: the whole B operand, one warp per block
            const int bw = warp < kTmaWarp ? warp : warp - 1;
            constexpr int nbw = kThr / 32 - 1;
            constexpr int kG = 4;                          // blocks a warp loads before converting
            constexpr int kV = QT == MUSER_Q4_K ? 2 : 4;   // float4 per lane and block
            for (int sb0 = bw; sb0 < nsb; sb0 += kG * nbw) {
                float4 raw[kG][kV];
#pragma unroll
                for (int j = 0; j < kG; ++j)
                    if (sb0 + j * nbw < nsb) block_x_load<QT>(p.x + (sb0 + j * nbw) * 256, lane, raw[j]);
#pragma unroll
                for (int j = 0; j < kG; ++j) {
                const int sb = sb0 + j * nbw;
                if (sb >= nsb) break;
                const BlockX<QT> bx = block_x<QT>(raw[j], lane);
                if constexpr (QT == MUSER_Q4_K) {
                    const int c = lane >> 3, t = lane & 7;
                    uint8_t* ch = B + 32 * (sb * 32 + 8 * c + t);
                    *reinterpret_cast<uint4*>(ch) = bx.hi0;
                    *reinterpret_cast<uint4*>(ch + 16) = bx.lo0;
                    if (t == 0) {
                        X[sb * 8 + 2 * c] = bx.sa;
                        X[sb * 8 + 2 * c + 1] = bx.sb;
                    }
                } else if (lane < 16) {
                    const int h = lane >> 3, i = lane & 7;
                    uint8_t* ch = B + 32 * (sb * 32 + 16 * h + 2 * i);
                    *reinterpret_cast<uint4*>(ch) = bx.hi0;
                    *reinterpret_cast<uint4*>(ch + 16) = bx.lo0;
                    *reinterpret_cast<uint4*>(ch + 32) = bx.hi1;
                    *reinterpret_cast<uint4*>(ch + 48) = bx.lo1;
                }
                if (lane == 0) esc[sb] = bx.esc;
                }
            }
            if (bw == 0) reinterpret_cast<uint4*>(B + nsb * 1024)[lane] = make_uint4(0u, 0u, 0u, 0u);  // slack
            fence_proxy_async_smem();
            named_sync(kBarBuild, nbw * 32);
        }

        if (warp == kMmaWarp) {
            // ----------------------------------------------- MMA issue
            if (lane == 0) {
                UnitIter<QT> it(u0, nsb);
                Ring ra, rd, rb;
                for (int i = 0; i < nunits && ok; ++i, it.next(), ra.next(kNA), rd.next(kND), rb.next(kNB)) {
                    const int a = ra.slot, db = rd.slot;
                    ok = mbar_wait_bounded(&afull[a], ra.phase, p.status, kDevStatusWaitTimeout);
                    if (MULTI && ok) ok = mbar_wait_bounded(&bfull[rb.slot], rb.phase, p.status, kDevStatusWaitTimeout);
                    if (ok && i >= kND) ok = mbar_wait_bounded(&dempty[db], rd.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t dcol = tmem + kDCol0 + kDCols * db, acol = tmem + 128u * a;
                    if constexpr (MULTI) {
                        // slab: K chunk stride 512 B, N-group stride 128 B
                        const uint32_t bbase = smem_u32(B) + kSlab * rb.slot;
                        mma_chain16(dcol, acol, smem_desc(bbase, 512u, 128u), kIdesc, 1024u >> 4);
                    } else {
                        // compact: two rows per 32-byte chunk, chunks overlap
                        const uint32_t bbase = smem_u32(B) + 1024u * it.sb;
                        mma_chain16(dcol, acol, smem_desc(bbase, 32u, 256u), kIdesc, 64u >> 4);
                    }
                    mma_commit(&dfull[db]);
                }
            }
            __syncwarp();
        } else if (warp < kDeqWarps) {
            // ------------------------------------- dequantisation warps
            const int q = warp & 3, hf = warp >> 2;
            const int l = 32 * q + lane;  // this thread's TMEM lane in every tile
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
            UnitIter<QT> it(u0, nsb);
            Ring rs, ra, rd;
            int cur_t = -1, cls_off = 0;  // Q6_K: (class * row bytes) mod 16 of the current tile
            for (int i = 0; i < nunits; ++i, it.next(), rs.next(NS), ra.next(kNA), rd.next(kND)) {
                const int s = rs.slot, a = ra.slot, db = rd.slot;
                if (ok) ok = mbar_wait_bounded(&full[s], rs.phase, p.status, kDevStatusWaitTimeout);
                if (ok && i >= kNA) ok = mbar_wait_bounded(&dfull[a], ra.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                const uint8_t* rbuf = stages + static_cast<size_t>(s) * kStage + l * RS;
                const uint32_t ta = tq + 128u * a;
                const int sb = it.sb;
                float4 sc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (ok) {
                    if constexpr (QT == MUSER_Q4_K) {
                        q4k_dequant_half(rbuf, hf, ta);
                        if (hf == 0) {
                            if constexpr (MULTI) {
                                uint32_t m03, m47;
                                q4k_block_dmins(rbuf, sc.x, sc.y, m03, m47);
                                sc.z = __uint_as_float(m03);
                                sc.w = __uint_as_float(m47);
                            } else {
                                q4k_block_scales(rbuf, X + 8 * sb, sc.x, sc.y);
                                sc.x *= esc[sb];
                            }
                        }
                    } else {
                        if (it.t != cur_t) {
                            cur_t = it.t;
                            cls_off = static_cast<int>((static_cast<int64_t>(cur_t % p.P) * rowbytes) & 15);
                        }
                        const int delta = (cls_off + 2 * sb) & 15;  // 210 = 2 mod 16
                        float d = 0.0f;
                        uint32_t bad = 0u;
                        q6k_dequant_half(rbuf, hf, delta, ta, d, bad);
                        if (bad) atomicOr(p.status, kDevStatusQ6kScale);
                        sc.x = MULTI ? d : d * esc[sb];
                    }
                    tc_wait_st();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&afull[a]);
                    mbar_arrive(&empty[s]);
                }
                if (hf == 0) {
                    // hand this unit's block scales to the readback warp of the quadrant
                    if (ok && i >= kND) ok = mbar_wait_bounded(&dempty[db], rd.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                    scr[db * 128 + l] = sc;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sfull[db]);
                }
            }
        } else if (MULTI && warp >= kBldWarp0 && p.bimg != nullptr) {
            // -------- several rows of x, B image prebuilt: per unit, one
            // bulk copy of the super-block's slab and of its sums and scales
            // (the image is the previous kernel's output: read after the PDL
            // wait above).  Warp kBldWarp0 copies, the other only arrives.
            const int bw = warp - kBldWarp0;
            UnitIter<QT> it(u0, nsb);
            Ring rb, rd;
            for (int i = 0; i < nunits; ++i, it.next(), rb.next(kNB), rd.next(kND)) {
                if (ok && i >= kNB) ok = mbar_wait_bounded(&dfull[rb.slot], rb.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                if (ok && i >= kND) ok = mbar_wait_bounded(&dempty[rd.slot], rd.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                if (bw == 0) {
                    if (ok && lane == 0) {
                        const uint8_t* src = p.bimg + static_cast<size_t>(it.sb) * kBImg;
                        mbar_arrive_expect_tx(&xfull[rb.slot], kBImg);
                        tma_load_1d(B + kSlab * rb.slot, src, kSlabBytes, &xfull[rb.slot]);
                        tma_load_1d(xr + kXr * rd.slot, src + kSlabBytes, kXrBytes, &xfull[rb.slot]);
                    }
                    if (ok) ok = mbar_wait_bounded(&xfull[rb.slot], rb.phase, p.status, kDevStatusWaitTimeout);
                }
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bfull[rb.slot]);
                    mbar_arrive(&sfull[rd.slot]);
                }
            }
        } else if (MULTI && warp >= kBldWarp0) {
            // -------- several rows of x: per-unit B slabs, scales and sums
            // Builder warp bw owns rows 8bw..8bw+7 of x; its slots of x are
            // filled by 2-D tensor copies (rows past M read as zero), kNB
            // units ahead.
            const int bw = warp - kBldWarp0;
            const int mlo = 8 * bw, mhi = min(M, mlo + 8);
            uint64_t* xf = xfull + kNB * bw;
            uint8_t* xs0 = xring + static_cast<size_t>(bw) * kNB * kXSlot;
            auto load_x = [&](int slot, int sb) {
                mbar_arrive_expect_tx(&xf[slot], kXSlot);
                tma_load_2d(xs0 + slot * kXSlot, &mapx, sb * 256, mlo, &xf[slot]);
            };
            if (lane == 0 && mlo < M) {
                UnitIter<QT> ahead(u0, nsb);
                for (int j = 0; j < kNB && j < nunits; ++j, ahead.next()) load_x(j, ahead.sb);
            }
            UnitIter<QT> it(u0, nsb), ahead(u0, nsb);
            for (int j = 0; j < kNB; ++j) ahead.next();
            Ring rb, rd;
            for (int i = 0; i < nunits; ++i, it.next(), ahead.next(), rb.next(kNB), rd.next(kND)) {
                if (ok && i >= kNB) ok = mbar_wait_bounded(&dfull[rb.slot], rb.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                if (ok && i >= kND) ok = mbar_wait_bounded(&dempty[rd.slot], rd.phase ^ 1u, p.status, kDevStatusWaitTimeout);
                if (ok && mlo < M) ok = mbar_wait_bounded(&xf[rb.slot], rb.phase, p.status, kDevStatusWaitTimeout);
                uint8_t* slab = B + kSlab * rb.slot;
                float* xu = xr + kXr * rd.slot;
                const float* xs = reinterpret_cast<const float*>(xs0 + rb.slot * kXSlot);
                if (ok && mlo < M) {
                    // lane (m, q): row m = mlo + lane / 4, quarter q = lane % 4
                    const int ml = lane >> 2, q = lane & 3, m = mlo + ml;
                    float xs8[8];
                    const float e2 = build_row_quarter<QT>(xs + ml * 256, q, slab,
                                                           (m >> 2) * 128 + (2 * m & 7) * 16, xs8);
                    if (m < mhi && q == 0) {
                        xu[8 * MB + m] = e2;
                        if constexpr (QT == MUSER_Q4_K) {
                            *reinterpret_cast<float4*>(xu + 8 * m) = make_float4(xs8[0], xs8[1], xs8[2], xs8[3]);
                            *reinterpret_cast<float4*>(xu + 8 * m + 4) = make_float4(xs8[4], xs8[5], xs8[6], xs8[7]);
                        }
                    }
                }
                fence_proxy_async_smem();  // slab for the MMA; x slot for the next copy
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bfull[rb.slot]);
                    mbar_arrive(&sfull[rd.slot]);
                    if (mlo < M && i + kNB < nunits) load_x(rb.slot, ahead.sb);
                }
            }
        } else if (warp >= kRbWarp0 && warp < kRbWarp0 + 4) {
            // ------------------------------ readback and epilogue warps
            const int q = warp & 3;
            const int l = 32 * q + lane;
            const uint32_t tq = tmem + (static_cast<uint32_t>(32 * q) << 16);
            float yacc[MB];
#pragma unroll
            for (int m = 0; m < MB; ++m) yacc[m] = 0.0f;
            UnitIter<QT> it(u0, nsb);
            Ring rd;
            for (int i = 0; i < nunits; ++i, it.next(), rd.next(kND)) {
                const int db = rd.slot;
                if (ok) ok = mbar_wait_bounded(&dfull[db], rd.phase, p.status, kDevStatusWaitTimeout);
                if (ok) ok = mbar_wait_bounded(&sfull[db], rd.phase, p.status, kDevStatusWaitTimeout);
                const float4 sc = lds_f4(&scr[db * 128 + l]);
                if constexpr (MULTI) {
                    uint32_t dv[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) dv[j] = 0u;
                    if (ok) {
                        tc_fence_after();
                        tmem_ld32(tq + kDCol0 + kDCols * db, dv);
                        tc_wait_ld();
                    }
                    const float* xu = xr + kXr * db;
                    float mins[8];
                    if constexpr (QT == MUSER_Q4_K) {
                        const uint32_t m03 = __float_as_uint(sc.z), m47 = __float_as_uint(sc.w);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            mins[j] = static_cast<float>((m03 >> (8 * j)) & 0xFFu);
                            mins[j + 4] = static_cast<float>((m47 >> (8 * j)) & 0xFFu);
                        }
                    }
#pragma unroll
                    for (int m4 = 0; m4 < MB; m4 += 4) {
                        if (m4 >= M) break;
                        const float4 e4 = lds_f4(xu + 8 * MB + m4);
                        const float ev[4] = {e4.x, e4.y, e4.z, e4.w};
#pragma unroll
                        for (int mm = 0; mm < 4; ++mm) {
                            const int m = m4 + mm;
                            const float dd = __uint_as_float(dv[2 * m]) + __uint_as_float(dv[2 * m + 1]) * (1.0f / 2048.0f);
                            float v = dd * (sc.x * ev[mm]);
                            if constexpr (QT == MUSER_Q4_K) {
                                const float4 xa = lds_f4(xu + 8 * m);
                                const float4 xb = lds_f4(xu + 8 * m + 4);
                                float s = mins[0] * xa.x;
                                s = fmaf(mins[1], xa.y, s);
                                s = fmaf(mins[2], xa.z, s);
                                s = fmaf(mins[3], xa.w, s);
                                s = fmaf(mins[4], xb.x, s);
                                s = fmaf(mins[5], xb.y, s);
                                s = fmaf(mins[6], xb.z, s);
                                s = fmaf(mins[7], xb.w, s);
                                v = fmaf(-sc.y, s, v);
                            }
                            yacc[m] += v;  // rows m >= M stay zero-weighted and are never stored
                        }
                    }
                } else {
                    uint32_t r0 = 0, r1 = 0;
                    if (ok) {
                        tc_fence_after();
                        tmem_ld2(tq + kDCol0 + kDCols * db, r0, r1);
                        tc_wait_ld();
                    }
                    yacc[0] += fmaf(__uint_as_float(r0) + __uint_as_float(r1) * (1.0f / 2048.0f), sc.x, -sc.y);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&dempty[db]);
                const int t = it.t;
                if (it.k != nsb - 1 && i != nunits - 1) continue;
                // ---- the tile's last unit in this CTA
                int c0 = blockIdx.x, c1 = blockIdx.x;
                if (p.tiles_per_cta == 0) {
                    c0 = cta_of(static_cast<int64_t>(t) * nsb, U, G);
                    c1 = cta_of(static_cast<int64_t>(t + 1) * nsb - 1, U, G);
                }
                float val[MB];
#pragma unroll
                for (int m = 0; m < MB; ++m) {
                    val[m] = yacc[m];
                    yacc[m] = 0.0f;
                }
                if (c1 > c0) {
                    // Tile t's part from CTA c sits in slot t + c (MB x 128 floats):
                    // CTAs take the units in order, so no two (tile, CTA) pairs share a slot.
                    float* own = p.part + static_cast<size_t>(t + blockIdx.x) * MB * 128;
#pragma unroll
                    for (int m = 0; m < MB; ++m)
                        if (m < M) own[m * 128 + l] = val[m];
                    // the ticket after the readback warps' barrier, with
                    // acquire-release semantics: it releases their part and
                    // the last CTA's acquire covers every other part
                    named_sync(kBarReadback, 128);
                    if (l == 0)
                        flags[1] = (atom_add_acq_rel_gpu(&p.tick[t], 1u) == static_cast<unsigned>(c1 - c0)) ? 1 : 0;
                    named_sync(kBarReadback, 128);
                    const bool last = flags[1] != 0;
                    named_sync(kBarReadback, 128);
                    if (!last) continue;
#pragma unroll
                    for (int m = 0; m < MB; ++m) val[m] = 0.0f;
                    // The parts in order (the sum does not depend on timing),
                    // two at a time and loads only, so their L2 round trips
                    // overlap; the zeroing stores follow in a pass of their own.
                    const int np = c1 - c0 + 1;
                    const float* part0 = p.part + static_cast<size_t>(t + c0) * MB * 128 + l;
                    int pp = 0;
                    for (; pp + 1 < np; pp += 2) {
                        const float* s0 = part0 + static_cast<size_t>(pp) * MB * 128;
                        const float* s1 = s0 + MB * 128;
                        float a0[MB], a1[MB];
#pragma unroll
                        for (int m = 0; m < MB; ++m) {
                            a0[m] = m < M ? __ldcg(s0 + m * 128) : 0.0f;
                            a1[m] = m < M ? __ldcg(s1 + m * 128) : 0.0f;
                        }
#pragma unroll
                        for (int m = 0; m < MB; ++m) val[m] = (val[m] + a0[m]) + a1[m];
                    }
                    if (pp < np) {
                        const float* s0 = part0 + static_cast<size_t>(pp) * MB * 128;
#pragma unroll
                        for (int m = 0; m < MB; ++m)
                            if (m < M) val[m] += __ldcg(s0 + m * 128);
                    }
                    // leave the scratch zeroed
                    for (int q = 0; q < np; ++q) {
                        float* s0 = p.part + static_cast<size_t>(t + c0 + q) * MB * 128 + l;
#pragma unroll
                        for (int m = 0; m < MB; ++m)
                            if (m < M) s0[m * 128] = 0.0f;
                    }
                    if (l == 0) p.tick[t] = 0u;
                }
                int mat;
                const int64_t row = tm.row(t, l, mat);
                if constexpr (EPI == kEpiSiluMul) {
#pragma unroll
                    for (int m = 0; m < MB; ++m)
                        if (m < M) xch[m * 128 + l] = val[m];
                    named_sync(kBarReadback, 128);
                    if (l < 64 && row < p.rows) {
                        for (int m = 0; m < M; ++m)
                            p.y[static_cast<int64_t>(m) * p.rows + row] = silu_mul_f(xch[m * 128 + l], xch[m * 128 + l + 64]);
                    }
                    named_sync(kBarReadback, 128);
                } else if (EPI == kEpiStore && p.nseg > 0) {
                    int sg = 0;
                    while (sg + 1 < p.nseg && t >= p.seg_t0[sg + 1]) ++sg;
                    const int64_t srow = static_cast<int64_t>(t - p.seg_t0[sg]) * 128 + l, nrows = p.seg_rows[sg];
                    if (srow < nrows) {
#pragma unroll
                        for (int m = 0; m < MB; ++m)
                            if (m < M) p.seg_y[sg][static_cast<int64_t>(m) * nrows + srow] = val[m];
                    }
                } else {
                    if (row < p.rows) {
#pragma unroll
                        for (int m = 0; m < MB; ++m)
                            if (m < M) p.y[static_cast<int64_t>(m) * p.rows + row] = val[m];
                    }
                    if constexpr (EPI == kEpiTail) {
                        named_sync(kBarReadback, 128);
                        if (l == 0 && atom_add_acq_rel_gpu(&p.tick[p.ntiles], 1u) == static_cast<unsigned>(p.ntiles - 1))
                            flags[0] = 1;
                    }
                }
            }
        }
    }
    tc_fence_before();
    ok = __syncthreads_and(ok);
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if constexpr (EPI == kEpiTail && !MULTI) {
        if (ok && flags[0]) {
            block_dual_tail_row(p.resid, p.y, p.out, p.w1, p.w2, static_cast<int>(p.rows), p.eps1, p.eps2, red);
            if (tid == 0) p.tick[p.ntiles] = 0u;
        }
    }
}

// Several rows of x: the B image of super-block blockIdx.x (its slab, the
// rows' sub-block sums of x and scales), built by two warps exactly as the
// builder warps of mvt_kernel build it per unit.  Rows past M convert zeros.
template <int QT>
__global__ void __launch_bounds__(64) mvt_prep_kernel(const float* __restrict__ x, int M, int nsb, uint8_t* img) {
    __shared__ __align__(16) float xs[16 * 256];
    const int sb = blockIdx.x, tid = threadIdx.x;
    pdl_launch_dependents();
    pdl_wait();  // x is the previous kernel's output
    const int64_t K = static_cast<int64_t>(nsb) * kQK;
    // all sixteen loads of a thread in flight at once, then the stores; x is
    // read through L2 (a non-coherent load counts as invariant and may be
    // moved above the wait for the kernel that writes x)
    float4 v[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const int i = tid + 64 * k, m = i >> 6;
        v[k] = m < M ? __ldcg(reinterpret_cast<const float4*>(x + m * K + static_cast<int64_t>(sb) * kQK) + (i & 63))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) reinterpret_cast<float4*>(xs)[tid + 64 * k] = v[k];
    __syncthreads();
    const int lane = tid & 31, m = 8 * (tid >> 5) + (lane >> 2), q = lane & 3;
    uint8_t* base = img + static_cast<size_t>(sb) * kBImg;
    float* xr = reinterpret_cast<float*>(base + kSlabBytes);
    float xs8[8];
    const float e2 = build_row_quarter<QT>(xs + m * 256, q, base, (m >> 2) * 128 + (2 * m & 7) * 16, xs8);
    if (q == 0) {
        xr[8 * 16 + m] = e2;
        if constexpr (QT == MUSER_Q4_K) {
            *reinterpret_cast<float4*>(xr + 8 * m) = make_float4(xs8[0], xs8[1], xs8[2], xs8[3]);
            *reinterpret_cast<float4*>(xr + 8 * m + 4) = make_float4(xs8[4], xs8[5], xs8[6], xs8[7]);
        }
    }
}

// The dual-eps tail of row m = blockIdx.x (dual_tail_row_reg) that also
// writes row m of every super-block's B image from the row's x, held in
// shared memory: quad (sb, q) of the first four warps converts quarter q of
// block sb as the prep kernel does.  Rows of the image past M stay as the
// zero-filled scratch has them, which the matvec reads as rows of zeros.
// 512 threads, so that a thread may hold the conversion's 64 inputs in
// registers (with 1,024 it spilled).
constexpr int kTailImageThreads = 512;
template <int QT, int V>
__global__ void __launch_bounds__(kTailImageThreads) mvt_tail_image_kernel(float* resid, const float* src, float* out,
                                                              const float* w1, const float* w2, int n, float eps1,
                                                              float eps2, uint8_t* img) {
    extern __shared__ __align__(16) float xrow[];  // n floats
    __shared__ float red[33];
    const int m = blockIdx.x, tid = threadIdx.x, n4 = n >> 2, nsb = n / kQK;
    const int64_t off = static_cast<int64_t>(m) * n;
    float4 xv[V];
    dual_tail_row_reg<V>(resid + off, src + off, out + off, w1, w2, n, eps1, eps2, red, xv);
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = tid + u * kTailImageThreads;
        if (i < n4) reinterpret_cast<float4*>(xrow)[i] = xv[u];
    }
    __syncthreads();
    if (tid < 128) {
        const uint32_t rowoff = static_cast<uint32_t>((m >> 2) * 128 + (2 * m & 7) * 16);
        for (int sb0 = 0; sb0 < nsb; sb0 += 32) {
            const int sbq = sb0 + (tid >> 2), q = tid & 3;
            const bool valid = sbq < nsb;
            const int sb = valid ? sbq : nsb - 1;  // past the row: shuffles only
            uint8_t* base = img + static_cast<size_t>(sb) * kBImg;
            float xs8[8];
            const float e2 = build_row_quarter<QT>(xrow + sb * kQK, q, base, rowoff, xs8, valid);
            if (valid && q == 0) {
                float* xr = reinterpret_cast<float*>(base + kSlabBytes);
                xr[8 * 16 + m] = e2;
                if constexpr (QT == MUSER_Q4_K) {
                    *reinterpret_cast<float4*>(xr + 8 * m) = make_float4(xs8[0], xs8[1], xs8[2], xs8[3]);
                    *reinterpret_cast<float4*>(xr + 8 * m + 4) = make_float4(xs8[4], xs8[5], xs8[6], xs8[7]);
                }
            }
        }
    }
}

// Zeroes the B image after the matvec has read it (the caller's scratch is
// left zero-filled).
__global__ void __launch_bounds__(256) mvt_clear_kernel(uint8_t* img, int nsb) {
    pdl_launch_dependents();
    pdl_wait();  // the matvec that reads the image is complete
    uint4* p = reinterpret_cast<uint4*>(img + static_cast<size_t>(blockIdx.x) * kBImg);
    for (int i = threadIdx.x; i < static_cast<int>(kBImg / 16); i += blockDim.x) p[i] = make_uint4(0u, 0u, 0u, 0u);
}

}  // namespace

// ------------------------------------------------------------------ host
namespace {

constexpr int kMaxGrid = 256;  // bound on the grid, so scratch sizes need no device query
// The B image costs two small launches; it pays when every CTA has enough
// units to amortise them (measured: the 19968 x 6656 gate/up, 53 units per
// CTA, and the 6656 x 19968 down projection, 27; not the 1-15 MB attention
// projections, 1-6).
constexpr int64_t kImgMinUnitsPerCta = 8;

struct MvtGeo {
    int P = 1, ntiles = 0, grid = 0, maxparts = 1, ns = 0, tiles_per_cta = 0;
    uint32_t x_off = 0, b_off = 0, stage_off = 0, xch_off = 0, smem = 0;
};

int gcd_int(int64_t a, int64_t b) {
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return static_cast<int>(a);
}

int tile_count(int nmat, int64_t rows, int P) {
    return nmat == 2 ? static_cast<int>((rows + 63) / 64) : static_cast<int>(P * ((rows + 128 * P - 1) / (128 * P)));
}

// Geometry of one launch; false if the shape does not fit this kernel.
// img: several rows of x with the B image built once per call (the builders
// need no ring of x).
bool mvt_geometry(int qtype, int nmat, int64_t rows, int64_t cols, int M, MvtGeo& g, bool whole_tiles,
                  bool img = false) {
    if (qtype != MUSER_Q4_K && qtype != MUSER_Q6_K) return false;
    if (nmat == 2 && qtype != MUSER_Q4_K) return false;
    if (cols % kQK != 0 || rows < 1 || M < 1 || M > 16) return false;
    const bool multi = M > 1;
    const int64_t nsb = cols / kQK;
    const int blk = qtype == MUSER_Q4_K ? kQ4KBytes : kQ6KBytes;
    const int64_t rowbytes = nsb * blk;
    if ((rows * rowbytes) % 16 != 0) return false;  // 16-byte copies never pass the matrix end
    g.P = nmat == 2 ? 1 : 16 / gcd_int(rowbytes, 16);
    if (rows % g.P != 0) return false;  // the class view of the matrix must be exact
    g.ntiles = tile_count(nmat, rows, g.P);
    const int sms = std::min(sm_count(), kMaxGrid);
    if (sms <= 0) return false;
    const int64_t U = static_cast<int64_t>(g.ntiles) * nsb;
    if (whole_tiles) {
        g.tiles_per_cta = (g.ntiles + sms - 1) / sms;
        g.grid = (g.ntiles + g.tiles_per_cta - 1) / g.tiles_per_cta;
        g.maxparts = 1;
    } else {
        g.grid = static_cast<int>(std::min<int64_t>(sms, U));
        auto cta_of_h = [&](int64_t u) { return static_cast<int>(((u + 1) * g.grid - 1) / U); };
        g.maxparts = 1;
        for (int t = 0; t < g.ntiles; ++t)
            g.maxparts = std::max(g.maxparts, cta_of_h(static_cast<int64_t>(t + 1) * nsb - 1) -
                                                  cta_of_h(static_cast<int64_t>(t) * nsb) + 1);
    }
    // barriers, TMEM address, flags (0..511), red (512..767), scale ring
    // (1280 + kND * 128 * 16), tile exchange, x scales and sums, B, stages
    const int MB = multi ? 16 : 1;
    g.xch_off = 1280 + kND * 128 * 16;
    g.x_off = g.xch_off + MB * 128 * 4;
    const uint32_t xbytes = multi ? static_cast<uint32_t>(kND * (MB * 8 + MB) * 4)
                                  : static_cast<uint32_t>(((nsb + 3) & ~3) * 4 + (qtype == MUSER_Q4_K ? nsb * 8 * 4 : 0));
    g.b_off = (g.x_off + xbytes + 127) / 128 * 128;
    // several rows: kNB B slabs, then two builder warps' kNB slots of 8 rows of x
    const uint32_t bbytes = multi ? static_cast<uint32_t>(kNB * 16384 + (img ? 0 : 2 * kNB * 8192))
                                  : static_cast<uint32_t>(nsb * 1024 + 512);
    g.stage_off = (g.b_off + bbytes + 1023) / 1024 * 1024;
    const uint32_t stage = 128u * (qtype == MUSER_Q4_K ? 144u : 240u);
    const int64_t budget = max_smem_optin();
    if (budget <= g.stage_off) return false;
    g.ns = static_cast<int>(std::min<int64_t>(kMaxStages, (budget - g.stage_off) / stage));
    if (g.ns < 3) return false;
    g.smem = g.stage_off + static_cast<uint32_t>(g.ns) * stage;
    return true;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A 2-D byte-array view of a matrix: `outer` rows of `inner` bytes, `stride`
// bytes apart, copied in boxes of box_x bytes x box_y rows.
int encode_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t stride, uint32_t box_x,
               uint32_t box_y) {
    auto fn = encode_fn();
    if (fn == nullptr) return set_error(MUSER_ERR_CUDA, "mvt: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MUSER_ERR_CUDA, "mvt: cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return MUSER_OK;
}

// A row-major binary32 matrix of `outer` rows of `inner` elements.
int encode_map_f32(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t stride_bytes,
                   uint32_t box_x, uint32_t box_y) {
    auto fn = encode_fn();
    if (fn == nullptr) return set_error(MUSER_ERR_CUDA, "mvt: cuTensorMapEncodeTiled is not available");
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {stride_bytes};
    const cuuint32_t box[2] = {box_x, box_y};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return set_error(MUSER_ERR_CUDA, "mvt: cuTensorMapEncodeTiled (x) failed (%d)", static_cast<int>(r));
    return MUSER_OK;
}

// A small kernel launched with programmatic stream serialization.
template <typename... KArgs, typename... Args>
int launch_pdl(void (*kern)(KArgs...), int grid, int threads, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    if (e != cudaSuccess) return cuda_fail(e, "mvt: cudaLaunchKernelEx (B image)");
    return check_launch("mvt B image");
}

template <int QT, int EPI, bool MULTI>
int launch_mvt_t(MvtArgs a, const MvtGeo& g, cudaStream_t stream) {
    constexpr int NMAT = (EPI == kEpiSiluMul) ? 2 : 1;
    const uint64_t rowbytes = static_cast<uint64_t>(a.nsb) * (QT == MUSER_Q4_K ? kQ4KBytes : kQ6KBytes);
    const uint64_t rows = static_cast<uint64_t>(a.rows);
    CUtensorMap m0, m1, m2, m3;
    if constexpr (QT == MUSER_Q4_K) {
        const uint32_t box_y = NMAT == 2 ? 64u : 128u;
        if (a.nseg > 0) {
            CUtensorMap* ms[kMvtMaxSeg] = {&m0, &m1, &m2, &m3};
            for (int i = 0; i < kMvtMaxSeg; ++i) {
                const int j = i < a.nseg ? i : 0;
                MUSER_TRY(encode_map(ms[i], a.seg_W[j], rowbytes, static_cast<uint64_t>(a.seg_rows[j]), rowbytes,
                                     kQ4KBytes, 128u));
            }
        } else {
            MUSER_TRY(encode_map(&m0, a.W[0], rowbytes, rows, rowbytes, kQ4KBytes, box_y));
            MUSER_TRY(encode_map(&m1, a.W[NMAT - 1], rowbytes, rows, rowbytes, kQ4KBytes, box_y));
            m2 = m3 = m0;
        }
    } else {
        const uint64_t P = static_cast<uint64_t>(g.P);
        MUSER_TRY(encode_map(&m0, a.W[0], P * rowbytes, rows / P, P * rowbytes, 240u, 128u));
        m1 = m2 = m3 = m0;
    }
    CUtensorMap mx = m0;
    if constexpr (MULTI) {
        // x as M rows of K floats, copied in boxes of one block x eight rows
        const uint64_t K = static_cast<uint64_t>(a.nsb) * kQK;
        MUSER_TRY(encode_map_f32(&mx, a.x, K, static_cast<uint64_t>(a.M), K * 4, 256u, 8u));
    }
    auto kern = mvt_kernel<QT, EPI, MULTI>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(g.smem));
    if (e != cudaSuccess) return cuda_fail(e, "mvt: cudaFuncSetAttribute");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(g.grid);
    cfg.blockDim = dim3(mvt_threads(MULTI));
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a, m0, m1, mx, m2, m3);
    if (e != cudaSuccess) return cuda_fail(e, "mvt: cudaLaunchKernelEx");
    return check_launch("mvt_kernel");
}

}  // namespace

bool mvt_supported(int qtype, int nmat, int64_t rows, int64_t cols, int M) {
    MvtGeo g;
    return mvt_geometry(qtype, nmat, rows, cols, M, g, true);
}

int64_t mvt_group_rows(int n, const int64_t* rows) {
    int64_t t = 0;
    for (int i = 0; i < n; ++i) t += (rows[i] + 127) / 128;
    return t * 128;
}

// Launches of one launch_mvt call with scratch of mvt_scratch_bytes(): three
// with the B image (built before, cleared after), else one; 0 if unsupported.
int mvt_launches(int qtype, int nmat, int64_t rows, int64_t cols, int M) {
    MvtGeo g;
    if (!mvt_geometry(qtype, nmat, rows, cols, M, g, false)) return 0;
    return M > 1 && static_cast<int64_t>(g.ntiles) * (cols / kQK) >= kImgMinUnitsPerCta * g.grid ? 3 : 1;
}

// Scratch of the even split: per-tile tickets and the tail counter, then
// ntiles + grid - 1 partial slots of 128 floats per row of x.  Depends only
// on the tile count and the grid bound, not on the device.
size_t mvt_scratch_bytes(int qtype, int nmat, int64_t rows, int64_t cols, int M) {
    const size_t split = mvt_split_scratch_bytes(qtype, nmat, rows, cols, M);
    return split && M > 1 ? split + static_cast<size_t>(cols / kQK) * kBImg : split;
}

size_t mvt_split_scratch_bytes(int qtype, int nmat, int64_t rows, int64_t cols, int M) {
    if (qtype != MUSER_Q4_K && qtype != MUSER_Q6_K) return 0;
    if (cols % kQK != 0 || rows < 1 || M < 1 || M > 16) return 0;
    const int64_t rowbytes = (cols / kQK) * (qtype == MUSER_Q4_K ? kQ4KBytes : kQ6KBytes);
    const int P = nmat == 2 ? 1 : 16 / gcd_int(rowbytes, 16);
    const int64_t ntiles = tile_count(nmat, rows, P);
    const size_t ticks = (static_cast<size_t>(ntiles) + 1) * sizeof(unsigned);
    const int MB = M > 1 ? 16 : 1;
    return (ticks + 255) / 256 * 256 + static_cast<size_t>(ntiles + kMaxGrid) * MB * 128 * sizeof(float);
}

// Where the B image sits in the even split's scratch: after the tile
// tickets and the partial slots.
uint8_t* image_of(void* scratch, int ntiles) {
    const size_t ticks = (static_cast<size_t>(ntiles) + 1) * sizeof(unsigned);
    return static_cast<uint8_t*>(scratch) + (ticks + 255) / 256 * 256 +
           static_cast<size_t>(ntiles + kMaxGrid) * 16 * 128 * sizeof(float);
}

// scratch == nullptr: whole tiles per CTA (no partial sums).  Otherwise the
// even split, with `scratch` of mvt_scratch_bytes(), zero-filled, left zeroed.
// The tail epilogue is for one row of x and needs scratch.
int launch_mvt(int qtype, int epi, MvtArgs a, void* scratch, size_t scratch_bytes, cudaStream_t s) {
    const int nmat = epi == kEpiSiluMul ? 2 : 1;
    const int64_t cols = static_cast<int64_t>(a.nsb) * kQK;
    MvtGeo g;
    if (!mvt_geometry(qtype, nmat, a.rows, cols, a.M, g, scratch == nullptr))
        return set_error(MUSER_ERR_UNSUPPORTED, "mvt: shape not supported");
    const bool img = scratch != nullptr && a.M > 1 &&
                     scratch_bytes >= mvt_scratch_bytes(qtype, nmat, a.rows, cols, a.M) &&
                     static_cast<int64_t>(g.ntiles) * a.nsb >= kImgMinUnitsPerCta * g.grid;
    if (img && !mvt_geometry(qtype, nmat, a.rows, cols, a.M, g, false, true))
        return set_error(MUSER_ERR_UNSUPPORTED, "mvt: shape not supported");
    if (epi == kEpiTail && (scratch == nullptr || a.M != 1))
        return set_error(MUSER_ERR_UNSUPPORTED, "mvt: the tail epilogue needs scratch and one row of x");
    a.ntiles = g.ntiles;
    a.P = g.P;
    a.maxparts = g.maxparts;
    a.ns = g.ns;
    a.tiles_per_cta = g.tiles_per_cta;
    a.x_off = g.x_off;
    a.b_off = g.b_off;
    a.stage_off = g.stage_off;
    a.xch_off = g.xch_off;
    if (a.nseg > 0) {
        if (qtype != MUSER_Q4_K || epi != kEpiStore || a.M < 2 || a.nseg > kMvtMaxSeg)
            return set_error(MUSER_ERR_UNSUPPORTED, "mvt: a group needs Q4_K, the store epilogue and 2..16 rows of x");
        a.seg_t0[0] = 0;
        for (int i = 0; i < a.nseg; ++i) a.seg_t0[i + 1] = a.seg_t0[i] + static_cast<int>((a.seg_rows[i] + 127) / 128);
        if (static_cast<int64_t>(a.seg_t0[a.nseg]) * 128 != a.rows)
            return set_error(MUSER_ERR_INVALID_ARG, "mvt: group rows must be the tile-aligned total");
    }
    a.bimg = nullptr;
    if (scratch != nullptr) {
        const size_t ticks = (static_cast<size_t>(g.ntiles) + 1) * sizeof(unsigned);
        a.tick = static_cast<unsigned*>(scratch);
        a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + (ticks + 255) / 256 * 256);
        if (img) a.bimg = image_of(scratch, g.ntiles);
    }
    if (a.image_ready && a.bimg == nullptr)
        return set_error(MUSER_ERR_INVALID_ARG, "mvt: a prebuilt B image for a launch that reads none");
    if (a.status == nullptr) a.status = device_status_word();
    if (a.status == nullptr) return set_error(MUSER_ERR_CUDA, "mvt: no device status word");
    const bool multi = a.M > 1;
    if (a.bimg != nullptr) {
        // the B image: built before the matvec, zeroed after it
        uint8_t* img = const_cast<uint8_t*>(a.bimg);
        if (!a.image_ready)
            MUSER_TRY(qtype == MUSER_Q4_K ? launch_pdl(mvt_prep_kernel<MUSER_Q4_K>, a.nsb, 64, s, a.x, a.M, a.nsb, img)
                                          : launch_pdl(mvt_prep_kernel<MUSER_Q6_K>, a.nsb, 64, s, a.x, a.M, a.nsb, img));
        int r = MUSER_ERR_UNSUPPORTED;
        if (qtype == MUSER_Q4_K && epi == kEpiSiluMul) r = launch_mvt_t<MUSER_Q4_K, kEpiSiluMul, true>(a, g, s);
        else if (qtype == MUSER_Q4_K && epi == kEpiStore) r = launch_mvt_t<MUSER_Q4_K, kEpiStore, true>(a, g, s);
        else if (qtype == MUSER_Q6_K && epi == kEpiStore) r = launch_mvt_t<MUSER_Q6_K, kEpiStore, true>(a, g, s);
        else return set_error(MUSER_ERR_UNSUPPORTED, "mvt: no kernel for qtype %d epilogue %d", qtype, epi);
        MUSER_TRY(r);
        return launch_pdl(mvt_clear_kernel, a.nsb, 256, s, img, a.nsb);
    }
    if (qtype == MUSER_Q4_K) {
        if (epi == kEpiSiluMul)
            return multi ? launch_mvt_t<MUSER_Q4_K, kEpiSiluMul, true>(a, g, s) : launch_mvt_t<MUSER_Q4_K, kEpiSiluMul, false>(a, g, s);
        if (epi == kEpiStore)
            return multi ? launch_mvt_t<MUSER_Q4_K, kEpiStore, true>(a, g, s) : launch_mvt_t<MUSER_Q4_K, kEpiStore, false>(a, g, s);
        if (epi == kEpiTail) return launch_mvt_t<MUSER_Q4_K, kEpiTail, false>(a, g, s);
    } else {
        if (epi == kEpiStore)
            return multi ? launch_mvt_t<MUSER_Q6_K, kEpiStore, true>(a, g, s) : launch_mvt_t<MUSER_Q6_K, kEpiStore, false>(a, g, s);
        if (epi == kEpiTail) return launch_mvt_t<MUSER_Q6_K, kEpiTail, false>(a, g, s);
    }
    return set_error(MUSER_ERR_UNSUPPORTED, "mvt: no kernel for qtype %d epilogue %d", qtype, epi);
}

bool mvt_tail_image_fits(int qtype, int nmat, int64_t rows, int64_t cols, int M, size_t scratch_bytes) {
    MvtGeo g;
    return M >= 2 && M <= 16 && cols % kQK == 0 && cols <= 8192 && (qtype == MUSER_Q4_K || qtype == MUSER_Q6_K) &&
           mvt_supported(qtype, nmat, rows, cols, M) && mvt_geometry(qtype, nmat, rows, cols, M, g, false) &&
           scratch_bytes >= mvt_scratch_bytes(qtype, nmat, rows, cols, M) &&
           static_cast<int64_t>(g.ntiles) * (cols / kQK) >= kImgMinUnitsPerCta * g.grid &&
           mvt_geometry(qtype, nmat, rows, cols, M, g, false, true);
}

int launch_mvt_tail_image(int qtype, int nmat, int64_t rows, int64_t cols, int M, float* resid, const float* src,
                          float* out, const float* w1, const float* w2, float eps1, float eps2, void* scratch,
                          size_t scratch_bytes, cudaStream_t s) {
    if (scratch == nullptr || !mvt_tail_image_fits(qtype, nmat, rows, cols, M, scratch_bytes))
        return MUSER_ERR_UNSUPPORTED;  // no image for this launch: the caller runs the plain tail
    MvtGeo g;
    (void)mvt_geometry(qtype, nmat, rows, cols, M, g, false, true);
    uint8_t* img = image_of(scratch, g.ntiles);
    const int n = static_cast<int>(cols), v = (n / 4 + kTailImageThreads - 1) / kTailImageThreads;
    const size_t smem = sizeof(float) * static_cast<size_t>(n);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(kTailImageThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    auto kern = [&](auto k) { return cudaLaunchKernelEx(&cfg, k, resid, src, out, w1, w2, n, eps1, eps2, img); };
    if (qtype == MUSER_Q4_K)
        e = v <= 2 ? kern(mvt_tail_image_kernel<MUSER_Q4_K, 2>) : kern(mvt_tail_image_kernel<MUSER_Q4_K, 4>);
    else
        e = v <= 2 ? kern(mvt_tail_image_kernel<MUSER_Q6_K, 2>) : kern(mvt_tail_image_kernel<MUSER_Q6_K, 4>);
    if (e != cudaSuccess) return cuda_fail(e, "mvt_tail_image: cudaLaunchKernelEx");
    return check_launch("mvt_tail_image");
}

}  // namespace muser
