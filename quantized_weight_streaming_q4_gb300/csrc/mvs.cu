// mvs.cu -- the one-token decode-FFN stack as one persistent kernel: every
// layer's gate/up/SiLU (Muser book Ch 10 §10.3 (d)), down projection (Ch 19
// §19.5) and dual-eps tail (Ch 19 §19.4) for one row of x, in the order of
// the book's layer loop (Ch 10 §10.3-§10.4), in a single cooperative launch
// with one block per SM.
//
// Why one launch: the weight stream is the whole cost of a decode token
// (Ch 19 §19.6).  With one kernel per projection the stream drains at every
// kernel boundary: the next kernel's blocks start only as the previous
// kernel's blocks leave their SMs, wait for the whole previous grid, load and
// convert their input, and only then run at the stream's rate.  Here each
// block's copy warp streams the weights of every phase back to back through
// one ring of stage buffers; it never waits for another block.  Only the
// consumer warps wait, at a grid barrier, for the activations the previous
// phase produced; meanwhile the ring keeps filling with the next phase's
// weights.
//
// Phases per layer l: GU(l) streams W_gate and W_up (Q4_K, two matrices,
// SiLU epilogue into `mid`); D(l) streams W_down (Q6_K, into `proj`).
// Consumer prologues:
//  * GU(0): x = rms_norm(residual) (the entry norm); GU(l > 0): the tail of
//    layer l - 1, computed by every block from `proj` and the residual, as in
//    the one-token kernel's fused prologue.  The updated residual goes to the
//    other buffer of a two-buffer relay, each block writing its share, so no
//    block overwrites a row another block still reads.
//  * D(l): x = mid.  The gate/up reducers store mid slice-major: input k of
//    the down-phase slice owned by consumer thread t sits at float4
//    (k / 4) * TGd + t, so each consumer thread loads its 64 inputs with 16
//    coalesced 16-byte loads and converts them to the 24-bit digits of the
//    one-token kernel's Q6_K dot in registers.  Nothing goes through shared
//    memory, so the whole ring stays free for weights.
// After the last layer every block computes the last tail and writes its
// share of the residual and of `out`.
//
// Warp roles (480 threads): 13 consumer warps (gate/up uses all of them in
// four row groups; down uses 12: one row group of 320 threads split by block
// parity, and two warps that mirror the first two warps' slices and take half
// their rows, so the four schedulers carry equal work); one copy warp; one
// reducer warp.  (With 480 threads a thread may hold 136
// registers: the two phases' slices and dot products fit without spills.)  Barriers: full/empty
// per stage buffer, pfull/reduced per partial slot, as in the one-token
// kernel, with ring positions counted across phases.  Every wait is bounded
// in time; a block that gives up sets the device status word and a global
// abort flag, and every other wait then returns at once.
#include <algorithm>
#include <cstdio>

#include "common.cuh"
#include "kernels.cuh"
#include "mv1_core.cuh"

namespace muser {
namespace {

constexpr int kCW = 13;             // consumer warps
constexpr int kTmaWarp = kCW;       // copy warp
constexpr int kRedWarp = kCW + 1;   // reducer warp
constexpr int kThreads = (kCW + 2) * 32;
constexpr int kHead = 1024;         // barriers, reduction scratch, flags
constexpr uint64_t kWaitNs = 1000000000ull;      // 1 s per barrier wait
constexpr uint64_t kGridWaitNs = 2000000000ull;  // 2 s per grid barrier

// sync words (zeroed by the launcher before every launch)
constexpr int kSyncCount = 0;   // grid barrier arrivals
constexpr int kSyncAbort = 1;   // set by a block that gave up a wait
constexpr int kSyncWords = 64;  // 256 bytes

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_volatile(const unsigned* p) {
    return *reinterpret_cast<const volatile unsigned*>(p);
}

// Gives up everything this block still waits for: the status bit for the
// host, the global flag for the other blocks, the local flag for this one.
__device__ __forceinline__ void give_up(const MvsArgs& p, volatile int* abort_s) {
    atomicOr(p.status, kDevStatusWaitTimeout);
    atomicExch(p.sync + kSyncAbort, 1u);
    *abort_s = 1;
}

// mbarrier wait bounded in time that also returns (false) once the block
// has given up.
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity, const MvsArgs& p, volatile int* abort_s) {
    if (*abort_s) return false;
    if (mbar_try_wait(bar, parity, 1000000u)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity, 200000u)) return true;
        if (*abort_s) return false;
        if (global_ns() - t0 > kWaitNs) {
            give_up(p, abort_s);
            return false;
        }
    }
}

// One thread: wait until the grid barrier count reaches `target` (every
// block has arrived that often), bounded in time; watches the abort flags.
__device__ __forceinline__ bool grid_wait(const MvsArgs& p, unsigned target, volatile int* abort_s) {
    if (*abort_s) return false;
    const uint64_t t0 = global_ns();
    for (int it = 0;; ++it) {
        if (ld_acquire(p.sync + kSyncCount) >= target) return true;
        if ((it & 31) == 31) {
            if (*abort_s) return false;
            if (ld_volatile(p.sync + kSyncAbort) != 0u) {
                *abort_s = 1;
                return false;
            }
            if (global_ns() - t0 > kGridWaitNs) {
                give_up(p, abort_s);
                return false;
            }
        }
    }
}

// The consumer warps wait for the grid barrier: thread 0 polls, the others
// wait on named barrier 1.  Returns false if the block gave up; the value is
// the same in every consumer thread (a broadcast), so it may decide whether
// the block runs code with block-wide barriers.
__device__ __forceinline__ bool consumers_grid_wait(const MvsArgs& p, unsigned target, volatile int* abort_s,
                                                    int* flag) {
    if (threadIdx.x == 0) *flag = grid_wait(p, target, abort_s) ? 1 : 0;
    named_barrier_sync(1, kCW * 32);
    const bool ok = *flag != 0;
    named_barrier_sync(1, kCW * 32);
    return ok;
}

// Residual buffer t of the relay: R(t) holds the residual after t tails;
// R(nl) must be the caller's buffer.
__device__ __forceinline__ float* relay(const MvsArgs& p, int t) {
    return ((p.nl - t) % 2 == 0) ? p.resid : p.resid_ws;
}

// ------------------------------------------------------ down-phase input
// Where the gate/up reducer stores input `row` of mid (slice-major, see the
// file comment): the Q6_K slice (b, c = 2h + j) holding it is owned by
// down-phase consumer thread t = (b odd ? HPd : 0) + 4 (b / 2) + c, as
// slice_of lays the threads out, and the input is element k = 16g + l of
// that slice (row = 256b + 128h + 32g + 16j + l).
__device__ __forceinline__ int64_t xperm_index(int64_t row, int HPd, int TGd) {
    const int64_t b = row >> 8;
    const int w = static_cast<int>(row & 255);
    const int h = w >> 7, g = (w >> 5) & 3, j = (w >> 4) & 1, l = w & 15;
    const int64_t t = ((b & 1) ? HPd : 0) + 4 * (b >> 1) + 2 * h + j;
    const int k = 16 * g + l;
    return ((k >> 2) * static_cast<int64_t>(TGd) + t) * 4 + (k & 3);
}

// The Q6_K slice of consumer thread t, loaded from the slice-major mid and
// converted in registers as the one-token kernel converts a slot
// (load_slice_q6): one power of two for the slice, digit words rotated by two
// bytes when the thread's blocks sit two bytes past a word (odd b).  mid was
// written by other blocks in this launch: loads bypass L1.
__device__ __forceinline__ void load_slice_q6_mem(SliceQ6& s, const float4* xperm, int t, int TGd, bool rot) {
    float v[4][16];
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float4 f = __ldcg(xperm + (4 * g + q) * TGd + t);
            v[g][4 * q + 0] = f.x;
            v[g][4 * q + 1] = f.y;
            v[g][4 * q + 2] = f.z;
            v[g][4 * q + 3] = f.w;
        }
    float m = 0.0f;
#pragma unroll
    for (int g = 0; g < 4; ++g)
#pragma unroll
        for (int l = 0; l < 16; ++l) m = fmaxf(m, fabsf(v[g][l]));
    const int e = slice_exponent(m);
    const float p2e = pow2f(e);
    s.inv = pow2f(-e);
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

// --------------------------------------------------------- the row tails
// The two norm weights of a tail, this thread's share (float4 j = tid +
// 416u, zeros past the row).  They do not depend on other blocks, so they are
// loaded before the grid barrier.  Every element is set on every path: an
// array set on some paths only would stay live across the layer loop.
__device__ __forceinline__ void load_tail_weights(const MvsArgs& p, const float* w1, const float* w2, float4* av,
                                                  float4* bv) {
    const int tid = threadIdx.x, n4 = p.hidden >> 2, nthr = kCW * 32;
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int j = tid + u * nthr;
        const bool in = j < n4;
        av[u] = __ldg(reinterpret_cast<const float4*>(w1) + (in ? j : 0));
        bv[u] = __ldg(reinterpret_cast<const float4*>(w2) + (in ? j : 0));
        if (!in) av[u] = bv[u] = z;
    }
}

// The tail of Ch 19 §19.4 for one row of `n` inputs, computed by the
// consumer warps of a block from proj and the residual R(t): Σp², h = r +
// w1·p·inv1, Σh², x = w2·h·inv2, each thread holding at most 4 float4 of each
// vector (float4 j = tid + 416u; av, bv from load_tail_weights).  The block
// writes its share of h to R(t + 1).  Returns 1/rms of h in inv2; h is left
// in rv.
__device__ __forceinline__ void block_tail(const MvsArgs& p, int t, const float4* av, float4* rv, float& inv2,
                                           float* red) {
    const int tid = threadIdx.x, n4 = p.hidden >> 2, nthr = kCW * 32;
    const float n = static_cast<float>(p.hidden);
    const float4* p4 = reinterpret_cast<const float4*>(p.proj);
    const float4* r4 = reinterpret_cast<const float4*>(relay(p, t));
    float4 pv[4];
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int j = tid + u * nthr;
        const bool in = j < n4;
        pv[u] = __ldcg(p4 + (in ? j : 0));
        rv[u] = __ldcg(r4 + (in ? j : 0));
        if (!in) pv[u] = rv[u] = z;
    }
    float ss = 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        ss = fmaf(pv[u].x, pv[u].x, ss);
        ss = fmaf(pv[u].y, pv[u].y, ss);
        ss = fmaf(pv[u].z, pv[u].z, ss);
        ss = fmaf(pv[u].w, pv[u].w, ss);
    }
    ss = warps_sum(ss, red, kCW);
    const float inv1 = 1.0f / sqrtf(ss / n + p.eps_post);
    float sh = 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float4 hh;  // zero past the row (all four vectors are zero there)
        hh.x = fmaf(pv[u].x * inv1, av[u].x, rv[u].x);
        hh.y = fmaf(pv[u].y * inv1, av[u].y, rv[u].y);
        hh.z = fmaf(pv[u].z * inv1, av[u].z, rv[u].z);
        hh.w = fmaf(pv[u].w * inv1, av[u].w, rv[u].w);
        sh = fmaf(hh.x, hh.x, sh);
        sh = fmaf(hh.y, hh.y, sh);
        sh = fmaf(hh.z, hh.z, sh);
        sh = fmaf(hh.w, hh.w, sh);
        rv[u] = hh;
    }
    sh = warps_sum(sh, red, kCW);
    inv2 = 1.0f / sqrtf(sh / n + p.eps_norm);
    // this block's share of the updated residual
    const int j0 = static_cast<int>(static_cast<int64_t>(n4) * blockIdx.x / gridDim.x);
    const int j1 = static_cast<int>(static_cast<int64_t>(n4) * (blockIdx.x + 1) / gridDim.x);
    float4* h4 = reinterpret_cast<float4*>(relay(p, t + 1));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int j = tid + u * nthr;
        if (j >= j0 && j < j1) h4[j] = rv[u];
    }
}

// ------------------------------------------------------------ consumers
// Shared-memory layout (offsets from the dynamic base): barriers full[8],
// empty[8], pfull[16], reduced[16] at 0; red (64 floats) at 512; the local
// abort flag at 768 and a broadcast flag at 776; partial slots at part_off
// (the gate/up input slots overlay them); the ring of stage buffers at
// ring_off.
struct Smem {
    uint64_t *full, *empty, *pfull, *reduced;
    float* red;
    volatile int* abort_s;
    int* flag;
    float* part;
    uint8_t* xslots;
    uint8_t* ring;
};
__device__ __forceinline__ Smem smem_of(uint8_t* smem, const MvsArgs& p) {
    Smem m;
    m.full = reinterpret_cast<uint64_t*>(smem);
    m.empty = m.full + 8;
    m.pfull = m.full + 16;
    m.reduced = m.full + 32;
    m.red = reinterpret_cast<float*>(smem + 512);
    m.abort_s = reinterpret_cast<volatile int*>(smem + 768);
    m.flag = reinterpret_cast<int*>(smem + 776);
    m.part = reinterpret_cast<float*>(smem + p.part_off);
    m.xslots = smem + p.part_off;
    m.ring = smem + p.ring_off;
    return m;
}

// The gate/up input of layer l (consumer warps): the entry norm (layer 0)
// or the previous layer's tail, written into the input slots and converted
// there, a quarter slot per thread.  Runs once per layer.  Returns false if
// the block gave up a wait.
template <int GQ>
__device__ __forceinline__ bool gu_prologue(const MvsArgs& p, int l, bool ok, uint8_t* smem_base) {
    const Smem m = smem_of(smem_base, p);
    const int tid = threadIdx.x;
    const int nbc_g = (p.hidden / kQK) * 4, TGg = nbc_g;
    float4 av[4], bv[4];  // the previous layer's norm weights (or the entry norm's, in bv)
    if (l > 0) load_tail_weights(p, p.layer[l - 1].w1, p.layer[l - 1].w2, av, bv);
    else load_tail_weights(p, p.w_in, p.w_in, av, bv);
    if (l > 0) ok = consumers_grid_wait(p, gridDim.x * static_cast<unsigned>(2 * l), m.abort_s, m.flag) && ok;
    const int n4 = p.hidden >> 2, nthr = kCW * 32;
    if (l == 0) {
        // the entry norm; the relay starts in the workspace when the layer
        // count is odd, and then this block copies its share of the row there
        const float4* r4 = reinterpret_cast<const float4*>(p.resid);
        float4 rv[4];
        float ss = 0.0f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = tid + u * nthr;
            rv[u] = __ldcg(r4 + (j < n4 ? j : 0));
            if (j >= n4) rv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            ss = fmaf(rv[u].x, rv[u].x, ss);
            ss = fmaf(rv[u].y, rv[u].y, ss);
            ss = fmaf(rv[u].z, rv[u].z, ss);
            ss = fmaf(rv[u].w, rv[u].w, ss);
        }
        ss = warps_sum(ss, m.red, kCW);
        const float inv = 1.0f / sqrtf(ss / static_cast<float>(p.hidden) + p.eps_norm);
        const int j0 = static_cast<int>(static_cast<int64_t>(n4) * blockIdx.x / gridDim.x);
        const int j1 = static_cast<int>(static_cast<int64_t>(n4) * (blockIdx.x + 1) / gridDim.x);
        float* R0 = relay(p, 0);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = tid + u * nthr;
            if (j < n4) {
                const float4 w = bv[u];
                sts_float4(m.xslots + xslot_offset(j, true, false, 0),
                           make_float4((rv[u].x * inv) * w.x, (rv[u].y * inv) * w.y, (rv[u].z * inv) * w.z,
                                       (rv[u].w * inv) * w.w));
                if (R0 != p.resid && j >= j0 && j < j1) reinterpret_cast<float4*>(R0)[j] = rv[u];
            }
        }
    } else {
        float4 rv[4];
        float inv2;
        block_tail(p, l - 1, av, rv, inv2, m.red);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = tid + u * nthr;
            if (j < n4)
                sts_float4(m.xslots + xslot_offset(j, true, false, 0),
                           make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y,
                                       (rv[u].z * inv2) * bv[u].z, (rv[u].w * inv2) * bv[u].w));
        }
    }
    named_barrier_sync(1, kCW * 32);
    // every slot converted once, a quarter per thread
    for (int q0 = 0; q0 < 4 * TGg; q0 += nthr) {
        const int q = q0 + tid, sq = q >> 2;
        int bq = 0, cq = 0;
        const bool valid = q < 4 * TGg && slice_of(sq, nbc_g, false, 0, bq, cq);
        convert_quarter<GQ>(m.xslots + (valid ? sq : 0) * kXSlot, q & 3, valid, false);
    }
    named_barrier_sync(1, kCW * 32);
    return ok;
}

// A consumer thread's ring position, packed: stage buffer, lap within the
// ring, partial slot, barrier phase bit and the thread's ok flag.
__device__ __forceinline__ uint32_t ring_pack(int buf, int lap, int slot, uint32_t phase, bool ok) {
    return static_cast<uint32_t>(buf) | (static_cast<uint32_t>(lap) << 8) | (static_cast<uint32_t>(slot) << 16) |
           (phase << 24) | (ok ? 0u : (1u << 25));
}
__device__ __forceinline__ int ring_buf(uint32_t s) { return static_cast<int>(s & 0xFFu); }
__device__ __forceinline__ int ring_lap(uint32_t s) { return static_cast<int>((s >> 8) & 0xFFu); }
__device__ __forceinline__ int ring_slot(uint32_t s) { return static_cast<int>((s >> 16) & 0xFFu); }
__device__ __forceinline__ uint32_t ring_phase(uint32_t s) { return (s >> 24) & 1u; }
__device__ __forceinline__ bool ring_ok(uint32_t s) { return ((s >> 25) & 1u) == 0u; }

// Down projection of layer l (consumer warps): each thread loads its slice's
// record of mid, then every stage of this block's rows.  st: the ring
// position (ring_pack), returned advanced.
template <int DQ>
__device__ __forceinline__ uint32_t d_phase(const MvsArgs& p, int l, uint32_t st, uint8_t* smem) {
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 8;
    uint64_t* pfull = full + 16;
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + 768);
    int* flag = reinterpret_cast<int*>(smem + 776);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    uint8_t* ring = smem + p.ring_off;
    constexpr int kBd = kBlockBytes<DQ>;
    const int tid = threadIdx.x, lane = tid & 31;
    const int NS = p.ns, NP = p.np;
    const int nsb_d = p.ffn / kQK, nbc_d = nsb_d * 4;
    const uint32_t rb_d = static_cast<uint32_t>(nsb_d) * kBd;
    const int64_t d0 = static_cast<int64_t>(p.hidden) * blockIdx.x / gridDim.x;
    const int64_t d1 = static_cast<int64_t>(p.hidden) * (blockIdx.x + 1) / gridDim.x;
    const int nloc_d = static_cast<int>(d1 - d0), RSd = p.RSd, nd = (nloc_d + RSd - 1) / RSd;
    int buf = ring_buf(st), lap = ring_lap(st), slot = ring_slot(st);
    uint32_t phase = ring_phase(st);
    bool ok = ring_ok(st);

                // Scheduler balance at the model's shape (320 slice threads,
                // 4 rows a stage): the 10 busy warps would put 3/3/2/2 on the
                // schedulers.  Warps 10 and 11 (idle otherwise, on schedulers
                // 2 and 3) hold copies of warps 0 and 1's slices and take the
                // second row pair of each stage from them: 5/5/5/5 row pairs.
                const bool bal = p.TGd == 320 && RSd == 4;
                const bool helper = bal && tid >= 320 && tid < 384;
                const int t = helper ? tid - 320 : tid;   // the slice this thread holds
                const int pair0 = helper ? 2 : 0;                    // first row of the thread's pairs
                const int pair_end = (bal && tid < 64) ? 2 : RSd;    // warps 0, 1: first pair only
                int b = 0, c = 0;
                const bool active = t < p.TGd && slice_of(t, nbc_d, true, p.HPd, b, c);
                if (!active) b = c = 0;
                const int bc = b * 4 + c;
                ok = consumers_grid_wait(p, gridDim.x * static_cast<unsigned>(2 * l + 1), abort_s, flag) && ok;
                // every thread converts a slice (inactive ones block 0's, unused)
                SliceQ6 sl;
                load_slice_q6_mem(sl, p.xperm, active ? t : 0, p.TGd, (b & 1) != 0);
                const uint32_t jq = static_cast<uint32_t>(c & 1);
                const uint32_t sel_sc = jq | ((jq + 2) << 4) | ((jq + 4) << 8) | ((jq + 6) << 12);
                const bool aligned = (b % 2) == 0;
                const uintptr_t wbase = reinterpret_cast<uintptr_t>(p.layer[l].wd);
                const uint8_t* rb = ring + static_cast<uint32_t>(b) * kBd;
#pragma unroll 1
                for (int s = 0; s < nd; ++s) {
                    const int rows_here = min(RSd, nloc_d - s * RSd);
                    if (ok) ok = wait_bar(&full[buf], phase, p, abort_s);
                    if (active && ok) {
                        float* pk = part + slot * p.part_stride;
                        // the stage's copy starts at the 16-byte boundary below its first row
                        const uint32_t delta = static_cast<uint32_t>(
                            (wbase + static_cast<uint64_t>(d0 + static_cast<int64_t>(s) * RSd) * rb_d) & 15u);
                        const uint8_t* sb = rb + static_cast<size_t>(buf) * p.sb + delta;
                        for (int rs = pair0; rs < min(rows_here, pair_end); rs += 2) {
                            const uint8_t* blk[2] = {sb + rs * rb_d, sb + (rs + 1) * rb_d};
                            float v[2];
                            if (rs + 1 < rows_here) {
                                if (aligned) dot_q6<2, kAlign>(sl, blk, c, sel_sc, v);
                                else dot_q6<2, kRotated>(sl, blk, c, sel_sc, v);
                                pk[rs * nbc_d + bc] = v[0];
                                pk[(rs + 1) * nbc_d + bc] = v[1];
                            } else {
                                if (aligned) dot_q6<1, kAlign>(sl, blk, c, sel_sc, v);
                                else dot_q6<1, kRotated>(sl, blk, c, sel_sc, v);
                                pk[rs * nbc_d + bc] = v[0];
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[buf]);
                        mbar_arrive(&pfull[slot]);
                    }
                    if (++buf == NS) buf = 0;
                    if (++lap == NS) {
                        lap = 0;
                        phase ^= 1u;
                    }
                    if (++slot == NP) slot = 0;
                }
    return ring_pack(buf, lap, slot, phase, ok);
}

// After the last layer (consumer warps): the last tail, each block writing
// its share of the residual (the relay ends in the caller's buffer) and of
// `out`.
__device__ __forceinline__ void last_tail(const MvsArgs& p, uint8_t* smem_base) {
    const Smem m = smem_of(smem_base, p);
    float4 av[4], bv[4], rv[4];
    load_tail_weights(p, p.layer[p.nl - 1].w1, p.layer[p.nl - 1].w2, av, bv);
    // a block-uniform decision: block_tail has block-wide barriers
    if (!consumers_grid_wait(p, gridDim.x * static_cast<unsigned>(2 * p.nl), m.abort_s, m.flag)) return;
    float inv2;
    block_tail(p, p.nl - 1, av, rv, inv2, m.red);
    const int tid = threadIdx.x, n4 = p.hidden >> 2, nthr = kCW * 32;
    const int j0 = static_cast<int>(static_cast<int64_t>(n4) * blockIdx.x / gridDim.x);
    const int j1 = static_cast<int>(static_cast<int64_t>(n4) * (blockIdx.x + 1) / gridDim.x);
    float4* o4 = reinterpret_cast<float4*>(p.out);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int j = tid + u * nthr;
        if (j >= j0 && j < j1)
            o4[j] = make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y,
                                (rv[u].z * inv2) * bv[u].z, (rv[u].w * inv2) * bv[u].w);
    }
}

// ---------------------------------------------------------------- kernel
template <int GQ, int DQ>
__global__ void __launch_bounds__(kThreads, 1) mvs_kernel(const __grid_constant__ MvsArgs p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + 8;
    uint64_t* pfull = full + 16;
    uint64_t* reduced = full + 32;
    volatile int* abort_s = reinterpret_cast<volatile int*>(smem + 768);
    float* part = reinterpret_cast<float*>(smem + p.part_off);
    uint8_t* xslots = smem + p.part_off;  // gate/up input slots over the partial slots
    uint8_t* ring = smem + p.ring_off;

    constexpr int kBg = kBlockBytes<GQ>, kBd = kBlockBytes<DQ>;
    const int nl = p.nl, NS = p.ns, NP = p.np;
    const int nsb_g = p.hidden / kQK, nbc_g = nsb_g * 4;
    const int nsb_d = p.ffn / kQK, nbc_d = nsb_d * 4;
    const uint32_t rb_g = static_cast<uint32_t>(nsb_g) * kBg, rb_d = static_cast<uint32_t>(nsb_d) * kBd;
    const int RSg = p.RSg, RSd = p.RSd;
    const int64_t g0 = static_cast<int64_t>(p.ffn) * blockIdx.x / gridDim.x;
    const int64_t g1 = static_cast<int64_t>(p.ffn) * (blockIdx.x + 1) / gridDim.x;
    const int64_t d0 = static_cast<int64_t>(p.hidden) * blockIdx.x / gridDim.x;
    const int64_t d1 = static_cast<int64_t>(p.hidden) * (blockIdx.x + 1) / gridDim.x;
    const int nloc_g = static_cast<int>(g1 - g0), nloc_d = static_cast<int>(d1 - d0);
    const int ng = (nloc_g + RSg - 1) / RSg, nd = (nloc_d + RSd - 1) / RSd;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kCW);
        }
        for (int i = 0; i < NP; ++i) {
            mbar_init(&pfull[i], kCW);
            mbar_init(&reduced[i], 1);
        }
        *abort_s = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kTmaWarp) {
        // ------------------------------------------------------- copy warp
        // Every phase's stages in order, into buffer k % NS, as soon as that
        // buffer has been read (stage k - NS) and the partial slot of stage k
        // has been reduced (stage k - NP).  Never waits for another block.
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int k = 0;
            bool ok = true;
            for (int l = 0; l < nl && ok; ++l) {
                const MvsLayer& L = p.layer[l];
                for (int ph = 0; ph < 2 && ok; ++ph) {
                    const int n = ph == 0 ? ng : nd;
                    for (int s = 0; s < n; ++s, ++k) {
                        const int buf = k % NS;
                        if (k >= NS) ok = wait_bar(&empty[buf], static_cast<uint32_t>((k / NS - 1) & 1), p, abort_s);
                        if (ok && k >= NP)
                            ok = wait_bar(&reduced[k % NP], static_cast<uint32_t>((k / NP - 1) & 1), p, abort_s);
                        if (!ok) break;
                        uint8_t* dst = ring + static_cast<size_t>(buf) * p.sb;
                        fence_proxy_async_smem();  // earlier generic writes to the buffer come first
                        if (ph == 0) {
                            const int64_t r0 = g0 + static_cast<int64_t>(s) * RSg;
                            const int64_t rows = std::min<int64_t>(RSg, g1 - r0);
                            const uint32_t bytes = static_cast<uint32_t>(rows * rb_g);
                            mbar_arrive_expect_tx(&full[buf], 2u * bytes);
                            tma_load_1d_hint(dst, L.wg + r0 * rb_g, bytes, &full[buf], pol);
                            tma_load_1d_hint(dst + p.sbm_g, L.wu + r0 * rb_g, bytes, &full[buf], pol);
                        } else {
                            const int64_t r0 = d0 + static_cast<int64_t>(s) * RSd;
                            const int64_t rows = std::min<int64_t>(RSd, d1 - r0);
                            const uint8_t* start = L.wd + r0 * rb_d;
                            const uint8_t* end = start + rows * rb_d;
                            const uint8_t* matend = L.wd + static_cast<int64_t>(p.hidden) * rb_d;
                            const uint8_t* s16 = reinterpret_cast<const uint8_t*>(
                                reinterpret_cast<uintptr_t>(start) & ~static_cast<uintptr_t>(15));
                            uintptr_t e16 = (reinterpret_cast<uintptr_t>(end) + 15) & ~static_cast<uintptr_t>(15);
                            const uintptr_t mend16 = reinterpret_cast<uintptr_t>(matend) & ~static_cast<uintptr_t>(15);
                            if (e16 > mend16) e16 = mend16;  // never read past the matrix
                            for (const uint8_t* q = reinterpret_cast<const uint8_t*>(e16); q < end; ++q)
                                dst[q - s16] = static_cast<uint8_t>(ldg_u8(q));
                            const uint32_t bytes = static_cast<uint32_t>(e16 - reinterpret_cast<uintptr_t>(s16));
                            mbar_arrive_expect_tx(&full[buf], bytes);
                            if (bytes) tma_load_1d_hint(dst, s16, bytes, &full[buf], pol);
                        }
                    }
                }
            }
            if (!ok) {
                // copies may still be landing in this block's buffers: give
                // the last NS a bounded chance before the block exits
                for (int kk = std::max(0, k - NS); kk < k; ++kk)
                    (void)mbar_wait_bounded(&full[kk % NS], static_cast<uint32_t>((kk / NS) & 1), p.status,
                                            kDevStatusTxTimeout, 200000000ull);
            }
        }
    } else if (warp >= kRedWarp) {
        // ---------------------------------------------------- reducer warp
        // Adds each row's partials of every stage in a fixed order
        // (deterministic) and writes the output.  At the end of a phase the
        // block arrives at the grid barrier.
        int k = 0;
        bool ok = true;
        for (int l = 0; l < nl; ++l) {
            for (int ph = 0; ph < 2; ++ph) {
                const bool gu = ph == 0;
                const int n = gu ? ng : nd;
                const int NMAT = gu ? 2 : 1;
                const int RS = gu ? RSg : RSd;
                const int nbc = gu ? nbc_g : nbc_d;
                const int nloc = gu ? nloc_g : nloc_d;
                const int64_t base = gu ? g0 : d0;
                int L = 32;
                while (L > 1 && L * RS * NMAT > 32) L >>= 1;
                const int n4 = nbc / 4;
                for (int s = 0; s < n; ++s, ++k) {
                    const int slot = k % NP;
                    if (ok) ok = wait_bar(&pfull[slot], static_cast<uint32_t>((k / NP) & 1), p, abort_s);
                    if (ok) {
                        const int lr0 = s * RS;
                        const int rows_here = std::min(RS, nloc - lr0);
                        const float* pk = part + slot * p.part_stride;
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
                            const float other = __shfl_down_sync(0xffffffffu, acc, L);
                            if (sub == 0 && rs < rows_here && m == 0) {
                                const int64_t row = base + lr0 + rs;
                                if (gu) reinterpret_cast<float*>(p.xperm)[xperm_index(row, p.HPd, p.TGd)] = silu_mul_f(acc, other);
                                else p.proj[row] = acc;
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&reduced[slot]);
                }
                // phase done in this block: one release arrival (the warp's
                // outputs, and the consumers' residual shares ordered before
                // them through the stage barriers, come first)
                __syncwarp();
                if (lane == 0 && ok && !*abort_s) red_release_add(p.sync + kSyncCount, 1u);
            }
        }
    } else {
        // --------------------------------------------------- consumer warps
        uint32_t st = 0u;  // the consumer's ring state (Ring, packed)
#pragma unroll 1
        for (int l = 0; l < nl; ++l) {
            int buf = ring_buf(st), lap = ring_lap(st), slot = ring_slot(st);
            uint32_t phase = ring_phase(st);
            bool ok = ring_ok(st);
            // ------------------------------------------ gate/up + SiLU (Q4_K)
            {
                const int TGg = nbc_g, Gg = (kCW * 32) / TGg;
                const int g = tid / TGg, idx = tid - g * TGg;
                int b, c;
                const bool active = slice_of(idx, nbc_g, false, 0, b, c) && g < Gg;
                if (!active) b = c = 0;
                const int bc = b * 4 + c;
                ok = gu_prologue<GQ>(p, l, ok, smem);
                // every thread loads a record (inactive ones slot 0's, unused):
                // a slice set on some paths only would stay live across the
                // layer loop and crowd the registers
                SliceQ4 sl;
                load_record(sl, xslots + (active ? idx : 0) * kXSlot);
                named_barrier_sync(1, kCW * 32);  // the slots are partial slots again
                const uint32_t sel_lo = 0x7540u | static_cast<uint32_t>(2 * (c & 1));
                const uint32_t sel_hi = 0x7540u | static_cast<uint32_t>(2 * (c & 1) + 1);
                const uint8_t* rb = ring + static_cast<uint32_t>(b) * kBg;
#pragma unroll 1
                for (int s = 0; s < ng; ++s) {
                    const int rows_here = min(RSg, nloc_g - s * RSg);
                    if (ok) ok = wait_bar(&full[buf], phase, p, abort_s);
                    if (active && ok) {
                        float* pk = part + slot * p.part_stride;
                        const uint8_t* sb0 = rb + static_cast<size_t>(buf) * p.sb;
                        const uint8_t* sb1 = sb0 + p.sbm_g;
                        for (int rs = g; rs < rows_here; rs += Gg) {
                            const uint8_t* blk[2] = {sb0 + rs * rb_g, sb1 + rs * rb_g};
                            float v[2];
                            dot_q4<2>(sl, blk, c, sel_lo, sel_hi, v);
                            pk[rs * nbc_g + bc] = v[0];
                            pk[(RSg + rs) * nbc_g + bc] = v[1];
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&empty[buf]);
                        mbar_arrive(&pfull[slot]);
                    }
                    if (++buf == NS) buf = 0;
                    if (++lap == NS) {
                        lap = 0;
                        phase ^= 1u;
                    }
                    if (++slot == NP) slot = 0;
                }
            }
            st = ring_pack(buf, lap, slot, phase, ok);
            st = d_phase<DQ>(p, l, st, smem);
        }
        last_tail(p, smem);
    }
}

// ----------------------------------------------------------------- geometry
struct MvsGeo {
    int RSg, RSd, ns, np, part_stride, part_off, ring_off, TGd, HPd;
    uint32_t sb, sbm_g;
    size_t smem;
};

bool mvs_geometry(int64_t hidden, int64_t ffn, int grid, int budget, MvsGeo& g) {
    if (hidden % kQK || ffn % (2 * kQK) || hidden < kQK || ffn < 2 * kQK) return false;
    // every block owns at least one row of each phase (it orders its input
    // writes before its grid-barrier arrivals through its own stages)
    if (hidden < grid || ffn < grid) return false;
    const int nsb_g = static_cast<int>(hidden / kQK), nbc_g = 4 * nsb_g;
    const int nsb_d = static_cast<int>(ffn / kQK), nbc_d = 4 * nsb_d;
    if (nbc_g > kCW * 32) return false;
    // the tails keep at most 4 float4 of each vector per consumer thread
    if (hidden / 4 > 4 * kCW * 32) return false;
    g.HPd = (nbc_d / 2 + 31) / 32 * 32;
    g.TGd = 2 * g.HPd;
    if (g.TGd > kCW * 32) return false;
    const int Gg = (kCW * 32) / nbc_g;
    const int64_t rb_g = static_cast<int64_t>(nsb_g) * kQ4KBytes, rb_d = static_cast<int64_t>(nsb_d) * kQ6KBytes;
    // rows per stage: gate/up a multiple of the row groups, about 60 KB over
    // both matrices; down in pairs, about 64 KB; neither beyond a block's rows
    int64_t rsg = std::max<int64_t>(1, (60 * 1024) / (2 * rb_g * Gg)) * Gg;
    const int64_t gpc = (ffn + grid - 1) / grid;
    rsg = std::min<int64_t>(rsg, (gpc + Gg - 1) / Gg * Gg);
    int64_t rsd = std::max<int64_t>(1, (64 * 1024) / (2 * rb_d)) * 2;
    const int64_t dpc = (hidden + grid - 1) / grid;
    rsd = std::min<int64_t>(rsd, (dpc + 1) / 2 * 2);
    g.RSg = static_cast<int>(rsg);
    g.RSd = static_cast<int>(rsd);
    g.sbm_g = static_cast<uint32_t>((rsg * rb_g + 127) / 128 * 128);
    const uint32_t sbd = static_cast<uint32_t>((rsd * rb_d + 32 + 127) / 128 * 128);
    g.sb = std::max(2 * g.sbm_g, sbd);
    g.part_stride = static_cast<int>(std::max<int64_t>(2 * rsg * nbc_g, rsd * nbc_d));
    const int64_t ps = static_cast<int64_t>(g.part_stride) * 4;
    const int64_t xbytes = static_cast<int64_t>(nbc_g) * kXSlot;
    g.part_off = kHead;
    for (int ns = 8; ns >= 2; --ns) {
        const int np = static_cast<int>(std::max<int64_t>(ns + 2, (xbytes + ps - 1) / ps));
        if (np > 16) continue;
        const int64_t ring_off = (kHead + np * ps + 127) / 128 * 128;
        const int64_t total = ring_off + static_cast<int64_t>(ns) * g.sb;
        if (total <= budget) {
            g.ns = ns;
            g.np = np;
            g.ring_off = static_cast<int>(ring_off);
            g.smem = static_cast<size_t>(total);
            return true;
        }
    }
    return false;
}

}  // namespace

size_t mvs_scratch_bytes(int64_t hidden, int64_t ffn) {
    if (hidden < 1 || ffn < 1) return 0;
    // the sync words, then mid stored slice-major (16 float4 per down-phase thread)
    const int64_t nbc_d = 4 * (ffn / kQK);
    const int64_t tgd = 2 * ((nbc_d / 2 + 31) / 32 * 32);
    return kSyncWords * sizeof(unsigned) + static_cast<size_t>(16 * tgd) * sizeof(float4);
}

bool mvs_supported(int gu_qtype, int down_qtype, int64_t hidden, int64_t ffn, int n_layers, int M) {
    if (M != 1 || gu_qtype != MUSER_Q4_K || down_qtype != MUSER_Q6_K) return false;
    if (n_layers < 1 || n_layers > kMvsMaxLayers) return false;
    const int sms = sm_count(), budget = max_smem_optin();
    if (sms <= 0 || budget <= 0) return false;
    MvsGeo g;
    return mvs_geometry(hidden, ffn, sms, budget, g);
}

int launch_mvs(MvsArgs a, void* scratch, cudaStream_t s) {
    const int sms = sm_count(), budget = max_smem_optin();
    if (sms <= 0 || budget <= 0) return set_error(MUSER_ERR_CUDA, "mvs: cannot query the device");
    MvsGeo g;
    if (!mvs_geometry(a.hidden, a.ffn, sms, budget, g)) return set_error(MUSER_ERR_UNSUPPORTED, "mvs: shape");
    a.RSg = g.RSg;
    a.RSd = g.RSd;
    a.ns = g.ns;
    a.np = g.np;
    a.sb = g.sb;
    a.sbm_g = g.sbm_g;
    a.part_off = g.part_off;
    a.ring_off = g.ring_off;
    a.part_stride = g.part_stride;
    a.HPd = g.HPd;
    a.TGd = g.TGd;
    const size_t sync = kSyncWords * sizeof(unsigned);
    a.sync = static_cast<unsigned*>(scratch);
    a.xperm = reinterpret_cast<float4*>(static_cast<uint8_t*>(scratch) + sync);
    a.status = device_status_word();
    if (a.status == nullptr) return set_error(MUSER_ERR_CUDA, "mvs: no device status word");
    // the barrier count and the abort flag start at zero
    cudaError_t e = cudaMemsetAsync(scratch, 0, sync, s);
    if (e != cudaSuccess) return cuda_fail(e, "mvs: cudaMemsetAsync");
    auto kern = mvs_kernel<MUSER_Q4_K, MUSER_Q6_K>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(g.smem));
    if (e != cudaSuccess) return cuda_fail(e, "mvs: cudaFuncSetAttribute");
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, g.smem);
    if (e != cudaSuccess) return cuda_fail(e, "mvs: occupancy query");
    if (per_sm < 1) return set_error(MUSER_ERR_UNSUPPORTED, "mvs: one block per SM does not fit");
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = g.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;  // every block resident at once (grid barriers)
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return cuda_fail(e, "mvs: cudaLaunchKernelEx");
    return check_launch("mvs_kernel");
}

}  // namespace muser
