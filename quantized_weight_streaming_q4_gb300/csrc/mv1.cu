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
#include "mv1_core.cuh"

namespace muser {

// Device status word of this library's bounded waits (see read_device_status).
__device__ unsigned g_device_status = 0u;

namespace {

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
// by every block from p.x (= projected), p.resid, p.w1, p.w2.  With a
// separate output row (p.resid_out) block 0 writes the updated row there (and
// x to p.out) as soon as it has it.  In place, no block may write the
// residual before every block has read it: once its consumers hold their
// slices (they read the row before), each block's copy warp takes a ticket
// (p.xticket) and looks at the answer only after its last copy request, so
// the ticket's round trip (many blocks update one counter) stays off the
// stream; at its end the block that took the last ticket recomputes the
// updated row with the consumers' 1/rms values (the same operations, so the
// same bits), writes it (and x to p.out) and re-zeroes the ticket.
// ONEG: one row group spans the row (G == 1; the down projections): each
// warp copies and converts its own input slots.  A separate instantiation,
// so the other shapes' code is not touched by that path.
template <int QT, int NMAT, int EPI, int XS, bool ONEG>
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
    // kXTail: consumer thread 0 leaves inv1, inv2 of the tail in red[60..61]
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
        // One row group (the long rows of a down projection): while the
        // consumers still wait for the previous kernel (x not yet requested),
        // the stream need not idle, so each time the last request has landed
        // the next free buffer is requested (bounded in time).  Measured
        // faster for the stand-alone 6656 x 19968 down projections; with the
        // previous tail in the prologue the extra requests delay the tail's
        // loads (slower), and the shorter plain projections gain nothing.
        int issued = lead;
        if (ONEG && lane == 0 && issued > 0) {
            const uint64_t t0 = global_ns();
            while (issued < early && !mbar_try_wait(xissued, 0, 0u)) {
                if (mbar_try_wait(&full[issued - 1 + rot], 0, 200u)) {
                    issue(issued, issued + rot);
                    ++issued;
                } else if (global_ns() - t0 > 1000000000ull) {
                    break;
                }
            }
        }
        issued = __shfl_sync(0xffffffffu, issued, 0);
        ok = mbar_wait_bounded(xissued, 0, &g_device_status, kDevStatusWaitTimeout);
        if (ok && lane == 0)
            for (int k = issued; k < early; ++k) issue(k, k + rot);
        __syncwarp();
        // The rest of the first NS stages once the slots are free again.
        if (ok) ok = mbar_wait_bounded(xready, 0, &g_device_status, kDevStatusWaitTimeout);
        // kXTail: every consumer has read the residual; take the ticket now
        // (release: this block's reads; acquire: the others'), look at the
        // answer after the last copy request.
        unsigned tk = 0u;
        if (XS == kXTail && p.resid_out == nullptr && ok && lane == 0) tk = atom_add_acq_rel_gpu(p.xticket, 1u);
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
        if (XS == kXTail && lane == 0) *flag = (ok && tk == gridDim.x - 1) ? 1 : 0;
    } else if (warp > ncw) {
        // ----------------------------------------------------- reducer warps
        // Two warps take alternate stages (the 2*NS partial slots alternate
        // with them, so each slot has one reducer).
        pdl_launch_dependents();
        pdl_wait();  // outputs of the previous kernel are complete before ours are written
        const int n4 = nbc / 4;
        if constexpr (EPI == kEpiTail) {
            // the last block reads this block's rows of the residual and both
            // norm weights: bring them to L2 while the stream runs
            if (warp == ncw + 1) {
                const char* vecs[3] = {reinterpret_cast<const char*>(p.resid), reinterpret_cast<const char*>(p.w1),
                                       reinterpret_cast<const char*>(p.w2)};
                const int64_t lo = (r0 * 4) & ~int64_t{127}, hi = (r0 + nloc) * 4;
                for (int64_t o = lo + 128 * lane; o < hi; o += 32 * 128)
#pragma unroll
                    for (int v = 0; v < 3; ++v) prefetch_l2(vecs[v] + o);
            }
        }
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
                    if constexpr (EPI == kEpiTail) tss = fmaf(acc, acc, tss);
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
            float inv2;
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
            inv2 = 1.0f / sqrtf(sh / n + p.eps2);
            if (tid == 0) {  // for the block that writes the updated row (kernel end)
                red[60] = inv1;
                red[61] = inv2;
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int j = tid + u * nthr;
                if (j < n4) {
                    const int i = xi(j);
                    const float4 xv = make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y,
                                                  (rv[u].z * inv2) * bv[u].z, (rv[u].w * inv2) * bv[u].w);
                    sts_float4(xslots + xslot_offset(i, QT != MUSER_Q6_K, parity_split, p.HP), xv);
                    // a separate output row: nobody reads it here, block 0 writes it now
                    if (p.resid_out != nullptr && blockIdx.x == 0) {
                        reinterpret_cast<float4*>(p.resid_out)[i] = rv[u];
                        if (p.out) reinterpret_cast<float4*>(p.out)[i] = xv;
                    }
                }
            }
        } else if constexpr (ONEG) {
            // One row group: thread tid owns slot tid, and warp w's 32 slots
            // are the four slices of eight super-blocks.  Each warp copies
            // those blocks' inputs (coalesced, 1 KB per block) and converts
            // its own slots, so no warp waits for another before its loop.
            pdl_wait();  // x is the previous kernel's output
            const float4* x4 = reinterpret_cast<const float4*>(p.x);
#pragma unroll
            for (int k0 = 0; k0 < 8; ++k0) {
                const int k = (k0 + blockIdx.x) & 7;  // blocks start at different lines
                int bk, ck;
                if (slice_of(warp * 32 + 4 * k, nbc, parity_split, p.HP, bk, ck)) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int i = bk * 64 + lane + 32 * h;
                        cp_async16(xslots + xslot_offset(i, QT != MUSER_Q6_K, parity_split, p.HP), x4 + i);
                    }
                }
            }
            cp_async_commit();
            __syncwarp();
            if (lane == 0) mbar_arrive(xissued);
            cp_async_wait_all();
            __syncwarp();
            if (active) {
                if constexpr (QT == MUSER_Q6_K)
                    load_slice_q6(sl, reinterpret_cast<const float*>(xslots + idx * kXSlot), parity_split && (b & 1));
                else
                    load_slice_q4(sl, reinterpret_cast<const float*>(xslots + idx * kXSlot));
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
        if constexpr (!ONEG) named_barrier_sync(1, ncw * 32);  // the consumer warps only
        if constexpr (ONEG) {
            // converted above, each thread its own slot
        } else if (QT != MUSER_Q6_K || G > 1) {
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
    if constexpr (XS == kXTail) {
        // In place (no p.resid_out): the block that took the last ticket.
        // Every block has read the residual, so the updated row replaces it
        // (h = r + p * inv1 * w1 as in the prologue, bit for bit) and x goes
        // to p.out.
        if (ok && p.resid_out == nullptr && *flag) {
            const float inv1 = red[60], inv2 = red[61];
            const int n4 = nbc * 16;
            const float4* p4 = reinterpret_cast<const float4*>(p.x);
            float4* r4 = reinterpret_cast<float4*>(p.resid);
            const float4* a4 = reinterpret_cast<const float4*>(p.w1);
            const float4* b4 = reinterpret_cast<const float4*>(p.w2);
            for (int i = tid; i < n4; i += blockDim.x) {
                const float4 pv = __ldcg(p4 + i), rv = __ldcg(r4 + i), av = __ldg(a4 + i), bv = __ldg(b4 + i);
                float4 h;
                h.x = fmaf(pv.x * inv1, av.x, rv.x);
                h.y = fmaf(pv.y * inv1, av.y, rv.y);
                h.z = fmaf(pv.z * inv1, av.z, rv.z);
                h.w = fmaf(pv.w * inv1, av.w, rv.w);
                r4[i] = h;
                if (p.out)
                    reinterpret_cast<float4*>(p.out)[i] =
                        make_float4((h.x * inv2) * bv.x, (h.y * inv2) * bv.y, (h.z * inv2) * bv.z, (h.w * inv2) * bv.w);
            }
            if (tid == 0) *p.xticket = 0u;
        }
    }
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
        // The ticket is taken after a block barrier with acquire-release
        // semantics: it releases every write of this block (projected, the
        // partial) and the last block acquires all the others'.
        if (tid == 0) {
            if (p.tail_part) p.tail_part[blockIdx.x] = red[40] + red[41];
            const unsigned t = atom_add_acq_rel_gpu(p.ticket, 1u);
            *flag = (t == gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (*flag) {
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

template <int QT, int NMAT, int EPI, int XS, bool ONEG = false>
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
    if (XS == kXTail && a.resid_out == nullptr && a.xticket == nullptr)
        return set_error(MUSER_ERR_INVALID_ARG, "mv1: the fused tail in place needs its ticket");
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
    if (ONEG != (geo.G == 1 && XS == kXMemory && NMAT == 1))
        return set_error(MUSER_ERR_UNSUPPORTED, "mv1: one-row-group instantiation for the wrong geometry");
    auto kern = mv1_kernel<QT, NMAT, EPI, XS, ONEG>;
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
    }
    // one row group (the down projections' rows): the ONEG instantiations
    const bool oneg = xs == kXMemory && nmat == 1 && mv1_geom(qtype, a.nsb).G == 1;
    if (oneg) {
        if (qtype == MUSER_Q4_K && epi == kEpiStore) return launch_mv1_t<MUSER_Q4_K, 1, kEpiStore, kXMemory, true>(a, s);
        if (qtype == MUSER_Q4_K && epi == kEpiTail) return launch_mv1_t<MUSER_Q4_K, 1, kEpiTail, kXMemory, true>(a, s);
        if (qtype == MUSER_Q5_K && epi == kEpiStore) return launch_mv1_t<MUSER_Q5_K, 1, kEpiStore, kXMemory, true>(a, s);
        if (qtype == MUSER_Q6_K && epi == kEpiStore) return launch_mv1_t<MUSER_Q6_K, 1, kEpiStore, kXMemory, true>(a, s);
        if (qtype == MUSER_Q6_K && epi == kEpiTail) return launch_mv1_t<MUSER_Q6_K, 1, kEpiTail, kXMemory, true>(a, s);
        if (qtype == MUSER_Q6_K && epi == kEpiSoftcap)
            return launch_mv1_t<MUSER_Q6_K, 1, kEpiSoftcap, kXMemory, true>(a, s);
        if (qtype == MUSER_Q4_K && epi == kEpiSoftcap)
            return launch_mv1_t<MUSER_Q4_K, 1, kEpiSoftcap, kXMemory, true>(a, s);
    } else if (xs == kXMemory && qtype == MUSER_Q4_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q4_K, 1, kEpiStore, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q4_K, 1, kEpiTail, kXMemory>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q4_K, 2, kEpiSiluMul, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiSoftcap) return launch_mv1_t<MUSER_Q4_K, 1, kEpiSoftcap, kXMemory>(a, s);
    } else if (xs == kXMemory && qtype == MUSER_Q5_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q5_K, 1, kEpiStore, kXMemory>(a, s);
    } else if (xs == kXMemory && qtype == MUSER_Q6_K) {
        if (nmat == 1 && epi == kEpiStore) return launch_mv1_t<MUSER_Q6_K, 1, kEpiStore, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiTail) return launch_mv1_t<MUSER_Q6_K, 1, kEpiTail, kXMemory>(a, s);
        if (nmat == 2 && epi == kEpiSiluMul) return launch_mv1_t<MUSER_Q6_K, 2, kEpiSiluMul, kXMemory>(a, s);
        if (nmat == 1 && epi == kEpiSoftcap) return launch_mv1_t<MUSER_Q6_K, 1, kEpiSoftcap, kXMemory>(a, s);
    }
    return set_error(MUSER_ERR_UNSUPPORTED, "mv1: no kernel for qtype %d nmat %d epilogue %d", qtype, nmat, epi);
}

}  // namespace muser
