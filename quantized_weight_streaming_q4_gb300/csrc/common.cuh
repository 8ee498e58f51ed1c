// common.cuh -- host error plumbing and device helpers shared by libmuser's
// translation units (CUDA, sm_103a).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "muser.h"

namespace muser {

// ------------------------------------------------------------------- host
// Records a printf-style message for muser_last_error() on this thread and
// returns `status`.
int set_error(int status, const char* fmt, ...);
void clear_error();
// Maps a CUDA error to MUSER_ERR_CUDA with a message naming `what`.
int cuda_fail(cudaError_t e, const char* what);
// Checks cudaGetLastError() after a launch.
int check_launch(const char* what);
// SM count of the current device (cached per device).
int sm_count();
// Max dynamic shared memory per block of the current device (opt-in limit).
int max_smem_optin();

// Returns the status of `expr` from the enclosing function unless it is MUSER_OK.
#define MUSER_TRY(expr)                  \
    do {                                 \
        const int _rc = (expr);          \
        if (_rc != MUSER_OK) return _rc; \
    } while (0)

inline bool is_aligned(const void* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}
inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Device-side status word: kernels that give up a bounded wait set a bit
// here instead of hanging; the host can read and clear it.
// kDevStatusQ6kScale: a Q6_K sub-block scale outside [-62, 62] reached the
// tensor-core kernel, whose binary16 products are exact only inside it.
enum : unsigned { kDevStatusWaitTimeout = 1u, kDevStatusTxTimeout = 2u, kDevStatusQ6kScale = 4u };
unsigned read_device_status(bool reset);

// ------------------------------------------------------------------ device
constexpr int kQK = 256;          // weights per super-block
constexpr int kQ4KBytes = 144;    // Q4_K super-block bytes
constexpr int kQ6KBytes = 210;    // Q6_K super-block bytes
constexpr int kQ5KBytes = 176;    // Q5_K super-block bytes
// Super-block bytes of a quant type known at compile time.
template <int QT>
constexpr int kBlockBytes = QT == MUSER_Q4_K ? kQ4KBytes : (QT == MUSER_Q5_K ? kQ5KBytes : kQ6KBytes);

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Deterministic block-wide sum: per-warp shuffle trees, then thread 0 adds
// the warp partials in warp order.  `red` needs 33 floats of shared memory.
// Every thread of the block must call it; all get the same value.
__device__ __forceinline__ float block_sum(float v, float* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nwarps = (blockDim.x + 31) >> 5;
    v = warp_sum(v);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.0f;
        for (int w = 0; w < nwarps; ++w) t += red[w];
        red[32] = t;
    }
    __syncthreads();
    const float t = red[32];
    __syncthreads();
    return t;
}

// Read-only global loads.  *_stream bypasses L1 allocation (weights are read
// once); plain nc loads keep L1 allocation.
__device__ __forceinline__ uint4 ldg_stream16(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u32(const void* p) {
    uint32_t v;
    asm volatile("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u16(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_u8(const void* p) {
    unsigned short v;
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=h"(v) : "l"(p));
    return v & 0xffu;
}

// Binary16 bits -> binary32 (exact).
__device__ __forceinline__ float h2f(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16 & 0xffffu)));
}

// The float whose bit pattern is `bits`.  With only the low 23 bits set it is
// a subnormal: bits * 2^-149, exactly.
__device__ __forceinline__ float bits_f(uint32_t bits) { return __uint_as_float(bits); }

// Small unsigned byte -> float through the 2^23 magic exponent: the float
// with bits 0x4B0000XX is 2^23 + XX, exactly.
__device__ __forceinline__ float byte_to_f(uint32_t word, uint32_t sel_with_magic) {
    return __uint_as_float(__byte_perm(word, 0x4B000000u, sel_with_magic)) - 8388608.0f;
}

__device__ __forceinline__ uint4 lds_uint4(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))));
    return v;
}
__device__ __forceinline__ void sts_uint4(void* p, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))),
                 "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}
// 16-byte shared-memory store (p 16-byte aligned, in shared memory).
__device__ __forceinline__ void sts_float4(void* p, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
                 : "memory");
}
// Bring the 128-byte line holding p into L2 (no register result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// 16-byte asynchronous copy global -> shared (both 16-byte aligned), and
// the waits on this thread's copies.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Barrier `id` (1..15) over the first `nthreads` threads of the block (a
// multiple of 32; every warp taking part calls it).
__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------- TMA / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// 16-byte shared-memory load (p 16-byte aligned, in shared memory).
__device__ __forceinline__ float4 lds_float4(const void* p) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes).
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void* dst, const void* src, uint32_t bytes,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// L2 policy for data read exactly once (the weight stream): its lines are
// the first candidates for eviction, so the stream does not displace the
// activations or the kernels' code from L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// 1-D bulk copy with an L2 cache policy (see tma_load_1d).
__device__ __forceinline__ void tma_load_1d_hint(void* dst, const void* src, uint32_t bytes,
                                                 uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// One wait attempt: the warp may be suspended in hardware for up to
// `hint_ns` nanoseconds and resumes as soon as the phase completes.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}
// Nanoseconds of the GPU's global timer.
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Bounded wait on an mbarrier phase: suspended attempts until the phase
// completes or `limit_ns` of global time (1 s by default) have passed; the
// bound is in time, so it holds however early an attempt returns.  Returns
// false and sets `flag` in the device status word *status on giving up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned* status,
                                                  unsigned flag, uint64_t limit_ns = 1000000000ull) {
    if (mbar_try_wait(bar, parity, 1000000u)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try_wait(bar, parity, 1000000u)) return true;
        if (global_ns() - t0 > limit_ns) break;
    }
    atomicOr(status, flag);
    return false;
}

// Atomic add at GPU scope with acquire-release semantics: the calling
// thread's earlier accesses (and those ordered before them by a block or warp
// barrier) are visible to a thread that later observes the result, and
// accesses other threads released before the values this one observes are
// visible to the caller afterwards.  Returns the old value.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Programmatic dependent launch controls (no-ops without the launch attribute).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------- dual-eps tail
// One row of the dual-eps tail (Muser book Ch 19 §19.4): three passes over
// the row by the whole block, float4 strides, deterministic reductions.
//   pass 1: inv1 = 1/sqrt(mean(src^2) + eps1)
//   pass 2: resid = resid + (src*inv1)*w1, stored; accumulate resid^2
//   pass 3: out = (resid*inv2)*w2 with inv2 = 1/sqrt(mean(resid^2) + eps2)
// `src` may have been written by other blocks of the same grid (read with
// .cg loads that bypass L1).  `red` needs 33 floats of shared memory.
__device__ __forceinline__ void block_dual_tail_row(float* resid, const float* src, float* out,
                                                    const float* w1, const float* w2, int n,
                                                    float eps1, float eps2, float* red) {
    const int n4 = n >> 2;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* r4 = reinterpret_cast<float4*>(resid);
    float4* o4 = reinterpret_cast<float4*>(out);
    const float4* a4 = reinterpret_cast<const float4*>(w1);
    const float4* b4 = reinterpret_cast<const float4*>(w2);
    float ss = 0.0f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = __ldcg(s4 + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
    ss = block_sum(ss, red);
    const float inv1 = 1.0f / sqrtf(ss / static_cast<float>(n) + eps1);
    float sh = 0.0f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = __ldcg(s4 + i);
        const float4 r = __ldcg(r4 + i);
        const float4 w = __ldg(a4 + i);
        float4 h;
        h.x = fmaf(v.x * inv1, w.x, r.x);
        h.y = fmaf(v.y * inv1, w.y, r.y);
        h.z = fmaf(v.z * inv1, w.z, r.z);
        h.w = fmaf(v.w * inv1, w.w, r.w);
        r4[i] = h;
        sh = fmaf(h.x, h.x, sh);
        sh = fmaf(h.y, h.y, sh);
        sh = fmaf(h.z, h.z, sh);
        sh = fmaf(h.w, h.w, sh);
    }
    sh = block_sum(sh, red);
    const float inv2 = 1.0f / sqrtf(sh / static_cast<float>(n) + eps2);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 h = r4[i];  // this thread's own pass-2 stores
        const float4 w = __ldg(b4 + i);
        o4[i] = make_float4((h.x * inv2) * w.x, (h.y * inv2) * w.y, (h.z * inv2) * w.z,
                            (h.w * inv2) * w.w);
    }
}

// The same row with the vectors in registers, for a kernel whose one
// block per row starts before the previous kernel ends (programmatic
// launch): w1 is read before the wait on it, src and the residual after it,
// w2 while the second sum is reduced.  Thread t holds float4 t + u * nt (u
// < V; n / 4 <= V * nt); the per-thread partial sums take its elements in
// the same order as block_dual_tail_row and the block sums are the same, so
// the results are equal.  x = w2 * h * inv2 also comes back in xv (zero past
// the row).
template <int V>
__device__ __forceinline__ void dual_tail_row_reg(float* resid, const float* src, float* out, const float* w1,
                                                  const float* w2, int n, float eps1, float eps2, float* red,
                                                  float4* xv) {
    const int n4 = n >> 2, tid = threadIdx.x, nt = blockDim.x;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* r4 = reinterpret_cast<float4*>(resid);
    float4* o4 = reinterpret_cast<float4*>(out);
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 pv[V], rv[V], av[V], bv[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = tid + u * nt;
        av[u] = i < n4 ? __ldg(reinterpret_cast<const float4*>(w1) + i) : z;
    }
    pdl_launch_dependents();
    pdl_wait();  // src and the residual are the previous kernels' outputs
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = tid + u * nt;
        pv[u] = i < n4 ? __ldcg(s4 + i) : z;
        rv[u] = i < n4 ? __ldcg(r4 + i) : z;
    }
    float ss = 0.0f;
#pragma unroll
    for (int u = 0; u < V; ++u) {
        ss = fmaf(pv[u].x, pv[u].x, ss);
        ss = fmaf(pv[u].y, pv[u].y, ss);
        ss = fmaf(pv[u].z, pv[u].z, ss);
        ss = fmaf(pv[u].w, pv[u].w, ss);
    }
    ss = block_sum(ss, red);
    const float inv1 = 1.0f / sqrtf(ss / static_cast<float>(n) + eps1);
    float sh = 0.0f;
#pragma unroll
    for (int u = 0; u < V; ++u) {
        float4 h;  // zero past the row
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
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = tid + u * nt;
        bv[u] = i < n4 ? __ldg(reinterpret_cast<const float4*>(w2) + i) : z;
    }
    sh = block_sum(sh, red);
    const float inv2 = 1.0f / sqrtf(sh / static_cast<float>(n) + eps2);
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = tid + u * nt;
        xv[u] = make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y, (rv[u].z * inv2) * bv[u].z,
                            (rv[u].w * inv2) * bv[u].w);
        if (i < n4) {
            r4[i] = rv[u];
            o4[i] = xv[u];
        }
    }
}

// The same row of the dual-eps tail when every block of the grid has left
// its share of sum(src^2) in parts[0..nparts) (the block that wrote those
// rows of src summed their squares): the first pass is a sum of nparts
// values, and the row (at most 4 float4 of each vector per thread) stays in
// registers between the two remaining steps.  Needs n / 4 <= 4 * blockDim.x.
__device__ __forceinline__ void block_dual_tail_row_parts(float* resid, const float* src, float* out,
                                                          const float* w1, const float* w2, int n,
                                                          float eps1, float eps2, const float* parts,
                                                          int nparts, float* red) {
    constexpr int V = 4;
    const int n4 = n >> 2;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4* r4 = reinterpret_cast<float4*>(resid);
    float4* o4 = reinterpret_cast<float4*>(out);
    const float4* a4 = reinterpret_cast<const float4*>(w1);
    const float4* b4 = reinterpret_cast<const float4*>(w2);
    // the row's loads go out first: the partials' sum waits on its own loads
    float4 pv[V], rv[V], av[V], bv[V];
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < n4) {
            pv[u] = __ldcg(s4 + i);
            rv[u] = __ldcg(r4 + i);
            av[u] = __ldg(a4 + i);
            bv[u] = __ldg(b4 + i);
        }
    }
    float ss = 0.0f;
    for (int i = threadIdx.x; i < nparts; i += blockDim.x) ss += __ldcg(parts + i);
    ss = block_sum(ss, red);
    const float inv1 = 1.0f / sqrtf(ss / static_cast<float>(n) + eps1);
    float sh = 0.0f;
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < n4) {
            float4 h;
            h.x = fmaf(pv[u].x * inv1, av[u].x, rv[u].x);
            h.y = fmaf(pv[u].y * inv1, av[u].y, rv[u].y);
            h.z = fmaf(pv[u].z * inv1, av[u].z, rv[u].z);
            h.w = fmaf(pv[u].w * inv1, av[u].w, rv[u].w);
            r4[i] = h;
            sh = fmaf(h.x, h.x, sh);
            sh = fmaf(h.y, h.y, sh);
            sh = fmaf(h.z, h.z, sh);
            sh = fmaf(h.w, h.w, sh);
            rv[u] = h;
        }
    }
    sh = block_sum(sh, red);
    const float inv2 = 1.0f / sqrtf(sh / static_cast<float>(n) + eps2);
#pragma unroll
    for (int u = 0; u < V; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i < n4)
            o4[i] = make_float4((rv[u].x * inv2) * bv[u].x, (rv[u].y * inv2) * bv[u].y,
                                (rv[u].z * inv2) * bv[u].z, (rv[u].w * inv2) * bv[u].w);
    }
}

// The LM head's logit scale and soft cap in binary32 (Ch 10 Figure 10.1 box
// 15): cap * tanh(l * scale / cap), with CUDA's tanhf.
__device__ __forceinline__ float softcap_f(float l, float scale, float cap) {
    return cap * tanhf((l * scale) / cap);
}

// SiLU(g) * u in binary32 (z/(1+exp(-z)) with CUDA's expf and IEEE division).
__device__ __forceinline__ float silu_mul_f(float g, float u) {
    return (g / (1.0f + expf(-g))) * u;
}

}  // namespace muser
