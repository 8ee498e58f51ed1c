// misc.cu -- the small kernels of the path: exact dequantisation (the
// bit-exact test hook), RMSNorm, SiLU gating, the standalone dual-eps tail,
// the f16 K/V ring store, and a bounded spin used to test muser_sync.
#include "common.cuh"
#include "kernels.cuh"

namespace muser {

namespace {

// ----------------------------------------------------------- dequantize
// One thread per 32-weight sub-block slot (see mvM.cu for the same slot
// arithmetic): value = the exactly rounded binary32 of the block formula.
__global__ void dequant_q4k_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                   float* __restrict__ out) {
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= nblocks * 8) return;
    const int64_t blkno = gid >> 3;
    const int j = static_cast<int>(gid & 7);
    const uint8_t* blk = W + blkno * kQ4KBytes;
    const uint4 hd = *reinterpret_cast<const uint4*>(blk);
    const int c = j >> 1;
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 32 + 32 * c);
    uint32_t sc, mn;
    if (j < 4) {
        sc = (hd.y >> (8 * j)) & 63u;
        mn = (hd.z >> (8 * j)) & 63u;
    } else {
        const int jj = j - 4;
        sc = ((hd.w >> (8 * jj)) & 0x0Fu) | (((hd.y >> (8 * jj + 6)) & 3u) << 4);
        mn = ((hd.w >> (8 * jj + 4)) & 0x0Fu) | (((hd.z >> (8 * jj + 6)) & 3u) << 4);
    }
    const float dsc = __fmul_rn(h2f(hd.x), static_cast<float>(sc));
    const float ndm = -__fmul_rn(h2f(hd.x >> 16), static_cast<float>(mn));
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const int sh = (j & 1) ? 4 : 0;
    float* o = out + blkno * kQK + 32 * j;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q4 = (words[t] >> sh) & 0x0F0F0F0Fu;
        float4 v;
        v.x = __fmaf_rn(dsc, static_cast<float>(q4 & 0xFFu), ndm);
        v.y = __fmaf_rn(dsc, static_cast<float>((q4 >> 8) & 0xFFu), ndm);
        v.z = __fmaf_rn(dsc, static_cast<float>((q4 >> 16) & 0xFFu), ndm);
        v.w = __fmaf_rn(dsc, static_cast<float>(q4 >> 24), ndm);
        reinterpret_cast<float4*>(o)[t] = v;
    }
}

// Q5_K: as Q4_K, with the codes at byte 48 and a fifth code bit, bit
// 2c + (j & 1) of qh[l] (bytes 16..47), for weight l of sub-block j.
__global__ void dequant_q5k_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                   float* __restrict__ out) {
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= nblocks * 8) return;
    const int64_t blkno = gid >> 3;
    const int j = static_cast<int>(gid & 7);
    const uint8_t* blk = W + blkno * kQ5KBytes;
    const uint4 hd = *reinterpret_cast<const uint4*>(blk);
    const int c = j >> 1;
    const uint4 ha = *reinterpret_cast<const uint4*>(blk + 16);
    const uint4 hb = *reinterpret_cast<const uint4*>(blk + 32);
    const uint4 qa = *reinterpret_cast<const uint4*>(blk + 48 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4*>(blk + 64 + 32 * c);
    uint32_t sc, mn;
    if (j < 4) {
        sc = (hd.y >> (8 * j)) & 63u;
        mn = (hd.z >> (8 * j)) & 63u;
    } else {
        const int jj = j - 4;
        sc = ((hd.w >> (8 * jj)) & 0x0Fu) | (((hd.y >> (8 * jj + 6)) & 3u) << 4);
        mn = ((hd.w >> (8 * jj + 4)) & 0x0Fu) | (((hd.z >> (8 * jj + 6)) & 3u) << 4);
    }
    const float dsc = __fmul_rn(h2f(hd.x), static_cast<float>(sc));
    const float ndm = -__fmul_rn(h2f(hd.x >> 16), static_cast<float>(mn));
    const uint32_t words[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    const uint32_t hbits[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
    const int sh = (j & 1) ? 4 : 0;
    const int hsh = 2 * c + (j & 1);
    float* o = out + blkno * kQK + 32 * j;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const uint32_t q5 = ((words[t] >> sh) & 0x0F0F0F0Fu) | (((hbits[t] >> hsh) & 0x01010101u) << 4);
        float4 v;
        v.x = __fmaf_rn(dsc, static_cast<float>(q5 & 0xFFu), ndm);
        v.y = __fmaf_rn(dsc, static_cast<float>((q5 >> 8) & 0xFFu), ndm);
        v.z = __fmaf_rn(dsc, static_cast<float>((q5 >> 16) & 0xFFu), ndm);
        v.w = __fmaf_rn(dsc, static_cast<float>(q5 >> 24), ndm);
        reinterpret_cast<float4*>(o)[t] = v;
    }
}

__global__ void dequant_q6k_kernel(const uint8_t* __restrict__ W, int64_t nblocks,
                                   float* __restrict__ out) {
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (gid >= nblocks * 8) return;
    const int64_t blkno = gid >> 3;
    const int j8 = static_cast<int>(gid & 7);
    const int h = j8 >> 2, g = j8 & 3;
    const uint8_t* blk = W + blkno * kQ6KBytes;
    const float d = h2f(ldg_u16(blk + 208));
    const float dsc0 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(ldg_u8(blk + 192 + 8 * h + 2 * g))));
    const float dsc1 = __fmul_rn(d, static_cast<float>(static_cast<int8_t>(ldg_u8(blk + 193 + 8 * h + 2 * g))));
    const uint8_t* ql = blk + 64 * h + 32 * (g & 1);
    const uint8_t* qh = blk + 128 + 32 * h;
    float* o = out + blkno * kQK + 128 * h + 32 * g;
    for (int l = 0; l < 32; ++l) {
        const uint32_t lb = ldg_u8(ql + l), hb = ldg_u8(qh + l);
        const uint32_t q = ((g & 2) ? (lb >> 4) : (lb & 0x0Fu)) | (((hb >> (2 * g)) & 3u) << 4);
        o[l] = __fmul_rn(l < 16 ? dsc0 : dsc1, static_cast<float>(static_cast<int>(q) - 32));
    }
}

// ------------------------------------------------------------ RMSNorm
// One block per row (Muser book Ch 2 §2.6 rms_norm_batch):
// out = (x * inv) * w, inv = 1/sqrt(mean(x^2) + eps).
__global__ void rms_norm_kernel(const float* x, const float* __restrict__ w, float* out, int n,
                                float eps) {
    __shared__ float red[33];
    const float4* x4 = reinterpret_cast<const float4*>(x + static_cast<int64_t>(blockIdx.x) * n);
    float4* o4 = reinterpret_cast<float4*>(out + static_cast<int64_t>(blockIdx.x) * n);
    const float4* w4 = reinterpret_cast<const float4*>(w);
    const int n4 = n >> 2;
    float ss = 0.0f;
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = x4[i];
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
    ss = block_sum(ss, red);
    const float inv = 1.0f / sqrtf(ss / static_cast<float>(n) + eps);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
        const float4 v = x4[i];
        const float4 ww = __ldg(w4 + i);
        o4[i] = make_float4((v.x * inv) * ww.x, (v.y * inv) * ww.y, (v.z * inv) * ww.z,
                            (v.w * inv) * ww.w);
    }
}

__global__ void scale_softcap_kernel(float* l, int64_t n, float scale, float cap) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        l[i] = softcap_f(l[i], scale, cap);
}

__global__ void silu_mul_kernel(const float* a, const float* b, float* out, int64_t n) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        out[i] = silu_mul_f(a[i], b[i]);
}

// One block per row; the page's kernel uses one 1,024-thread group per row.
__global__ void dual_tail_kernel(float* resid, const float* src, float* out, const float* w1,
                                 const float* w2, int n, float eps1, float eps2) {
    __shared__ float red[33];
    pdl_launch_dependents();
    pdl_wait();  // src and the residual are the previous kernels' outputs
    const int64_t off = static_cast<int64_t>(blockIdx.x) * n;
    block_dual_tail_row(resid + off, src + off, out + off, w1, w2, n, eps1, eps2, red);
}

// The same row with the vectors in registers (dual_tail_row_reg; n / 4 <=
// V * 1024, V <= 3; longer rows take dual_tail_kernel): one round of loads
// instead of three passes, with the results of dual_tail_kernel.
template <int V>  // float4 of each vector per thread: n / 4 <= V * 1024
__global__ void __launch_bounds__(1024) dual_tail_reg_kernel(float* resid, const float* src, float* out,
                                                              const float* w1, const float* w2, int n, float eps1,
                                                              float eps2) {
    __shared__ float red[33];
    const int64_t off = static_cast<int64_t>(blockIdx.x) * n;
    float4 xv[V];
    dual_tail_row_reg<V>(resid + off, src + off, out + off, w1, w2, n, eps1, eps2, red, xv);
}

// -------------------------------------------------------------- KV store
// Muser book Ch 15 §15.4 (muser_kv_store_batch_f16): source row t of the batch
// (t >= src_first) lands in physical row (phys_of_first + t) % capacity; the
// binary32 -> binary16 conversion rounds to nearest even.
__global__ void kv_store_kernel(uint16_t* key, uint16_t* value, const float* k, const float* v,
                                int64_t kv_dim, int64_t head_dim, int head_major,
                                int64_t capacity, int64_t phys_of_first, int64_t src_first,
                                int64_t nrows) {
    const int64_t total = nrows * kv_dim;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t t = src_first + i / kv_dim;
        const int64_t e = i % kv_dim;
        const int64_t phys = (phys_of_first + t) % capacity;
        int64_t dst = phys * kv_dim + e;
        if (head_major) dst = ((e / head_dim) * capacity + phys) * head_dim + e % head_dim;
        const int64_t s = t * kv_dim + e;
        key[dst] = __half_as_ushort(__float2half_rn(k[s]));
        value[dst] = __half_as_ushort(__float2half_rn(v[s]));
    }
}

// Muser book Ch 15 §15.6: moves `count` token rows between a K/V plane pair
// and detached token-major rows.  Row j of the window <-> physical slot
// (phys0 + j) % capacity, in either plane layout (§15.3 Figure 15.1).  This
// is the element form, one half per thread, for shapes or buffers that the
// 16-byte form below does not take.
template <bool TO_PLANE>
__global__ void kv_window_kernel(uint16_t* __restrict__ pk, uint16_t* __restrict__ pv,
                                 uint16_t* __restrict__ rk, uint16_t* __restrict__ rv,
                                 int64_t kv_dim, int64_t head_dim, int head_major,
                                 int64_t capacity, int64_t phys0, int64_t count) {
    const int64_t total = count * kv_dim;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t j = i / kv_dim;
        const int64_t e = i - j * kv_dim;
        const int64_t p = (phys0 + j) % capacity;
        const int64_t pi =
            head_major ? ((e / head_dim) * capacity + p) * head_dim + e % head_dim : p * kv_dim + e;
        if constexpr (TO_PLANE) {
            pk[pi] = rk[i];
            pv[pi] = rv[i];
        } else {
            rk[i] = pk[pi];
            rv[i] = pv[pi];
        }
    }
}

// The 16-byte form, one warp per token row: the row's slot is computed once
// per row, the lanes take the row's 16-byte chunks (kv_dim / 8 of them), and
// two rows are in flight per warp (both rows' loads before their stores).
template <bool TO_PLANE>
__global__ void kv_window_rows_kernel(uint16_t* __restrict__ pk, uint16_t* __restrict__ pv,
                                      uint16_t* __restrict__ rk, uint16_t* __restrict__ rv,
                                      int kv_dim, int head_dim, int head_major, int64_t capacity,
                                      int64_t phys0, int64_t count) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
    const int nch = kv_dim >> 3;
    auto plane_index = [&](int64_t p, int e) -> int64_t {
        if (!head_major) return p * kv_dim + e;
        const int h = e / head_dim;
        return (static_cast<int64_t>(h) * capacity + p) * head_dim + (e - h * head_dim);
    };
    for (int64_t j0 = warp; j0 < count; j0 += 2 * nwarps) {
        const int64_t j1 = j0 + nwarps;
        const bool two = j1 < count;
        const int64_t p0 = (phys0 + j0) % capacity;
        const int64_t p1 = two ? (phys0 + j1) % capacity : 0;
        for (int c = lane; c < nch; c += 32) {
            const int e = c << 3;
            const int64_t r0 = j0 * kv_dim + e, r1 = j1 * kv_dim + e;
            const int64_t q0 = plane_index(p0, e), q1 = two ? plane_index(p1, e) : 0;
            uint4 k0, v0, k1 = make_uint4(0, 0, 0, 0), v1 = k1;
            if constexpr (TO_PLANE) {
                k0 = *reinterpret_cast<const uint4*>(rk + r0);
                v0 = *reinterpret_cast<const uint4*>(rv + r0);
                if (two) {
                    k1 = *reinterpret_cast<const uint4*>(rk + r1);
                    v1 = *reinterpret_cast<const uint4*>(rv + r1);
                }
                *reinterpret_cast<uint4*>(pk + q0) = k0;
                *reinterpret_cast<uint4*>(pv + q0) = v0;
                if (two) {
                    *reinterpret_cast<uint4*>(pk + q1) = k1;
                    *reinterpret_cast<uint4*>(pv + q1) = v1;
                }
            } else {
                k0 = *reinterpret_cast<const uint4*>(pk + q0);
                v0 = *reinterpret_cast<const uint4*>(pv + q0);
                if (two) {
                    k1 = *reinterpret_cast<const uint4*>(pk + q1);
                    v1 = *reinterpret_cast<const uint4*>(pv + q1);
                }
                *reinterpret_cast<uint4*>(rk + r0) = k0;
                *reinterpret_cast<uint4*>(rv + r0) = v0;
                if (two) {
                    *reinterpret_cast<uint4*>(rk + r1) = k1;
                    *reinterpret_cast<uint4*>(rv + r1) = v1;
                }
            }
        }
    }
}

// Busy-waits on the global nanosecond timer; returns after `ns` (bounded).
__global__ void spin_kernel(uint64_t ns) {
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        __nanosleep(1000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns);
}

// Holds its SM (through its shared memory) for `ns` of global time.
__global__ void occupy_kernel(uint64_t ns) {
    extern __shared__ uint8_t hold[];
    uint64_t t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    do {
        __nanosleep(1000);
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    } while (t - t0 < ns);
    if (t == 0) hold[threadIdx.x] = 0;  // never true: keeps the allocation referenced
}

}  // namespace

int launch_dequantize(int qtype, const uint8_t* W, int64_t rows, int64_t cols, float* out,
                      cudaStream_t s) {
    const int64_t nblocks = rows * (cols / kQK);
    const int64_t threads = nblocks * 8;
    if (threads == 0) return MUSER_OK;
    const int bs = 256;
    const int64_t grid = (threads + bs - 1) / bs;
    if (qtype == MUSER_Q4_K) dequant_q4k_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(W, nblocks, out);
    else if (qtype == MUSER_Q5_K) dequant_q5k_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(W, nblocks, out);
    else dequant_q6k_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(W, nblocks, out);
    return check_launch("dequantize");
}

int launch_rms_norm(const float* x, const float* w, float* out, int n, int M, float eps,
                    cudaStream_t s) {
    rms_norm_kernel<<<M, 1024, 0, s>>>(x, w, out, n, eps);
    return check_launch("rms_norm");
}

int launch_scale_softcap(float* logits, int64_t n, float scale, float cap, cudaStream_t s) {
    if (n == 0) return MUSER_OK;
    const int bs = 256;
    const int64_t grid = std::min<int64_t>((n + bs - 1) / bs, static_cast<int64_t>(sm_count()) * 16);
    scale_softcap_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(logits, n, scale, cap);
    return check_launch("scale_softcap");
}

int launch_silu_mul(const float* a, const float* b, float* out, int64_t n, cudaStream_t s) {
    if (n == 0) return MUSER_OK;
    const int bs = 256;
    const int64_t grid = std::min<int64_t>((n + bs - 1) / bs, static_cast<int64_t>(sm_count()) * 16);
    silu_mul_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(a, b, out, n);
    return check_launch("silu_mul");
}

int launch_dual_tail(float* resid, const float* src, float* out, const float* w1,
                     const float* w2, int n, int M, float eps1, float eps2, cudaStream_t s) {
    // programmatic serialization: the next kernel may start its own
    // independent work while this one runs
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(M));
    cfg.blockDim = dim3(1024);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const int v = ((n >> 2) + 1023) / 1024;
    cudaError_t e;
    if (v <= 1) e = cudaLaunchKernelEx(&cfg, dual_tail_reg_kernel<1>, resid, src, out, w1, w2, n, eps1, eps2);
    else if (v == 2) e = cudaLaunchKernelEx(&cfg, dual_tail_reg_kernel<2>, resid, src, out, w1, w2, n, eps1, eps2);
    else if (v == 3) e = cudaLaunchKernelEx(&cfg, dual_tail_reg_kernel<3>, resid, src, out, w1, w2, n, eps1, eps2);
    else e = cudaLaunchKernelEx(&cfg, dual_tail_kernel, resid, src, out, w1, w2, n, eps1, eps2);
    if (e != cudaSuccess) return cuda_fail(e, "dual_tail: cudaLaunchKernelEx");
    return check_launch("dual_tail");
}

int launch_kv_store(uint16_t* key, uint16_t* value, const float* k, const float* v,
                    int64_t kv_dim, int64_t head_dim, int head_major, int64_t capacity,
                    int64_t phys_of_first, int64_t src_first, int64_t nrows, cudaStream_t s) {
    const int64_t total = nrows * kv_dim;
    if (total == 0) return MUSER_OK;
    const int bs = 256;
    const int64_t grid = std::min<int64_t>((total + bs - 1) / bs, static_cast<int64_t>(sm_count()) * 8);
    kv_store_kernel<<<static_cast<unsigned>(grid), bs, 0, s>>>(
        key, value, k, v, kv_dim, head_dim, head_major, capacity, phys_of_first, src_first, nrows);
    return check_launch("kv_store");
}

int launch_kv_window(uint16_t* key, uint16_t* value, uint16_t* k_rows, uint16_t* v_rows,
                     int64_t kv_dim, int64_t head_dim, int head_major, int64_t capacity,
                     int64_t phys0, int64_t count, bool to_plane, cudaStream_t s) {
    if (count == 0) return MUSER_OK;
    const auto a16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; };
    const bool vec = kv_dim % 8 == 0 && (!head_major || head_dim % 8 == 0) && a16(key) &&
                     a16(value) && a16(k_rows) && a16(v_rows);
    const int bs = 256;
    if (vec) {
        // one warp per row, two rows per warp per pass
        const int64_t warps = (count + 1) / 2;
        const int64_t grid = std::min<int64_t>((warps * 32 + bs - 1) / bs, static_cast<int64_t>(sm_count()) * 8);
        const unsigned g = static_cast<unsigned>(grid);
        const int kd = static_cast<int>(kv_dim), hd = static_cast<int>(head_dim);
        if (to_plane)
            kv_window_rows_kernel<true><<<g, bs, 0, s>>>(key, value, k_rows, v_rows, kd, hd, head_major,
                                                         capacity, phys0, count);
        else
            kv_window_rows_kernel<false><<<g, bs, 0, s>>>(key, value, k_rows, v_rows, kd, hd, head_major,
                                                          capacity, phys0, count);
        return check_launch("kv_window");
    }
    const int64_t total = count * kv_dim;
    const int64_t grid = std::min<int64_t>((total + bs - 1) / bs, static_cast<int64_t>(sm_count()) * 8);
    const unsigned g = static_cast<unsigned>(grid);
    if (to_plane)
        kv_window_kernel<true><<<g, bs, 0, s>>>(key, value, k_rows, v_rows, kv_dim, head_dim,
                                                  head_major, capacity, phys0, count);
    else
        kv_window_kernel<false><<<g, bs, 0, s>>>(key, value, k_rows, v_rows, kv_dim, head_dim,
                                                   head_major, capacity, phys0, count);
    return check_launch("kv_window");
}

int launch_occupy(int ctas, int64_t microseconds, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(occupy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kOccupySmemBytes);
    if (e != cudaSuccess) return cuda_fail(e, "occupy: cudaFuncSetAttribute");
    occupy_kernel<<<ctas, 32, kOccupySmemBytes, s>>>(static_cast<uint64_t>(microseconds) * 1000ull);
    return check_launch("occupy");
}

int launch_spin(int64_t microseconds, cudaStream_t s) {
    spin_kernel<<<1, 1, 0, s>>>(static_cast<uint64_t>(microseconds) * 1000ull);
    return check_launch("spin");
}

}  // namespace muser
