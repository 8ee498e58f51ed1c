// api.cu -- the C ABI of libmuser (declared in include/muser.h): argument
// validation on the host, then launches on the caller's stream.  Nothing here
// allocates device memory.
#include <time.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace muser {

static thread_local char g_err[512];

int set_error(int status, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof g_err, fmt, ap);
    va_end(ap);
    return status;
}
void clear_error() { g_err[0] = 0; }
int cuda_fail(cudaError_t e, const char* what) {
    return set_error(MUSER_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}
int check_launch(const char* what) {
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MUSER_OK : cuda_fail(e, what);
}

namespace {
constexpr int kMaxDev = 64;
std::mutex g_attr_mu;
int g_sm[kMaxDev] = {0};
int g_smem[kMaxDev] = {0};

int device_attr(int* cache, cudaDeviceAttr attr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
    std::lock_guard<std::mutex> lk(g_attr_mu);
    if (cache[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess) return -1;
        cache[dev] = v;
    }
    return cache[dev];
}

// The FFN, tail, group and LM-head calls take Q4_K and Q6_K; the plain
// matvec and dequantisation take Q5_K as well.
bool known_qtype(int q) { return q == MUSER_Q4_K || q == MUSER_Q6_K; }
bool matvec_qtype(int q) { return known_qtype(q) || q == MUSER_Q5_K; }
size_t block_bytes_of(int q) {
    return q == MUSER_Q4_K ? static_cast<size_t>(kQ4KBytes)
                           : q == MUSER_Q5_K ? static_cast<size_t>(kQ5KBytes)
                                             : (q == MUSER_Q6_K ? static_cast<size_t>(kQ6KBytes) : 0);
}

// Shared checks of a quantized matrix operand.
int check_matrix(const char* fn, int qtype, const void* W, int64_t rows, int64_t cols,
                 bool allow_q5 = false) {
    if (!(allow_q5 ? matvec_qtype(qtype) : known_qtype(qtype)))
        return set_error(MUSER_ERR_UNSUPPORTED, "%s: unsupported quant type %d (Q4_K=12, %sQ6_K=14)", fn,
                         qtype, allow_q5 ? "Q5_K=13, " : "");
    if (W == nullptr) return set_error(MUSER_ERR_INVALID_ARG, "%s: weight pointer is NULL", fn);
    if (rows < 1 || rows > (int64_t{1} << 31))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: rows = %lld out of range", fn, (long long)rows);
    if (cols < kQK || cols % kQK != 0 || cols > (int64_t{1} << 28))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: cols = %lld must be a positive multiple of 256", fn, (long long)cols);
    if (!is_aligned(W, 16))
        return set_error(MUSER_ERR_MISALIGNED, "%s: weight pointer not 16-byte aligned", fn);
    return MUSER_OK;
}

int check_f32(const char* fn, const char* name, const void* p) {
    if (p == nullptr) return set_error(MUSER_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
    if (!is_aligned(p, 16)) return set_error(MUSER_ERR_MISALIGNED, "%s: %s not 16-byte aligned", fn, name);
    return MUSER_OK;
}

// The ticket scratch of the fused layer-boundary calls.
int check_boundary_scratch(const char* fn, const void* scratch, size_t scratch_bytes) {
    MUSER_TRY(check_f32(fn, "scratch", scratch));
    if (scratch_bytes < MUSER_BOUNDARY_SCRATCH_BYTES)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: scratch_bytes %zu < %u", fn, scratch_bytes,
                         static_cast<unsigned>(MUSER_BOUNDARY_SCRATCH_BYTES));
    return MUSER_OK;
}

// The updated-residual output of the fused boundary calls: null (in place,
// the ticket scratch required) or a row distinct from the other operands.
int check_residual_out(const char* fn, const float* residual_out, const float* residual, const float* projected,
                       const float* x_out, const void* scratch, size_t scratch_bytes) {
    if (residual_out == nullptr) return check_boundary_scratch(fn, scratch, scratch_bytes);
    MUSER_TRY(check_f32(fn, "residual_out", residual_out));
    if (residual_out == residual || residual_out == projected || residual_out == x_out)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: residual_out must be distinct from residual, projected and x_out",
                         fn);
    return MUSER_OK;
}

int check_M(const char* fn, int M) {
    if (M < 1 || M > MUSER_MAX_M)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: M = %d outside 1..%d", fn, M, MUSER_MAX_M);
    return MUSER_OK;
}


// Scratch of the one-token down + tail kernel: its ticket, then (from byte
// kTailPartOffset) the blocks' sums of projected^2.
constexpr size_t kTailPartOffset = 256;
constexpr size_t kScratchBytes = kTailPartOffset + sizeof(float) * kMv1TailParts;
// Route one-token calls to the tensor-core kernel (mvt) instead of mv1.
// mv1 measures faster for one row of x (one launch and inside the stack).
constexpr bool kTensorCoreM1 = false;

// Scratch of the fused down projection + tail: the CUDA-core kernel's ticket
// and per-block sums (kScratchBytes), then the tensor-core kernel's tickets
// and partial sums.
// The bound holds for every row length (a one-block Q6_K row has the most
// tiles).
size_t down_scratch_bytes(int64_t hidden, int M) {
    return kScratchBytes + mvt_split_scratch_bytes(MUSER_Q6_K, 1, hidden, kQK, M);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Workspace {
    float* xa;
    float* xb;
    float* mid;
    float* proj;
    float* resid_ws;   // the second buffer of the residual relay
    void* mvs;         // the one-launch stack's sync words and input records
    void* scratch;     // down + tail scratch, down_scratch_bytes(hidden)
    void* gu_scratch;  // gate/up tensor-core scratch (null if the shape has none)
    size_t scratch_bytes;
    size_t total;
};
Workspace carve(void* base, int64_t hidden, int64_t ffn, int M) {
    Workspace w{};
    uint8_t* p = static_cast<uint8_t*>(base);
    size_t off = 0;
    const size_t hb = round_up(sizeof(float) * static_cast<size_t>(hidden) * M, 256);
    const size_t fb = round_up(sizeof(float) * static_cast<size_t>(ffn) * M, 256);
    w.xa = reinterpret_cast<float*>(p + off);
    off += hb;
    w.xb = reinterpret_cast<float*>(p + off);
    off += hb;
    w.mid = reinterpret_cast<float*>(p + off);
    off += fb;
    w.proj = reinterpret_cast<float*>(p + off);
    off += hb;
    w.resid_ws = reinterpret_cast<float*>(p + off);
    off += hb;
    w.mvs = p + off;
    off += round_up(mvs_scratch_bytes(hidden, ffn), 256);
    w.scratch = p + off;
    // with several rows of x, also room for the tensor-core kernel's B image
    // of a down projection over ffn inputs
    size_t down = down_scratch_bytes(hidden, M);
    if (M > 1)
        for (int qt : {MUSER_Q4_K, MUSER_Q6_K})
            down = std::max(down, kScratchBytes + mvt_scratch_bytes(qt, 1, hidden, ffn, M));
    w.scratch_bytes = round_up(down, 256);
    off += w.scratch_bytes;
    const size_t gu = mvt_scratch_bytes(MUSER_Q4_K, 2, ffn, hidden, M);
    w.gu_scratch = gu ? p + off : nullptr;
    off += round_up(gu, 256);
    w.total = off;
    return w;
}

// The gate/up launch that follows a multi-row down projection + tail in a
// stack: its tail can also write that launch's B image.
struct NextImage {
    int qtype;
    void* scratch;
    size_t scratch_bytes;
    bool* built;  // set when the tail wrote it
};

// Launch the matvec + tail on validated arguments.
int down_tail_launch(int qtype, const void* Wdown, int64_t hidden, int64_t ffn, const float* mid,
                     int M, float* projected, float* residual, float* out, const float* w1,
                     const float* w2, float eps1, float eps2, void* scratch, size_t scratch_bytes,
                     cudaStream_t s, const NextImage* next = nullptr) {
    if (next != nullptr) *next->built = false;
    // One token: the CUDA-core kernel mv1 is measured faster than the
    // tensor-core kernel on this shape, so it takes M = 1.
    const bool tc_ok = mvt_supported(qtype, 1, hidden, ffn, M);
    const bool tc_fits = tc_ok && scratch_bytes >= kScratchBytes + mvt_split_scratch_bytes(qtype, 1, hidden, ffn, M);
    if (M > 1 && tc_ok) {
        // several rows: the tensor-core matvec into `projected`, then the tail
        // per row.  With room for its partial sums the matvec spreads its
        // units over every SM; otherwise each SM takes whole row tiles.
        MvtArgs a{};
        a.W[0] = static_cast<const uint8_t*>(Wdown);
        a.W[1] = a.W[0];
        a.rows = hidden;
        a.nsb = static_cast<int>(ffn / kQK);
        a.x = mid;
        a.M = M;
        a.y = projected;
        MUSER_TRY(launch_mvt(qtype, kEpiStore, a, tc_fits ? static_cast<uint8_t*>(scratch) + kScratchBytes : nullptr,
                             tc_fits ? scratch_bytes - kScratchBytes : 0, s));
        if (next != nullptr) {
            const int r = launch_mvt_tail_image(next->qtype, 2, ffn, hidden, M, residual, projected, out, w1, w2, eps1,
                                                eps2, next->scratch, next->scratch_bytes, s);
            if (r != MUSER_ERR_UNSUPPORTED) {
                *next->built = r == MUSER_OK;
                return r;
            }
        }
        return launch_dual_tail(residual, projected, out, w1, w2, static_cast<int>(hidden), M, eps1, eps2, s);
    }
    if (kTensorCoreM1 && M == 1 && tc_fits) {
        MvtArgs a{};
        a.W[0] = static_cast<const uint8_t*>(Wdown);
        a.W[1] = a.W[0];
        a.rows = hidden;
        a.nsb = static_cast<int>(ffn / kQK);
        a.x = mid;
        a.y = projected;
        a.resid = residual;
        a.out = out;
        a.w1 = w1;
        a.w2 = w2;
        a.eps1 = eps1;
        a.eps2 = eps2;
        a.M = 1;
        return launch_mvt(qtype, kEpiTail, a, static_cast<uint8_t*>(scratch) + kScratchBytes, scratch_bytes - kScratchBytes,
                          s);
    }
    if (M == 1 && mv1_supported(qtype, ffn)) {
        Mv1Args a{};
        a.W[0] = static_cast<const uint8_t*>(Wdown);
        a.W[1] = a.W[0];
        a.rows = hidden;
        a.nsb = static_cast<int>(ffn / kQK);
        a.x = mid;
        a.y0 = projected;
        a.resid = residual;
        a.out = out;
        a.w1 = w1;
        a.w2 = w2;
        a.eps1 = eps1;
        a.eps2 = eps2;
        a.ticket = static_cast<unsigned*>(scratch);
        // with room for the blocks' sums the tail skips its first pass
        a.tail_part = scratch_bytes >= kScratchBytes
                          ? reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + kTailPartOffset)
                          : nullptr;
        return launch_mv1(qtype, 1, kEpiTail, a, s);
    }
    MvMArgs a{};
    a.W[0] = static_cast<const uint8_t*>(Wdown);
    a.W[1] = a.W[0];
    a.rows = hidden;
    a.nsb = static_cast<int>(ffn / kQK);
    a.x = mid;
    a.M = M;
    a.y0 = projected;
    MUSER_TRY(launch_mvM(qtype, 1, kEpiStore, a, s));
    return launch_dual_tail(residual, projected, out, w1, w2, static_cast<int>(hidden), M, eps1,
                            eps2, s);
}

// Whether muser_ffn_stack runs the whole stack in one persistent launch.
bool stack_one_launch(const muser_ffn_layer* layers, int n_layers, int64_t hidden, int64_t ffn, int M) {
    if (M != 1 || n_layers < 1) return false;
    for (int l = 0; l < n_layers; ++l)
        if (layers[l].gate_up_qtype != MUSER_Q4_K || layers[l].down_qtype != MUSER_Q6_K) return false;
    return mvs_supported(MUSER_Q4_K, MUSER_Q6_K, hidden, ffn, n_layers, M);
}

// The tail of the previous layer fused into this layer's gate/up kernel.
bool gate_up_tail_fused(int qtype, int64_t hidden, int M) {
    return M == 1 && mv1_tail_prologue_supported(qtype, hidden);
}

int gate_up_launch(int qtype, const void* Wg, const void* Wu, int64_t ffn, int64_t hidden,
                   const float* x, int M, float* mid, void* scratch, cudaStream_t s, bool image_ready = false);

// The tail with its residual going to resid_out (distinct) or, when that is
// null, updated in place.
int dual_tail_to(float* residual, float* resid_out, const float* src, float* out, const float* w1, const float* w2,
                 int n, int M, float eps1, float eps2, cudaStream_t s) {
    if (resid_out != nullptr) {
        const cudaError_t e = cudaMemcpyAsync(resid_out, residual, sizeof(float) * static_cast<size_t>(n) * M,
                                              cudaMemcpyDeviceToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(residual)");
        residual = resid_out;
    }
    return launch_dual_tail(residual, src, out, w1, w2, n, M, eps1, eps2, s);
}

// The layer boundary (previous tail, then gate/up) on validated arguments.
// resid_out: a separate output row for the updated residual, or null (in
// place; ticket: MUSER_BOUNDARY_SCRATCH_BYTES of zero-filled caller scratch).
int gate_up_tail_launch(int qtype, const void* Wg, const void* Wu, int64_t ffn, int64_t hidden,
                        const float* projected, float* residual, float* resid_out, const float* w1, const float* w2,
                        float eps1, float eps2, float* x_out, int M, float* mid, unsigned* ticket,
                        cudaStream_t s) {
    if (gate_up_tail_fused(qtype, hidden, M)) {
        Mv1Args a{};
        a.W[0] = static_cast<const uint8_t*>(Wg);
        a.W[1] = static_cast<const uint8_t*>(Wu);
        a.rows = ffn;
        a.nsb = static_cast<int>(hidden / kQK);
        a.x = projected;
        a.y0 = mid;
        a.resid = residual;
        a.out = x_out;
        a.w1 = w1;
        a.w2 = w2;
        a.eps1 = eps1;
        a.eps2 = eps2;
        a.resid_out = resid_out;
        a.xticket = ticket;
        return launch_mv1(qtype, 2, kEpiSiluMul, a, s, kXTail);
    }
    MUSER_TRY(dual_tail_to(residual, resid_out, projected, x_out, w1, w2, static_cast<int>(hidden), M, eps1, eps2, s));
    return gate_up_launch(qtype, Wg, Wu, ffn, hidden, x_out, M, mid, nullptr, s);
}

// scratch: the tensor-core kernel's even-split scratch, or null (whole tiles).
int gate_up_launch(int qtype, const void* Wg, const void* Wu, int64_t ffn, int64_t hidden,
                   const float* x, int M, float* mid, void* scratch, cudaStream_t s, bool image_ready) {
    if ((M > 1 || kTensorCoreM1) && mvt_supported(qtype, 2, ffn, hidden, M)) {
        MvtArgs a{};
        a.W[0] = static_cast<const uint8_t*>(Wg);
        a.W[1] = static_cast<const uint8_t*>(Wu);
        a.rows = ffn;
        a.nsb = static_cast<int>(hidden / kQK);
        a.x = x;
        a.M = M;
        a.y = mid;
        a.image_ready = image_ready ? 1 : 0;  // written by the previous layer's tail
        return launch_mvt(qtype, kEpiSiluMul, a, scratch, scratch ? mvt_scratch_bytes(qtype, 2, ffn, hidden, M) : 0, s);
    }
    if (M == 1 && mv1_supported(qtype, hidden)) {
        Mv1Args a{};
        a.W[0] = static_cast<const uint8_t*>(Wg);
        a.W[1] = static_cast<const uint8_t*>(Wu);
        a.rows = ffn;
        a.nsb = static_cast<int>(hidden / kQK);
        a.x = x;
        a.y0 = mid;
        return launch_mv1(qtype, 2, kEpiSiluMul, a, s);
    }
    MvMArgs a{};
    a.W[0] = static_cast<const uint8_t*>(Wg);
    a.W[1] = static_cast<const uint8_t*>(Wu);
    a.rows = ffn;
    a.nsb = static_cast<int>(hidden / kQK);
    a.x = x;
    a.M = M;
    a.y0 = mid;
    return launch_mvM(qtype, 2, kEpiSiluMul, a, s);
}

}  // namespace

int sm_count() { return device_attr(g_sm, cudaDevAttrMultiProcessorCount); }
int max_smem_optin() { return device_attr(g_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin); }

// Scratch of muser_qmatvec_residual_dual_rmsnorm_static: the tail's
// completion counter in the first kStaticCounterBytes, then the projected
// rows.  It is part of the library image, so every GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[MUSER_STATIC_SCRATCH_BYTES];

namespace {
constexpr size_t kStaticCounterBytes = 256;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDev] = {nullptr};

// Device address of g_static_scratch on the current device.  The lookup
// runs once per device, with that device current; later calls reuse it.
int static_scratch(const char* fn, unsigned char** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDev)
        return set_error(MUSER_ERR_UNSUPPORTED, "%s: device %d beyond the library's %d", fn, dev, kMaxDev);
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (g_static_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
        if (p == nullptr) return set_error(MUSER_ERR_CUDA, "%s: static scratch has no device address", fn);
        g_static_ptr[dev] = p;
    }
    *ptr = static_cast<unsigned char*>(g_static_ptr[dev]);
    return MUSER_OK;
}
}  // namespace

}  // namespace muser

using namespace muser;

extern "C" {

int muser_version(void) { return MUSER_ABI_VERSION; }

const char* muser_last_error(void) { return g_err; }

size_t muser_block_bytes(int qtype) { return block_bytes_of(qtype); }

size_t muser_matrix_bytes(int qtype, int64_t rows, int64_t cols) {
    if (!matvec_qtype(qtype) || rows < 0 || cols < 0 || cols % kQK) return 0;
    return static_cast<size_t>(rows) * static_cast<size_t>(cols / kQK) * block_bytes_of(qtype);
}

int muser_dequantize(int qtype, const void* W, int64_t rows, int64_t cols, float* out,
                     void* stream) {
    clear_error();
    MUSER_TRY(check_matrix("muser_dequantize", qtype, W, rows, cols, true));
    MUSER_TRY(check_f32("muser_dequantize", "out", out));
    return launch_dequantize(qtype, static_cast<const uint8_t*>(W), rows, cols, out,
                             as_stream(stream));
}

int muser_qmatvec(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, int M,
                  float* y, void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec";
    MUSER_TRY(check_matrix(fn, qtype, W, rows, cols, true));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "y", y));
    if (M == 1 && mv1_supported(qtype, cols)) {
        Mv1Args a{};
        a.W[0] = static_cast<const uint8_t*>(W);
        a.W[1] = a.W[0];
        a.rows = rows;
        a.nsb = static_cast<int>(cols / kQK);
        a.x = x;
        a.y0 = y;
        return launch_mv1(qtype, 1, kEpiStore, a, as_stream(stream));
    }
    if (mvt_supported(qtype, 1, rows, cols, M)) {
        // several rows of x: the tensor-core kernel (whole row tiles per CTA)
        MvtArgs t{};
        t.W[0] = static_cast<const uint8_t*>(W);
        t.W[1] = t.W[0];
        t.rows = rows;
        t.nsb = static_cast<int>(cols / kQK);
        t.x = x;
        t.M = M;
        t.y = y;
        return launch_mvt(qtype, kEpiStore, t, nullptr, 0, as_stream(stream));
    }
    MvMArgs a{};
    a.W[0] = static_cast<const uint8_t*>(W);
    a.W[1] = a.W[0];
    a.rows = rows;
    a.nsb = static_cast<int>(cols / kQK);
    a.x = x;
    a.M = M;
    a.y0 = y;
    return launch_mvM(qtype, 1, kEpiStore, a, as_stream(stream));
}

size_t muser_qmatvec_scratch_bytes(int qtype, int64_t rows, int64_t cols, int M) {
    // one row of x runs on the one-token kernel, which needs none
    if (M < 2 || M > MUSER_MAX_M || !mvt_supported(qtype, 1, rows, cols, M)) return 0;
    return mvt_scratch_bytes(qtype, 1, rows, cols, M);
}

int muser_qmatvec_scratch(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, int M,
                          float* y, void* scratch, size_t scratch_bytes, void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_scratch";
    MUSER_TRY(check_matrix(fn, qtype, W, rows, cols, true));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "y", y));
    const size_t need = muser_qmatvec_scratch_bytes(qtype, rows, cols, M);
    if (need == 0) return muser_qmatvec(qtype, W, rows, cols, x, M, y, stream);
    MUSER_TRY(check_f32(fn, "scratch", scratch));
    if (scratch_bytes < need)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: scratch_bytes %zu < %zu", fn, scratch_bytes, need);
    // several rows of x: the tensor-core kernel with the (tile, super-block)
    // units spread evenly over the SMs
    MvtArgs t{};
    t.W[0] = static_cast<const uint8_t*>(W);
    t.W[1] = t.W[0];
    t.rows = rows;
    t.nsb = static_cast<int>(cols / kQK);
    t.x = x;
    t.M = M;
    t.y = y;
    return launch_mvt(qtype, kEpiStore, t, scratch, scratch_bytes, as_stream(stream));
}

int muser_rms_norm(const float* x, const float* w, float* out, int n, int M, float eps,
                   void* stream) {
    clear_error();
    const char* fn = "muser_rms_norm";
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "w", w));
    MUSER_TRY(check_f32(fn, "out", out));
    if (n < 4 || n % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: n = %d must be a positive multiple of 4", fn, n);
    if (M < 1 || M > 65535) return set_error(MUSER_ERR_INVALID_ARG, "%s: M = %d out of range", fn, M);
    if (!(eps > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    return launch_rms_norm(x, w, out, n, M, eps, as_stream(stream));
}

int muser_silu_mul(const float* a, const float* b, float* out, int64_t n, void* stream) {
    clear_error();
    const char* fn = "muser_silu_mul";
    if (n < 0) return set_error(MUSER_ERR_INVALID_ARG, "%s: n < 0", fn);
    if (n == 0) return MUSER_OK;
    if (!a || !b || !out) return set_error(MUSER_ERR_INVALID_ARG, "%s: NULL pointer", fn);
    if (!is_aligned(a, 4) || !is_aligned(b, 4) || !is_aligned(out, 4))
        return set_error(MUSER_ERR_MISALIGNED, "%s: pointers must be 4-byte aligned", fn);
    return launch_silu_mul(a, b, out, n, as_stream(stream));
}

int muser_ffn_gate_up_silu(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                           int64_t hidden, const float* x, int M, float* mid, void* stream) {
    clear_error();
    const char* fn = "muser_ffn_gate_up_silu";
    MUSER_TRY(check_matrix(fn, qtype, Wg, ffn, hidden));
    MUSER_TRY(check_matrix(fn, qtype, Wu, ffn, hidden));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "mid", mid));
    return gate_up_launch(qtype, Wg, Wu, ffn, hidden, x, M, mid, nullptr, as_stream(stream));
}

size_t muser_gate_up_scratch_bytes(int qtype, int64_t ffn, int64_t hidden, int M) {
    if (M < 1 || M > MUSER_MAX_M) return 0;
    return mvt_scratch_bytes(qtype, 2, ffn, hidden, M);
}

int muser_ffn_gate_up_silu_scratch(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                                   int64_t hidden, const float* x, int M, float* mid, void* scratch,
                                   size_t scratch_bytes, void* stream) {
    clear_error();
    const char* fn = "muser_ffn_gate_up_silu_scratch";
    MUSER_TRY(check_matrix(fn, qtype, Wg, ffn, hidden));
    MUSER_TRY(check_matrix(fn, qtype, Wu, ffn, hidden));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "mid", mid));
    const size_t need = mvt_scratch_bytes(qtype, 2, ffn, hidden, M);
    if (need > 0) {
        MUSER_TRY(check_f32(fn, "scratch", scratch));
        if (scratch_bytes < need)
            return set_error(MUSER_ERR_INVALID_ARG, "%s: scratch_bytes %zu < %zu", fn, scratch_bytes, need);
    }
    return gate_up_launch(qtype, Wg, Wu, ffn, hidden, x, M, mid, need > 0 ? scratch : nullptr, as_stream(stream));
}

int muser_ffn_gate_up_silu_tail(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                                int64_t hidden, const float* projected, float* residual, float* residual_out,
                                const float* w1, const float* w2, float eps1, float eps2,
                                float* x_out, int M, float* mid, void* scratch, size_t scratch_bytes,
                                void* stream) {
    clear_error();
    const char* fn = "muser_ffn_gate_up_silu_tail";
    MUSER_TRY(check_matrix(fn, qtype, Wg, ffn, hidden));
    MUSER_TRY(check_matrix(fn, qtype, Wu, ffn, hidden));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "projected", projected));
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "w1", w1));
    MUSER_TRY(check_f32(fn, "w2", w2));
    MUSER_TRY(check_f32(fn, "x_out", x_out));
    MUSER_TRY(check_f32(fn, "mid", mid));
    if (hidden % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: hidden must be a multiple of 4", fn);
    if (!(eps1 > 0.0f) || !(eps2 > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    if (x_out == residual || x_out == projected || projected == residual)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: projected, residual and x_out must be distinct", fn);
    MUSER_TRY(check_residual_out(fn, residual_out, residual, projected, x_out, scratch, scratch_bytes));
    return gate_up_tail_launch(qtype, Wg, Wu, ffn, hidden, projected, residual, residual_out, w1, w2, eps1, eps2,
                               x_out, M, mid, static_cast<unsigned*>(scratch), as_stream(stream));
}

// Validation shared by the two group calls.
static int check_group(const char* fn, int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                       const float* x, int M, float* const* y) {
    if (n < 1 || n > kMv1MaxSeg || W == nullptr || rows == nullptr || y == nullptr)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: need 1..%d matrices with their rows and outputs", fn, kMv1MaxSeg);
    for (int i = 0; i < n; ++i) {
        MUSER_TRY(check_matrix(fn, qtype, W[i], rows[i], cols));
        MUSER_TRY(check_f32(fn, "y", y[i]));
    }
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    return MUSER_OK;
}

// Scratch of the grouped tensor-core launch (0: the group does not take it).
static size_t group_scratch_bytes(int qtype, int n, const int64_t* rows, int64_t cols, int M) {
    if (qtype != MUSER_Q4_K || M < 2 || M > MUSER_MAX_M || n < 1 || n > kMvtMaxSeg || rows == nullptr) return 0;
    for (int i = 0; i < n; ++i)
        if (rows[i] < 1) return 0;
    const int64_t vrows = mvt_group_rows(n, rows);
    if (!mvt_supported(qtype, 1, vrows, cols, M)) return 0;
    return mvt_scratch_bytes(qtype, 1, vrows, cols, M);
}

// One launch over the group's rows when one row of x, Q4_K (rows of whole
// 16-byte units) and the one-token kernel fit; with 2..16 rows of x, Q4_K and
// enough scratch, one tensor-core launch over the group's row tiles;
// otherwise one call per matrix.
static int group_launch(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                        int M, float* const* y, const float* projected, float* residual, float* resid_out,
                        const float* w1, const float* w2, float eps1, float eps2, float* x_out, unsigned* ticket,
                        cudaStream_t s, void* gscratch = nullptr, size_t gscratch_bytes = 0) {
    const bool tail = projected != nullptr;
    const bool fused = M == 1 && qtype == MUSER_Q4_K &&
                       (tail ? mv1_tail_prologue_supported(qtype, cols) : mv1_supported(qtype, cols));
    if (fused) {
        Mv1Args a{};
        a.nseg = n;
        int64_t r = 0;
        for (int i = 0; i < n; ++i) {
            a.segW[i] = static_cast<const uint8_t*>(W[i]);
            a.seg0[i] = r;
            a.segY[i] = y[i];
            r += rows[i];
        }
        a.seg0[n] = r;
        a.rows = r;
        a.nsb = static_cast<int>(cols / kQK);
        a.x = tail ? projected : x;
        if (tail) {
            a.resid = residual;
            a.out = x_out;
            a.w1 = w1;
            a.w2 = w2;
            a.eps1 = eps1;
            a.eps2 = eps2;
            a.resid_out = resid_out;
            a.xticket = ticket;
        }
        return launch_mv1(qtype, 1, kEpiStore, a, s, tail ? kXTail : kXMemory);
    }
    const float* xin = x;
    const size_t gneed = group_scratch_bytes(qtype, n, rows, cols, M);
    const bool grouped = gneed > 0 && gscratch != nullptr && gscratch_bytes >= gneed;
    bool image_ready = false;
    if (tail) {
        // several rows: the tail, which also builds the grouped launch's B
        // image of its output when that launch takes one
        int r = MUSER_ERR_UNSUPPORTED;
        if (grouped) {
            float* res = residual;
            if (resid_out != nullptr) {
                const cudaError_t e = cudaMemcpyAsync(resid_out, residual, sizeof(float) * static_cast<size_t>(cols) * M,
                                                      cudaMemcpyDeviceToDevice, s);
                if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync(residual)");
                res = resid_out;
            }
            r = launch_mvt_tail_image(qtype, 1, mvt_group_rows(n, rows), cols, M, res, projected, x_out, w1, w2, eps1,
                                      eps2, gscratch, gscratch_bytes, s);
            if (r != MUSER_OK && r != MUSER_ERR_UNSUPPORTED) return r;
            if (r == MUSER_ERR_UNSUPPORTED) r = launch_dual_tail(res, projected, x_out, w1, w2, static_cast<int>(cols),
                                                                 M, eps1, eps2, s);
            else image_ready = true;
            MUSER_TRY(r);
        } else {
            MUSER_TRY(dual_tail_to(residual, resid_out, projected, x_out, w1, w2, static_cast<int>(cols), M, eps1, eps2,
                                   s));
        }
        xin = x_out;
    }
    if (grouped) {
        MvtArgs t{};
        t.nseg = n;
        for (int i = 0; i < n; ++i) {
            t.seg_W[i] = static_cast<const uint8_t*>(W[i]);
            t.seg_rows[i] = rows[i];
            t.seg_y[i] = y[i];
        }
        t.W[0] = t.W[1] = t.seg_W[0];
        t.rows = mvt_group_rows(n, rows);
        t.nsb = static_cast<int>(cols / kQK);
        t.x = xin;
        t.M = M;
        t.image_ready = image_ready ? 1 : 0;
        return launch_mvt(qtype, kEpiStore, t, gscratch, gscratch_bytes, s);
    }
    for (int i = 0; i < n; ++i) MUSER_TRY(muser_qmatvec(qtype, W[i], rows[i], cols, xin, M, y[i], s));
    return MUSER_OK;
}

size_t muser_qmatvec_group_scratch_bytes(int qtype, int n, const int64_t* rows, int64_t cols, int M) {
    return group_scratch_bytes(qtype, n, rows, cols, M);
}

int muser_qmatvec_group_scratch(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                                const float* x, int M, float* const* y, void* scratch, size_t scratch_bytes,
                                void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_group_scratch";
    MUSER_TRY(check_group(fn, qtype, n, W, rows, cols, x, M, y));
    const size_t need = group_scratch_bytes(qtype, n, rows, cols, M);
    if (need > 0) {
        MUSER_TRY(check_f32(fn, "scratch", scratch));
        if (scratch_bytes < need)
            return set_error(MUSER_ERR_INVALID_ARG, "%s: scratch_bytes %zu < %zu", fn, scratch_bytes, need);
    }
    return group_launch(qtype, n, W, rows, cols, x, M, y, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f, 0.f,
                        nullptr, nullptr, as_stream(stream), scratch, scratch_bytes);
}

int muser_qmatvec_group(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols, const float* x,
                        int M, float* const* y, void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_group";
    MUSER_TRY(check_group(fn, qtype, n, W, rows, cols, x, M, y));
    return group_launch(qtype, n, W, rows, cols, x, M, y, nullptr, nullptr, nullptr, nullptr, nullptr, 0.f, 0.f,
                        nullptr, nullptr, as_stream(stream));
}

int muser_qmatvec_group_tail(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                             const float* projected, float* residual, float* residual_out, const float* w1,
                             const float* w2, float eps1, float eps2, float* x_out, int M, float* const* y,
                             void* scratch, size_t scratch_bytes, void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_group_tail";
    MUSER_TRY(check_group(fn, qtype, n, W, rows, cols, x_out, M, y));
    MUSER_TRY(check_f32(fn, "projected", projected));
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "w1", w1));
    MUSER_TRY(check_f32(fn, "w2", w2));
    if (cols % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: cols must be a multiple of 4", fn);
    if (!(eps1 > 0.0f) || !(eps2 > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    if (x_out == residual || x_out == projected || projected == residual)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: projected, residual and x_out must be distinct", fn);
    MUSER_TRY(check_residual_out(fn, residual_out, residual, projected, x_out, scratch, scratch_bytes));
    // several rows of x: the tail runs on its own, and scratch of
    // muser_qmatvec_group_scratch_bytes() or more takes the grouped launch
    return group_launch(qtype, n, W, rows, cols, nullptr, M, y, projected, residual, residual_out, w1, w2, eps1, eps2,
                        x_out, static_cast<unsigned*>(scratch), as_stream(stream), M > 1 ? scratch : nullptr,
                        M > 1 ? scratch_bytes : 0);
}

int muser_scale_softcap(float* logits, int64_t n, float scale, float cap, void* stream) {
    clear_error();
    const char* fn = "muser_scale_softcap";
    MUSER_TRY(check_f32(fn, "logits", logits));
    if (n < 0) return set_error(MUSER_ERR_INVALID_ARG, "%s: n must be >= 0", fn);
    if (!(cap > 0.0f) || !std::isfinite(cap) || !std::isfinite(scale))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: cap must be > 0 and finite, scale finite", fn);
    return launch_scale_softcap(logits, n, scale, cap, as_stream(stream));
}

int muser_lm_head(int qtype, const void* W, int64_t vocab, int64_t hidden, const float* x, int M, float* logits,
                  float scale, float cap, void* stream) {
    clear_error();
    const char* fn = "muser_lm_head";
    MUSER_TRY(check_matrix(fn, qtype, W, vocab, hidden));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "x", x));
    MUSER_TRY(check_f32(fn, "logits", logits));
    if (!(cap > 0.0f) || !std::isfinite(cap) || !std::isfinite(scale))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: cap must be > 0 and finite, scale finite", fn);
    const cudaStream_t s = as_stream(stream);
    if (M == 1 && mv1_supported(qtype, hidden)) {
        // one row of x: the cap is the one-token kernel's epilogue
        Mv1Args a{};
        a.W[0] = static_cast<const uint8_t*>(W);
        a.W[1] = a.W[0];
        a.rows = vocab;
        a.nsb = static_cast<int>(hidden / kQK);
        a.x = x;
        a.y0 = logits;
        a.scale = scale;
        a.cap = cap;
        return launch_mv1(qtype, 1, kEpiSoftcap, a, s);
    }
    MUSER_TRY(muser_qmatvec(qtype, W, vocab, hidden, x, M, logits, stream));
    return launch_scale_softcap(logits, vocab * M, scale, cap, s);
}

int muser_fused_residual_dual_rmsnorm(float* residual, const float* src, float* out,
                                      const float* w1, const float* w2, int n, int M, float eps1,
                                      float eps2, void* stream) {
    clear_error();
    const char* fn = "muser_fused_residual_dual_rmsnorm";
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "src", src));
    MUSER_TRY(check_f32(fn, "out", out));
    MUSER_TRY(check_f32(fn, "w1", w1));
    MUSER_TRY(check_f32(fn, "w2", w2));
    if (n < 4 || n % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: n = %d must be a positive multiple of 4", fn, n);
    if (M < 1 || M > 65535) return set_error(MUSER_ERR_INVALID_ARG, "%s: M = %d out of range", fn, M);
    if (!(eps1 > 0.0f) || !(eps2 > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    if (out == residual || out == src)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: out must not alias residual or src", fn);
    return launch_dual_tail(residual, src, out, w1, w2, n, M, eps1, eps2, as_stream(stream));
}

size_t muser_scratch_bytes(int64_t hidden, int M) {
    (void)M;
    if (hidden < 1 || M < 1 || M > MUSER_MAX_M) return kScratchBytes;
    return down_scratch_bytes(hidden, M);
}

int muser_qmatvec_residual_dual_rmsnorm(int qtype, const void* Wdown, int64_t hidden, int64_t ffn,
                                        const float* mid, int M, float* projected,
                                        float* residual, float* out, const float* w1,
                                        const float* w2, float eps1, float eps2, void* scratch,
                                        size_t scratch_bytes, void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_residual_dual_rmsnorm";
    MUSER_TRY(check_matrix(fn, qtype, Wdown, hidden, ffn));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "mid", mid));
    MUSER_TRY(check_f32(fn, "projected", projected));
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "out", out));
    MUSER_TRY(check_f32(fn, "w1", w1));
    MUSER_TRY(check_f32(fn, "w2", w2));
    MUSER_TRY(check_f32(fn, "scratch", scratch));
    if (hidden % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: hidden must be a multiple of 4", fn);
    // 256 bytes (the ticket) suffice; muser_scratch_bytes() also leaves room
    // for the blocks' sums (a shorter tail) and the tensor-core kernel
    if (scratch_bytes < kTailPartOffset)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: scratch_bytes %zu < %zu", fn, scratch_bytes, kTailPartOffset);
    if (!(eps1 > 0.0f) || !(eps2 > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    if (out == residual || out == projected || projected == residual)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: projected, residual and out must be distinct", fn);
    return down_tail_launch(qtype, Wdown, hidden, ffn, mid, M, projected, residual, out, w1, w2,
                            eps1, eps2, scratch, scratch_bytes, as_stream(stream));
}

int muser_qmatvec_residual_dual_rmsnorm_static(int qtype, const void* Wdown, int64_t hidden,
                                               int64_t ffn, const float* mid, int M,
                                               float* residual, float* out, const float* w1,
                                               const float* w2, float eps1, float eps2,
                                               void* stream) {
    clear_error();
    const char* fn = "muser_qmatvec_residual_dual_rmsnorm_static";
    MUSER_TRY(check_matrix(fn, qtype, Wdown, hidden, ffn));
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "mid", mid));
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "out", out));
    MUSER_TRY(check_f32(fn, "w1", w1));
    MUSER_TRY(check_f32(fn, "w2", w2));
    if (hidden % 4) return set_error(MUSER_ERR_INVALID_ARG, "%s: hidden must be a multiple of 4", fn);
    const size_t need = kStaticCounterBytes + sizeof(float) * static_cast<size_t>(hidden) * M;
    if (need > MUSER_STATIC_SCRATCH_BYTES)
        return set_error(MUSER_ERR_INVALID_ARG,
                         "%s: M * hidden = %lld needs %zu bytes of scratch, more than the library's "
                         "fixed %zu (M * hidden <= %zu)",
                         fn, static_cast<long long>(hidden) * M, need,
                         static_cast<size_t>(MUSER_STATIC_SCRATCH_BYTES),
                         (static_cast<size_t>(MUSER_STATIC_SCRATCH_BYTES) - kStaticCounterBytes) / sizeof(float));
    if (!(eps1 > 0.0f) || !(eps2 > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    if (out == residual) return set_error(MUSER_ERR_INVALID_ARG, "%s: out must not alias residual", fn);
    unsigned char* base = nullptr;
    MUSER_TRY(static_scratch(fn, &base));
    const cudaStream_t s = as_stream(stream);
    // The array keeps the last call's bytes: the completion counter must read
    // zero when this call's kernels start, whatever an earlier call left.
    const cudaError_t e = cudaMemsetAsync(base, 0, kStaticCounterBytes, s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(static scratch counter)");
    float* projected = reinterpret_cast<float*>(base + kStaticCounterBytes);
    return down_tail_launch(qtype, Wdown, hidden, ffn, mid, M, projected, residual, out, w1, w2,
                            eps1, eps2, base, kStaticCounterBytes, s);
}

size_t muser_ffn_workspace_bytes(int64_t hidden, int64_t ffn, int M) {
    if (hidden < 1 || ffn < 1 || M < 1) return 0;
    return carve(nullptr, hidden, ffn, M).total;
}

int muser_ffn_stack_launches(const muser_ffn_layer* layers, int n_layers, int64_t hidden, int64_t ffn, int M) {
    clear_error();
    if (layers == nullptr || n_layers < 1 || M < 1 || M > MUSER_MAX_M) return -1;
    if (stack_one_launch(layers, n_layers, hidden, ffn, M)) return 1;
    bool fused = true;
    for (int l = 0; l < n_layers && fused; ++l)
        fused = gate_up_tail_fused(layers[l].gate_up_qtype, hidden, M) && mv1_supported(layers[l].down_qtype, ffn);
    // the entry norm, two kernels per layer, and (fused boundaries) the last tail
    if (fused) return 2 + 2 * n_layers;
    if (M == 1) return 1 + 2 * n_layers;
    // several rows: gate/up, the down projection and its tail; a tensor-core
    // matvec with its B image is three launches (built before, cleared
    // after), or two when the previous layer's tail built the image
    int n = 1;
    const size_t gu_bytes = mvt_scratch_bytes(MUSER_Q4_K, 2, ffn, hidden, M);
    bool image_ready = false;
    for (int l = 0; l < n_layers; ++l) {
        const int gu = mvt_launches(layers[l].gate_up_qtype, 2, ffn, hidden, M);
        const int dn = mvt_launches(layers[l].down_qtype, 1, hidden, ffn, M);
        n += (gu > 0 ? gu - (image_ready ? 1 : 0) : 1) + (dn > 0 ? dn : 1) + 1;
        image_ready = l + 1 < n_layers && M > 1 && mvt_supported(layers[l].down_qtype, 1, hidden, ffn, M) &&
                      gu_bytes > 0 &&
                      mvt_tail_image_fits(layers[l + 1].gate_up_qtype, 2, ffn, hidden, M, gu_bytes);
    }
    return n;
}

int muser_ffn_stack(const muser_ffn_layer* layers, int n_layers, const float* entry_norm,
                    int64_t hidden, int64_t ffn, int M, float* residual, float* out,
                    float eps_norm, float eps_post, void* workspace, size_t workspace_bytes,
                    void* stream) {
    clear_error();
    const char* fn = "muser_ffn_stack";
    if (layers == nullptr || n_layers < 1)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: need at least one layer", fn);
    MUSER_TRY(check_M(fn, M));
    MUSER_TRY(check_f32(fn, "entry_norm", entry_norm));
    MUSER_TRY(check_f32(fn, "residual", residual));
    MUSER_TRY(check_f32(fn, "out", out));
    MUSER_TRY(check_f32(fn, "workspace", workspace));
    if (out == residual) return set_error(MUSER_ERR_INVALID_ARG, "%s: out must not alias residual", fn);
    if (hidden % 4 || hidden > (int64_t{1} << 30))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: hidden must be a multiple of 4", fn);
    if (!(eps_norm > 0.0f) || !(eps_post > 0.0f)) return set_error(MUSER_ERR_INVALID_ARG, "%s: eps must be > 0", fn);
    const Workspace ws = carve(workspace, hidden, ffn, M);
    if (workspace_bytes < ws.total)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: workspace_bytes %zu < %zu", fn, workspace_bytes, ws.total);
    for (int l = 0; l < n_layers; ++l) {
        const muser_ffn_layer& L = layers[l];
        MUSER_TRY(check_matrix(fn, L.gate_up_qtype, L.w_gate, ffn, hidden));
        MUSER_TRY(check_matrix(fn, L.gate_up_qtype, L.w_up, ffn, hidden));
        MUSER_TRY(check_matrix(fn, L.down_qtype, L.w_down, hidden, ffn));
        MUSER_TRY(check_f32(fn, "post_norm", L.post_norm));
        MUSER_TRY(check_f32(fn, "next_norm", L.next_norm));
    }
    cudaStream_t s = as_stream(stream);
    if (stack_one_launch(layers, n_layers, hidden, ffn, M)) {
        // One row of x, Q4_K gate/up and Q6_K down: the whole stack in one
        // persistent launch (mvs.cu).
        MvsArgs a{};
        a.nl = n_layers;
        a.hidden = static_cast<int>(hidden);
        a.ffn = static_cast<int>(ffn);
        a.eps_norm = eps_norm;
        a.eps_post = eps_post;
        a.w_in = entry_norm;
        a.resid = residual;
        a.resid_ws = ws.resid_ws;
        a.out = out;
        a.proj = ws.proj;
        for (int l = 0; l < n_layers; ++l) {
            a.layer[l].wg = static_cast<const uint8_t*>(layers[l].w_gate);
            a.layer[l].wu = static_cast<const uint8_t*>(layers[l].w_up);
            a.layer[l].wd = static_cast<const uint8_t*>(layers[l].w_down);
            a.layer[l].w1 = layers[l].post_norm;
            a.layer[l].w2 = layers[l].next_norm;
        }
        return launch_mvs(a, ws.mvs, s);
    }
    MUSER_TRY(launch_rms_norm(residual, entry_norm, ws.xa, static_cast<int>(hidden), M, eps_norm, s));
    // One row of x: each layer's tail runs in the next layer's gate/up kernel
    // and the down projection only stores `projected`; the last tail runs on
    // its own.
    bool fused = true;
    for (int l = 0; l < n_layers && fused; ++l)
        fused = gate_up_tail_fused(layers[l].gate_up_qtype, hidden, M) && mv1_supported(layers[l].down_qtype, ffn);
    if (fused) {
        for (int l = 0; l < n_layers; ++l) {
            const muser_ffn_layer& L = layers[l];
            if (l == 0) {
                MUSER_TRY(gate_up_launch(L.gate_up_qtype, L.w_gate, L.w_up, ffn, hidden, ws.xa, M, ws.mid, nullptr, s));
            } else {
                // the residual relays between the caller's buffer and the
                // workspace (tail t reads buffer t % 2, writes the other), so
                // no block overwrites the row the others still read
                const muser_ffn_layer& P = layers[l - 1];
                float* r_in = (l - 1) % 2 == 0 ? residual : ws.resid_ws;
                float* r_out = (l - 1) % 2 == 0 ? ws.resid_ws : residual;
                MUSER_TRY(gate_up_tail_launch(L.gate_up_qtype, L.w_gate, L.w_up, ffn, hidden, ws.proj, r_in, r_out,
                                              P.post_norm, P.next_norm, eps_post, eps_norm, ws.xb, M, ws.mid,
                                              nullptr, s));
            }
            Mv1Args d{};
            d.W[0] = static_cast<const uint8_t*>(L.w_down);
            d.W[1] = d.W[0];
            d.rows = hidden;
            d.nsb = static_cast<int>(ffn / kQK);
            d.x = ws.mid;
            d.y0 = ws.proj;
            MUSER_TRY(launch_mv1(L.down_qtype, 1, kEpiStore, d, s));
        }
        // the last tail reads buffer (n_layers - 1) % 2 and ends in the caller's
        const muser_ffn_layer& Z = layers[n_layers - 1];
        float* r_last = (n_layers - 1) % 2 == 0 ? residual : ws.resid_ws;
        return dual_tail_to(r_last, r_last == residual ? nullptr : residual, ws.proj, out, Z.post_norm, Z.next_norm,
                            static_cast<int>(hidden), M, eps_post, eps_norm, s);
    }
    // Several rows: each layer's tail also writes the next gate/up launch's B
    // image of its output, where that launch takes one.
    float* x = ws.xa;
    float* xnext = ws.xb;
    bool image_ready = false;
    const size_t gu_bytes = ws.gu_scratch ? mvt_scratch_bytes(MUSER_Q4_K, 2, ffn, hidden, M) : 0;
    for (int l = 0; l < n_layers; ++l) {
        const muser_ffn_layer& L = layers[l];
        MUSER_TRY(gate_up_launch(L.gate_up_qtype, L.w_gate, L.w_up, ffn, hidden, x, M, ws.mid, ws.gu_scratch, s,
                                 image_ready));
        float* dst = (l == n_layers - 1) ? out : xnext;
        NextImage next{l + 1 < n_layers ? layers[l + 1].gate_up_qtype : 0, ws.gu_scratch, gu_bytes, &image_ready};
        MUSER_TRY(down_tail_launch(L.down_qtype, L.w_down, hidden, ffn, ws.mid, M, ws.proj,
                                   residual, dst, L.post_norm, L.next_norm, eps_post, eps_norm,
                                   ws.scratch, ws.scratch_bytes, s,
                                   l + 1 < n_layers && ws.gu_scratch ? &next : nullptr));
        std::swap(x, xnext);
    }
    return MUSER_OK;
}

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
static bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

// Detached rows (count rows of kv_dim halves each) must not overlap the planes.
static bool rows_overlap_plane(const muser_kv_plane& P, const void* k_rows, const void* v_rows, int64_t count) {
    const size_t nr = static_cast<size_t>(count) * static_cast<size_t>(P.kv_dim) * 2u;
    const size_t np = static_cast<size_t>(P.capacity) * static_cast<size_t>(P.kv_dim) * 2u;
    for (const void* r : {k_rows, v_rows})
        for (const void* q : {static_cast<const void*>(P.key), static_cast<const void*>(P.value)})
            if (ranges_overlap(r, nr, q, np)) return true;
    return ranges_overlap(k_rows, nr, v_rows, nr);
}

// The plane checks shared by the K/V calls (Ch 15 §15.2 metadata invariants).
static int check_plane(const muser_kv_plane* plane, const char* fn) {
    if (plane == nullptr) return set_error(MUSER_ERR_INVALID_ARG, "%s: plane is NULL", fn);
    const muser_kv_plane& P = *plane;
    if (P.key == nullptr || P.value == nullptr)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: plane buffers are NULL", fn);
    if (!is_aligned(P.key, 2) || !is_aligned(P.value, 2))
        return set_error(MUSER_ERR_MISALIGNED, "%s: plane buffers must be 2-byte aligned", fn);
    if (P.capacity < 1 || P.len < 0 || P.len > P.capacity || P.origin_logical < 0 ||
        P.origin_physical < 0 || P.origin_physical >= P.capacity)
        return set_error(MUSER_ERR_INVALID_ARG, "%s: inconsistent ring metadata", fn);
    if (P.kv_dim < 1 || (P.head_major && (P.head_dim < 1 || P.kv_dim % P.head_dim != 0)))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: bad kv_dim/head_dim", fn);
    return MUSER_OK;
}

int muser_kv_ring_write(muser_kv_plane* plane, const float* k, const float* v, int64_t position,
                        int64_t count, int64_t* first_physical, void* stream) {
    clear_error();
    const char* fn = "muser_kv_ring_write";
    MUSER_TRY(check_plane(plane, fn));
    muser_kv_plane& P = *plane;
    if (count < 0) return set_error(MUSER_ERR_INVALID_ARG, "%s: count < 0", fn);
    const int64_t expected = P.origin_logical + P.len;
    if (position != expected)
        return set_error(MUSER_ERR_CACHE_DISCONTINUITY,
                         "%s: cache discontinuity: expected position %lld, got %lld", fn,
                         (long long)expected, (long long)position);
    const int64_t phys_first = (P.origin_physical + P.len) % P.capacity;
    if (count == 0) {
        if (first_physical) *first_physical = phys_first;
        return MUSER_OK;
    }
    if (!k || !v) return set_error(MUSER_ERR_INVALID_ARG, "%s: k/v NULL", fn);
    if (!is_aligned(k, 4) || !is_aligned(v, 4))
        return set_error(MUSER_ERR_MISALIGNED, "%s: k/v must be 4-byte aligned", fn);
    // Sequential appends: only the last `capacity` rows of the batch survive.
    const int64_t src_first = std::max<int64_t>(0, count - P.capacity);
    MUSER_TRY(launch_kv_store(P.key, P.value, k, v, P.kv_dim, P.head_dim, P.head_major,
                              P.capacity, phys_first, src_first, count - src_first,
                              as_stream(stream)));
    const int64_t total = P.len + count;
    if (total <= P.capacity) {
        P.len = total;
    } else {
        const int64_t advance = total - P.capacity;
        P.len = P.capacity;
        P.origin_logical += advance;
        P.origin_physical = (P.origin_physical + advance) % P.capacity;
    }
    if (first_physical) *first_physical = phys_first;
    return MUSER_OK;
}

int muser_kv_snapshot(const muser_kv_plane* plane, int64_t first_logical, int64_t count,
                      uint16_t* k_rows, uint16_t* v_rows, void* stream) {
    clear_error();
    const char* fn = "muser_kv_snapshot";
    MUSER_TRY(check_plane(plane, fn));
    const muser_kv_plane& P = *plane;
    if (count < 0 || count > P.len || first_logical < P.origin_logical ||
        first_logical - P.origin_logical > P.len - count)
        return set_error(MUSER_ERR_INVALID_ARG,
                         "%s: rows %lld..+%lld are outside the live window %lld..+%lld", fn,
                         (long long)first_logical, (long long)count, (long long)P.origin_logical,
                         (long long)P.len);
    if (count == 0) return MUSER_OK;
    if (!k_rows || !v_rows) return set_error(MUSER_ERR_INVALID_ARG, "%s: k_rows/v_rows NULL", fn);
    if (!is_aligned(k_rows, 2) || !is_aligned(v_rows, 2))
        return set_error(MUSER_ERR_MISALIGNED, "%s: k_rows/v_rows must be 2-byte aligned", fn);
    if (rows_overlap_plane(P, k_rows, v_rows, count))
        return set_error(MUSER_ERR_INVALID_ARG, "%s: k_rows, v_rows and the planes must not overlap", fn);
    const int64_t phys0 = (P.origin_physical + (first_logical - P.origin_logical)) % P.capacity;
    return launch_kv_window(P.key, P.value, k_rows, v_rows, P.kv_dim, P.head_dim, P.head_major,
                            P.capacity, phys0, count, false, as_stream(stream));
}

int muser_kv_restore(muser_kv_plane* plane, const uint16_t* k_rows, const uint16_t* v_rows,
                     int64_t origin_logical, int64_t len, void* stream) {
    clear_error();
    const char* fn = "muser_kv_restore";
    MUSER_TRY(check_plane(plane, fn));
    muser_kv_plane& P = *plane;
    if (origin_logical < 0 || len < 0 || len > P.capacity)
        return set_error(MUSER_ERR_INVALID_ARG,
                         "%s: a window of %lld rows from origin %lld does not fit capacity %lld", fn,
                         (long long)len, (long long)origin_logical, (long long)P.capacity);
    const int64_t rotation = origin_logical % P.capacity;
    if (len > 0) {
        if (!k_rows || !v_rows) return set_error(MUSER_ERR_INVALID_ARG, "%s: k_rows/v_rows NULL", fn);
        if (!is_aligned(k_rows, 2) || !is_aligned(v_rows, 2))
            return set_error(MUSER_ERR_MISALIGNED, "%s: k_rows/v_rows must be 2-byte aligned", fn);
        if (rows_overlap_plane(P, k_rows, v_rows, len))
            return set_error(MUSER_ERR_INVALID_ARG, "%s: k_rows, v_rows and the planes must not overlap", fn);
        MUSER_TRY(launch_kv_window(P.key, P.value, const_cast<uint16_t*>(k_rows),
                                   const_cast<uint16_t*>(v_rows), P.kv_dim, P.head_dim,
                                   P.head_major, P.capacity, rotation, len, true,
                                   as_stream(stream)));
    }
    P.len = len;
    P.origin_logical = origin_logical;
    P.origin_physical = rotation;
    return MUSER_OK;
}

int muser_sync(void* stream, int timeout_ms) {
    clear_error();
    cudaEvent_t ev;
    cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
    if (e != cudaSuccess) return cuda_fail(e, "muser_sync: cudaEventCreate");
    e = cudaEventRecord(ev, as_stream(stream));
    if (e != cudaSuccess) {
        cudaEventDestroy(ev);
        return cuda_fail(e, "muser_sync: cudaEventRecord");
    }
    timespec t0;
    clock_gettime(CLOCK_MONOTONIC, &t0);
    int rc = MUSER_OK;
    for (;;) {
        e = cudaEventQuery(ev);
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) {
            rc = cuda_fail(e, "muser_sync: cudaEventQuery");
            break;
        }
        if (timeout_ms >= 0) {
            timespec t;
            clock_gettime(CLOCK_MONOTONIC, &t);
            const double ms = (t.tv_sec - t0.tv_sec) * 1e3 + (t.tv_nsec - t0.tv_nsec) * 1e-6;
            if (ms >= timeout_ms) {
                rc = set_error(MUSER_ERR_TIMEOUT, "muser_sync: stream still busy after %d ms", timeout_ms);
                break;
            }
        }
        const timespec nap{0, 20000};
        nanosleep(&nap, nullptr);
    }
    cudaEventDestroy(ev);
    return rc;
}

int muser_debug_spin(int64_t microseconds, void* stream) {
    clear_error();
    if (microseconds < 0 || microseconds > 10 * 1000 * 1000)
        return set_error(MUSER_ERR_INVALID_ARG, "muser_debug_spin: 0..10 s only");
    return launch_spin(microseconds, as_stream(stream));
}

int muser_debug_occupy(int ctas, int64_t microseconds, void* stream) {
    clear_error();
    if (ctas < 1 || ctas > 4096 || microseconds < 0 || microseconds > 10 * 1000 * 1000)
        return set_error(MUSER_ERR_INVALID_ARG, "muser_debug_occupy: 1..4096 blocks for 0..10 s only");
    return launch_occupy(ctas, microseconds, as_stream(stream));
}

int muser_device_sm_count(void) { return sm_count(); }

unsigned muser_device_status(int reset) { return read_device_status(reset != 0); }

}  // extern "C"
