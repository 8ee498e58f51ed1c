/*
 * muser.h -- C ABI of libmuser, the GB300 (sm_103a) decode-FFN weight-streaming
 * library.
 *
 * The operations are those of the Muser engine's decode hot path as the book
 * "How to Write an Inference Engine -- the Muser book" describes it: the
 * one-token quantized matvec over ggml-style Q4_K / Q6_K super-blocks
 * (Ch 19 §19.3, §19.5), the FFN gate/up/SiLU step (Ch 10 Figure 10.1 box 11,
 * §10.3 (d)), the dual-epsilon fused residual tail (Ch 19 §19.4; Ch 10 §10.4
 * Figure 10.2) and the f16 K/V ring store (Ch 15 §15.4-§15.5).  Around it:
 * the attention-side projection group of the same layer (Ch 10 Figure 10.1
 * box 4, §10.3 (e)), the LM head with its logit scale and soft cap (boxes 14
 * and 15), Q5_K matrices (the third k-quant of the kernel registry, Ch 4
 * §4.4), and the K/V window snapshot and rotation-preserving restore
 * (Ch 15 §15.6).
 *
 * Conventions shared by every entry point:
 *  - Ownership: the caller owns every buffer.  No entry point allocates or
 *    frees device memory.  Pointers marked "device" must point to memory of
 *    the current CUDA device; "host" pointers to ordinary host memory.
 *  - Streams: `stream` is a cudaStream_t (NULL = the legacy default stream).
 *    Work is enqueued asynchronously on it; nothing synchronises the host
 *    except muser_sync().
 *  - Errors: every entry point returns a muser_status.  Arguments are checked
 *    on the host before anything is launched; on any error nothing is
 *    launched and no output buffer is touched (the book's fail-closed rule,
 *    Ch 4 §4.4 and Ch 10 §10.9).  muser_last_error() returns a description of
 *    the calling thread's most recent error.
 *  - Types: activations and norm weights are binary32 ("f32"), row-major.
 *    A quantized matrix W with `rows` outputs and `cols` inputs is stored as
 *    rows of cols/256 consecutive super-blocks: rows*(cols/256)*block_bytes
 *    bytes, block_bytes = 144 (Q4_K), 176 (Q5_K) or 210 (Q6_K).
 *  - Quant types: every matvec entry point takes Q4_K and Q6_K.
 *    muser_dequantize and muser_qmatvec also take Q5_K, the third k-quant of
 *    the book's kernel registry (Ch 4 §4.4; ggml layout: f16 d and dmin,
 *    Q4_K's packed scales and mins, 32 bytes of fifth code bits, 128 code
 *    bytes).  Any other type, or Q5_K elsewhere, is MUSER_ERR_UNSUPPORTED.
 *  - Alignment: f32 pointers and quantized matrices 16-byte aligned (any
 *    cudaMalloc/torch allocation is).  Misaligned pointers return
 *    MUSER_ERR_MISALIGNED.
 *  - Activation rows: M is the number of activation rows (1 for one-token
 *    decode, up to MUSER_MAX_M = 16 for the speculative-verify shape,
 *    Ch 10 §10.1 MAX_DFLASH_BLOCK).
 *  - Scratch: calls that take caller scratch want it zero-filled before its
 *    first use and leave it zero-filled after every call that completes.  A
 *    kernel that gives up a bounded wait (muser_device_status() non-zero)
 *    may leave counters in it: zero-fill it again before reusing it.
 */
#ifndef MUSER_H
#define MUSER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MUSER_ABI_VERSION 2
#define MUSER_MAX_M 16
/* Scratch of the fused layer-boundary calls (muser_ffn_gate_up_silu_tail,
 * muser_qmatvec_group_tail) when they update the residual in place: the
 * blocks' ticket. */
#define MUSER_BOUNDARY_SCRATCH_BYTES 256u

/* ggml type ids, informational */
typedef enum { MUSER_Q4_K = 12, MUSER_Q5_K = 13, MUSER_Q6_K = 14 } muser_qtype;

typedef enum {
    MUSER_OK = 0,
    MUSER_ERR_INVALID_ARG = -1,        /* a size, count or pointer is invalid */
    MUSER_ERR_UNSUPPORTED = -2,        /* quant type or shape the library does not handle */
    MUSER_ERR_MISALIGNED = -3,         /* a pointer breaks the alignment rule above */
    MUSER_ERR_CACHE_DISCONTINUITY = -4,/* KV append at a position other than origin_logical+len */
    MUSER_ERR_CUDA = -5,               /* a CUDA runtime call or launch failed */
    MUSER_ERR_TIMEOUT = -6             /* muser_sync gave up before the stream drained */
} muser_status;

/* ABI version (MUSER_ABI_VERSION of the built library). */
int muser_version(void);

/* Description of the calling thread's last error ("" if none).  The string
 * stays valid until the next failing call on the same thread. */
const char* muser_last_error(void);

/* Bytes of one super-block of `qtype` (144, 176, 210; 0 if unknown). */
size_t muser_block_bytes(int qtype);

/* Bytes of a rows x cols matrix of `qtype` (0 if cols % 256 != 0 or the type
 * is unknown). */
size_t muser_matrix_bytes(int qtype, int64_t rows, int64_t cols);

/*
 * muser_dequantize -- out[r*cols + k] = the binary32 value of weight (r, k).
 *   Q4_K: d*scale_j*q - dmin*min_j of sub-block j = k%256/32 (Q5_K the
 *   same with q = 0..31, its fifth bit from qh); Q6_K:
 *   d*scale_s*(q-32) of sub-block s = k%256/16 (block layouts: Ch 19 §19.3,
 *   ggml super-block bit positions).  Each value is the exactly rounded
 *   binary32 of that expression; this is the bit-exact test hook of the
 *   path (the matvec kernels never materialise these values).
 *   W: device, rows x cols matrix; out: device f32 [rows*cols].
 */
int muser_dequantize(int qtype, const void* W, int64_t rows, int64_t cols, float* out,
                     void* stream);

/*
 * muser_qmatvec -- y[m*rows + r] = sum_k w(r,k) * x[m*cols + k], m < M
 *   (Ch 19 §19.1 operation 1; the decode projection of Ch 1).  Weights are
 *   dequantised in registers straight from HBM; sums are binary32.
 *   W: device matrix; x: device f32 [M*cols]; y: device f32 [M*rows].
 *   1 <= M <= 16, cols % 256 == 0, rows >= 1.  x and y must not overlap.
 *   Q6_K with 2..16 rows of x runs on the tensor cores with the products
 *   sc * (q - 32) in binary16, exact for sub-block scales in [-62, 62] (the
 *   book's workloads draw them on [-32, 31]); a scale outside that range sets
 *   bit 4 of muser_device_status().  One row of x takes any int8 scale.
 *   Intermediate sums are binary32: above |x| of about 1e34 the Q4_K/Q5_K
 *   min terms (a 32-input sum of x times a min of up to 63) can overflow.
 */
int muser_qmatvec(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, int M,
                  float* y, void* stream);

/* Scratch bytes muser_qmatvec_scratch needs (0: the call needs none, as for
 * one row of x and for shapes the tensor-core kernel does not take).  It
 * covers the tile tickets, the partial sums and, for 2..16 rows of x, the
 * call's B operand image (x split into binary16 parts once per call, about
 * 17 KB per 256 inputs, when every SM has enough units to amortise building
 * it). */
size_t muser_qmatvec_scratch_bytes(int qtype, int64_t rows, int64_t cols, int M);

/*
 * muser_qmatvec_scratch -- the same result as muser_qmatvec.  With 2..16 rows
 *   of x and caller scratch the tensor-core kernel spreads the (row tile,
 *   super-block) units of the matrix evenly over the SMs and sums a tile's
 *   parts in a fixed order; without it each SM takes whole 128-row tiles,
 *   which leaves most SMs idle on matrices of few tiles (the attention-side
 *   projections of the book's model are 2 to 52 tiles).
 *   scratch: device memory of at least muser_qmatvec_scratch_bytes(...)
 *   bytes, 16-byte aligned, owned by the caller, zero-filled before its first
 *   use; every successful call leaves it zero-filled again.  Calls that can
 *   run at the same time must not share it.  When the size is 0, scratch is
 *   not used and may be NULL.  Other arguments as muser_qmatvec.
 */
int muser_qmatvec_scratch(int qtype, const void* W, int64_t rows, int64_t cols, const float* x, int M,
                          float* y, void* scratch, size_t scratch_bytes, void* stream);

/*
 * muser_rms_norm -- out[m*n+i] = w[i] * x[m*n+i] / sqrt(mean_i(x[m*n+i]^2) + eps)
 *   (Ch 2 §2.6 rms_norm_batch; the layer-0 input norm of Ch 10 Figure 10.1).
 *   x, out: device f32 [M*n] (may alias); w: device f32 [n].  n % 4 == 0,
 *   eps > 0, 1 <= M.
 */
int muser_rms_norm(const float* x, const float* w, float* out, int n, int M, float eps,
                   void* stream);

/*
 * muser_silu_mul -- out[i] = silu(a[i]) * b[i], silu(z) = z/(1+exp(-z))
 *   (muser_silu_mul_inplace, Ch 10 Figure 10.1 box 11).  Device f32 arrays of
 *   n elements; out may alias a or b.
 */
int muser_silu_mul(const float* a, const float* b, float* out, int64_t n, void* stream);

/*
 * muser_ffn_gate_up_silu -- mid[m*ffn + r] = silu(g) * u with
 *   g = sum_k wg(r,k) x[m*hidden+k] and u = sum_k wu(r,k) x[m*hidden+k]
 *   (both binary32), computed in one pass that streams both matrices
 *   (the book's opt-in ffn_q4k_gate_up_silu fusion, Ch 10 §10.3 (d)).
 *   Wg, Wu: device matrices [ffn x hidden] of `qtype`; x: device f32
 *   [M*hidden]; mid: device f32 [M*ffn].
 */
int muser_ffn_gate_up_silu(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                           int64_t hidden, const float* x, int M, float* mid, void* stream);

/* Scratch bytes muser_ffn_gate_up_silu_scratch needs (0: the call needs
 * none); as for muser_qmatvec_scratch_bytes, including the B operand image. */
size_t muser_gate_up_scratch_bytes(int qtype, int64_t ffn, int64_t hidden, int M);

/*
 * muser_ffn_gate_up_silu_scratch -- the same result as muser_ffn_gate_up_silu.
 *   With caller scratch the tensor-core kernel (2..16 rows of x) can split a
 *   row tile's super-blocks over several SMs and sum the parts in a fixed
 *   order; without it each SM takes whole tiles, which leaves SMs idle when
 *   the tile count is not a multiple of the SM count.
 *   scratch: device memory of at least muser_gate_up_scratch_bytes(...) bytes,
 *   16-byte aligned, owned by the caller, zero-filled before its first use;
 *   every successful call leaves it zero-filled again.  Calls that can run at
 *   the same time must not share it.  Other arguments as
 *   muser_ffn_gate_up_silu.
 */
int muser_ffn_gate_up_silu_scratch(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                                   int64_t hidden, const float* x, int M, float* mid, void* scratch,
                                   size_t scratch_bytes, void* stream);

/*
 * muser_fused_residual_dual_rmsnorm -- the dual-eps tail (Ch 19 §19.4,
 *   muser_fused_norm_residual_rms_norm_32sg; Ch 10 Figure 10.2), per row m:
 *     residual += w1 * src / sqrt(mean(src^2) + eps1)      (in place)
 *     out       = w2 * residual / sqrt(mean(residual^2) + eps2)
 *   The updated residual is stored as binary32 and the second norm reads the
 *   stored value (the book's device-memory rounding point, §19.7).
 *   residual: device f32 [M*n] in/out; src, out: device f32 [M*n]; w1, w2:
 *   device f32 [n].  n % 4 == 0; eps1, eps2 > 0; out must not alias
 *   residual or src.
 */
int muser_fused_residual_dual_rmsnorm(float* residual, const float* src, float* out,
                                      const float* w1, const float* w2, int n, int M, float eps1,
                                      float eps2, void* stream);

/*
 * muser_qmatvec_group -- n (1..4) matvecs of one input, y_i = W_i . x, as the
 *   book issues the attention projections Q, K, V and gate: one concurrent
 *   group reading one shared normed input (Ch 10 Figure 10.1 box 4, §10.3
 *   (e)).  W[i]: device matrices [rows[i] x cols] of `qtype`; x: device f32
 *   [M*cols]; y[i]: device f32 [M*rows[i]].  W, rows and y are host arrays of
 *   n entries.  For one row of x and Q4_K the n matrices stream in one launch,
 *   their rows taken as one matrix; otherwise each runs as muser_qmatvec.
 *   Results are those of n muser_qmatvec calls.  Fail-closed like
 *   muser_qmatvec.
 */
int muser_qmatvec_group(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                        const float* x, int M, float* const* y, void* stream);

/* Scratch bytes muser_qmatvec_group_scratch needs for one tensor-core launch
 * over the whole group (0: the group runs as muser_qmatvec_group: one row of
 * x, a type other than Q4_K, or a shape the tensor-core kernel does not take).
 * rows: host array of n entries. */
size_t muser_qmatvec_group_scratch_bytes(int qtype, int n, const int64_t* rows, int64_t cols, int M);

/*
 * muser_qmatvec_group_scratch -- the same results as muser_qmatvec_group.
 *   With 2..16 rows of x, Q4_K and caller scratch of at least
 *   muser_qmatvec_group_scratch_bytes(...) bytes, the n matrices run as one
 *   tensor-core launch: each matrix's rows start a 128-row tile of one
 *   virtual matrix, the (tile, super-block) units spread over every SM and x
 *   is converted once for all of them (Ch 10 Figure 10.1 box 4: one group on
 *   one input).  Otherwise as muser_qmatvec_group (scratch unused, may be
 *   NULL).  scratch: 16-byte aligned, owned by the caller, zero-filled before
 *   its first use and left zero-filled by every call; calls that can run at
 *   the same time must not share it.
 */
int muser_qmatvec_group_scratch(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                                const float* x, int M, float* const* y, void* scratch, size_t scratch_bytes,
                                void* stream);

/*
 * muser_qmatvec_group_tail -- the previous sub-block's dual-eps tail, then
 *   the group on its output: as muser_fused_residual_dual_rmsnorm (src =
 *   projected, out = x_out, n = cols) followed by muser_qmatvec_group with
 *   x = x_out.  With one row of x and Q4_K the tail runs inside the group's
 *   launch, every block for itself.  residual_out, residual and scratch as
 *   for muser_ffn_gate_up_silu_tail: a distinct residual_out takes the
 *   updated residual; NULL updates `residual` in place through the ticket in
 *   `scratch`.  With 2..16 rows of x the tail runs as a kernel of its own,
 *   and scratch of at least muser_qmatvec_group_scratch_bytes(...) bytes
 *   takes the group's one tensor-core launch (as
 *   muser_qmatvec_group_scratch); when that launch reads its B operand from
 *   an image in the scratch (Q4_K groups large enough to give every SM at
 *   least 8 units of 128 rows x 256 inputs, cols <= 8192), the tail kernel
 *   writes the image of x_out itself, saving the kernel that would build it.
 *   projected, residual, x_out (and residual_out): device f32 [M*cols],
 *   distinct; w1, w2: device f32 [cols]; cols % 4 == 0; eps1, eps2 > 0.
 */
int muser_qmatvec_group_tail(int qtype, int n, const void* const* W, const int64_t* rows, int64_t cols,
                             const float* projected, float* residual, float* residual_out, const float* w1,
                             const float* w2, float eps1, float eps2, float* x_out, int M, float* const* y,
                             void* scratch, size_t scratch_bytes, void* stream);

/*
 * muser_scale_softcap -- logits[i] = cap * tanh(logits[i] * scale / cap), in
 *   place (the book's muser_scale_softcap_inplace, Ch 10 Figure 10.1 box 15:
 *   scale 0.196116 = 1/sqrt(26), cap 20).  logits: device f32 [n]; cap > 0
 *   and finite; scale finite.
 */
int muser_scale_softcap(float* logits, int64_t n, float scale, float cap, void* stream);

/*
 * muser_lm_head -- the LM head (Ch 10 Figure 10.1 boxes 14 and 15): binary32
 *   logits = W . x (the final normed hidden row), then the scale and soft cap
 *   above.  W: device matrix [vocab x hidden] of `qtype` (the book's model:
 *   202,048 x 6,656); x: device f32 [M*hidden]; logits: device f32
 *   [M*vocab].  For one row of x the cap is the matvec kernel's epilogue;
 *   otherwise the two run one after the other.  Fail-closed like
 *   muser_qmatvec.
 */
int muser_lm_head(int qtype, const void* W, int64_t vocab, int64_t hidden, const float* x, int M,
                  float* logits, float scale, float cap, void* stream);

/*
 * muser_ffn_gate_up_silu_tail -- the boundary between two decode layers in
 *   one call: the previous layer's dual-eps tail (Ch 19 §19.4, as
 *   muser_fused_residual_dual_rmsnorm with src = projected, out = x_out),
 *   then this layer's gate/up/SiLU on its output (Ch 10 §10.3 (d), as
 *   muser_ffn_gate_up_silu with x = x_out).  Per row m, with R the updated
 *   residual (written to residual_out, or to residual when residual_out is
 *   NULL):
 *     R     = residual + w1 * projected / sqrt(mean(projected^2) + eps1)
 *     x_out = w2 * R / sqrt(mean(R^2) + eps2)
 *     mid   = silu(Wg . x_out) * (Wu . x_out)
 *   w2 is the next norm of the previous layer, i.e. this layer's input norm
 *   (Ch 10 §10.4).  The rounding points are those of the two calls: the
 *   residual and x_out are binary32 values.  For one row of x with a short
 *   enough row (hidden <= 6656 for Q4_K gate/up) the tail runs inside the
 *   gate/up kernel, so the layer boundary costs no separate launch; other
 *   shapes run the two calls.  Inside the kernel every block computes the
 *   tail for itself from the whole residual row.
 *   - residual_out != NULL (a row distinct from the others): the updated
 *     residual goes there and `residual` is only read; no block can write a
 *     row another block reads.  This is the fast form; a layer loop
 *     alternates two residual buffers.  scratch is not used (may be NULL).
 *   - residual_out == NULL: the residual is updated in place.  No block may
 *     overwrite the row while another still has to read it, so each block
 *     takes a ticket in `scratch` once it has read the row, and the block
 *     that takes the last ticket writes the updated residual and x_out at its
 *     end.  scratch: device memory of at least MUSER_BOUNDARY_SCRATCH_BYTES
 *     bytes, 16-byte aligned, owned by the caller, zero-filled before its
 *     first use and left zero-filled by every call; calls that can run at the
 *     same time must not share it.
 *   projected, residual, x_out (and residual_out): device f32 [M*hidden],
 *   distinct; w1, w2: device f32 [hidden]; Wg, Wu: device matrices
 *   [ffn x hidden]; mid: device f32 [M*ffn].
 *   hidden % 4 == 0; eps1, eps2 > 0.  Fail-closed like the two calls.
 */
int muser_ffn_gate_up_silu_tail(int qtype, const void* Wg, const void* Wu, int64_t ffn,
                                int64_t hidden, const float* projected, float* residual, float* residual_out,
                                const float* w1, const float* w2, float eps1, float eps2,
                                float* x_out, int M, float* mid, void* scratch, size_t scratch_bytes,
                                void* stream);

/* Scratch bytes muser_qmatvec_residual_dual_rmsnorm should get: 1 KiB for the
 * one-row kernel (its completion ticket, then one sum of projected^2 per
 * block, which spares the tail one pass over the row) plus the tensor-core
 * kernel's tickets and partial sums for several rows.  256 bytes (the ticket)
 * is the minimum the call accepts.  With 1 KiB more than
 * muser_qmatvec_scratch_bytes(qtype, hidden, ffn, M), several rows of x also
 * take the B operand image described there. */
size_t muser_scratch_bytes(int64_t hidden, int M);

/*
 * muser_qmatvec_residual_dual_rmsnorm -- the layer exit of Ch 19 §19.5 in one
 *   call: projected = W_down . mid (binary32, written to `projected`), then
 *   the dual-eps tail above with src = projected.
 *   Wdown: device matrix [hidden x ffn]; mid: device f32 [M*ffn];
 *   projected: device f32 [M*hidden] (output); residual: device f32
 *   [M*hidden] in/out; out: device f32 [M*hidden]; w1, w2: device f32
 *   [hidden].
 *   scratch: device memory of at least muser_scratch_bytes(hidden, M) bytes,
 *   16-byte aligned, owned by the caller, zero-filled before its first use;
 *   every successful call leaves it zero-filled again.  One scratch buffer
 *   must not be used by two calls that can run at the same time.
 */
int muser_qmatvec_residual_dual_rmsnorm(int qtype, const void* Wdown, int64_t hidden, int64_t ffn,
                                        const float* mid, int M, float* projected,
                                        float* residual, float* out, const float* w1,
                                        const float* w2, float eps1, float eps2, void* scratch,
                                        size_t scratch_bytes, void* stream);

/* Size of the library's own scratch array (1 MiB), see the call below. */
#define MUSER_STATIC_SCRATCH_BYTES (1u << 20)

/*
 * muser_qmatvec_residual_dual_rmsnorm_static -- the same down projection and
 *   dual-eps tail as muser_qmatvec_residual_dual_rmsnorm, for callers that
 *   cannot hand the library any device memory of their own.  The Muser book
 *   has no counterpart to this call; it is a convenience of this library.
 *
 *   Who needs it: a host that embeds the library but owns no allocator (its
 *   device memory was carved up front into weights, KV cache and activations
 *   by someone else, and nothing is left to lend), and a token loop that must
 *   not call cudaMalloc or cudaFree between tokens, because those calls can
 *   wait for the whole device and so stall the stream it is feeding.
 *
 *   Instead of `projected` and `scratch`, the call uses an array that is
 *   compiled into the library: MUSER_STATIC_SCRATCH_BYTES bytes of device
 *   memory on every GPU that loads the library, held until the process
 *   exits.  Its first 256 bytes hold the tail's completion counter and the
 *   rest holds the projected rows, so M * hidden * 4 + 256 must not exceed
 *   MUSER_STATIC_SCRATCH_BYTES (M * hidden <= 262080); larger sizes fail
 *   with MUSER_ERR_INVALID_ARG and a message naming the limit.  The call
 *   never calls cudaMalloc, cudaFree or any routine that allocates.
 *
 *   The first call on each device looks up the array's device address, with
 *   that device current, and keeps it; make that first call before starting
 *   any stream capture.  Every call clears the completion counter on
 *   `stream` before its kernels run; the projected rows are overwritten.
 *
 *   All calls in the process share the one array of their device, and it
 *   keeps whatever the last call left in it.  Calls whose work can overlap
 *   on the GPU (on streams with no ordering between them) race on it and
 *   give wrong results: issue them on one stream, or order them with events.
 *
 *   With one row of x the down projection and the tail run on the same
 *   one-token kernel as muser_qmatvec_residual_dual_rmsnorm; the tail then
 *   takes one more pass over the row, since the array has no room for the
 *   blocks' partial sums.  With 2..16 rows the tensor-core kernel runs with
 *   whole 128-row tiles per SM (its even split over every SM needs partial
 *   sums the array has no room for), then the tail per row.
 *
 *   Other arguments, alignment and errors as muser_qmatvec_residual_dual_rmsnorm.
 */
int muser_qmatvec_residual_dual_rmsnorm_static(int qtype, const void* Wdown, int64_t hidden,
                                               int64_t ffn, const float* mid, int M,
                                               float* residual, float* out, const float* w1,
                                               const float* w2, float eps1, float eps2,
                                               void* stream);

/*
 * One decode-FFN layer's parameters (Ch 10 Figure 10.1 boxes 11-13): gate and
 * up [ffn x hidden], down [hidden x ffn], the post-FFN norm weight (w1, eps1)
 * and the next norm's weight (w2, eps2): the next layer's input norm, or the
 * output norm after the last layer (§10.3 (c)).  All pointers are device
 * pointers; the struct itself is host memory.
 */
typedef struct {
    const void* w_gate;
    const void* w_up;
    const void* w_down;
    const float* post_norm;
    const float* next_norm;
    int32_t gate_up_qtype;
    int32_t down_qtype;
} muser_ffn_layer;

/* Bytes of workspace muser_ffn_stack needs: two normed-input buffers, the
 * FFN intermediate, the projected buffer, a second residual buffer, the
 * one-launch stack's synchronisation words and input records, and the tail
 * scratch. */
size_t muser_ffn_workspace_bytes(int64_t hidden, int64_t ffn, int M);

/* Number of kernel launches one muser_ffn_stack call with these arguments
 * makes (1 when the whole stack runs as one persistent launch); -1 for
 * arguments the call would reject outright. */
int muser_ffn_stack_launches(const muser_ffn_layer* layers, int n_layers, int64_t hidden, int64_t ffn, int M);

/*
 * muser_ffn_stack -- `n_layers` decode-FFN layers over M residual rows
 *   (Ch 10 §10.3-§10.4): the entry RMSNorm (weight entry_norm, eps_norm) runs
 *   once; then per layer l: mid = silu(Wg.x) * (Wu.x); projected = Wd.mid;
 *   residual += post_norm * rms_norm(projected, eps_post); x = next_norm *
 *   rms_norm(residual, eps_norm).  `out` receives the last layer's x.
 *   layers: host array of n_layers structs; entry_norm: device f32 [hidden];
 *   residual: device f32 [M*hidden] in/out; out: device f32 [M*hidden];
 *   workspace: device memory of muser_ffn_workspace_bytes(hidden, ffn, M)
 *   bytes, 16-byte aligned, zero-filled before its first use.
 *   n_layers == 1 is one decode-FFN block.
 *   One row of x with Q4_K gate/up and Q6_K down (up to 128 layers, hidden up
 *   to 6656, ffn a multiple of 512 up to 24576) runs as one persistent
 *   kernel: one block per SM, launched cooperatively so that every block is
 *   resident; each block streams every layer's weights through one ring of
 *   shared-memory stages, and its compute warps wait at grid barriers
 *   (bounded in time) only for the activations each phase needs.  The
 *   residual is relayed through a second buffer in the workspace, so no block
 *   overwrites a row another block still reads; the result is left in
 *   `residual`.  The call also clears a few synchronisation words of the
 *   workspace on `stream` before the kernel.  Other shapes run one launch per
 *   projection.
 */
int muser_ffn_stack(const muser_ffn_layer* layers, int n_layers, const float* entry_norm,
                    int64_t hidden, int64_t ffn, int M, float* residual, float* out,
                    float eps_norm, float eps_post, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * K/V plane metadata (Ch 15 §15.2 MetalKvPlane).  key/value are device
 * binary16 planes of capacity*kv_dim halves.  Token-major index:
 * physical*kv_dim + e; head-major: (e/head_dim*capacity + physical)*head_dim
 * + e%head_dim (§15.3 Figure 15.1).  The struct is host memory; the library
 * updates len/origin_* on success only.
 */
typedef struct {
    uint16_t* key;
    uint16_t* value;
    int64_t capacity;
    int64_t len;
    int64_t origin_logical;
    int64_t origin_physical;
    int32_t kv_dim;
    int32_t head_dim;
    int32_t head_major;
    int32_t reserved;
} muser_kv_plane;

/*
 * muser_kv_ring_write -- append `count` token rows at logical positions
 *   position..position+count-1 (Ch 15 §15.5 append / append_batch): the
 *   physical row comes from the plane's explicit origins, never from the
 *   absolute position; K and V are stored as binary16 rounded to nearest
 *   even.  position != origin_logical + len returns
 *   MUSER_ERR_CACHE_DISCONTINUITY and leaves the plane and its metadata
 *   untouched.  When count > capacity only the last `capacity` rows survive,
 *   as with sequential appends.
 *   plane: host struct (updated on success); k, v: device f32
 *   [count*kv_dim]; first_physical: host, receives the physical row of
 *   `position` (may be NULL).
 */
int muser_kv_ring_write(muser_kv_plane* plane, const float* k, const float* v, int64_t position,
                        int64_t count, int64_t* first_physical, void* stream);

/*
 * muser_kv_snapshot -- copy the live logical rows first_logical ..
 *   first_logical+count-1 out of a plane pair as a detached window (Ch 15
 *   §15.6, the snapshot a restore replays).  The row of logical position q
 *   sits in slot (origin_physical + q - origin_logical) % capacity.
 *   plane: host struct, read only; k_rows, v_rows: device binary16
 *   [count*kv_dim], token-major, in logical order, 2-byte aligned (16-byte
 *   alignment with kv_dim, and head_dim for head-major planes, multiples of 8
 *   takes 16-byte copies), not overlapping the planes or each other
 *   (MUSER_ERR_INVALID_ARG).  count == 0 launches nothing.  A range outside
 *   [origin_logical, origin_logical+len) returns MUSER_ERR_INVALID_ARG and
 *   writes nothing.
 */
int muser_kv_snapshot(const muser_kv_plane* plane, int64_t first_logical, int64_t count,
                      uint16_t* k_rows, uint16_t* v_rows, void* stream);

/*
 * muser_kv_restore -- install a detached window of `len` logical rows starting
 *   at logical position origin_logical at the rotation a ring built by
 *   sequential appends holds there (Ch 15 §15.6; Ch 10 §10.7): rotation =
 *   origin_logical % capacity, logical row j goes to slot (rotation + j) %
 *   capacity, and on success the metadata becomes len = len, origin_logical =
 *   origin_logical, origin_physical = rotation.  Attention scans slots in
 *   physical order, so this placement keeps a restored session's sums, and
 *   their rounding, those of the live one.  Slots outside the window are not
 *   written; a NoPE plane (origin 0) gets the plain layout.
 *   plane: host struct (updated on success); k_rows, v_rows: device binary16
 *   [len*kv_dim], token-major, as muser_kv_snapshot writes them, not
 *   overlapping the planes or each other (MUSER_ERR_INVALID_ARG).
 *   origin_logical < 0, len < 0 or len > capacity
 *   returns MUSER_ERR_INVALID_ARG and changes nothing.  len == 0 only sets the
 *   metadata.
 */
int muser_kv_restore(muser_kv_plane* plane, const uint16_t* k_rows, const uint16_t* v_rows,
                     int64_t origin_logical, int64_t len, void* stream);

/*
 * muser_sync -- wait until all work enqueued on `stream` has finished, for at
 *   most timeout_ms milliseconds (the book's bounded wait_for_completion,
 *   Ch 2 §2.10).  Returns MUSER_OK, MUSER_ERR_TIMEOUT (the work keeps
 *   running) or MUSER_ERR_CUDA.  timeout_ms < 0 waits without a limit.
 */
int muser_sync(void* stream, int timeout_ms);

/*
 * muser_debug_spin -- enqueue a kernel that busy-waits `microseconds` on the
 *   GPU's global timer and then returns (bounded by construction, at most
 *   10 s).  Exists to exercise muser_sync's timeout path without stalling the
 *   GPU.
 */
int muser_debug_spin(int64_t microseconds, void* stream);

/*
 * muser_debug_occupy -- enqueue `ctas` (1..4096) blocks that each hold 160 KB
 *   of shared memory, so that no block of this library's weight-streaming
 *   kernels fits beside one on the same SM, and busy-wait `microseconds`
 *   (0..10 s) on the GPU's global timer.  Bounded by construction.  Run on
 *   another stream, it keeps SMs busy while a kernel under test starts, so
 *   that some of that kernel's blocks start late: the tests use it to check
 *   that no block depends on when the others start.
 */
int muser_debug_occupy(int ctas, int64_t microseconds, void* stream);

/* Number of SMs of the current device (for reports); -1 on error. */
int muser_device_sm_count(void);

/*
 * muser_device_status -- the library's device status word (0 = clean).  Bit 1:
 *   a kernel gave up a bounded wait on a weight-tile transfer and returned
 *   without finishing its outputs; bit 2: its clean-up wait also gave up;
 *   bit 4: a Q6_K sub-block scale outside [-62, 62] reached the tensor-core
 *   kernel (2..16 rows of x), whose results are then not exact.
 *   Synchronous (reads device memory); reset != 0 clears the word afterwards.
 *   Returns 0xFFFFFFFF if the word cannot be read.
 */
unsigned muser_device_status(int reset);

#ifdef __cplusplus
}
#endif

#endif /* MUSER_H */
