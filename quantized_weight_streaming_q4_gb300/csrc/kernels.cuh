// kernels.cuh -- launch interfaces between libmuser's translation units.
#pragma once

#include "common.cuh"

namespace muser {

enum EpiKind { kEpiStore = 0, kEpiSiluMul = 1, kEpiTail = 2, kEpiSoftcap = 3 };
// Where the one-token kernel's x comes from: memory, or the previous layer's
// dual-eps tail computed in its prologue (x = p.x is then `projected`).
enum XSource { kXMemory = 0, kXTail = 1 };

// One-token matvec (mv1.cu).  W[0..NMAT-1] share rows x (nsb*256) and x.
constexpr int kMv1MaxSeg = 4;
struct Mv1Args {
    const uint8_t* W[2];
    int64_t rows;
    int nsb;
    const float* x;
    float* y0;  // store: y of W[0]; silu: mid; tail: projected
    float* y1;  // store with two matrices: y of W[1]
    // tail epilogue
    float* resid;
    float* out;
    const float* w1;
    const float* w2;
    float eps1, eps2;
    float scale, cap;  // soft-cap epilogue: y = cap * tanh(y * scale / cap)
    unsigned* ticket;
    float* tail_part;  // per-block sums of projected^2 (kMv1TailParts floats), or null
    // x from the previous layer's tail (kXTail): the updated residual goes to
    // resid_out when that is set (a row distinct from resid); otherwise it
    // replaces resid, written by the block that takes the last ticket in
    // xticket, which it re-zeroes
    float* resid_out;
    unsigned* xticket;
    // Row segments (Q4_K, one matrix, store epilogue; Q4_K rows are whole 16-byte units):
    // rows [seg0[s], seg0[s+1]) of the virtual matrix are rows of segW[s],
    // and their results go to segY[s].  nseg == 0: W[0] and y0 as usual.
    int nseg;
    const uint8_t* segW[kMv1MaxSeg];
    int64_t seg0[kMv1MaxSeg + 1];
    float* segY[kMv1MaxSeg];
    // geometry, filled by the launcher
    int G, RS, ns, nconsumer_warps;
    int TG;  // consumer threads per row group
    int HP;  // Q6_K parity split: first thread of the odd-block half
    uint32_t stage_bytes;
    int part_off, stage_off;
    int x_off;  // input slots (shared memory offset)
    int rot;    // stage buffers under the input slots; stage k uses buffer (k + rot) % ns
    int lead;   // stages requested before the loads of x
};
// Blocks whose share of the tail's first sum fits in Mv1Args::tail_part.
constexpr int kMv1TailParts = 192;
bool mv1_supported(int qtype, int64_t cols);
bool mv1_tail_prologue_supported(int qtype, int64_t cols);
int launch_mv1(int qtype, int nmat, int epi, const Mv1Args& a, cudaStream_t s, int xs = kXMemory);

// Multi-row matvec (mvM.cu): y[m*rows + r], m < M <= 16.
struct MvMArgs {
    const uint8_t* W[2];
    int64_t rows;
    int nsb;
    const float* x;
    int M;
    float* y0;
    float* y1;
};
int launch_mvM(int qtype, int nmat, int epi, const MvMArgs& a, cudaStream_t s);

constexpr int kMvtMaxSeg = 4;
// One-token matvec on the tensor cores (mvt.cu).  Gate+up Q4_K with the SiLU
// epilogue (two matrices), or one Q4_K/Q6_K matrix with the store or tail
// epilogue.  Work is split into (row tile, super-block) units over all SMs;
// tiles shared by several CTAs are summed through `part`/`tick` scratch.
struct MvtArgs {
    const uint8_t* W[2];
    int64_t rows;  // rows of each matrix
    int nsb;       // super-blocks per row
    const float* x;  // [M][nsb*256]
    int M;           // rows of x (1..16)
    float* y;        // [M][rows]; store: y; silu: mid; tail: projected
    float* resid;
    float* out;
    const float* w1;
    const float* w2;
    float eps1, eps2;
    float* part;      // scratch: partial sums, 128 floats per slot; tile t from CTA c in slot t + c
    unsigned* tick;   // scratch: per-tile tickets [ntiles], then the tail counter
    unsigned* status; // device status word
    // several rows of x with scratch: the B operand of every super-block,
    // built once per call by a prep kernel (slab, then the x sums and scales)
    const uint8_t* bimg;
    // the image is already in the scratch (launch_mvt_tail_image wrote it
    // for this x): no prep launch
    int image_ready;
    // A group of Q4_K matrices on one x (store epilogue; nseg > 0): segment s
    // has seg_rows[s] rows (weights seg_W[s], results seg_y[s]) and owns tiles
    // [seg_t0[s], seg_t0[s+1]) of 128 rows; `rows` is then the tile total * 128.
    int nseg;
    const uint8_t* seg_W[kMvtMaxSeg];
    int64_t seg_rows[kMvtMaxSeg];
    float* seg_y[kMvtMaxSeg];
    int seg_t0[kMvtMaxSeg + 1];
    // geometry, filled by the launcher
    int ntiles, P, maxparts, ns, tiles_per_cta;
    uint32_t x_off, b_off, stage_off, xch_off;
};
bool mvt_supported(int qtype, int nmat, int64_t rows, int64_t cols, int M);
// Scratch of the even split: tickets and partial sums, and for several rows
// of x the B image after them (mvt_split_scratch_bytes: without the image).
size_t mvt_scratch_bytes(int qtype, int nmat, int64_t rows, int64_t cols, int M);
size_t mvt_split_scratch_bytes(int qtype, int nmat, int64_t rows, int64_t cols, int M);
// scratch == nullptr: whole tiles per CTA; else the even split over all SMs
// with `scratch` (zero-filled, left zeroed) of scratch_bytes >=
// mvt_split_scratch_bytes(); from mvt_scratch_bytes() on, several rows of x
// take the prebuilt B image.
int launch_mvt(int qtype, int epi, MvtArgs a, void* scratch, size_t scratch_bytes, cudaStream_t s);
// The dual-eps tail of M rows (as launch_dual_tail, cols inputs) that also
// writes the B image of its output `out` into `scratch` for a launch_mvt of
// (qtype, nmat, rows, cols, M) with that scratch, which then takes
// image_ready.  MUSER_ERR_UNSUPPORTED, with nothing launched, when that
// launch builds no image or the row is longer than 8,192.
int launch_mvt_tail_image(int qtype, int nmat, int64_t rows, int64_t cols, int M, float* resid, const float* src,
                          float* out, const float* w1, const float* w2, float eps1, float eps2, void* scratch,
                          size_t scratch_bytes, cudaStream_t s);
// Whether launch_mvt_tail_image takes that shape (with scratch_bytes of scratch).
bool mvt_tail_image_fits(int qtype, int nmat, int64_t rows, int64_t cols, int M, size_t scratch_bytes);
// Launches one launch_mvt call makes with scratch of mvt_scratch_bytes() (0: unsupported).
int mvt_launches(int qtype, int nmat, int64_t rows, int64_t cols, int M);
// Rows of the tile-aligned matrix a group of Q4_K matrices forms in one
// launch (each matrix starts a 128-row tile).
int64_t mvt_group_rows(int n, const int64_t* rows);
// Device address of the status word (mv1.cu), for kernels in other units.
unsigned* device_status_word();

// The one-token decode-FFN stack as one persistent kernel (mvs.cu): every
// layer's gate/up (Q4_K), down (Q6_K) and dual-eps tail for one row of x.
constexpr int kMvsMaxLayers = 128;
struct MvsLayer {
    const uint8_t* wg;
    const uint8_t* wu;
    const uint8_t* wd;
    const float* w1;  // post-FFN norm
    const float* w2;  // next norm (the next layer's input norm, or the output norm)
};
struct MvsArgs {
    int nl;
    int hidden, ffn;
    float eps_norm, eps_post;
    const float* w_in;  // entry norm
    float* resid;       // caller's residual row (in/out)
    float* resid_ws;    // the relay's other residual buffer
    float* out;         // the last layer's next-norm output
    float* proj;        // [hidden]
    // filled by the launcher
    unsigned* sync;     // grid barrier count, abort flag
    float4* xperm;      // mid, slice-major for the down phase's threads
    unsigned* status;   // device status word
    int RSg, RSd, ns, np, part_stride, part_off, ring_off, HPd, TGd;
    uint32_t sb, sbm_g;
    MvsLayer layer[kMvsMaxLayers];
};
bool mvs_supported(int gu_qtype, int down_qtype, int64_t hidden, int64_t ffn, int n_layers, int M);
// Scratch of launch_mvs: its synchronisation words and the slice-major mid.
size_t mvs_scratch_bytes(int64_t hidden, int64_t ffn);
int launch_mvs(MvsArgs a, void* scratch, cudaStream_t s);

// misc.cu
int launch_dequantize(int qtype, const uint8_t* W, int64_t rows, int64_t cols, float* out,
                      cudaStream_t s);
int launch_rms_norm(const float* x, const float* w, float* out, int n, int M, float eps,
                    cudaStream_t s);
int launch_silu_mul(const float* a, const float* b, float* out, int64_t n, cudaStream_t s);
int launch_scale_softcap(float* logits, int64_t n, float scale, float cap, cudaStream_t s);
int launch_dual_tail(float* resid, const float* src, float* out, const float* w1,
                     const float* w2, int n, int M, float eps1, float eps2, cudaStream_t s);
int launch_kv_store(uint16_t* key, uint16_t* value, const float* k, const float* v,
                    int64_t kv_dim, int64_t head_dim, int head_major, int64_t capacity,
                    int64_t phys_of_first, int64_t src_first, int64_t nrows, cudaStream_t s);
// Ch 15 §15.6: rows j < count of a window <-> plane slot (phys0 + j) % capacity;
// to_plane restores detached rows into the plane, else snapshots them out.
int launch_kv_window(uint16_t* key, uint16_t* value, uint16_t* k_rows, uint16_t* v_rows,
                     int64_t kv_dim, int64_t head_dim, int head_major, int64_t capacity,
                     int64_t phys0, int64_t count, bool to_plane, cudaStream_t s);
int launch_spin(int64_t microseconds, cudaStream_t s);
// `ctas` blocks that each hold kOccupySmemBytes of shared memory (one block
// per SM) and busy-wait `microseconds` on the global timer.
constexpr int kOccupySmemBytes = 160 * 1024;
int launch_occupy(int ctas, int64_t microseconds, cudaStream_t s);

}  // namespace muser
