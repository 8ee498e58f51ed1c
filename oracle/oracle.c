/*
 * oracle.c -- plain, slow, fp64 CPU oracle for the decode-FFN quantized weight
 * stream of the Muser engine ("How to Write an Inference Engine -- the Muser
 * book").
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
 * its Python binding) may link, load or call this file.  Only the tests, the
 * GPU smoke check and the CPU-baseline leg of the benchmark use it.  It shares
 * no code, header, table or constant with the CUDA path.
 *
 * Every function computes a plain definition, in double precision, and rounds
 * to binary32 only where the book stores a binary32 buffer.  The steps follow
 * the book's order; there is no blocking, fusion or reordering beyond that.
 * OpenMP only splits independent output rows across threads: each row's sum
 * is the same sequential fp64 loop whichever thread runs it.
 *
 * Readings of the pages (the pages are silent on these points; see DESIGN):
 *  - The Q4_K / Q5_K / Q6_K bit layouts are the ggml/GGUF super-block conventions that
 *    the book's "ggml-style" blocks name; the book gives only the block sizes
 *    (144 B and 210 B per 256 weights, Ch 19 §19.3) and field lists.
 *  - Q4_K value = d*scale*q - dmin*min (ggml form of the book's
 *    "scale x index + min", Ch 5 §5.5).
 *  - SiLU(z) = z / (1 + exp(-z)), the logistic form of the book's sigmoid gate
 *    kernel (Ch 2 §2.7) times z.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_Q4_K 12
#define ORC_Q5_K 13
#define ORC_Q6_K 14
#define ORC_OK 0
#define ORC_ERR_ARG -1
#define ORC_ERR_DISCONTINUITY -4

int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ binary16
 * IEEE 754 binary16 (Ch 5 §5.2, Figure 5.3: 1 sign bit, 5 exponent bits, 10
 * mantissa bits).  Normal: (1 + m/1024) * 2^(e-15); subnormal: m * 2^-24. */
double orc_f16_to_f64(uint16_t h) {
    int sign = h >> 15;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)m, -24);
    } else if (e == 31) {
        v = (m == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + m), e - 25);
    }
    return sign ? -v : v;
}

/* binary32 -> binary16, round to nearest, ties to even, overflow to infinity.
 * This is the conversion the book's KV store performs when it assigns an f32
 * activation to a half plane (Ch 15 §15.4).  rint() rounds in the default
 * to-nearest-even mode. */
uint16_t orc_f32_to_f16(float f) {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t sign = (uint16_t)((bits >> 16) & 0x8000u);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs((double)f);
    /* 65520 is half-way between the largest finite half (65504) and 2^16;
     * ties go to the even neighbour, 2^16, which is out of range. */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u);
    if (a < ldexp(1.0, -14)) {
        /* zero or subnormal: an integer multiple of 2^-24 (1024 carries into
         * the smallest normal, whose encoding is exactly 0x0400) */
        double m = rint(ldexp(a, 24));
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e2;
    (void)frexp(a, &e2);           /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;                /* unbiased exponent */
    double m = rint(ldexp(a, 10 - E)); /* significand with 10 fraction bits */
    if (m == 2048.0) {
        m = 1024.0;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(((E + 15) << 10) | ((int)m - 1024)));
}

void orc_f16_to_f64_array(const uint16_t* h, double* out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_to_f64(h[i]);
}

void orc_f32_to_f16_array(const float* f, uint16_t* out, int64_t n) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(f[i]);
}

static uint16_t rd_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* ---------------------------------------------------------------- Q4_K block
 * 256 weights in 144 bytes: f16 d, f16 dmin, 12 bytes packing eight 6-bit
 * sub-block scales and eight 6-bit sub-block mins, 128 bytes of 4-bit codes.
 * Weight i belongs to sub-block j = i / 32.  Codes: in code byte 32c + l
 * (c = 0..3, l = 0..31) the low nibble is weight 64c + l and the high nibble
 * weight 64c + 32 + l.  Scales/mins of sub-blocks 0..3 are the low six bits
 * of packed bytes j and j+4; those of sub-blocks 4..7 take their low four bits
 * from byte j+4 (low nibble: scale, high nibble: min) and their top two bits
 * from the top two bits of bytes j-4 (scale) and j (min). */
void orc_q4k_scale_min(const uint8_t* s, int j, int* sc, int* mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 0x0f) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

void orc_q4k_block(const uint8_t* blk, float* out) {
    const double d = orc_f16_to_f64(rd_u16(blk));
    const double dmin = orc_f16_to_f64(rd_u16(blk + 2));
    const uint8_t* s = blk + 4;
    const uint8_t* qs = blk + 16;
    for (int i = 0; i < 256; ++i) {
        const int c = i / 64;
        const int hi = (i % 64) >= 32;
        const int l = i % 32;
        const int byte = qs[32 * c + l];
        const int q = hi ? (byte >> 4) : (byte & 0x0f);
        int sc, mn;
        orc_q4k_scale_min(s, i / 32, &sc, &mn);
        /* d*sc*q and dmin*mn are integer multiples of 2^-24 below 2^26, so the
         * difference is exact in fp64; the cast is the one rounding. */
        out[i] = (float)(d * sc * q - dmin * mn);
    }
}

/* ---------------------------------------------------------------- Q5_K block
 * The third k-quant of the book's kernel registry (Ch 4 §4.4), which names the
 * type but not its layout; the layout is the ggml/GGUF one.  256 weights in
 * 176 bytes: f16 d, f16 dmin, the same 12 packed bytes of 6-bit scales and
 * mins as Q4_K, 32 bytes of fifth code bits (qh), 128 bytes of 4-bit codes.
 * Weight i = 64c + 32h + l (c = 0..3, h = 0/1, l = 0..31) belongs to sub-block
 * 2c + h; its low four bits are the low (h = 0) or high (h = 1) nibble of code
 * byte 32c + l, its fifth bit is bit 2c + h of qh[l], and its value is
 * d*sc*q - dmin*min with q = 0..31. */
void orc_q5k_block(const uint8_t* blk, float* out) {
    const double d = orc_f16_to_f64(rd_u16(blk));
    const double dmin = orc_f16_to_f64(rd_u16(blk + 2));
    const uint8_t* s = blk + 4;
    const uint8_t* qh = blk + 16;
    const uint8_t* qs = blk + 48;
    for (int i = 0; i < 256; ++i) {
        const int c = i / 64;
        const int h = (i % 64) >= 32;
        const int l = i % 32;
        const int byte = qs[32 * c + l];
        const int low = h ? (byte >> 4) : (byte & 0x0f);
        const int top = (qh[l] >> (2 * c + h)) & 1;
        const int q = low | (top << 4);
        int sc, mn;
        orc_q4k_scale_min(s, i / 32, &sc, &mn);
        /* as for Q4_K: both products are integer multiples of 2^-24 below
         * 2^27, so the difference is exact in fp64 and the cast rounds once */
        out[i] = (float)(d * sc * q - dmin * mn);
    }
}

/* ---------------------------------------------------------------- Q6_K block
 * 256 weights in 210 bytes: 128 bytes of low 4-bit codes (ql), 64 bytes of
 * high 2-bit codes (qh), 16 int8 sub-block scales, f16 d.  Weight i: half
 * h = i / 128, group g = (i % 128) / 32, l = i % 32.  Its low nibble is the
 * low (g = 0, 1) or high (g = 2, 3) nibble of ql[64h + 32*(g&1) + l]; its high
 * two bits are bits 2g..2g+1 of qh[32h + l].  The 6-bit code q is offset by 32
 * and scaled by scale[i / 16] and d. */
void orc_q6k_block(const uint8_t* blk, float* out) {
    const uint8_t* ql = blk;
    const uint8_t* qh = blk + 128;
    const int8_t* sc = (const int8_t*)(blk + 192);
    const double d = orc_f16_to_f64(rd_u16(blk + 208));
    for (int i = 0; i < 256; ++i) {
        const int h = i / 128;
        const int g = (i % 128) / 32;
        const int l = i % 32;
        const int lo = ql[64 * h + 32 * (g & 1) + l];
        const int nib = (g & 2) ? (lo >> 4) : (lo & 0x0f);
        const int top = (qh[32 * h + l] >> (2 * g)) & 3;
        const int q = nib | (top << 4);
        out[i] = (float)(d * (double)sc[i / 16] * (double)(q - 32));
    }
}

static int block_bytes(int qtype) {
    return qtype == ORC_Q4_K ? 144 : (qtype == ORC_Q5_K ? 176 : (qtype == ORC_Q6_K ? 210 : 0));
}

static void decode_block(int qtype, const uint8_t* blk, float* out) {
    if (qtype == ORC_Q4_K) orc_q4k_block(blk, out);
    else if (qtype == ORC_Q5_K) orc_q5k_block(blk, out);
    else orc_q6k_block(blk, out);
}

/* out[r*cols + k] = binary32 dequantised weight (row-major). */
int orc_dequantize(int qtype, const uint8_t* W, int64_t rows, int64_t cols, float* out) {
    const int bb = block_bytes(qtype);
    if (!bb || cols % 256 || rows < 0) return ORC_ERR_ARG;
    const int64_t nsb = cols / 256;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t b = 0; b < nsb; ++b)
            decode_block(qtype, W + (r * nsb + b) * bb, out + r * cols + b * 256);
    return ORC_OK;
}

/* ------------------------------------------------------------------ matvec
 * y[m][r] = sum_k w[r][k] * x[m][k] (Ch 19 §19.1 operation 1; Ch 1's
 * one-token projection).  The binary32 dequantised weights times the binary32
 * inputs, summed in fp64 in k order, rounded once to binary32.
 * Layout: W rows of consecutive super-blocks; x and y row-major [M][.]. */
static void matvec_row(int qtype, const uint8_t* Wrow, int64_t cols, const float* x, int64_t M,
                       double* acc) {
    const int bb = block_bytes(qtype);
    float w[256];
    for (int64_t m = 0; m < M; ++m) acc[m] = 0.0;
    for (int64_t b = 0; b < cols / 256; ++b) {
        decode_block(qtype, Wrow + b * bb, w);
        for (int64_t m = 0; m < M; ++m) {
            const float* xm = x + m * cols + b * 256;
            double s = acc[m];
            for (int i = 0; i < 256; ++i) s += (double)w[i] * (double)xm[i];
            acc[m] = s;
        }
    }
}

int orc_qmatvec(int qtype, const uint8_t* W, int64_t rows, int64_t cols, const float* x, int64_t M,
                float* y) {
    const int bb = block_bytes(qtype);
    if (!bb || cols % 256 || M < 1 || M > 64) return ORC_ERR_ARG;
    const int64_t row_bytes = (cols / 256) * bb;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double acc[64];
        matvec_row(qtype, W + r * row_bytes, cols, x, M, acc);
        for (int64_t m = 0; m < M; ++m) y[m * rows + r] = (float)acc[m];
    }
    return ORC_OK;
}

/* The same sums for a chosen subset of output rows: y[m][i] for row ridx[i]. */
int orc_qmatvec_rows(int qtype, const uint8_t* W, int64_t rows, int64_t cols, const int64_t* ridx,
                     int64_t nr, const float* x, int64_t M, float* y) {
    const int bb = block_bytes(qtype);
    if (!bb || cols % 256 || M < 1 || M > 64) return ORC_ERR_ARG;
    const int64_t row_bytes = (cols / 256) * bb;
    for (int64_t i = 0; i < nr; ++i)
        if (ridx[i] < 0 || ridx[i] >= rows) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nr; ++i) {
        double acc[64];
        matvec_row(qtype, W + ridx[i] * row_bytes, cols, x, M, acc);
        for (int64_t m = 0; m < M; ++m) y[m * nr + i] = (float)acc[m];
    }
    return ORC_OK;
}

/* ----------------------------------------------------------------- RMSNorm
 * out_i = w_i * x_i / sqrt(mean(x^2) + eps), per row of n (Ch 2 §2.6,
 * rms_norm_batch: the eps is added to the mean inside the root). */
void orc_rms_norm(const float* x, const float* w, int64_t n, int64_t M, double eps, float* out) {
    for (int64_t m = 0; m < M; ++m) {
        const float* xr = x + m * n;
        double ss = 0.0;
        for (int64_t i = 0; i < n; ++i) ss += (double)xr[i] * (double)xr[i];
        const double inv = 1.0 / sqrt(ss / (double)n + eps);
        for (int64_t i = 0; i < n; ++i) out[m * n + i] = (float)((double)w[i] * (double)xr[i] * inv);
    }
}

/* ------------------------------------------------------ dual-eps fused tail
 * Ch 19 §19.1 operation 2 and §19.4 (muser_fused_norm_residual_rms_norm_32sg),
 * Ch 10 Figure 10.2:
 *     hidden += w1 * rms_norm(src, eps1)       (residual update, in place)
 *     out     = w2 * rms_norm(hidden, eps2)
 * The updated residual is a binary32 buffer that the second norm reads back
 * (§19.7: a fusion may delete dispatches, not rounding points), so h is
 * rounded to binary32 before its mean square is taken. */
void orc_dual_tail(const float* r_in, const float* src, const float* w1, const float* w2, int64_t n,
                   int64_t M, double eps1, double eps2, float* r_out, float* out) {
    for (int64_t m = 0; m < M; ++m) {
        const float* p = src + m * n;
        const float* r = r_in + m * n;
        float* h = r_out + m * n;
        double sp = 0.0;
        for (int64_t i = 0; i < n; ++i) sp += (double)p[i] * (double)p[i];
        const double inv1 = 1.0 / sqrt(sp / (double)n + eps1);
        for (int64_t i = 0; i < n; ++i)
            h[i] = (float)((double)r[i] + (double)w1[i] * (double)p[i] * inv1);
        double sh = 0.0;
        for (int64_t i = 0; i < n; ++i) sh += (double)h[i] * (double)h[i];
        const double inv2 = 1.0 / sqrt(sh / (double)n + eps2);
        for (int64_t i = 0; i < n; ++i) out[m * n + i] = (float)((double)w2[i] * (double)h[i] * inv2);
    }
}

/* -------------------------------------------------------------------- SiLU */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

void orc_silu_mul(const float* a, const float* b, int64_t n, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)(orc_silu((double)a[i]) * (double)b[i]);
}

/* ---------------------------------------------- LM head scale + soft cap */
/* Ch 10 Figure 10.1 boxes 14 and 15: the LM head is a matvec of the final
 * normed hidden row (its binary32 logits are written out), then
 * muser_scale_softcap_inplace multiplies each logit by the logit scale and
 * caps it as cap * tanh(l / cap).  Here the scaled and capped value is taken
 * in fp64 from the binary32 logit and rounded once. */
double orc_softcap(double l, double scale, double cap) { return cap * tanh(l * scale / cap); }

void orc_scale_softcap(const float* logits, int64_t n, double scale, double cap, float* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = (float)orc_softcap((double)logits[i], scale, cap);
}

/* FFN gate/up/SiLU (Ch 10 Figure 10.1 box 11): g = Wg.x and u = Wu.x are
 * binary32 activations (the book's default route writes both, then applies
 * SiLU in place), mid = silu(g) * u.  mid is [M][ffn]. */
int orc_gate_up_silu(int qtype, const uint8_t* Wg, const uint8_t* Wu, int64_t ffn, int64_t hidden,
                     const float* x, int64_t M, float* mid) {
    float* g = (float*)malloc(sizeof(float) * (size_t)(ffn * M));
    float* u = (float*)malloc(sizeof(float) * (size_t)(ffn * M));
    if (!g || !u) {
        free(g);
        free(u);
        return ORC_ERR_ARG;
    }
    int rc = orc_qmatvec(qtype, Wg, ffn, hidden, x, M, g);
    if (rc == ORC_OK) rc = orc_qmatvec(qtype, Wu, ffn, hidden, x, M, u);
    if (rc == ORC_OK) orc_silu_mul(g, u, ffn * M, mid);
    free(g);
    free(u);
    return rc;
}

/* --------------------------------------------------------------- KV ring
 * Ch 15 §15.5, append: the write row for `position` comes from explicit ring
 * metadata, never from the absolute position.  A position other than
 * origin_logical + len is a cache discontinuity and changes nothing. */
typedef struct {
    int64_t capacity, len, origin_logical, origin_physical;
} orc_ring;

int orc_ring_append(orc_ring* r, int64_t position, int64_t* write) {
    const int64_t expected = r->origin_logical + r->len;
    if (position != expected) return ORC_ERR_DISCONTINUITY;
    if (r->len < r->capacity) {
        *write = (r->origin_physical + r->len) % r->capacity;
        r->len += 1;
    } else {
        *write = r->origin_physical;
        r->origin_logical += 1;
        r->origin_physical = (r->origin_physical + 1) % r->capacity;
    }
    return ORC_OK;
}

/* Store `count` consecutive token rows of K and V (binary32, [count][kv_dim])
 * into binary16 planes, one append per row (Ch 15 §15.5 append_batch is the
 * chunked form of the same sequence).  Token-major destination:
 * physical*kv_dim + e; head-major: (e/head_dim * capacity + physical) *
 * head_dim + e%head_dim (Ch 15 §15.3, Figure 15.1). */
int orc_kv_write(orc_ring* r, uint16_t* key, uint16_t* value, int64_t kv_dim, int64_t head_dim,
                 int head_major, const float* k, const float* v, int64_t position, int64_t count,
                 int64_t* first_write) {
    if (count < 0 || kv_dim <= 0 || (head_major && (head_dim <= 0 || kv_dim % head_dim)))
        return ORC_ERR_ARG;
    if (position != r->origin_logical + r->len) return ORC_ERR_DISCONTINUITY;
    for (int64_t t = 0; t < count; ++t) {
        int64_t w;
        int rc = orc_ring_append(r, position + t, &w);
        if (rc != ORC_OK) return rc;
        if (t == 0 && first_write) *first_write = w;
        for (int64_t e = 0; e < kv_dim; ++e) {
            int64_t dst = w * kv_dim + e;
            if (head_major) dst = ((e / head_dim) * r->capacity + w) * head_dim + e % head_dim;
            key[dst] = orc_f32_to_f16(k[t * kv_dim + e]);
            value[dst] = orc_f32_to_f16(v[t * kv_dim + e]);
        }
    }
    return ORC_OK;
}

/* Element e of the token row held in physical slot p, in either layout
 * (Ch 15 §15.3, Figure 15.1). */
static int64_t orc_kv_index(int64_t p, int64_t e, int64_t kv_dim, int64_t head_dim, int head_major,
                            int64_t capacity) {
    return head_major ? ((e / head_dim) * capacity + p) * head_dim + e % head_dim : p * kv_dim + e;
}

/* Detached copy of live rows (Ch 15 §15.6): logical rows first..first+count-1,
 * which must lie inside the live window [origin_logical, origin_logical+len),
 * are written in logical order as token-major binary16 rows [count][kv_dim].
 * The row of logical position q sits in slot
 * (origin_physical + q - origin_logical) % capacity. */
int orc_kv_snapshot(const orc_ring* r, const uint16_t* key, const uint16_t* value, int64_t kv_dim,
                    int64_t head_dim, int head_major, int64_t first, int64_t count, uint16_t* k_rows,
                    uint16_t* v_rows) {
    if (count < 0 || kv_dim <= 0 || (head_major && (head_dim <= 0 || kv_dim % head_dim)))
        return ORC_ERR_ARG;
    if (first < r->origin_logical || first + count > r->origin_logical + r->len) return ORC_ERR_ARG;
    for (int64_t j = 0; j < count; ++j) {
        const int64_t p = (r->origin_physical + (first + j - r->origin_logical)) % r->capacity;
        for (int64_t e = 0; e < kv_dim; ++e) {
            const int64_t src = orc_kv_index(p, e, kv_dim, head_dim, head_major, r->capacity);
            k_rows[j * kv_dim + e] = key[src];
            v_rows[j * kv_dim + e] = value[src];
        }
    }
    return ORC_OK;
}

/* Rotation-preserving restore (Ch 15 §15.6; Ch 10 §10.7): a detached window of
 * `len` logical rows starting at logical position `origin` is installed at the
 * rotation a ring built by sequential appends from position 0 holds there,
 * origin % capacity.  Logical row j goes to slot (origin % capacity + j) %
 * capacity, and the metadata becomes (len, origin, origin % capacity).  Slots
 * outside the window are not written.  A NoPE plane (origin 0) reduces to the
 * plain layout. */
int orc_kv_restore(orc_ring* r, uint16_t* key, uint16_t* value, int64_t kv_dim, int64_t head_dim,
                   int head_major, const uint16_t* k_rows, const uint16_t* v_rows, int64_t origin,
                   int64_t len) {
    if (kv_dim <= 0 || (head_major && (head_dim <= 0 || kv_dim % head_dim))) return ORC_ERR_ARG;
    if (origin < 0 || len < 0 || len > r->capacity) return ORC_ERR_ARG;
    const int64_t rotation = origin % r->capacity;
    for (int64_t j = 0; j < len; ++j) {
        const int64_t p = (rotation + j) % r->capacity;
        for (int64_t e = 0; e < kv_dim; ++e) {
            const int64_t dst = orc_kv_index(p, e, kv_dim, head_dim, head_major, r->capacity);
            key[dst] = k_rows[j * kv_dim + e];
            value[dst] = v_rows[j * kv_dim + e];
        }
    }
    r->len = len;
    r->origin_logical = origin;
    r->origin_physical = rotation;
    return ORC_OK;
}
