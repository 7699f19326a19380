/*
 * splitkv_oracle.c -- fp64 CPU oracle for split-KV flash attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA library is checked against.  Only the test suite, the smoke check and
 * the benchmark's CPU-baseline leg load it; the library never does, and this
 * file includes nothing of the library (no shared headers, helpers or tables).
 *
 * What it computes, and where each definition comes from:
 *
 *  - Cache row layout and GQA mapping: a cache row holds all KV heads of one
 *    position, cell-major ("Rolling KV -- position-windowed KV residency",
 *    opencoti patch 0070, KV-cache window/tail tensors); q head h reads KV head
 *    h / (H/Hk) (same page, streaming_lse_kernel's head mapping).
 *  - The paged host layout [block][Hk][page_rows][D] of the block-cache
 *    workload ("Strata compare", KV streaming, KvHostPools identity layout).
 *  - q8_0 / q4_0 decoding: value = d*q and value = d*(u-8) with a per-32-value
 *    fp16 scale d.  The pages name the types and their 32-value blocks (patch
 *    0070 sizer; patch 0102 on raw quant bytes) but print no byte layout; this
 *    oracle reads the usual ggml block layout (2-byte fp16 scale, then the
 *    codes; q4_0 keeps value j in the low nibble of byte j and value j+16 in
 *    the high nibble).
 *  - Row indirection: key j of sequence s reads cache row kv_rows[s][j]; a
 *    negative entry is padding and the key is absent ("llama + CUDA:
 *    flash_attn_ext_rows (fix unified kv for multi-seq)", the op's doc comment).
 *  - Attention: s_j = scale * q.k_j + mask_j; O = sum_j e^{s_j-M} v_j / Z,
 *    lse = M + ln Z, M = max_j s_j, Z = sum_j e^{s_j-M}; an all-masked row
 *    gives O = 0 and lse = -inf (patch 0070, streaming_lse_kernel and the
 *    tail-partial conversion kernel's empty-row convention).  Computed in two
 *    passes over the keys (max, then sums), not online.
 *  - Combine: M = max_t lse_t; w_t = e^{lse_t-M} (0 when lse_t = -inf);
 *    O = sum_t w_t O_t / sum_t w_t; lse = M + ln sum_t w_t (patch 0070,
 *    fattn.cu key-axis tiling comment and streaming_combine_kernel; the lse
 *    output of the combine is this library's addition).
 *
 * Parallelism: OpenMP over independent (sequence, token, q-head) rows only;
 * each row's arithmetic is sequential in key order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F16 = 0, ORC_Q8_0 = 1, ORC_Q4_0 = 2 };
enum { ORC_CELL_MAJOR = 0, ORC_PAGED = 1 };

/* IEEE 754 binary16 -> double, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_half_to_double(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);            /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/2^10) * 2^(e-15) */
    return sign ? -v : v;
}

static uint16_t rd_u16(const uint8_t *p)
{
    /* little-endian two-byte load */
    return (uint16_t)(p[0] | ((uint16_t)p[1] << 8));
}

/* Bytes that one head's D values occupy in a row of the given type. */
int64_t orc_segment_bytes(int type, int D)
{
    switch (type) {
    case ORC_F16: return 2 * (int64_t)D;
    case ORC_Q8_0: return 34 * (int64_t)(D / 32);
    case ORC_Q4_0: return 18 * (int64_t)(D / 32);
    default: return -1;
    }
}

/* Decode n values (n a multiple of 32 for the quantised types). */
static void decode_values(int type, const uint8_t *src, int64_t n, double *out)
{
    if (type == ORC_F16) {
        for (int64_t i = 0; i < n; ++i)
            out[i] = orc_half_to_double(rd_u16(src + 2 * i));
    } else if (type == ORC_Q8_0) {
        for (int64_t b = 0; b < n / 32; ++b) {
            const uint8_t *blk = src + 34 * b;
            const double d = orc_half_to_double(rd_u16(blk));
            for (int i = 0; i < 32; ++i)
                out[32 * b + i] = d * (double)(int8_t)blk[2 + i];
        }
    } else if (type == ORC_Q4_0) {
        for (int64_t b = 0; b < n / 32; ++b) {
            const uint8_t *blk = src + 18 * b;
            const double d = orc_half_to_double(rd_u16(blk));
            for (int j = 0; j < 16; ++j) {
                const int lo = blk[2 + j] & 0x0f;
                const int hi = (blk[2 + j] >> 4) & 0x0f;
                out[32 * b + j] = d * (double)(lo - 8);
                out[32 * b + j + 16] = d * (double)(hi - 8);
            }
        }
    }
}

/* Exported: decode n_values quantised (or fp16) values into doubles. */
int orc_dequant(int type, const void *src, int64_t n_values, double *out)
{
    if (type != ORC_F16 && (n_values % 32) != 0) return 1;
    if (type < ORC_F16 || type > ORC_Q4_0) return 1;
    decode_values(type, (const uint8_t *)src, n_values, out);
    return 0;
}

/* A key source: one cache region, cell-major [row][Hk][seg] with a row stride
 * in bytes, or paged [row/page_rows][Hk][page_rows][seg]. */
typedef struct {
    const uint8_t *base;
    int64_t n_rows;
    int64_t row_bytes;   /* cell-major stride between rows */
    int layout;          /* ORC_CELL_MAJOR or ORC_PAGED */
    int page_rows;       /* paged layout only */
} orc_source;

static const uint8_t *source_segment(const orc_source *src, int64_t row, int head,
                                     int Hk, int64_t seg)
{
    if (src->layout == ORC_PAGED) {
        const int64_t blk = row / src->page_rows;
        const int64_t in_blk = row % src->page_rows;
        return src->base + ((blk * Hk + head) * src->page_rows + in_blk) * seg;
    }
    return src->base + row * src->row_bytes + (int64_t)head * seg;
}

/*
 * Attention of every (s, t, h) row over a logical key list.
 *
 * Logical rows: index x < n_rows of region 0 addresses region 0; index x >= that
 * addresses region 1 at x - n_rows0 (the device window [0, wc) followed by the
 * host tail [wc, n_kv) of patch 0070's two-region forward).
 * Key j (0 <= j < n_keys) of sequence s (and KV head k when rows_per_head):
 *   row_j = kv_rows ? kv_rows[(s*RH + k)*n_keys + j] : j,   RH = rows_per_head ? Hk : 1
 *   row_j < 0  -> padding, absent.
 *   causal (q_pos != NULL): key visible iff key_pos0 + j <= q_pos[s*nq + t].
 *   mask (fp16 bits, NULL allowed): additive term mask[(s*nq + t)*n_keys + j].
 * Outputs: O[(s*nq + t)*H + h][D] and lse[(s*nq + t)*H + h], fp64.
 */
int orc_attention(int S, int nq, int H, int Hk, int D, double scale,
                  const uint16_t *q, int k_type, int v_type,
                  const void *k0, const void *v0, int64_t n_rows0,
                  int64_t k_row_bytes0, int64_t v_row_bytes0,
                  const void *k1, const void *v1, int64_t n_rows1,
                  int64_t k_row_bytes1, int64_t v_row_bytes1,
                  int layout, int page_rows,
                  int64_t n_keys, const int32_t *kv_rows, int rows_per_head,
                  const uint16_t *mask, const int32_t *q_pos, int64_t key_pos0,
                  double *out_o, double *out_lse)
{
    if (S <= 0 || nq <= 0 || H <= 0 || Hk <= 0 || D <= 0 || H % Hk != 0) return 1;
    if ((k_type != ORC_F16 || v_type != ORC_F16) && D % 32 != 0) return 1;
    const int G = H / Hk;
    const int64_t segk = orc_segment_bytes(k_type, D);
    const int64_t segv = orc_segment_bytes(v_type, D);
    if (segk < 0 || segv < 0) return 1;
    orc_source ks[2] = {{(const uint8_t *)k0, n_rows0, k_row_bytes0, layout, page_rows},
                        {(const uint8_t *)k1, n_rows1, k_row_bytes1, layout, page_rows}};
    orc_source vs[2] = {{(const uint8_t *)v0, n_rows0, v_row_bytes0, layout, page_rows},
                        {(const uint8_t *)v1, n_rows1, v_row_bytes1, layout, page_rows}};
    const int64_t n_out = (int64_t)S * nq * H;
    int err = 0;

#pragma omp parallel
    {
        double *sc = (double *)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
        double *qv = (double *)malloc(sizeof(double) * (size_t)D);
        double *kv = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        if (!sc || !qv || !kv || !acc) {
#pragma omp atomic write
            err = 2;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t r = 0; r < n_out; ++r) {
                const int64_t st = r / H;          /* s*nq + t */
                const int h = (int)(r % H);
                const int s = (int)(st / nq);
                const int k = h / G;
                const int64_t list = rows_per_head ? ((int64_t)s * Hk + k) : s;
                for (int d = 0; d < D; ++d) qv[d] = orc_half_to_double(q[r * D + d]);

                /* pass 1: scores and their maximum */
                double M = -INFINITY;
                for (int64_t j = 0; j < n_keys; ++j) {
                    const int64_t row = kv_rows ? (int64_t)kv_rows[list * n_keys + j] : j;
                    int visible = row >= 0 && row < n_rows0 + n_rows1;
                    if (visible && q_pos && key_pos0 + j > (int64_t)q_pos[st]) visible = 0;
                    if (!visible) { sc[j] = -INFINITY; continue; }
                    const int reg = row < n_rows0 ? 0 : 1;
                    const int64_t lr = reg ? row - n_rows0 : row;
                    decode_values(k_type, source_segment(&ks[reg], lr, k, Hk, segk), D, kv);
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += qv[d] * kv[d];
                    double sj = scale * dot;
                    if (mask) sj += orc_half_to_double(mask[st * n_keys + j]);
                    sc[j] = sj;
                    if (sj > M) M = sj;
                }
                double *o = out_o + r * D;
                if (M == -INFINITY) {
                    for (int d = 0; d < D; ++d) o[d] = 0.0;
                    out_lse[r] = -INFINITY;
                    continue;
                }
                /* pass 2: normaliser and weighted sum of values */
                double Z = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int64_t j = 0; j < n_keys; ++j) {
                    if (sc[j] == -INFINITY) continue;
                    const double w = exp(sc[j] - M);
                    const int64_t row = kv_rows ? (int64_t)kv_rows[list * n_keys + j] : j;
                    const int reg = row < n_rows0 ? 0 : 1;
                    const int64_t lr = reg ? row - n_rows0 : row;
                    decode_values(v_type, source_segment(&vs[reg], lr, k, Hk, segv), D, kv);
                    Z += w;
                    for (int d = 0; d < D; ++d) acc[d] += w * kv[d];
                }
                for (int d = 0; d < D; ++d) o[d] = acc[d] / Z;
                out_lse[r] = M + log(Z);
            }
        }
        free(sc); free(qv); free(kv); free(acc);
    }
    return err;
}

/*
 * Log-sum-exp combine of n_parts partial results over disjoint key sets.
 * o_parts [n_parts][rows][D], lse_parts [n_parts][rows] -> o [rows][D], lse [rows].
 */
int orc_combine(int n_parts, int64_t rows, int D,
                const double *o_parts, const double *lse_parts,
                double *o, double *lse)
{
    if (n_parts < 0 || rows < 0 || D <= 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < n_parts; ++p)
            if (lse_parts[(int64_t)p * rows + r] > M) M = lse_parts[(int64_t)p * rows + r];
        double *out = o + r * D;
        if (M == -INFINITY) {
            for (int d = 0; d < D; ++d) out[d] = 0.0;
            lse[r] = -INFINITY;
            continue;
        }
        double W = 0.0;
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        for (int p = 0; p < n_parts; ++p) {
            const double l = lse_parts[(int64_t)p * rows + r];
            if (l == -INFINITY) continue;
            const double w = exp(l - M);
            W += w;
            const double *op = o_parts + ((int64_t)p * rows + r) * D;
            for (int d = 0; d < D; ++d) out[d] += w * op[d];
        }
        for (int d = 0; d < D; ++d) out[d] /= W;
        lse[r] = M + log(W);
    }
    return 0;
}

/* Threads the OpenMP runtime will use (1 without OpenMP). */
int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---- appending rows ------------------------------------------------------
 *
 * Definitions (write routing: "Rolling KV", opencoti patch 0070, the window /
 * host-tail split of the K/V copies; write-through: "Strata compare", KV
 * streaming, the kv_append writers and their identity-layout host copy;
 * quantisation: the same page's kv_append_q8 kernel):
 *  - fp16 rows: each fp32 value rounded to the nearest binary16, ties to even.
 *  - q8_0 block of 32 values, fp32 arithmetic: d = fp16(amax / 127);
 *    q = nearest integer (ties to even) of x / d, clamped to [-127, 127];
 *    d = 0 gives all codes 0.  The page's scale covers 64 values; the cache
 *    rows here are q8_0, whose scale covers 32.
 *  - q4_0 block: d = fp16(amax / 7); u = nearest integer of x / d, plus 8,
 *    clamped to [0, 15]; byte j holds u_j (low nibble) and u_{j+16} (high).
 *    The pages give no q4_0 quantiser: this reading keeps the q8 rule.
 */

/* fp32 -> IEEE 754 binary16, round to nearest, ties to even, from the format's
 * definition (value = 2^(e-15) * (1 + f/1024), subnormals 2^-24 * f).  The
 * scalings below are by powers of two, so they are exact in double. */
uint16_t orc_float_to_half(float xf)
{
    const double x = (double)xf;
    const uint16_t sign = signbit(x) ? 0x8000 : 0;
    const double a = fabs(x);
    if (isnan(a)) return sign | 0x7e00;
    if (isinf(a)) return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {                       /* subnormal range: units of 2^-24 */
        const double f = nearbyint(ldexp(a, 24));      /* 1024 here is the smallest normal */
        return sign | (uint16_t)f;
    }
    int e2;
    frexp(a, &e2);                                   /* a in [2^(e2-1), 2^e2) */
    int e = e2 - 1;
    double f = nearbyint(ldexp(a, 10 - e));          /* significand in units of 2^(e-10) */
    if (f == 2048.0) {                               /* rounded up to the next binade */
        f = 1024.0;
        e += 1;
    }
    if (e + 15 >= 31) return sign | 0x7c00;          /* overflow to infinity */
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)(f - 1024.0);
}

/* One 32-value block of q8_0 (34 bytes) or q4_0 (18 bytes). */
static void quantize_block(int type, const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) {
        const float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    const float qmax = type == ORC_Q8_0 ? 127.0f : 7.0f;
    const uint16_t dbits = orc_float_to_half(amax / qmax);
    const float d = (float)orc_half_to_double(dbits);
    blk[0] = (uint8_t)(dbits & 0xff);                /* little-endian fp16 scale */
    blk[1] = (uint8_t)(dbits >> 8);
    int code[32];
    for (int i = 0; i < 32; ++i) code[i] = d > 0.0f ? (int)rintf(x[i] / d) : 0;
    if (type == ORC_Q8_0) {
        for (int i = 0; i < 32; ++i) {
            int q = code[i];
            if (q < -127) q = -127;
            if (q > 127) q = 127;
            blk[2 + i] = (uint8_t)(int8_t)q;
        }
    } else {
        for (int j = 0; j < 16; ++j) {
            int lo = code[j] + 8, hi = code[j + 16] + 8;
            lo = lo < 0 ? 0 : (lo > 15 ? 15 : lo);
            hi = hi < 0 ? 0 : (hi > 15 ? 15 : hi);
            blk[2 + j] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* Encode D values (one head) into its segment of the given type. */
static void encode_segment(int type, const float *x, int D, uint8_t *seg)
{
    if (type == ORC_F16) {
        for (int d = 0; d < D; ++d) {
            const uint16_t b = orc_float_to_half(x[d]);
            seg[2 * d] = (uint8_t)(b & 0xff);
            seg[2 * d + 1] = (uint8_t)(b >> 8);
        }
        return;
    }
    const int blk = type == ORC_Q8_0 ? 34 : 18;
    for (int b = 0; b < D / 32; ++b) quantize_block(type, x + 32 * b, seg + (int64_t)b * blk);
}

/* Exported: encode n_values (a multiple of 32 for quantised types) values. */
int orc_quantize(int type, const float *x, int64_t n_values, void *out)
{
    if (orc_segment_bytes(type, 32) < 0 || n_values < 0 || (type != ORC_F16 && n_values % 32)) return 1;
    uint8_t *o = (uint8_t *)out;
    if (type == ORC_F16) {
        encode_segment(ORC_F16, x, (int)n_values, o);
        return 0;
    }
    const int blk = type == ORC_Q8_0 ? 34 : 18;
    for (int64_t b = 0; b < n_values / 32; ++b) quantize_block(type, x + 32 * b, o + b * blk);
    return 0;
}

/* Cell-major append: row i of x ([n][Hk][D] fp32) goes to cache position
 * positions[i]; p < n_rows0 is row p of region 0, otherwise row p - n_rows0 of
 * region 1 (row stride row_bytes, head k at byte k * segment).  Negative
 * positions are skipped; positions >= n_rows0 + n_rows1 are skipped and
 * counted.  Rows are written in order i = 0, 1, ...  Returns the count of
 * out-of-range positions, or -1 for bad arguments. */
int64_t orc_kv_append(int type, int Hk, int D, int64_t row_bytes, const float *x, const int32_t *positions,
                      int64_t n, void *dst0, int64_t n_rows0, void *dst1, int64_t n_rows1)
{
    const int64_t seg = orc_segment_bytes(type, D);
    if (seg < 0 || D % 32 || row_bytes < Hk * seg) return -1;
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t p = positions[i];
        if (p < 0) continue;
        if (p >= n_rows0 + n_rows1) {
            ++bad;
            continue;
        }
        uint8_t *row = p < n_rows0 ? (uint8_t *)dst0 + p * row_bytes : (uint8_t *)dst1 + (p - n_rows0) * row_bytes;
        for (int k = 0; k < Hk; ++k) encode_segment(type, x + (i * Hk + k) * D, D, row + k * seg);
    }
    return bad;
}

/* Paged append into a host copy laid out [n_blocks][Hk][block_rows][D] fp16:
 * position p, head k lands at page (p / block_rows) * Hk + k, row
 * p % block_rows.  Same skipping and return value as orc_kv_append. */
int64_t orc_paged_append(int Hk, int D, int block_rows, int64_t n_blocks, const float *x, const int32_t *positions,
                         int64_t n, uint16_t *host)
{
    if (Hk <= 0 || D <= 0 || block_rows <= 0) return -1;
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t p = positions[i];
        if (p < 0) continue;
        if (p >= n_blocks * block_rows) {
            ++bad;
            continue;
        }
        const int64_t blk = p / block_rows, in_blk = p % block_rows;
        for (int k = 0; k < Hk; ++k) {
            uint16_t *dst = host + (((blk * Hk + k) * block_rows) + in_blk) * D;
            for (int d = 0; d < D; ++d) dst[d] = orc_float_to_half(x[(i * Hk + k) * D + d]);
        }
    }
    return bad;
}
