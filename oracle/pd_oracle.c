/*
 * pd_oracle.c -- plain FP64 CPU oracle for paged-decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header or constant with the
 * CUDA library; the two are independent statements of the same definition.
 *
 * What it computes (written from the pages, not from any kernel):
 *
 *   For a sequence s and a query head h, with G = num_q_heads / num_kv_heads
 *   and kvh = h / G (consecutive query heads share one KV head), let the
 *   sequence's tokens be t = 0 .. L_s-1, where token t lives in physical block
 *   block_table[s][t / block_size] at row t % block_size of the paged cache
 *   [num_blocks, block_size, num_kv_heads, head_dim].  Then
 *
 *       x_t  = inv_sqrt_d * sum_d q[s,h,d] * K[t,kvh,d]
 *       out  = sum_t exp(x_t - max x) V[t,kvh,:] / sum_t exp(x_t - max x)
 *
 *   and out = 0 when the sequence has no token (the "0 where l is 0" rule of
 *   the tiled_attention.rs page, TiledAttention::finalize, and of the module
 *   doc of the same page).
 *
 *   Every BF16 input is widened exactly to double; inv_sqrt_d is the FP32
 *   value the caller passes, widened.  All arithmetic is FP64 in the plain
 *   order written above: no blocking, no reordering, no fusion.
 *
 *   orc_split_replay is a second mode used only to check split invariance:
 *   it takes the steps of the split-K method in the order the pages describe
 *   them (Module attn_splitk page: the split-K workspace of [o, m, l] slots
 *   and the non-associative merge; tiled_attention.rs page: the running
 *   (m, l, o) state set to (-inf, 0, 0), folded tile by tile, and finalised
 *   as o / l).  It is exact arithmetic re-association of the definition above.
 *
 *   orc_tiled_attn covers the begin_step / step_tile / finalize interface of
 *   the tiled_attention.rs page: the token set is every block named by the
 *   tiles of every step_tile call, the last block of a sequence's tile in a
 *   call holding last_block_valid_slots tokens (values outside
 *   1 .. block_size-1 mean a full block), K and V addressed through the
 *   (blk, tok, kvh) element strides the caller passes, and the scale
 *   1/sqrt(head_dim) rounded to FP32 because step_tile carries no scale.
 *   orc_tiled_attn_multi is the same with every call naming its own K and V
 *   pools and strides (the page's step_tile takes them per call, so one step
 *   may mix the paged layout and the scratch-pool layout).
 *
 *   orc_decode_attn_fp8 is the paged definition over an FP8 KV cache (the
 *   Module attn_splitk page names BF16 and FP8 paged-decode launches but no
 *   format or scale).  Reading: OCP FP8 E4M3 (sign, 4 exponent bits with bias
 *   7, 3 mantissa bits; no infinities; exponent 15 with mantissa 7 is NaN),
 *   one FP32 scale per tensor: K = e4m3(k_code) * k_scale, V = e4m3(v_code)
 *   * v_scale, both formed exactly in FP64; then the definition above.
 *
 * Return codes: 0 ok, -1 bad argument, -2 out of memory, -3 a block id or
 * context length outside the buffers the caller described.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* BF16 is the top half of an IEEE binary32; widening is exact. */
static double widen_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double dot_bf16(const uint16_t *a, const uint16_t *b, int n)
{
    double acc = 0.0;
    for (int d = 0; d < n; ++d)
        acc += widen_bf16(a[d]) * widen_bf16(b[d]);
    return acc;
}

/*
 * Softmax attention of one query row over an explicit list of key/value rows:
 * the definition in the file header, evaluated directly.
 * x: caller scratch of ntok doubles.  out: head_dim doubles.
 */
static void attend_direct(const uint16_t *qrow, const uint16_t *const *krows,
                          const uint16_t *const *vrows, int64_t ntok, int head_dim,
                          double scale, double *x, double *out)
{
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (ntok == 0)
        return; /* l = 0  ->  output 0 */

    double xmax = -INFINITY;
    for (int64_t t = 0; t < ntok; ++t) {
        x[t] = scale * dot_bf16(qrow, krows[t], head_dim);
        if (x[t] > xmax)
            xmax = x[t];
    }
    double den = 0.0;
    for (int64_t t = 0; t < ntok; ++t) {
        double w = exp(x[t] - xmax);
        den += w;
        for (int d = 0; d < head_dim; ++d)
            out[d] += w * widen_bf16(vrows[t][d]);
    }
    for (int d = 0; d < head_dim; ++d)
        out[d] /= den;
}

/*
 * The split-K method replayed in FP64: the token range is cut into chunks of
 * `chunk` tokens; each chunk keeps its own running (m, l, o) folded one token
 * at a time; the chunks' states are then merged into (M, L, O) and the result
 * is O / L, or 0 when L is 0.
 * part: caller scratch of nsplits * (head_dim + 2) doubles.
 */
static void attend_split_replay(const uint16_t *qrow, const uint16_t *const *krows,
                                const uint16_t *const *vrows, int64_t ntok, int head_dim,
                                double scale, int64_t chunk, double *part, double *out)
{
    int64_t nsplits = ntok == 0 ? 0 : (ntok + chunk - 1) / chunk;
    for (int64_t i = 0; i < nsplits; ++i) {
        double *o = part + i * (head_dim + 2);
        double m = -INFINITY, l = 0.0;
        for (int d = 0; d < head_dim; ++d)
            o[d] = 0.0;
        int64_t t1 = (i + 1) * chunk < ntok ? (i + 1) * chunk : ntok;
        for (int64_t t = i * chunk; t < t1; ++t) {
            double s = scale * dot_bf16(qrow, krows[t], head_dim);
            double m_new = s > m ? s : m;
            double c = (m == -INFINITY) ? 0.0 : exp(m - m_new);
            double e = exp(s - m_new);
            l = l * c + e;
            for (int d = 0; d < head_dim; ++d)
                o[d] = o[d] * c + e * widen_bf16(vrows[t][d]);
            m = m_new;
        }
        o[head_dim] = m;
        o[head_dim + 1] = l;
    }
    /* merge, in split order */
    double M = -INFINITY;
    for (int64_t i = 0; i < nsplits; ++i) {
        double m = part[i * (head_dim + 2) + head_dim];
        if (m > M)
            M = m;
    }
    double L = 0.0;
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    for (int64_t i = 0; i < nsplits; ++i) {
        const double *o = part + i * (head_dim + 2);
        double m = o[head_dim];
        if (m == -INFINITY)
            continue;
        double w = exp(m - M);
        L += o[head_dim + 1] * w;
        for (int d = 0; d < head_dim; ++d)
            out[d] += o[d] * w;
    }
    if (L > 0.0) {
        for (int d = 0; d < head_dim; ++d)
            out[d] /= L;
    } else {
        for (int d = 0; d < head_dim; ++d)
            out[d] = 0.0;
    }
}

static int check_heads(int num_q_heads, int num_kv_heads, int head_dim, int block_size)
{
    if (num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return -1;
    if (num_q_heads % num_kv_heads != 0)
        return -1;
    return 0;
}

/*
 * Token rows of sequence s / KV head kvh in the paged layout
 * [num_blocks, block_size, num_kv_heads, head_dim].
 */
static int paged_rows(const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_table, int64_t max_blocks_per_seq,
                      int64_t L, int s, int kvh, int num_kv_heads, int head_dim,
                      int block_size, int64_t num_blocks,
                      const uint16_t **krows, const uint16_t **vrows)
{
    for (int64_t t = 0; t < L; ++t) {
        int64_t j = t / block_size;
        if (j >= max_blocks_per_seq)
            return -3;
        int64_t blk = block_table[(int64_t)s * max_blocks_per_seq + j];
        if (blk < 0 || blk >= num_blocks)
            return -3;
        int64_t row = ((blk * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
        krows[t] = k_cache + row;
        vrows[t] = v_cache + row;
    }
    return 0;
}

static int64_t max_context(const int32_t *context_lens, int num_seqs)
{
    int64_t m = 0;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] > m)
            m = context_lens[s];
    return m;
}

/* Shared driver of the two paged modes; chunk <= 0 selects the direct form. */
static int paged_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                      const int32_t *block_table, int64_t max_blocks_per_seq,
                      const int32_t *context_lens, int num_seqs, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                      float inv_sqrt_d, int64_t chunk, double *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim, block_size) != 0 || num_seqs < 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] < 0)
            return -3;
    int64_t lmax = max_context(context_lens, num_seqs);
    int64_t nsplit_max = chunk > 0 ? (lmax + chunk - 1) / chunk + 1 : 1;
    const uint16_t **krows = malloc(sizeof(*krows) * (size_t)(lmax + 1));
    const uint16_t **vrows = malloc(sizeof(*vrows) * (size_t)(lmax + 1));
    double *x = malloc(sizeof(double) * (size_t)(lmax + 1));
    double *part = malloc(sizeof(double) * (size_t)(nsplit_max * (head_dim + 2)));
    int rc = 0;
    if (!krows || !vrows || !x || !part) {
        rc = -2;
        goto done;
    }
    int G = num_q_heads / num_kv_heads;
    double scale = (double)inv_sqrt_d;
    for (int s = 0; s < num_seqs && rc == 0; ++s) {
        int64_t L = context_lens[s];
        for (int h = 0; h < num_q_heads && rc == 0; ++h) {
            int kvh = h / G;
            rc = paged_rows(k_cache, v_cache, block_table, max_blocks_per_seq, L, s, kvh,
                            num_kv_heads, head_dim, block_size, num_blocks, krows, vrows);
            if (rc != 0)
                break;
            const uint16_t *qrow = q + ((int64_t)s * num_q_heads + h) * head_dim;
            double *o = out + ((int64_t)s * num_q_heads + h) * head_dim;
            if (chunk > 0)
                attend_split_replay(qrow, krows, vrows, L, head_dim, scale, chunk, part, o);
            else
                attend_direct(qrow, krows, vrows, L, head_dim, scale, x, o);
        }
    }
done:
    free(krows);
    free(vrows);
    free(x);
    free(part);
    return rc;
}

/*
 * Paged-decode attention by definition.
 * q [num_seqs, num_q_heads, head_dim] BF16 bits; k_cache, v_cache
 * [num_blocks, block_size, num_kv_heads, head_dim] BF16 bits; block_table
 * [num_seqs, max_blocks_per_seq] int32; context_lens [num_seqs] int32;
 * out [num_seqs, num_q_heads, head_dim] double.
 */
int orc_decode_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                    const int32_t *block_table, int64_t max_blocks_per_seq,
                    const int32_t *context_lens, int num_seqs, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                    float inv_sqrt_d, double *out)
{
    return paged_attn(q, k_cache, v_cache, block_table, max_blocks_per_seq, context_lens,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                      inv_sqrt_d, 0, out);
}

/*
 * The same attention, replayed as split-K: each sequence's range cut into
 * chunks of chunk_tokens[s] tokens (chunk_tokens[s] > 0), folded and merged.
 */
int orc_split_replay(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                     const int32_t *block_table, int64_t max_blocks_per_seq,
                     const int32_t *context_lens, const int64_t *chunk_tokens, int num_seqs,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, float inv_sqrt_d, double *out)
{
    for (int s = 0; s < num_seqs; ++s) {
        if (chunk_tokens[s] <= 0)
            return -1;
        int rc = paged_attn(q + (int64_t)s * num_q_heads * head_dim, k_cache, v_cache,
                            block_table + (int64_t)s * max_blocks_per_seq, max_blocks_per_seq,
                            context_lens + s, 1, num_q_heads, num_kv_heads, head_dim,
                            block_size, num_blocks, inv_sqrt_d, chunk_tokens[s],
                            out + (int64_t)s * num_q_heads * head_dim);
        if (rc != 0)
            return rc;
    }
    return 0;
}

/*
 * The tiled interface's result after begin_step, num_calls step_tile calls
 * and finalize.
 * tile_blocks [num_calls, num_seqs, tile_capacity] int32;
 * tile_block_counts [num_calls, num_seqs] int32;
 * last_block_valid_slots [num_calls] int32;
 * K row of (blk, tok, kvh) at k_pool + blk*blk_stride + tok*tok_stride + kvh*kvh_stride
 * (elements), V likewise from v_pool; pool_elems bounds both pools.
 */
int orc_tiled_attn(const uint16_t *q, const uint16_t *k_pool, const uint16_t *v_pool,
                   int64_t pool_elems, const int32_t *tile_blocks,
                   const int32_t *tile_block_counts, const int32_t *last_block_valid_slots,
                   int num_calls, int num_seqs, int num_q_heads, int num_kv_heads,
                   int head_dim, int block_size, int tile_capacity, int64_t blk_stride,
                   int64_t tok_stride, int64_t kvh_stride, double *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim, block_size) != 0 || num_seqs < 0 ||
        num_calls < 0 || tile_capacity < 0)
        return -1;
    int64_t max_tok = (int64_t)num_calls * tile_capacity * block_size;
    const uint16_t **krows = malloc(sizeof(*krows) * (size_t)(max_tok + 1));
    const uint16_t **vrows = malloc(sizeof(*vrows) * (size_t)(max_tok + 1));
    double *x = malloc(sizeof(double) * (size_t)(max_tok + 1));
    int rc = 0;
    if (!krows || !vrows || !x) {
        rc = -2;
        goto done;
    }
    int G = num_q_heads / num_kv_heads;
    double scale = (double)(float)(1.0 / sqrt((double)head_dim));
    for (int s = 0; s < num_seqs && rc == 0; ++s) {
        for (int h = 0; h < num_q_heads && rc == 0; ++h) {
            int kvh = h / G;
            int64_t n = 0;
            for (int c = 0; c < num_calls && rc == 0; ++c) {
                int cnt = tile_block_counts[(int64_t)c * num_seqs + s];
                if (cnt < 0 || cnt > tile_capacity) {
                    rc = -3;
                    break;
                }
                int lb = last_block_valid_slots[c];
                for (int i = 0; i < cnt; ++i) {
                    int64_t blk =
                        tile_blocks[((int64_t)c * num_seqs + s) * tile_capacity + i];
                    int ntok = block_size;
                    if (i == cnt - 1 && lb >= 1 && lb < block_size)
                        ntok = lb;
                    for (int t = 0; t < ntok; ++t) {
                        int64_t off = blk * blk_stride + (int64_t)t * tok_stride +
                                      (int64_t)kvh * kvh_stride;
                        if (blk < 0 || off < 0 || off + head_dim > pool_elems) {
                            rc = -3;
                            break;
                        }
                        krows[n] = k_pool + off;
                        vrows[n] = v_pool + off;
                        ++n;
                    }
                    if (rc != 0)
                        break;
                }
            }
            if (rc != 0)
                break;
            const uint16_t *qrow = q + ((int64_t)s * num_q_heads + h) * head_dim;
            double *o = out + ((int64_t)s * num_q_heads + h) * head_dim;
            attend_direct(qrow, krows, vrows, n, head_dim, scale, x, o);
        }
    }
done:
    free(krows);
    free(vrows);
    free(x);
    return rc;
}

/*
 * The tiled step over calls that each name their own source: call c reads K
 * from k_pools[c] and V from v_pools[c] (both bounded by pool_elems[c]
 * elements) at blk*strides[3c] + tok*strides[3c+1] + kvh*strides[3c+2], with
 * tile_blocks[c] [num_seqs, tile_capacity[c]], tile_block_counts[c]
 * [num_seqs] and last_block_valid_slots[c].  The token set and the scale are
 * those of orc_tiled_attn.
 */
int orc_tiled_attn_multi(const uint16_t *q, const uint16_t *const *k_pools,
                         const uint16_t *const *v_pools, const int64_t *pool_elems,
                         const int64_t *strides, const int32_t *const *tile_blocks,
                         const int32_t *const *tile_block_counts, const int32_t *tile_capacity,
                         const int32_t *last_block_valid_slots, int num_calls, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         double *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim, block_size) != 0 || num_seqs < 0 ||
        num_calls < 0)
        return -1;
    int64_t max_tok = 0;
    for (int c = 0; c < num_calls; ++c) {
        if (tile_capacity[c] < 0)
            return -1;
        max_tok += (int64_t)tile_capacity[c] * block_size;
    }
    const uint16_t **krows = malloc(sizeof(*krows) * (size_t)(max_tok + 1));
    const uint16_t **vrows = malloc(sizeof(*vrows) * (size_t)(max_tok + 1));
    double *x = malloc(sizeof(double) * (size_t)(max_tok + 1));
    int rc = 0;
    if (!krows || !vrows || !x) {
        rc = -2;
        goto done;
    }
    int G = num_q_heads / num_kv_heads;
    double scale = (double)(float)(1.0 / sqrt((double)head_dim));
    for (int s = 0; s < num_seqs && rc == 0; ++s) {
        for (int h = 0; h < num_q_heads && rc == 0; ++h) {
            int kvh = h / G;
            int64_t n = 0;
            for (int c = 0; c < num_calls && rc == 0; ++c) {
                int tcap = tile_capacity[c];
                int cnt = tile_block_counts[c][s];
                if (cnt < 0 || cnt > tcap) {
                    rc = -3;
                    break;
                }
                int lb = last_block_valid_slots[c];
                for (int i = 0; i < cnt; ++i) {
                    int64_t blk = tile_blocks[c][(int64_t)s * tcap + i];
                    int ntok = block_size;
                    if (i == cnt - 1 && lb >= 1 && lb < block_size)
                        ntok = lb;
                    for (int t = 0; t < ntok; ++t) {
                        int64_t off = blk * strides[3 * c] + (int64_t)t * strides[3 * c + 1] +
                                      (int64_t)kvh * strides[3 * c + 2];
                        if (blk < 0 || off < 0 || off + head_dim > pool_elems[c]) {
                            rc = -3;
                            break;
                        }
                        krows[n] = k_pools[c] + off;
                        vrows[n] = v_pools[c] + off;
                        ++n;
                    }
                    if (rc != 0)
                        break;
                }
            }
            if (rc != 0)
                break;
            const uint16_t *qrow = q + ((int64_t)s * num_q_heads + h) * head_dim;
            double *o = out + ((int64_t)s * num_q_heads + h) * head_dim;
            attend_direct(qrow, krows, vrows, n, head_dim, scale, x, o);
        }
    }
done:
    free(krows);
    free(vrows);
    free(x);
    return rc;
}

/* OCP FP8 E4M3 code -> value (exact in FP64). */
double orc_e4m3_value(uint8_t code)
{
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* m/8 * 2^-6 */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/*
 * Paged-decode attention by definition over an FP8 E4M3 cache with per-tensor
 * scales.  q [num_seqs, Hq, D] BF16 bits; k_cache, v_cache
 * [num_blocks, block_size, Hkv, D] E4M3 codes; the rest as orc_decode_attn.
 */
int orc_decode_attn_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                        float k_scale, float v_scale, const int32_t *block_table,
                        int64_t max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int64_t num_blocks, float inv_sqrt_d, double *out)
{
    if (check_heads(num_q_heads, num_kv_heads, head_dim, block_size) != 0 || num_seqs < 0)
        return -1;
    for (int s = 0; s < num_seqs; ++s)
        if (context_lens[s] < 0)
            return -3;
    int64_t lmax = max_context(context_lens, num_seqs);
    double *kr = malloc(sizeof(double) * (size_t)((lmax + 1) * head_dim));
    double *vr = malloc(sizeof(double) * (size_t)((lmax + 1) * head_dim));
    double *qd = malloc(sizeof(double) * (size_t)head_dim);
    double *x = malloc(sizeof(double) * (size_t)(lmax + 1));
    int rc = 0;
    if (!kr || !vr || !qd || !x) {
        rc = -2;
        goto done;
    }
    int G = num_q_heads / num_kv_heads;
    double scale = (double)inv_sqrt_d;
    double ks = (double)k_scale, vs = (double)v_scale;
    for (int s = 0; s < num_seqs && rc == 0; ++s) {
        int64_t L = context_lens[s];
        for (int kvh = 0; kvh < num_kv_heads && rc == 0; ++kvh) {
            /* the sequence's K and V rows for this KV head, dequantised */
            for (int64_t t = 0; t < L; ++t) {
                int64_t j = t / block_size;
                if (j >= max_blocks_per_seq) {
                    rc = -3;
                    break;
                }
                int64_t blk = block_table[(int64_t)s * max_blocks_per_seq + j];
                if (blk < 0 || blk >= num_blocks) {
                    rc = -3;
                    break;
                }
                int64_t row = ((blk * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
                for (int d = 0; d < head_dim; ++d) {
                    kr[t * head_dim + d] = orc_e4m3_value(k_cache[row + d]) * ks;
                    vr[t * head_dim + d] = orc_e4m3_value(v_cache[row + d]) * vs;
                }
            }
            if (rc != 0)
                break;
            for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
                const uint16_t *qrow = q + ((int64_t)s * num_q_heads + h) * head_dim;
                double *o = out + ((int64_t)s * num_q_heads + h) * head_dim;
                for (int d = 0; d < head_dim; ++d) {
                    qd[d] = widen_bf16(qrow[d]);
                    o[d] = 0.0;
                }
                if (L == 0)
                    continue; /* l = 0  ->  output 0 */
                double xmax = -INFINITY;
                for (int64_t t = 0; t < L; ++t) {
                    double acc = 0.0;
                    for (int d = 0; d < head_dim; ++d)
                        acc += qd[d] * kr[t * head_dim + d];
                    x[t] = scale * acc;
                    if (x[t] > xmax)
                        xmax = x[t];
                }
                double den = 0.0;
                for (int64_t t = 0; t < L; ++t) {
                    double w = exp(x[t] - xmax);
                    den += w;
                    for (int d = 0; d < head_dim; ++d)
                        o[d] += w * vr[t * head_dim + d];
                }
                for (int d = 0; d < head_dim; ++d)
                    o[d] /= den;
            }
        }
    }
done:
    free(kr);
    free(vr);
    free(qd);
    free(x);
    return rc;
}
