/*
 * Plain CPU reference ("oracle") for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The CUDA library never
 * links, includes or calls it, and it shares no code, header, table or
 * constant with the CUDA path.
 *
 * Everything is computed in double precision from the 16-bit inputs widened
 * exactly.  Nothing is blocked, fused or reordered beyond the definitions
 * cited at each function.  OpenMP (when available) only distributes
 * independent (sequence, query head) outputs over threads; every output is
 * computed by the same sequential loop whatever the thread count.
 *
 * Sources (web pages on vLLM / PagedAttention):
 *  - youngju.dev, "vLLM inference optimization" post, section "PagedAttention"
 *    (PagedAttentionManager: the cache tensors shaped
 *    [num_blocks, block_size, num_heads, head_dim], the free list, and
 *    append_token writing k_cache[last_block, slot_in_block]).
 *  - ta-paperlens, "LLM serving from scratch", section on fragmentation and
 *    PagedAttention: the attention kernel follows the logical->physical block
 *    table and gathers K and V while it computes.
 *  - Attention itself (softmax(scale * q.K^T) . V) is the textbook
 *    definition; the pages name it but never write it out.
 *
 * Readings taken where the pages are silent:
 *  - the table stores physical block ids, row b holds sequence b's logical
 *    blocks in order; token i of a sequence sits in block table[b][i / bs]
 *    at offset i % bs;
 *  - query head h reads KV head h / G with G = num_q_heads / num_kv_heads;
 *  - a slot number is physical_block * block_size + offset; a negative slot
 *    is padding and writes nothing;
 *  - an empty context yields a zero output.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_DTYPE_F16 0
#define OR_DTYPE_BF16 1

/* ---- exact widening of the 16-bit storage formats ---------------------- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-24 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(1024.0 + (double)f, e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 (8 exponent bits, bias 127,
 * 7 fraction bits). */
double oracle_bf16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);              /* subnormal: f * 2^-133 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp(128.0 + (double)f, e - 134);   /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* OCP FP8 E4M3 (the "fn" variant): 1 sign, 4 exponent (bias 7), 3 fraction
 * bits; no infinities; S.1111.111 is NaN; largest finite 448. */
double oracle_e4m3_to_f64(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int f = b & 0x7;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -9);                /* subnormal: f/8 * 2^-6 */
    } else if (e == 15 && f == 7) {
        v = NAN;
    } else {
        v = ldexp(8.0 + (double)f, e - 10);      /* (1 + f/8) * 2^(e-7) */
    }
    return sign ? -v : v;
}

/*
 * Nearest E4M3 code of a float, ties to the even code, magnitudes above 448
 * saturated to 448, NaN to the NaN code.  Found by comparing against every
 * finite positive code (exact in double).
 */
uint8_t oracle_f32_to_e4m3(float y) {
    if (y != y) return 0x7f;
    uint8_t sign = (y < 0.0f || (y == 0.0f && 1.0f / y < 0.0f)) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7e);
    int best = 0;
    double best_err = a;                         /* code 0 is +0 */
    for (int c = 1; c <= 0x7e; ++c) {
        double err = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

static double widen(uint16_t h, int dtype) {
    return dtype == OR_DTYPE_BF16 ? oracle_bf16_to_f64(h) : oracle_f16_to_f64(h);
}

void oracle_widen(const uint16_t* src, double* dst, int64_t n, int dtype) {
    for (int64_t i = 0; i < n; ++i) dst[i] = widen(src[i], dtype);
}

/* ---- cache write: append_token / reshape_and_cache --------------------- */

/*
 * For every new token t whose slot s = slot_mapping[t] is >= 0, copy its
 * num_kv_heads*head_dim key elements bit for bit into
 * k_cache[s / block_size][s % block_size][:][:], and its value elements into
 * v_cache at the same place (youngju.dev post, PagedAttentionManager
 * .append_token).  Returns the number of tokens whose slot lies past the
 * pool (those are not written), 0 when all slots were valid or padding.
 */
int64_t oracle_reshape_and_cache(const uint16_t* k, const uint16_t* v,
                                 const int64_t* slot_mapping,
                                 uint16_t* k_cache, uint16_t* v_cache,
                                 int64_t num_tokens, int num_kv_heads, int head_dim,
                                 int block_size, int64_t num_blocks) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;                              /* padding */
        int64_t blk = s / block_size;
        int64_t off = s % block_size;
        if (blk >= num_blocks) { ++bad; continue; }
        int64_t dst = (blk * block_size + off) * row;
        memcpy(k_cache + dst, k + t * row, (size_t)row * sizeof(uint16_t));
        memcpy(v_cache + dst, v + t * row, (size_t)row * sizeof(uint16_t));
    }
    return bad;
}

/*
 * FP8 cache write: each element of the new token's K (V) becomes the E4M3
 * code of x / k_scale (x / v_scale), the quotient taken in fp32.  Slots as
 * in oracle_reshape_and_cache.  Caches are [num_blocks][block_size][Hkv][D]
 * bytes.  Returns the number of tokens whose slot lies past the pool.
 */
int64_t oracle_reshape_and_cache_fp8(const uint16_t* k, const uint16_t* v,
                                     const int64_t* slot_mapping, uint8_t* k_cache,
                                     uint8_t* v_cache, int64_t num_tokens, int num_kv_heads,
                                     int head_dim, int block_size, int64_t num_blocks,
                                     int dtype, float k_scale, float v_scale) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0) continue;
        if (s / block_size >= num_blocks) { ++bad; continue; }
        for (int64_t i = 0; i < row; ++i) {
            float xk = (float)widen(k[t * row + i], dtype);
            float xv = (float)widen(v[t * row + i], dtype);
            k_cache[s * row + i] = oracle_f32_to_e4m3(xk / k_scale);
            v_cache[s * row + i] = oracle_f32_to_e4m3(xv / v_scale);
        }
    }
    return bad;
}

/* ---- whole-block copies: copy-on-write and swap ------------------------ */

/*
 * For each pair p: dst pool block mapping[2p+1] receives a bit copy of src
 * pool block mapping[2p], for K and V (a block is block_size * num_kv_heads
 * * head_dim elements).  Copy-on-write gives a request its own copy of a
 * shared block before it writes there (tcdigital article, memory sharing for
 * parallel sampling; youngju.dev post, Copy-on-Write); swapping moves blocks
 * between GPU and CPU pools (tcdigital article, --swap-space).  Pairs with
 * an id outside either pool are skipped and counted; the count is returned.
 */
int64_t oracle_copy_blocks(const uint16_t* k_src, const uint16_t* v_src, int64_t src_blocks,
                           uint16_t* k_dst, uint16_t* v_dst, int64_t dst_blocks,
                           const int64_t* mapping, int64_t num_pairs, int block_size,
                           int num_kv_heads, int head_dim) {
    int64_t elems = (int64_t)block_size * num_kv_heads * head_dim;
    int64_t bad = 0;
    for (int64_t p = 0; p < num_pairs; ++p) {
        int64_t s = mapping[2 * p], d = mapping[2 * p + 1];
        if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) { ++bad; continue; }
        memcpy(k_dst + d * elems, k_src + s * elems, (size_t)elems * sizeof(uint16_t));
        memcpy(v_dst + d * elems, v_src + s * elems, (size_t)elems * sizeof(uint16_t));
    }
    return bad;
}

/* ---- attention over one span of one sequence -------------------------- */

/*
 * Element (token i, kv head g, dim d) of the paged cache for sequence b:
 * physical block block_tables[b][i / bs], offset i % bs.
 */
static const uint16_t* paged_row(const uint16_t* cache, const int32_t* table_row,
                                 int64_t i, int g, int num_kv_heads, int head_dim,
                                 int block_size) {
    int64_t p = table_row[i / block_size];
    int64_t o = i % block_size;
    return cache + ((p * block_size + o) * num_kv_heads + g) * (int64_t)head_dim;
}

/*
 * Two-pass softmax attention of one query row over tokens [t0, t1) of one
 * sequence:
 *   s_i = scale * sum_d q[d] * K_i[d]
 *   m   = max_i s_i
 *   w_i = exp(s_i - m),  l = sum_i w_i
 *   o   = sum_i w_i * V_i / l
 * Writes o (head_dim doubles) and returns m and l through the pointers.
 */
static void attend_span(const double* qrow, const uint16_t* k_cache,
                        const uint16_t* v_cache, const int32_t* table_row,
                        int64_t t0, int64_t t1, int g, int num_kv_heads,
                        int head_dim, int block_size, int dtype, double scale,
                        double* o, double* m_out, double* l_out) {
    int64_t n = t1 - t0;
    double* s = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        const uint16_t* kr = paged_row(k_cache, table_row, t0 + i, g, num_kv_heads,
                                       head_dim, block_size);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d) dot += qrow[d] * widen(kr[d], dtype);
        s[i] = scale * dot;
        if (s[i] > m) m = s[i];
    }
    double l = 0.0;
    for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double w = exp(s[i] - m);
        l += w;
        const uint16_t* vr = paged_row(v_cache, table_row, t0 + i, g, num_kv_heads,
                                       head_dim, block_size);
        for (int d = 0; d < head_dim; ++d) o[d] += w * widen(vr[d], dtype);
    }
    if (n > 0) {
        for (int d = 0; d < head_dim; ++d) o[d] /= l;
    }
    free(s);
    *m_out = m;
    *l_out = l;
}

/*
 * Paged decode attention: for every sequence b and query head h,
 *   out[b][h][:] = softmax_i(scale * q[b][h] . K_i) . V_i,  i < context_lens[b],
 * with K_i, V_i reached through the block table (ta-paperlens page,
 * PagedAttention paragraph).  out is [num_seqs][num_q_heads][head_dim] doubles.
 * Returns -1 on a shape error, else 0.
 */
int oracle_paged_decode(const uint16_t* q, const uint16_t* k_cache,
                        const uint16_t* v_cache, const int32_t* block_tables,
                        const int32_t* context_lens, double scale, int num_seqs,
                        int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int max_blocks_per_seq, int dtype,
                        double* out) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    int G = num_q_heads / num_kv_heads;
    int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / num_q_heads);
        int h = (int)(bh % num_q_heads);
        double* qrow = (double*)malloc((size_t)head_dim * sizeof(double));
        const uint16_t* qsrc = q + bh * head_dim;
        for (int d = 0; d < head_dim; ++d) qrow[d] = widen(qsrc[d], dtype);
        double m, l;
        attend_span(qrow, k_cache, v_cache,
                    block_tables + (int64_t)b * max_blocks_per_seq, 0,
                    context_lens[b], h / G, num_kv_heads, head_dim, block_size,
                    dtype, scale, out + bh * head_dim, &m, &l);
        free(qrow);
    }
    return 0;
}

/*
 * Paged prefill / chunked prefill: sequence b has C_b = query_start[b+1] -
 * query_start[b] new tokens, the last C_b of its L_b = context_lens[b] tokens
 * (all already in the cache).  New token i sits at position
 * p = L_b - C_b + i and attends causally to positions 0..p:
 *   out[query_start[b] + i][h] = softmax_{j <= p}(scale * q . K_j) . V_j
 * (ta-paperlens page, prefill vs decode and chunked prefill; techfeed summary,
 * chunked prefill splits a long prompt across forward passes).  q and out are
 * [total_tokens][num_q_heads][head_dim].
 */
int oracle_paged_prefill(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                         const int32_t* block_tables, const int32_t* context_lens,
                         const int32_t* query_start, double scale, int num_seqs,
                         int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int max_blocks_per_seq, int dtype, double* out) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    int G = num_q_heads / num_kv_heads;
    int64_t total = query_start[num_seqs];
    int64_t rows = total * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t tok = r / num_q_heads;
        int h = (int)(r % num_q_heads);
        int b = 0;
        while (query_start[b + 1] <= tok) ++b;           /* the token's sequence */
        int64_t C = query_start[b + 1] - query_start[b];
        int64_t p = context_lens[b] - C + (tok - query_start[b]);
        double* qrow = (double*)malloc((size_t)head_dim * sizeof(double));
        for (int d = 0; d < head_dim; ++d) qrow[d] = widen(q[r * head_dim + d], dtype);
        double m, l;
        attend_span(qrow, k_cache, v_cache, block_tables + (int64_t)b * max_blocks_per_seq, 0,
                    p + 1, h / G, num_kv_heads, head_dim, block_size, dtype, scale,
                    out + r * head_dim, &m, &l);
        free(qrow);
    }
    return 0;
}

/*
 * Per-partition results of the context split: partition s of sequence b
 * covers tokens [s*P, min((s+1)*P, L_b)).  For each (b, h, s) with
 * s*P < L_b it writes
 *   part_max[b][h][s] = m_s = max_i s_i                (natural-log units)
 *   part_sum[b][h][s] = l_s = sum_i exp(s_i - m_s)
 *   part_out[b][h][s][:] = sum_i exp(s_i - m_s) V_i / l_s
 * and leaves partitions at or past L_b untouched.
 * part_out is [B][Hq][max_parts][D], the others [B][Hq][max_parts].
 */
int oracle_paged_decode_partitions(const uint16_t* q, const uint16_t* k_cache,
                                   const uint16_t* v_cache,
                                   const int32_t* block_tables,
                                   const int32_t* context_lens, double scale,
                                   int num_seqs, int num_q_heads, int num_kv_heads,
                                   int head_dim, int block_size,
                                   int max_blocks_per_seq, int dtype,
                                   int partition_size, int max_parts,
                                   double* part_out, double* part_max,
                                   double* part_sum) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    if (partition_size <= 0) return -1;
    int G = num_q_heads / num_kv_heads;
    int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / num_q_heads);
        int h = (int)(bh % num_q_heads);
        double* qrow = (double*)malloc((size_t)head_dim * sizeof(double));
        const uint16_t* qsrc = q + bh * head_dim;
        for (int d = 0; d < head_dim; ++d) qrow[d] = widen(qsrc[d], dtype);
        int64_t L = context_lens[b];
        for (int s = 0; s < max_parts; ++s) {
            int64_t t0 = (int64_t)s * partition_size;
            if (t0 >= L) break;
            int64_t t1 = t0 + partition_size < L ? t0 + partition_size : L;
            int64_t idx = bh * max_parts + s;
            attend_span(qrow, k_cache, v_cache,
                        block_tables + (int64_t)b * max_blocks_per_seq, t0, t1,
                        h / G, num_kv_heads, head_dim, block_size, dtype, scale,
                        part_out + idx * head_dim, part_max + idx, part_sum + idx);
        }
        free(qrow);
    }
    return 0;
}

/*
 * Paged decode attention over an FP8 (E4M3) cache with per-tensor scales:
 * K_i = e4m3(code) * k_scale, V_i = e4m3(code) * v_scale, then the same
 * two-pass softmax definition as oracle_paged_decode.  q is 16-bit (dtype).
 */
int oracle_paged_decode_fp8(const uint16_t* q, const uint8_t* k_cache,
                            const uint8_t* v_cache, const int32_t* block_tables,
                            const int32_t* context_lens, double scale, double k_scale,
                            double v_scale, int num_seqs, int num_q_heads, int num_kv_heads,
                            int head_dim, int block_size, int max_blocks_per_seq, int dtype,
                            double* out) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    int G = num_q_heads / num_kv_heads;
    int64_t pairs = (int64_t)num_seqs * num_q_heads;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < pairs; ++bh) {
        int b = (int)(bh / num_q_heads);
        int g = (int)(bh % num_q_heads) / G;
        const int32_t* table = block_tables + (int64_t)b * max_blocks_per_seq;
        int64_t L = context_lens[b];
        double* o = out + bh * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (L <= 0) continue;
        double* s = (double*)malloc((size_t)L * sizeof(double));
        double m = -INFINITY;
        for (int64_t i = 0; i < L; ++i) {
            int64_t base = ((int64_t)table[i / block_size] * block_size + i % block_size) *
                               num_kv_heads * head_dim + (int64_t)g * head_dim;
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += widen(q[bh * head_dim + d], dtype) *
                       (oracle_e4m3_to_f64(k_cache[base + d]) * k_scale);
            s[i] = scale * dot;
            if (s[i] > m) m = s[i];
        }
        double l = 0.0;
        for (int64_t i = 0; i < L; ++i) {
            int64_t base = ((int64_t)table[i / block_size] * block_size + i % block_size) *
                               num_kv_heads * head_dim + (int64_t)g * head_dim;
            double w = exp(s[i] - m);
            l += w;
            for (int d = 0; d < head_dim; ++d)
                o[d] += w * (oracle_e4m3_to_f64(v_cache[base + d]) * v_scale);
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= l;
        free(s);
    }
    return 0;
}

/*
 * Log-sum-exp merge of the partitions of each (b, h):
 *   M = max_s m_s,  w_s = l_s * exp(m_s - M),
 *   out = sum_s w_s o_s / sum_s w_s      (zero when L_b = 0).
 * Partitions s < min(ceil(L_b / P), max_parts) take part.
 */
int oracle_lse_merge(const double* part_out, const double* part_max,
                     const double* part_sum, const int32_t* context_lens,
                     int num_seqs, int num_q_heads, int head_dim,
                     int partition_size, int max_parts, double* out) {
    if (partition_size <= 0) return -1;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t L = context_lens[b];
        int64_t np = (L + partition_size - 1) / partition_size;
        if (np > max_parts) np = max_parts;
        for (int h = 0; h < num_q_heads; ++h) {
            int64_t bh = (int64_t)b * num_q_heads + h;
            double* o = out + bh * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (np <= 0) continue;
            double M = -INFINITY;
            for (int64_t s = 0; s < np; ++s)
                if (part_max[bh * max_parts + s] > M) M = part_max[bh * max_parts + s];
            double wsum = 0.0;
            for (int64_t s = 0; s < np; ++s) {
                int64_t idx = bh * max_parts + s;
                double w = part_sum[idx] * exp(part_max[idx] - M);
                wsum += w;
                for (int d = 0; d < head_dim; ++d) o[d] += w * part_out[idx * head_dim + d];
            }
            for (int d = 0; d < head_dim; ++d) o[d] /= wsum;
        }
    }
    return 0;
}

/*
 * Unpaged attention: the same definition over per-sequence contiguous K/V
 * arrays, k_seq/v_seq = [sum_b L_b][num_kv_heads][head_dim] with sequence b's
 * tokens starting at row seq_start[b].  No block table is involved; this is
 * the contiguous-reservation layout the pages contrast with paging.
 */
int oracle_contiguous_decode(const uint16_t* q, const uint16_t* k_seq,
                             const uint16_t* v_seq, const int64_t* seq_start,
                             const int32_t* context_lens, double scale,
                             int num_seqs, int num_q_heads, int num_kv_heads,
                             int head_dim, int dtype, double* out) {
    if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return -1;
    int G = num_q_heads / num_kv_heads;
    for (int b = 0; b < num_seqs; ++b) {
        int64_t L = context_lens[b];
        for (int h = 0; h < num_q_heads; ++h) {
            int64_t bh = (int64_t)b * num_q_heads + h;
            int g = h / G;
            double* o = out + bh * head_dim;
            for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
            if (L <= 0) continue;
            double* s = (double*)malloc((size_t)L * sizeof(double));
            double m = -INFINITY;
            for (int64_t i = 0; i < L; ++i) {
                const uint16_t* kr = k_seq + ((seq_start[b] + i) * num_kv_heads + g) * (int64_t)head_dim;
                double dot = 0.0;
                for (int d = 0; d < head_dim; ++d)
                    dot += widen(q[bh * head_dim + d], dtype) * widen(kr[d], dtype);
                s[i] = scale * dot;
                if (s[i] > m) m = s[i];
            }
            double l = 0.0;
            for (int64_t i = 0; i < L; ++i) {
                double w = exp(s[i] - m);
                l += w;
                const uint16_t* vr = v_seq + ((seq_start[b] + i) * num_kv_heads + g) * (int64_t)head_dim;
                for (int d = 0; d < head_dim; ++d) o[d] += w * widen(vr[d], dtype);
            }
            for (int d = 0; d < head_dim; ++d) o[d] /= l;
            free(s);
        }
    }
    return 0;
}

/* Threads the parallel loops above may use (1 without OpenMP). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
