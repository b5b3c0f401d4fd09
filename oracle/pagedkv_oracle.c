/*
 * CPU oracle for the paged KV cache hot path.  TEST INFRASTRUCTURE ONLY: it is
 * called by the tests, by the smoke check and by the benchmark's CPU-baseline
 * leg, never by the product path.  It shares no code, header or table with the
 * CUDA library.
 *
 * Plain C99, fp64 arithmetic, no blocking or fusion: every function is the
 * plain definition of what the pages describe, written out.
 *
 *  - slot indexing: token t of sequence s lives in physical block
 *    block_table[s][t / block_size] at in-block offset t % block_size
 *    ("Paged KV Cache 与 Packed Sequence", discosf.com, section 2.2; the
 *    block-table example of "PagedAttention 与前缀缓存", 2kiu.com, section 2.2).
 *  - append: the K/V of a new token is written at that (block, offset) and
 *    nowhere else (2kiu.com section 4.1 step 3, section 6.3; discosf.com
 *    section 4.3 step 2).  fp16/bf16 caches store the bits unchanged.  The FP8
 *    cache (2kiu.com section 1.1: one byte per element) stores
 *    E4M3(fp32(x) / scale) with the OCP 8-bit floating point E4M3 encoding,
 *    round-to-nearest-even, saturating to +-448 ("satfinite").
 *  - decode attention: for each sequence and query head, gather the keys and
 *    values of positions 0..L-1 through the block table, softmax of the scaled
 *    dot products, weighted sum of the values; positions >= L are never read
 *    (2kiu.com section 2.3 and its tail-block warning).  Grouped-query heads:
 *    query head h reads KV head h / (Hq / Hkv).
 *  - packed prefill: sequences packed back to back, sequence i owning rows
 *    [cu[i], cu[i+1]); a query attends to keys of its own sequence at an
 *    in-sequence position <= its own (block-diagonal causal mask, discosf.com
 *    sections 3.1-3.2).
 *  - prefill on a cached prefix: the same for the tail tokens of a prompt whose
 *    first ctx tokens are already in the sequence's blocks (2kiu.com section 4.3
 *    steps 2-4), every key read through the block table.
 *  - whole-block copy and swap: copy-on-write of shared blocks and moving block
 *    contents to CPU memory and back (2kiu.com sections 2.2, 4.3, 5.2).
 *
 * Readings where the pages are silent (all listed with the design notes):
 *  - softmax is the exact real-number definition, evaluated in fp64 with libm exp;
 *  - context_len == 0 gives an all-zero output row;
 *  - a NaN input to the FP8 encoder gives the canonical NaN code 0x7F;
 *  - a slot < 0 is a padding token and is skipped.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

/* ---------------------------------------------------------------- scalar formats */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double orc_f16_to_double(uint16_t h) {
    int sign = h >> 15, e = (h >> 10) & 31, f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP E4M3: 1 sign, 4 exponent (bias 7), 3 mantissa bits; no infinities;
 * S.1111.111 is NaN; largest finite 448 = 1.75 * 2^8; subnormals m * 2^-9. */
double orc_e4m3_to_double(uint8_t c) {
    int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a binary32 value to E4M3, nearest-even, saturating at +-448. */
uint8_t orc_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal spacing 2^-9; a result of 8 is the smallest normal (code 0x08) */
        double m = nearbyint(ldexp(a, 9));
        return (uint8_t)(sign | (int)m);
    }
    int e;
    frexp(a, &e);
    e -= 1; /* a = f * 2^e, f in [1, 2) */
    double m = nearbyint((ldexp(a, -e) - 1.0) * 8.0);
    if (m == 8.0) {
        m = 0.0;
        e += 1;
    }
    return (uint8_t)(sign | ((e + 7) << 3) | (int)m);
}

static double lut16[2][65536];
static double lut8[256];
static int lut_ready = 0;

static void build_luts(void) {
    if (lut_ready) return;
    for (int i = 0; i < 65536; ++i) {
        lut16[ORC_F16][i] = orc_f16_to_double((uint16_t)i);
        lut16[ORC_BF16][i] = orc_bf16_to_double((uint16_t)i);
    }
    for (int i = 0; i < 256; ++i) lut8[i] = orc_e4m3_to_double((uint8_t)i);
    lut_ready = 1;
}

void orc_init(void) { build_luts(); }

static double widen(uint16_t bits, int dtype) { return lut16[dtype][bits]; }

/* ---------------------------------------------------------------- slot indexing */

/* slot = block_table[s][p / bs] * bs + p % bs; -1 when the token has no block. */
int64_t orc_slot(const int32_t *tables, int64_t num_rows, int64_t max_blocks, int32_t s, int32_t p,
                 int64_t bs) {
    if (s < 0 || s >= num_rows || p < 0) return -1;
    int64_t logical = (int64_t)p / bs;
    if (logical >= max_blocks) return -1;
    int32_t b = tables[(int64_t)s * max_blocks + logical];
    if (b < 0) return -1;
    return (int64_t)b * bs + (int64_t)p % bs;
}

void orc_slot_mapping(const int32_t *tables, int64_t num_rows, int64_t max_blocks, const int32_t *seq_ids,
                      const int32_t *positions, int64_t n, int64_t bs, int64_t *slots) {
    for (int64_t i = 0; i < n; ++i) slots[i] = orc_slot(tables, num_rows, max_blocks, seq_ids[i], positions[i], bs);
}

/* ---------------------------------------------------------------- cache element access */

/* Element (block, kv, head, offset, dim) of the pool; strides in elements. */
static int64_t pool_index(const int64_t *st, int64_t b, int64_t kv, int64_t h, int64_t o, int64_t e) {
    return b * st[0] + kv * st[1] + h * st[2] + o * st[3] + e * st[4];
}

static double pool_value(const void *pool, const int64_t *st, int cache_dtype, const float *scale, int64_t b,
                         int64_t kv, int64_t h, int64_t o, int64_t e) {
    int64_t i = pool_index(st, b, kv, h, o, e);
    if (cache_dtype == ORC_E4M3) return lut8[((const uint8_t *)pool)[i]] * (double)scale[h];
    return lut16[cache_dtype][((const uint16_t *)pool)[i]];
}

/* ---------------------------------------------------------------- append */

/* Write token j's K and V ([n, hkv, d] source bits) at slot[j].  Returns the
 * number of tokens whose slot lies beyond the pool (those are skipped). */
int64_t orc_kv_append(void *pool, const int64_t *st, int cache_dtype, int64_t num_blocks, int64_t bs, int64_t hkv,
                      int64_t d, const uint16_t *k, const uint16_t *v, int src_dtype, const int64_t *slots, int64_t n,
                      const float *k_scale, const float *v_scale) {
    build_luts();
    int64_t bad = 0;
    for (int64_t j = 0; j < n; ++j) {
        int64_t sl = slots[j];
        if (sl < 0) continue;
        if (sl >= num_blocks * bs) {
            ++bad;
            continue;
        }
        int64_t b = sl / bs, o = sl % bs;
        for (int kv = 0; kv < 2; ++kv) {
            const uint16_t *src = kv ? v : k;
            const float *sc = kv ? v_scale : k_scale;
            for (int64_t h = 0; h < hkv; ++h)
                for (int64_t e = 0; e < d; ++e) {
                    uint16_t x = src[(j * hkv + h) * d + e];
                    int64_t i = pool_index(st, b, kv, h, o, e);
                    if (cache_dtype == ORC_E4M3) {
                        float xf = (float)widen(x, src_dtype); /* exact */
                        float y = xf / sc[h];                  /* IEEE binary32 division */
                        ((uint8_t *)pool)[i] = orc_e4m3_encode(y);
                    } else {
                        ((uint16_t *)pool)[i] = x;
                    }
                }
        }
    }
    return bad;
}

/* ---------------------------------------------------------------- decode attention */

/* out[s][h][:] = sum_t softmax_t(scale * q.K_t) V_t over t < context_lens[s], K_t/V_t read
 * from block tables[s][t / bs] at offset t % bs.  psum[s][h] = sum of the softmax weights.
 * Returns the number of table entries outside [0, num_blocks) that were needed. */
int64_t orc_paged_decode(const uint16_t *q, int q_dtype, const void *pool, const int64_t *st, int cache_dtype,
                         const float *k_scale, const float *v_scale, int64_t num_blocks, const int32_t *tables,
                         int64_t max_blocks, const int32_t *context_lens, int64_t S, int64_t hq, int64_t hkv,
                         int64_t d, int64_t bs, double scale, double *out, double *psum) {
    build_luts();
    int64_t group = hq / hkv, bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (int64_t sh = 0; sh < S * hq; ++sh) {
        int64_t s = sh / hq, h = sh % hq, g = h / group;
        int64_t L = context_lens[s];
        double *o = out + sh * d;
        for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
        if (psum) psum[sh] = 0.0;
        if (L <= 0) continue;
        double *x = (double *)malloc((size_t)L * sizeof(double));
        int64_t *blk = (int64_t *)malloc((size_t)L * sizeof(int64_t));
        const uint16_t *qv = q + sh * d;
        int ok = 1;
        for (int64_t t = 0; t < L; ++t) {
            int64_t lb = t / bs;
            int32_t b = lb < max_blocks ? tables[s * max_blocks + lb] : -1;
            if (b < 0 || b >= num_blocks) {
                ok = 0;
                break;
            }
            blk[t] = b;
            double dot = 0.0;
            for (int64_t e = 0; e < d; ++e)
                dot += widen(qv[e], q_dtype) * pool_value(pool, st, cache_dtype, k_scale, b, 0, g, t % bs, e);
            x[t] = scale * dot;
        }
        if (!ok) {
            ++bad;
            free(x);
            free(blk);
            continue;
        }
        double m = x[0];
        for (int64_t t = 1; t < L; ++t)
            if (x[t] > m) m = x[t];
        double den = 0.0;
        for (int64_t t = 0; t < L; ++t) {
            x[t] = exp(x[t] - m);
            den += x[t];
        }
        for (int64_t t = 0; t < L; ++t) {
            double p = x[t] / den;
            if (psum) psum[sh] += p;
            for (int64_t e = 0; e < d; ++e)
                o[e] += p * pool_value(pool, st, cache_dtype, v_scale, blk[t], 1, g, t % bs, e);
        }
        free(x);
        free(blk);
    }
    return bad;
}

/* ---------------------------------------------------------------- packed causal prefill */

/* out[cu[i]+r][h][:] = sum_{c<=r} softmax_c(scale * q[cu[i]+r][h] . k[cu[i]+c][g]) v[cu[i]+c][g]. */
void orc_packed_prefill(const uint16_t *q, const uint16_t *k, const uint16_t *v, int dtype, const int32_t *cu,
                        int64_t num_seqs, int64_t hq, int64_t hkv, int64_t d, double scale, double *out) {
    build_luts();
    int64_t group = hq / hkv;
#pragma omp parallel for schedule(dynamic)
    for (int64_t ih = 0; ih < num_seqs * hq; ++ih) {
        int64_t i = ih / hq, h = ih % hq, g = h / group;
        int64_t start = cu[i], n = (int64_t)cu[i + 1] - cu[i];
        if (n <= 0) continue;
        double *x = (double *)malloc((size_t)n * sizeof(double));
        for (int64_t r = 0; r < n; ++r) {
            const uint16_t *qr = q + ((start + r) * hq + h) * d;
            for (int64_t c = 0; c <= r; ++c) {
                const uint16_t *kc = k + ((start + c) * hkv + g) * d;
                double dot = 0.0;
                for (int64_t e = 0; e < d; ++e) dot += widen(qr[e], dtype) * widen(kc[e], dtype);
                x[c] = scale * dot;
            }
            double m = x[0];
            for (int64_t c = 1; c <= r; ++c)
                if (x[c] > m) m = x[c];
            double den = 0.0;
            for (int64_t c = 0; c <= r; ++c) {
                x[c] = exp(x[c] - m);
                den += x[c];
            }
            double *o = out + ((start + r) * hq + h) * d;
            for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
            for (int64_t c = 0; c <= r; ++c) {
                double p = x[c] / den;
                const uint16_t *vc = v + ((start + c) * hkv + g) * d;
                for (int64_t e = 0; e < d; ++e) o[e] += p * widen(vc[e], dtype);
            }
        }
        free(x);
    }
}

/* ---------------------------------------------------------------- whole-block copies */

/* Copy-on-write of shared blocks and swapping block contents to CPU memory ("PagedAttention 与前缀缓存",
 * 2kiu.com, section 2.2; section 4.3 step 3: a shared block is never rewritten in place, the
 * diverging path gets its own copy; section 5.2: preempted requests' blocks go to CPU memory).
 * A block is every element (K|V, head, slot, dim) of one physical block.  elt = bytes per element.
 * Pairs whose ids fall outside [0, num_blocks) are skipped and counted. */

static void copy_elem(void *dst, int64_t di, const void *src, int64_t si, int elt) {
    memcpy((char *)dst + di * elt, (const char *)src + si * elt, (size_t)elt);
}

/* block dst_ids[i] := block src_ids[i] (the caller keeps destinations distinct from sources). */
int64_t orc_block_copy(void *pool, const int64_t *st, int elt, int64_t num_blocks, int64_t bs, int64_t hkv, int64_t d,
                       const int32_t *src_ids, const int32_t *dst_ids, int64_t n) {
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t sb = src_ids[i], db = dst_ids[i];
        if (sb < 0 || sb >= num_blocks || db < 0 || db >= num_blocks) {
            ++bad;
            continue;
        }
        for (int kv = 0; kv < 2; ++kv)
            for (int64_t h = 0; h < hkv; ++h)
                for (int64_t o = 0; o < bs; ++o)
                    for (int64_t e = 0; e < d; ++e)
                        copy_elem(pool, pool_index(st, db, kv, h, o, e), pool, pool_index(st, sb, kv, h, o, e), elt);
    }
    return bad;
}

/* index of element (kv, h, o, e) of block i in a swap buffer: blocks back to back, each in the
 * documented pool order [K|V][head][slot][dim] */
static int64_t buf_index(int64_t i, int kv, int64_t h, int64_t o, int64_t e, int64_t bs, int64_t hkv, int64_t d) {
    return (((i * 2 + kv) * hkv + h) * bs + o) * d + e;
}

/* swap out: buffer block i := pool block ids[i] */
int64_t orc_block_swap_out(const void *pool, const int64_t *st, int elt, int64_t num_blocks, int64_t bs, int64_t hkv,
                           int64_t d, const int32_t *ids, int64_t n, void *buf) {
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = ids[i];
        if (b < 0 || b >= num_blocks) {
            ++bad;
            continue;
        }
        for (int kv = 0; kv < 2; ++kv)
            for (int64_t h = 0; h < hkv; ++h)
                for (int64_t o = 0; o < bs; ++o)
                    for (int64_t e = 0; e < d; ++e)
                        copy_elem(buf, buf_index(i, kv, h, o, e, bs, hkv, d), pool, pool_index(st, b, kv, h, o, e), elt);
    }
    return bad;
}

/* swap in: pool block ids[i] := buffer block i */
int64_t orc_block_swap_in(void *pool, const int64_t *st, int elt, int64_t num_blocks, int64_t bs, int64_t hkv,
                          int64_t d, const int32_t *ids, int64_t n, const void *buf) {
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t b = ids[i];
        if (b < 0 || b >= num_blocks) {
            ++bad;
            continue;
        }
        for (int kv = 0; kv < 2; ++kv)
            for (int64_t h = 0; h < hkv; ++h)
                for (int64_t o = 0; o < bs; ++o)
                    for (int64_t e = 0; e < d; ++e)
                        copy_elem(pool, pool_index(st, b, kv, h, o, e), buf, buf_index(i, kv, h, o, e, bs, hkv, d), elt);
    }
    return bad;
}

/* ---------------------------------------------------------------- prefill on a cached prefix */

/* The tail of a prompt after a prefix-cache hit ("PagedAttention 与前缀缓存", 2kiu.com, section 4.3
 * steps 2-4 and section 3.3: only the tokens past the hit are prefilled, the hit blocks are read):
 * sequence i already holds ctx[i] tokens in its blocks; its n_i = cu[i+1] - cu[i] new tokens sit
 * at positions ctx[i] .. ctx[i] + n_i - 1 and their K/V have been written at their slots (append).
 * New row r attends to every position c <= ctx[i] + r of the sequence, all read from the pool
 * through the table:
 *   out[cu[i] + r][h] = sum_{c <= ctx_i + r} softmax_c(scale * q[cu[i] + r][h] . K_c) V_c.
 * Returns the number of (row, head) outputs that needed a table entry outside [0, num_blocks). */
int64_t orc_prefill_ctx(const uint16_t *q, int q_dtype, const void *pool, const int64_t *st, int cache_dtype,
                        const float *k_scale, const float *v_scale, int64_t num_blocks, const int32_t *tables,
                        int64_t max_blocks, const int32_t *cu, const int32_t *ctx, int64_t num_seqs, int64_t hq,
                        int64_t hkv, int64_t d, int64_t bs, double scale, double *out) {
    build_luts();
    int64_t group = hq / hkv, bad = 0;
#pragma omp parallel for schedule(dynamic) reduction(+ : bad)
    for (int64_t ih = 0; ih < num_seqs * hq; ++ih) {
        int64_t i = ih / hq, h = ih % hq, g = h / group;
        int64_t start = cu[i], n = (int64_t)cu[i + 1] - cu[i], c0 = ctx[i];
        if (n <= 0) continue;
        int64_t total = c0 + n;
        double *x = (double *)malloc((size_t)total * sizeof(double));
        int64_t *blk = (int64_t *)malloc((size_t)total * sizeof(int64_t));
        int ok = 1;
        for (int64_t c = 0; c < total; ++c) {
            int64_t lb = c / bs;
            int32_t b = lb < max_blocks ? tables[i * max_blocks + lb] : -1;
            if (b < 0 || b >= num_blocks) {
                ok = 0;
                break;
            }
            blk[c] = b;
        }
        for (int64_t r = 0; r < n; ++r) {
            double *o = out + ((start + r) * hq + h) * d;
            for (int64_t e = 0; e < d; ++e) o[e] = 0.0;
            if (!ok) continue;
            const uint16_t *qr = q + ((start + r) * hq + h) * d;
            int64_t L = c0 + r + 1;
            for (int64_t c = 0; c < L; ++c) {
                double dot = 0.0;
                for (int64_t e = 0; e < d; ++e)
                    dot += widen(qr[e], q_dtype) * pool_value(pool, st, cache_dtype, k_scale, blk[c], 0, g, c % bs, e);
                x[c] = scale * dot;
            }
            double m = x[0];
            for (int64_t c = 1; c < L; ++c)
                if (x[c] > m) m = x[c];
            double den = 0.0;
            for (int64_t c = 0; c < L; ++c) {
                x[c] = exp(x[c] - m);
                den += x[c];
            }
            for (int64_t c = 0; c < L; ++c) {
                double p = x[c] / den;
                for (int64_t e = 0; e < d; ++e)
                    o[e] += p * pool_value(pool, st, cache_dtype, v_scale, blk[c], 1, g, c % bs, e);
            }
        }
        if (!ok) bad += n;
        free(x);
        free(blk);
    }
    return bad;
}

int orc_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
