/*
 * oracle.c -- plain, slow, fp64 CPU oracle for paged KV-cache decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file.  It shares no code, header, table or helper with the CUDA
 * library; the only thing the two sides have in common is the seeded input
 * generator that feeds both.
 *
 * What it follows:
 *  - "What Is vLLM: The Fast Inference Engine for Large Language Models",
 *    section "How does PagedAttention work?": the KV cache of each sequence
 *    is cut into fixed-size blocks; a per-sequence block table maps logical
 *    KV positions to physical blocks; to attend at position p the engine
 *    finds the physical block holding p and indexes into it.  Several
 *    sequences may point at the same physical block (reference counting,
 *    copy-on-write).
 *  - "vLLM in Production - PagedAttention, Continuous Batching, ...",
 *    sections "The KV Cache and the 60-80% Memory Tax" (each new token
 *    attends to every previous token through the cached keys and values) and
 *    "PagedAttention - Virtual Memory for the KV Cache" (blocks live anywhere
 *    in memory, the table grows one block at a time as tokens arrive).
 *  - "Serving models with vLLM", section "How it works: PagedAttention"
 *    (blocks of e.g. 16 tokens, a block table per request mapping logical
 *    positions to physical blocks, prefix sharing of physical blocks).
 *
 * The pages give no formula, layout or precision for the attention step, so
 * the readings taken here are:
 *  - pool layout  k_pool, v_pool : [num_blocks][num_kv_heads][block_size][head_dim]
 *  - position p of sequence s lives in block  block_tables[s][p / B]  at row p % B
 *  - q head h reads kv head h / (num_q_heads / num_kv_heads)  (contiguous groups)
 *  - attention = softmax(scale * q . K^T) V, computed from the definition in
 *    double: scores, their maximum, exp(score - max), the sum, the weighted
 *    sum of V rows divided by the sum.  context length 0 gives a zero row.
 *  - slot of position p = block_tables[s][p / B] * B + p % B;  slot < 0 skips.
 *
 * Every stored element is converted exactly to double (fp32, fp16 and bf16
 * are all exactly representable).  The partition/merge pair restates the
 * same definition over token ranges of P tokens and combines the partial
 * results by the log-sum-exp rule; a test checks it equals the plain form.
 *
 * Parallelism: independent (sequence, kv head) outputs may run on several
 * OpenMP threads; each output is still computed in the order written here.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_BLOCK = 2, ORC_ERR_NOMEM = 3 };

static int elem_bytes(int dtype) { return dtype == ORC_F32 ? 4 : 2; }

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24); /* subnormal: f * 2^(1-15-10) */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32. */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float x;
    memcpy(&x, &u, sizeof x);
    return (double)x;
}

static double load_as_double(const void* base, int dtype, int64_t i) {
    if (dtype == ORC_F32) return (double)((const float*)base)[i];
    uint16_t bits = ((const uint16_t*)base)[i];
    return dtype == ORC_F16 ? half_to_double(bits) : bf16_to_double(bits);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Element conversion exported on its own so that tests can pin it against
 * library conversions over every bit pattern. */
void oracle_convert_to_double(int dtype, const void* src, int64_t n, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = load_as_double(src, dtype, i);
}

/* Gather the first ctx positions of sequence s, kv head g, into contiguous
 * [ctx][D] double arrays, looking every position up through the block table.
 * Returns ORC_ERR_BLOCK if a table entry the positions need is outside the pool. */
static int gather_sequence(int dtype, const void* k_pool, const void* v_pool,
                           int32_t num_blocks, int32_t B, int32_t Hkv, int32_t D,
                           const int32_t* table_row, int32_t ctx, int32_t g,
                           double* Kc, double* Vc) {
    for (int32_t p = 0; p < ctx; ++p) {
        int32_t logical_block = p / B;
        int32_t row = p % B;
        int32_t phys = table_row[logical_block];
        if (phys < 0 || phys >= num_blocks) return ORC_ERR_BLOCK;
        int64_t base = (((int64_t)phys * Hkv + g) * B + row) * D;
        for (int32_t d = 0; d < D; ++d) {
            Kc[(int64_t)p * D + d] = load_as_double(k_pool, dtype, base + d);
            Vc[(int64_t)p * D + d] = load_as_double(v_pool, dtype, base + d);
        }
    }
    return ORC_OK;
}

/* x_i = scale * sum_d q_d K_i,d  for i < n, starting at position first. */
static void scores(const double* qd, const double* Kc, int32_t first, int32_t n, int32_t D,
                   double scale, double* x) {
    for (int32_t i = 0; i < n; ++i) {
        double dot = 0.0;
        const double* k = Kc + (int64_t)(first + i) * D;
        for (int32_t d = 0; d < D; ++d) dot += qd[d] * k[d];
        x[i] = scale * dot;
    }
}

static int check_common(int dtype, int32_t num_blocks, int32_t B, int32_t Hkv, int32_t D,
                        int32_t S, int32_t Hq, int32_t M) {
    if (dtype < ORC_F32 || dtype > ORC_BF16) return ORC_ERR_ARG;
    if (num_blocks <= 0 || B <= 0 || Hkv <= 0 || D <= 0 || S < 0 || Hq <= 0 || M <= 0)
        return ORC_ERR_ARG;
    if (Hq % Hkv != 0) return ORC_ERR_ARG;
    return ORC_OK;
}

/*
 * out[s][h][d] (double) = softmax(scale * q[s][h] . K_s^T) V_s  over the
 * context_lens[s] cached positions of sequence s, where K_s, V_s are the
 * sequence's keys and values gathered in logical order through its block table.
 */
int oracle_paged_decode(int dtype, const void* k_pool, const void* v_pool,
                        int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                        int32_t head_dim, const void* q, int32_t num_seqs, int32_t num_q_heads,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* context_lens, float scale, double* out) {
    const int32_t B = block_size, Hkv = num_kv_heads, D = head_dim, Hq = num_q_heads;
    int rc = check_common(dtype, num_blocks, B, Hkv, D, num_seqs, Hq, max_blocks_per_seq);
    if (rc) return rc;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t ctx = context_lens[s];
        if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * B) return ORC_ERR_ARG;
    }
    const int32_t G = Hq / Hkv;
    int err = ORC_OK;
    int64_t units = (int64_t)num_seqs * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int32_t s = (int32_t)(u / Hkv), g = (int32_t)(u % Hkv);
        int32_t ctx = context_lens[s];
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* x = (double*)malloc(sizeof(double) * ((size_t)ctx + 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        if (!Kc || !Vc || !x || !qd) {
#pragma omp atomic write
            err = ORC_ERR_NOMEM;
            free(Kc); free(Vc); free(x); free(qd);
            continue;
        }
        int grc = gather_sequence(dtype, k_pool, v_pool, num_blocks, B, Hkv, D,
                                  block_tables + (int64_t)s * max_blocks_per_seq, ctx, g, Kc, Vc);
        if (grc) {
#pragma omp atomic write
            err = grc;
        }
        for (int32_t j = 0; j < G && !grc; ++j) {
            int32_t h = g * G + j;
            double* o = out + ((int64_t)s * Hq + h) * D;
            for (int32_t d = 0; d < D; ++d)
                qd[d] = load_as_double(q, dtype, ((int64_t)s * Hq + h) * D + d);
            if (ctx == 0) {
                for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                continue;
            }
            scores(qd, Kc, 0, ctx, D, (double)scale, x);
            double m = x[0];
            for (int32_t i = 1; i < ctx; ++i) if (x[i] > m) m = x[i];
            double den = 0.0;
            for (int32_t i = 0; i < ctx; ++i) { x[i] = exp(x[i] - m); den += x[i]; }
            for (int32_t d = 0; d < D; ++d) {
                double acc = 0.0;
                for (int32_t i = 0; i < ctx; ++i) acc += x[i] * Vc[(int64_t)i * D + d];
                o[d] = acc / den;
            }
        }
        free(Kc); free(Vc); free(x); free(qd);
    }
    return err;
}

/*
 * The same attention over token ranges [k*P, min(ctx, (k+1)*P)).  For each
 * (s, h, k):  m = max score in the range, l = sum exp(score - m),
 * o[d] = sum exp(score - m) V[d]  (not divided by l).  Ranges past the end of
 * the context give m = -inf, l = 0, o = 0.  Outputs are [S][Hq][max_parts](+[D]).
 */
int oracle_partition_decode(int dtype, const void* k_pool, const void* v_pool,
                            int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                            int32_t head_dim, const void* q, int32_t num_seqs,
                            int32_t num_q_heads, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* context_lens, float scale,
                            int32_t partition_size, int32_t max_parts, double* m_out,
                            double* l_out, double* o_out) {
    const int32_t B = block_size, Hkv = num_kv_heads, D = head_dim, Hq = num_q_heads;
    const int32_t P = partition_size;
    int rc = check_common(dtype, num_blocks, B, Hkv, D, num_seqs, Hq, max_blocks_per_seq);
    if (rc) return rc;
    if (P <= 0 || max_parts <= 0) return ORC_ERR_ARG;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t ctx = context_lens[s];
        if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * B) return ORC_ERR_ARG;
        if ((int64_t)ctx > (int64_t)max_parts * P) return ORC_ERR_ARG;
    }
    const int32_t G = Hq / Hkv;
    int err = ORC_OK;
    int64_t units = (int64_t)num_seqs * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int32_t s = (int32_t)(u / Hkv), g = (int32_t)(u % Hkv);
        int32_t ctx = context_lens[s];
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* x = (double*)malloc(sizeof(double) * ((size_t)P + 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        if (!Kc || !Vc || !x || !qd) {
#pragma omp atomic write
            err = ORC_ERR_NOMEM;
            free(Kc); free(Vc); free(x); free(qd);
            continue;
        }
        int grc = gather_sequence(dtype, k_pool, v_pool, num_blocks, B, Hkv, D,
                                  block_tables + (int64_t)s * max_blocks_per_seq, ctx, g, Kc, Vc);
        if (grc) {
#pragma omp atomic write
            err = grc;
        }
        for (int32_t j = 0; j < G && !grc; ++j) {
            int32_t h = g * G + j;
            for (int32_t d = 0; d < D; ++d)
                qd[d] = load_as_double(q, dtype, ((int64_t)s * Hq + h) * D + d);
            for (int32_t k = 0; k < max_parts; ++k) {
                int64_t idx = ((int64_t)s * Hq + h) * max_parts + k;
                double* o = o_out + idx * D;
                int32_t first = k * P;
                int32_t n = ctx - first < P ? ctx - first : P;
                if (n <= 0) {
                    m_out[idx] = -INFINITY;
                    l_out[idx] = 0.0;
                    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                    continue;
                }
                scores(qd, Kc, first, n, D, (double)scale, x);
                double m = x[0];
                for (int32_t i = 1; i < n; ++i) if (x[i] > m) m = x[i];
                double l = 0.0;
                for (int32_t i = 0; i < n; ++i) { x[i] = exp(x[i] - m); l += x[i]; }
                for (int32_t d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int32_t i = 0; i < n; ++i) acc += x[i] * Vc[(int64_t)(first + i) * D + d];
                    o[d] = acc;
                }
                m_out[idx] = m;
                l_out[idx] = l;
            }
        }
        free(Kc); free(Vc); free(x); free(qd);
    }
    return err;
}

/*
 * Log-sum-exp combination of per-range partial results of one (s, h) row:
 * M = max_k m_k;  out = sum_k exp(m_k - M) o_k / sum_k exp(m_k - M) l_k.
 * Rows whose ranges are all empty (l = 0 everywhere) give zeros.
 * rows = number of (s, h) rows; partials are [rows][max_parts](+[D]).
 */
int oracle_lse_merge(int32_t rows, int32_t max_parts, int32_t head_dim, const double* m_in,
                     const double* l_in, const double* o_in, double* out) {
    if (rows < 0 || max_parts <= 0 || head_dim <= 0) return ORC_ERR_ARG;
    const int32_t D = head_dim;
    for (int32_t r = 0; r < rows; ++r) {
        const double* m = m_in + (int64_t)r * max_parts;
        const double* l = l_in + (int64_t)r * max_parts;
        double* o = out + (int64_t)r * D;
        double M = -INFINITY;
        for (int32_t k = 0; k < max_parts; ++k) if (l[k] > 0.0 && m[k] > M) M = m[k];
        if (M == -INFINITY) {
            for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
            continue;
        }
        double L = 0.0;
        for (int32_t k = 0; k < max_parts; ++k) if (l[k] > 0.0) L += exp(m[k] - M) * l[k];
        for (int32_t d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int32_t k = 0; k < max_parts; ++k)
                if (l[k] > 0.0) acc += exp(m[k] - M) * o_in[((int64_t)r * max_parts + k) * D + d];
            o[d] = acc / L;
        }
    }
    return ORC_OK;
}

/*
 * slot[t] = block_tables[s][p / B] * B + p % B  with s = token_seq[t] (or t
 * when token_seq is NULL) and p = positions[t];  p < 0 gives -1.
 * Returns ORC_ERR_BLOCK when p / B falls outside the table row.
 */
int oracle_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* positions, const int32_t* token_seq, int32_t num_tokens,
                        int32_t block_size, int64_t* slot_mapping) {
    if (max_blocks_per_seq <= 0 || block_size <= 0 || num_tokens < 0) return ORC_ERR_ARG;
    int rc = ORC_OK;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int32_t s = token_seq ? token_seq[t] : t;
        int32_t p = positions[t];
        if (p < 0) { slot_mapping[t] = -1; continue; }
        int32_t logical_block = p / block_size;
        if (logical_block >= max_blocks_per_seq) { slot_mapping[t] = -1; rc = ORC_ERR_BLOCK; continue; }
        int32_t phys = block_tables[(int64_t)s * max_blocks_per_seq + logical_block];
        slot_mapping[t] = (int64_t)phys * block_size + p % block_size;
    }
    return rc;
}

/*
 * Append: for every token t with slot >= 0, copy its K and V rows for all kv
 * heads into  pool[slot / B][h][slot % B][:]  (bit copy; no conversion).
 * new_k, new_v are [T][Hkv][D] in the pool's element type.
 */
int oracle_kv_cache_write(int dtype, void* k_pool, void* v_pool, int32_t num_blocks,
                          int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                          const void* new_k, const void* new_v, const int64_t* slot_mapping,
                          int32_t num_tokens) {
    if (dtype < ORC_F32 || dtype > ORC_BF16 || num_blocks <= 0 || block_size <= 0 ||
        num_kv_heads <= 0 || head_dim <= 0 || num_tokens < 0)
        return ORC_ERR_ARG;
    const int64_t e = elem_bytes(dtype);
    const int64_t row_bytes = (int64_t)head_dim * e;
    int rc = ORC_OK;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        int64_t blk = slot / block_size, row = slot % block_size;
        if (blk >= num_blocks) { rc = ORC_ERR_BLOCK; continue; }
        for (int32_t h = 0; h < num_kv_heads; ++h) {
            int64_t dst = ((blk * num_kv_heads + h) * block_size + row) * row_bytes;
            int64_t src = ((int64_t)t * num_kv_heads + h) * row_bytes;
            memcpy((char*)k_pool + dst, (const char*)new_k + src, (size_t)row_bytes);
            memcpy((char*)v_pool + dst, (const char*)new_v + src, (size_t)row_bytes);
        }
    }
    return rc;
}

/*
 * Copy-on-write block copy: for each pair (src, dst), the whole physical
 * block dst (all kv heads, all rows) of both pools becomes a copy of src.
 * pairs is [n][2] = {src, dst}.
 */
int oracle_copy_blocks(void* k_pool, void* v_pool, int32_t num_blocks, int64_t block_bytes,
                       const int32_t* pairs, int32_t num_pairs) {
    if (num_blocks <= 0 || block_bytes <= 0 || num_pairs < 0) return ORC_ERR_ARG;
    int rc = ORC_OK;
    for (int32_t i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { rc = ORC_ERR_BLOCK; continue; }
        memcpy((char*)k_pool + (int64_t)dst * block_bytes, (const char*)k_pool + (int64_t)src * block_bytes,
               (size_t)block_bytes);
        memcpy((char*)v_pool + (int64_t)dst * block_bytes, (const char*)v_pool + (int64_t)src * block_bytes,
               (size_t)block_bytes);
    }
    return rc;
}

/*
 * Swap between two pools of the same block geometry (for example the GPU pool
 * and a pool in host memory, as when a preempted sequence's KV cache is moved
 * to the CPU: "What Is vLLM", section "What is continuous batching in vLLM?").
 * For each pair (src, dst): block dst of the destination pools becomes a copy
 * of block src of the source pools, K and V.
 */
int oracle_swap_blocks(const void* src_k, const void* src_v, int32_t src_blocks, void* dst_k,
                       void* dst_v, int32_t dst_blocks, int64_t block_bytes, const int32_t* pairs,
                       int32_t num_pairs) {
    if (src_blocks <= 0 || dst_blocks <= 0 || block_bytes <= 0 || num_pairs < 0) return ORC_ERR_ARG;
    int rc = ORC_OK;
    for (int32_t i = 0; i < num_pairs; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) { rc = ORC_ERR_BLOCK; continue; }
        memcpy((char*)dst_k + (int64_t)dst * block_bytes, (const char*)src_k + (int64_t)src * block_bytes,
               (size_t)block_bytes);
        memcpy((char*)dst_v + (int64_t)dst * block_bytes, (const char*)src_v + (int64_t)src * block_bytes,
               (size_t)block_bytes);
    }
    return rc;
}

/*
 * Several new tokens per sequence (a chunked-prefill tail or speculative draft
 * tokens; "Serving models with vLLM", section "How it works: inference serving
 * with vLLM").  The last nq positions of sequence s are its new tokens; query j
 * sees positions [0, c_j) with c_j = context_lens[s] - nq + 1 + j, the causal
 * prefix up to and including itself, and its output is the plain attention over
 * those positions (zero when c_j <= 0).  q and out are [S][nq][Hq][D].
 */
int oracle_paged_decode_multi(int dtype, const void* k_pool, const void* v_pool,
                              int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                              int32_t head_dim, const void* q, int32_t num_seqs, int32_t nq,
                              int32_t num_q_heads, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* context_lens,
                              float scale, double* out) {
    const int32_t B = block_size, Hkv = num_kv_heads, D = head_dim, Hq = num_q_heads;
    int rc = check_common(dtype, num_blocks, B, Hkv, D, num_seqs, Hq, max_blocks_per_seq);
    if (rc) return rc;
    if (nq <= 0) return ORC_ERR_ARG;
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t ctx = context_lens[s];
        if (ctx < 0 || (int64_t)ctx > (int64_t)max_blocks_per_seq * B) return ORC_ERR_ARG;
    }
    const int32_t G = Hq / Hkv;
    int err = ORC_OK;
    int64_t units = (int64_t)num_seqs * Hkv;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
        int32_t s = (int32_t)(u / Hkv), g = (int32_t)(u % Hkv);
        int32_t ctx = context_lens[s];
        double* Kc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* Vc = (double*)malloc(sizeof(double) * ((size_t)ctx * D + 1));
        double* x = (double*)malloc(sizeof(double) * ((size_t)ctx + 1));
        double* qd = (double*)malloc(sizeof(double) * (size_t)D);
        if (!Kc || !Vc || !x || !qd) {
#pragma omp atomic write
            err = ORC_ERR_NOMEM;
            free(Kc); free(Vc); free(x); free(qd);
            continue;
        }
        int grc = gather_sequence(dtype, k_pool, v_pool, num_blocks, B, Hkv, D,
                                  block_tables + (int64_t)s * max_blocks_per_seq, ctx, g, Kc, Vc);
        if (grc) {
#pragma omp atomic write
            err = grc;
        }
        for (int32_t j = 0; j < nq && !grc; ++j) {
            int32_t c = ctx - nq + 1 + j;
            for (int32_t hh = 0; hh < G; ++hh) {
                int32_t h = g * G + hh;
                int64_t row = ((int64_t)s * nq + j) * Hq + h;
                double* o = out + row * D;
                if (c <= 0) {
                    for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
                    continue;
                }
                for (int32_t d = 0; d < D; ++d) qd[d] = load_as_double(q, dtype, row * D + d);
                scores(qd, Kc, 0, c, D, (double)scale, x);
                double m = x[0];
                for (int32_t i = 1; i < c; ++i) if (x[i] > m) m = x[i];
                double den = 0.0;
                for (int32_t i = 0; i < c; ++i) { x[i] = exp(x[i] - m); den += x[i]; }
                for (int32_t d = 0; d < D; ++d) {
                    double acc = 0.0;
                    for (int32_t i = 0; i < c; ++i) acc += x[i] * Vc[(int64_t)i * D + d];
                    o[d] = acc / den;
                }
            }
        }
        free(Kc); free(Vc); free(x); free(qd);
    }
    return err;
}

/*
 * Block bookkeeping, one sequence after another ("vLLM in Production",
 * section "PagedAttention - Virtual Memory for the KV Cache": a sequence grows
 * one block at a time as tokens arrive; "What Is vLLM", section "How does
 * PagedAttention work?": blocks allocated on demand, shared blocks reference
 * counted and copied on write).  State: a stack of free ids (free_ids[0 ..
 * *free_count)) and a reference count per block.
 */
void oracle_allocator_reset(int32_t* free_ids, int32_t* free_count, int32_t* refcount,
                            int32_t num_blocks) {
    for (int32_t i = 0; i < num_blocks; ++i) {
        free_ids[i] = num_blocks - 1 - i; /* the top of the stack is block 0 */
        refcount[i] = 0;
    }
    *free_count = num_blocks;
}

static int32_t take_free(int32_t* free_ids, int32_t* free_count) {
    if (*free_count <= 0) return -1;
    *free_count -= 1;
    return free_ids[*free_count];
}

/*
 * Sequence s grows from old_lens[s] to new_lens[s] tokens.  If its last block
 * is partly filled (old % B != 0) and referenced by others, the sequence gets
 * a private copy of it first (copy-on-write); then every new logical block
 * gets a free block.  status[s]: 0 done, 1 no free block left, 2 bad lengths.
 */
int oracle_allocate_for_append(int32_t* free_ids, int32_t* free_count, int32_t* refcount,
                               int32_t num_blocks, void* k_pool, void* v_pool, int64_t block_bytes,
                               int32_t B, int32_t* block_tables, int32_t M, const int32_t* old_lens,
                               const int32_t* new_lens, int32_t num_seqs, int32_t* status) {
    for (int32_t s = 0; s < num_seqs; ++s) {
        int32_t old_len = old_lens[s], new_len = new_lens[s];
        int32_t* row = block_tables + (int64_t)s * M;
        status[s] = 0;
        if (old_len < 0 || new_len < old_len || (int64_t)new_len > (int64_t)M * B) {
            status[s] = 2;
            continue;
        }
        if (new_len == old_len) continue;
        if (old_len % B != 0) {
            int32_t j = (old_len - 1) / B;
            int32_t b = row[j];
            if (b < 0 || b >= num_blocks) { status[s] = 2; continue; }
            if (refcount[b] > 1) {
                int32_t nb = take_free(free_ids, free_count);
                if (nb < 0) { status[s] = 1; continue; }
                memcpy((char*)k_pool + (int64_t)nb * block_bytes,
                       (const char*)k_pool + (int64_t)b * block_bytes, (size_t)block_bytes);
                memcpy((char*)v_pool + (int64_t)nb * block_bytes,
                       (const char*)v_pool + (int64_t)b * block_bytes, (size_t)block_bytes);
                refcount[b] -= 1;
                refcount[nb] = 1;
                row[j] = nb;
            }
        }
        for (int32_t j = (old_len + B - 1) / B; j < (new_len + B - 1) / B; ++j) {
            int32_t nb = take_free(free_ids, free_count);
            if (nb < 0) { status[s] = 1; break; }
            refcount[nb] = 1;
            row[j] = nb;
        }
    }
    return ORC_OK;
}

/* Sequence dst takes the first ceil(lens[i] / B) blocks of src; each gains a reference. */
int oracle_fork_sequences(int32_t* refcount, int32_t num_blocks, int32_t B, int32_t* block_tables,
                          int32_t M, const int32_t* pairs, const int32_t* lens, int32_t n) {
    int rc = ORC_OK;
    for (int32_t i = 0; i < n; ++i) {
        int32_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        int32_t nb = (lens[i] + B - 1) / B;
        if (lens[i] < 0 || nb > M) { rc = ORC_ERR_ARG; continue; }
        for (int32_t j = 0; j < nb; ++j) {
            int32_t b = block_tables[(int64_t)src * M + j];
            if (b < 0 || b >= num_blocks) { rc = ORC_ERR_BLOCK; continue; }
            block_tables[(int64_t)dst * M + j] = b;
            refcount[b] += 1;
        }
    }
    return rc;
}

/* Each listed sequence drops its references; blocks left unreferenced become free. */
int oracle_free_sequences(int32_t* free_ids, int32_t* free_count, int32_t* refcount,
                          int32_t num_blocks, int32_t B, int32_t* block_tables, int32_t M,
                          const int32_t* seqs, const int32_t* lens, int32_t n) {
    int rc = ORC_OK;
    for (int32_t i = 0; i < n; ++i) {
        int32_t* row = block_tables + (int64_t)seqs[i] * M;
        int32_t nb = (lens[i] + B - 1) / B;
        if (lens[i] < 0 || nb > M) { rc = ORC_ERR_ARG; continue; }
        for (int32_t j = 0; j < nb; ++j) {
            int32_t b = row[j];
            row[j] = -1;
            if (b < 0 || b >= num_blocks) { rc = ORC_ERR_BLOCK; continue; }
            refcount[b] -= 1;
            if (refcount[b] == 0) free_ids[(*free_count)++] = b;
        }
    }
    return rc;
}
