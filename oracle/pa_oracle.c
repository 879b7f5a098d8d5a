/*
 * pa_oracle.c -- plain fp64 CPU oracle for the paged KV-cache path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only tests/, the smoke check in __graft_entry__.py and the
 * CPU-baseline leg of bench.py use it.  It shares no code, header, table or
 * helper with the CUDA library; it reads the cache through its own index
 * arithmetic.
 *
 * Every function computes the plain definition of its step, slowly and in
 * the obvious order, in double precision.  bf16 inputs are widened exactly
 * (a bf16 value is the top 16 bits of an IEEE binary32).
 *
 * Sources (vLLM PagedAttention pages):
 *   - "vLLM 深度解析（二）：PagedAttention 核心机制", section 2.1 (exact
 *     attention S = QK^T, P = softmax(S), O = PV), section 2.2 (online
 *     softmax state (m, l, A)), section 3.1 (logical block, offset,
 *     physical block, slot), section 3.2.1 (the x-split K/V cache shapes),
 *     section 3.2.4/3.2.8 (masking past seq_len,
 *     zeroed V of out-of-context slots), section 3.2.9 (cross-partition
 *     merge), section 5.2 (query_start_loc packing).
 *   - "分块预填充与混合批处理", section 11.6 (varlen batch: cu_seqlens_q =
 *     query_start_loc, seqused_k = seq_lens counts this step's tokens).
 *   - "vllm 深度解析：一切从 PagedAttention 谈起", BlockTable walk-through
 *     (slot_id = physical_block * block_size + block_offset) and
 *     write_to_paged_cache / reshape_and_cache ([num_tokens, heads, dim]
 *     scattered to [blocks, block_size, heads, dim]).
 *   - "LLM 推理基础与 vLLM 内部机制", section 2 (KV bytes per token).
 *
 * Readings of points the pages leave open: cache layout [num_blocks, block_size, num_kv_heads, head_dim];
 * q head h reads kv head h / (num_heads / num_kv_heads); no epsilon in the
 * softmax denominator; a negative slot means "do not write"; query i of a
 * request with q_len new tokens sits at position seq_len - q_len + i and
 * sees keys 0 .. seq_len - q_len + i (bottom-right causal alignment); a slot
 * at or past num_blocks * block_size is not written either.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "pa_oracle.h"

/* Worker threads of the attention loops.  Every output row is computed by
 * one thread in the same order as on one thread, so the results do not
 * depend on the thread count (OpenMP only spreads independent rows). */
static int g_threads = 1;

void oracle_set_threads(int32_t n) { g_threads = n > 0 ? n : 1; }

int32_t oracle_max_threads(void) {
#ifdef _OPENMP
    return (int32_t)omp_get_num_procs();
#else
    return 1;
#endif
}

/* bf16 -> double, exact: the bf16 bit pattern is the high half of a binary32. */
static double bf16_to_double(uint16_t h) {
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* ---- Paged addressing (page 1 section 3.1; page 3 BlockTable walk-through) */

int64_t oracle_slot(const int32_t* block_table_row, int32_t block_size, int64_t position) {
    int64_t logical_block = position / block_size;
    int64_t offset = position % block_size;
    int64_t physical_block = block_table_row[logical_block];
    return physical_block * block_size + offset;
}

void oracle_query_start_loc(const int32_t* q_lens, int32_t num_seqs, int32_t* query_start_loc) {
    /* page 1 section 5.2: consecutive differences are the per-request q_len */
    query_start_loc[0] = 0;
    for (int32_t r = 0; r < num_seqs; ++r) query_start_loc[r + 1] = query_start_loc[r] + q_lens[r];
}

void oracle_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* query_start_loc, const int32_t* seq_lens,
                         int32_t num_seqs, int32_t block_size, int64_t* slot_mapping) {
    for (int32_t r = 0; r < num_seqs; ++r) {
        int32_t q_len = query_start_loc[r + 1] - query_start_loc[r];
        int64_t first_pos = (int64_t)seq_lens[r] - q_len;
        const int32_t* row = block_tables + (int64_t)r * max_blocks_per_seq;
        for (int32_t i = 0; i < q_len; ++i)
            slot_mapping[query_start_loc[r] + i] = oracle_slot(row, block_size, first_pos + i);
    }
}

/* ---- reshape_and_cache (page 3 write_to_paged_cache) ------------------- */

void oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim,
                              uint16_t* key_cache, uint16_t* value_cache,
                              int32_t num_blocks, int32_t block_size,
                              const int64_t* slot_mapping) {
    int64_t row = (int64_t)num_kv_heads * head_dim; /* one token's [heads, dim] */
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        /* a negative slot is padding; a slot past the pool's last block has
         * no place in the cache: neither is written */
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
        int64_t block = slot / block_size;
        int64_t offset = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t x = 0; x < head_dim; ++x) {
                int64_t dst = ((block * block_size + offset) * num_kv_heads + h) * head_dim + x;
                int64_t src = i * row + (int64_t)h * head_dim + x;
                key_cache[dst] = key[src];
                value_cache[dst] = value[src];
            }
    }
}

/* ---- KV bytes per token (page 1 section 1; page 4 section 2) ----------- */

int64_t oracle_kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t elem_bytes) {
    return 2LL * num_layers * num_kv_heads * head_dim * elem_bytes;
}

/* ---- Exact attention for one query row (page 1 section 2.1) ------------
 * Gathers keys 0 .. n_keys-1 of one request through its block-table row,
 * scores s_t = scale * <q, k_t>, takes the direct softmax (shift by the
 * max, exponentiate, sum, divide) and returns O = sum_t p_t v_t.        */
static void attend_row(double* out, const uint16_t* q_row, const uint16_t* key_cache,
                       const uint16_t* value_cache, const int32_t* table_row, int64_t n_keys,
                       int32_t kv_head, int32_t num_kv_heads, int32_t head_dim,
                       int32_t block_size, double scale, double* s) {
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t phys = table_row[t / block_size];
        int64_t off = t % block_size;
        const uint16_t* k = key_cache + ((phys * block_size + off) * num_kv_heads + kv_head) * head_dim;
        double dot = 0.0;
        for (int32_t x = 0; x < head_dim; ++x) dot += bf16_to_double(q_row[x]) * bf16_to_double(k[x]);
        s[t] = scale * dot;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n_keys; ++t) if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
    for (int32_t x = 0; x < head_dim; ++x) out[x] = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t phys = table_row[t / block_size];
        int64_t off = t % block_size;
        const uint16_t* v = value_cache + ((phys * block_size + off) * num_kv_heads + kv_head) * head_dim;
        double p = s[t] / l;
        for (int32_t x = 0; x < head_dim; ++x) out[x] += p * bf16_to_double(v[x]);
    }
}

/* ---- Paged decode (page 1 section 3.2; page 3 kernel summary) ----------
 * out[r][h][:] for the single query row of request r, over all seq_lens[r]
 * keys.  q is [num_seqs, num_heads, head_dim].                           */
int oracle_decode(double* out, const uint16_t* q, const uint16_t* key_cache,
                  const uint16_t* value_cache, const int32_t* block_tables,
                  int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    int32_t group = num_heads / num_kv_heads;
    int64_t max_len = 0;
    for (int32_t r = 0; r < num_seqs; ++r) if (seq_lens[r] > max_len) max_len = seq_lens[r];
    int failed = 0;
    /* one (request, q head) row per iteration; each thread its own scores */
#pragma omp parallel num_threads(g_threads) reduction(|| : failed)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t rh = 0; rh < (int64_t)num_seqs * num_heads; ++rh) {
                int32_t r = (int32_t)(rh / num_heads), h = (int32_t)(rh % num_heads);
                attend_row(out + ((int64_t)r * num_heads + h) * head_dim,
                           q + ((int64_t)r * num_heads + h) * head_dim, key_cache, value_cache,
                           block_tables + (int64_t)r * max_blocks_per_seq, seq_lens[r],
                           h / group, num_kv_heads, head_dim, block_size, scale, s);
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* ---- Varlen chunked prefill (page 2 section 11.6; page 1 section 5.2) ---
 * Request r owns query rows query_start_loc[r] .. query_start_loc[r+1]-1.
 * With q_len rows and K/V length seq_lens[r], row i sits at position
 * seq_lens[r] - q_len + i and attends keys 0 .. that position.  A q_len of
 * 1 is a decode row and sees all seq_lens[r] keys.                       */
int oracle_prefill_varlen(double* out, const uint16_t* q, const uint16_t* key_cache,
                          const uint16_t* value_cache, const int32_t* query_start_loc,
                          const int32_t* seq_lens, int32_t num_seqs,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    int32_t group = num_heads / num_kv_heads;
    int64_t max_len = 0;
    for (int32_t r = 0; r < num_seqs; ++r) if (seq_lens[r] > max_len) max_len = seq_lens[r];
    int failed = 0;
    /* one (request, q head) per iteration, its query rows in order */
#pragma omp parallel num_threads(g_threads) reduction(|| : failed)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t rh = 0; rh < (int64_t)num_seqs * num_heads; ++rh) {
                int32_t r = (int32_t)(rh / num_heads), h = (int32_t)(rh % num_heads);
                int32_t q_len = query_start_loc[r + 1] - query_start_loc[r];
                int64_t context = (int64_t)seq_lens[r] - q_len;
                for (int32_t i = 0; i < q_len; ++i) {
                    int64_t row = (int64_t)query_start_loc[r] + i;
                    attend_row(out + (row * num_heads + h) * head_dim,
                               q + (row * num_heads + h) * head_dim, key_cache, value_cache,
                               block_tables + (int64_t)r * max_blocks_per_seq, context + i + 1,
                               h / group, num_kv_heads, head_dim, block_size, scale, s);
                }
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* ---- Online softmax over tiles (page 1 section 2.2) --------------------
 * Scores s[0..n) and values v[n][dv] arrive in tiles [bounds[j],
 * bounds[j+1]).  State (m, l, A) starts at (-inf, 0, 0); each tile:
 *   m' = max(m, max s_j); l' = e^{m-m'} l + sum e^{s_j - m'};
 *   A' = e^{m-m'} A + sum e^{s_j - m'} v_j.
 * Returns O = A / l and the final (m, l).                                */
void oracle_online_softmax(const double* s, const double* v, int32_t n, int32_t dv,
                           const int32_t* bounds, int32_t num_tiles,
                           double* out, double* m_out, double* l_out) {
    double m = -INFINITY, l = 0.0;
    double* A = (double*)calloc((size_t)(dv > 0 ? dv : 1), sizeof(double));
    for (int32_t j = 0; j < num_tiles; ++j) {
        int32_t lo = bounds[j], hi = bounds[j + 1];
        if (hi > n) hi = n;
        if (lo >= hi) continue;
        double tile_max = -INFINITY;
        for (int32_t t = lo; t < hi; ++t) if (s[t] > tile_max) tile_max = s[t];
        double m_new = m > tile_max ? m : tile_max;
        double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
        l *= alpha;
        for (int32_t x = 0; x < dv; ++x) A[x] *= alpha;
        for (int32_t t = lo; t < hi; ++t) {
            double p = exp(s[t] - m_new);
            l += p;
            for (int32_t x = 0; x < dv; ++x) A[x] += p * v[(int64_t)t * dv + x];
        }
        m = m_new;
    }
    for (int32_t x = 0; x < dv; ++x) out[x] = A[x] / l;
    *m_out = m;
    *l_out = l;
    free(A);
}

/* ---- Cross-partition merge (page 1 section 3.2.9) ----------------------
 * Partition p holds its max m_p, exp-sum l_p and normalised output O_p.
 *   m = max_p m_p;  L = sum_p l_p e^{m_p - m};  O = sum_p O_p l_p e^{m_p - m} / L. */
void oracle_merge_partitions(const double* m_parts, const double* l_parts, const double* o_parts,
                             int32_t num_parts, int32_t dv, double* out) {
    double m = -INFINITY;
    for (int32_t p = 0; p < num_parts; ++p) if (m_parts[p] > m) m = m_parts[p];
    double L = 0.0;
    for (int32_t p = 0; p < num_parts; ++p) L += l_parts[p] * exp(m_parts[p] - m);
    for (int32_t x = 0; x < dv; ++x) out[x] = 0.0;
    for (int32_t p = 0; p < num_parts; ++p) {
        double w = l_parts[p] * exp(m_parts[p] - m) / L;
        for (int32_t x = 0; x < dv; ++x) out[x] += o_parts[(int64_t)p * dv + x] * w;
    }
}

/* map_to_kernel_blocks ("vllm 深度解析：一切从 PagedAttention 谈起",
 * BlockTable.map_to_kernel_blocks): every KV-manager block id b becomes the
 * kernel block ids b*k, b*k+1, ..., b*k+k-1, in order, for k kernel blocks
 * per manager block; with k == 1 the list is unchanged.  Negative entries
 * (table padding) become k entries of -1. */
void oracle_map_to_kernel_blocks(const int32_t* ids, int32_t n, int32_t k, int32_t* out) {
    int64_t w = 0;
    for (int32_t i = 0; i < n; ++i)
        for (int32_t j = 0; j < k; ++j)
            out[w++] = ids[i] < 0 ? -1 : (int32_t)((int64_t)ids[i] * k + j);
}

/* ---- FP8 (e4m3) KV cache ------------------------------------------------
 * "vLLM 深度解析（二）：PagedAttention 核心机制", section 3.2 (an FP8 KV
 * cache is loaded as quantized vectors and converted with the cache's
 * scale: fp8::scaled_convert) and "LLM 推理基础与 vLLM 内部机制", section 2
 * (FP8 halves the bytes per token).  The e4m3 format: 1 sign bit, 4
 * exponent bits (bias 7), 3 mantissa bits; exponent field 0 encodes the
 * subnormals m/8 * 2^-6; 0x7F / 0xFF are NaN; there is no infinity; the
 * largest finite magnitude is 1.75 * 2^8 = 448.
 * Readings: a cache value is e4m3(x / scale), the quotient taken in binary32
 * and rounded to the nearest e4m3 value, ties to the even mantissa, with
 * magnitudes beyond 448 saturated to 448 (NaN stays NaN); reading it back
 * gives decoded(e4m3) * scale. */

double oracle_e4m3_decode(uint8_t c) {
    int sign = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) a = 448.0;
    /* spacing of the e4m3 values around a */
    double quantum;
    if (a < ldexp(1.0, -6)) {
        quantum = ldexp(1.0, -9);
    } else {
        int ex;
        frexp(a, &ex);                 /* a = f * 2^ex, 0.5 <= f < 1 */
        quantum = ldexp(1.0, ex - 1 - 3);
    }
    double n = a / quantum;            /* exact: a and quantum are dyadic */
    double fl = floor(n);
    double r = n - fl;
    if (r > 0.5 || (r == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double v = fl * quantum;           /* <= 448: 448 is itself an e4m3 value */
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return (uint8_t)(sign | (uint8_t)(v / ldexp(1.0, -9)));
    int ex;
    double f = frexp(v, &ex);          /* v = f * 2^ex, mantissa 2f - 1 in [0, 1) */
    int e = ex - 1 + 7;
    int m = (int)((2.0 * f - 1.0) * 8.0);
    return (uint8_t)(sign | (uint8_t)(e << 3) | (uint8_t)m);
}

/* Quantizing cache write: like oracle_reshape_and_cache, the slot's row of
 * every kv head receives e4m3(x / scale) of the token's bf16 values. */
void oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, int32_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, uint8_t* key_cache,
                                  uint8_t* value_cache, int32_t num_blocks, int32_t block_size,
                                  const int64_t* slot_mapping, float k_scale, float v_scale) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
        for (int64_t x = 0; x < row; ++x) {
            float kf = (float)bf16_to_double(key[(int64_t)i * row + x]);
            float vf = (float)bf16_to_double(value[(int64_t)i * row + x]);
            key_cache[slot * row + x] = oracle_e4m3_encode(kf / k_scale);
            value_cache[slot * row + x] = oracle_e4m3_encode(vf / v_scale);
        }
    }
}

/* Paged decode over an e4m3 cache: the same exact attention as
 * oracle_decode with k_t = decoded(K) * k_scale and v_t = decoded(V) * v_scale. */
int oracle_decode_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                      const uint8_t* value_cache, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, double scale, double k_scale, double v_scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    int32_t heads_per_kv = num_heads / num_kv_heads;
    int64_t max_len = 1;
    for (int32_t r = 0; r < num_seqs; ++r) if (seq_lens[r] > max_len) max_len = seq_lens[r];
    int failed = 0;
    /* one (request, q head) row per iteration; each thread its own weights */
#pragma omp parallel num_threads(g_threads) reduction(|| : failed)
    {
    double* w = (double*)malloc(sizeof(double) * (size_t)max_len);
    if (!w) failed = 1;
#pragma omp for schedule(dynamic, 1)
    for (int64_t rh = 0; rh < (int64_t)num_seqs * num_heads; ++rh) {
        if (!w) continue;
        int32_t r = (int32_t)(rh / num_heads), h = (int32_t)(rh % num_heads);
        int64_t n = seq_lens[r];
        const int32_t* table = block_tables + (int64_t)r * max_blocks_per_seq;
        {
            const uint16_t* qh = q + ((int64_t)r * num_heads + h) * head_dim;
            int32_t kvh = h / heads_per_kv;
            double top = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                const uint8_t* kr = key_cache +
                    (((int64_t)table[t / block_size] * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
                double acc = 0.0;
                for (int32_t x = 0; x < head_dim; ++x)
                    acc += bf16_to_double(qh[x]) * (oracle_e4m3_decode(kr[x]) * k_scale);
                w[t] = acc * scale;
                if (w[t] > top) top = w[t];
            }
            double total = 0.0;
            for (int64_t t = 0; t < n; ++t) { w[t] = exp(w[t] - top); total += w[t]; }
            double* o = out + ((int64_t)r * num_heads + h) * head_dim;
            for (int32_t x = 0; x < head_dim; ++x) o[x] = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                const uint8_t* vr = value_cache +
                    (((int64_t)table[t / block_size] * block_size + t % block_size) * num_kv_heads + kvh) * head_dim;
                for (int32_t x = 0; x < head_dim; ++x)
                    o[x] += (w[t] / total) * (oracle_e4m3_decode(vr[x]) * v_scale);
            }
        }
    }
    free(w);
    }
    return failed ? -2 : 0;
}

/* ---- Varlen prefill over an FP8 (e4m3) cache (page 1 section 3.2:
 * fp8::scaled_convert inside the K/V load; "分块预填充与混合批处理" section
 * 11.6 for the varlen batch).  The same rows as oracle_prefill_varlen, with
 * key t read as e4m3_decode(K_t) * k_scale and value t as
 * e4m3_decode(V_t) * v_scale.                                            */
static void attend_row_fp8(double* out, const uint16_t* q_row, const uint8_t* key_cache,
                           const uint8_t* value_cache, const int32_t* table_row, int64_t n_keys,
                           int32_t kv_head, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, double scale, double k_scale, double v_scale,
                           double* s) {
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t phys = table_row[t / block_size];
        int64_t off = t % block_size;
        const uint8_t* k = key_cache + ((phys * block_size + off) * num_kv_heads + kv_head) * head_dim;
        double dot = 0.0;
        for (int32_t x = 0; x < head_dim; ++x)
            dot += bf16_to_double(q_row[x]) * (oracle_e4m3_decode(k[x]) * k_scale);
        s[t] = dot * scale;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n_keys; ++t) if (s[t] > m) m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
    for (int32_t x = 0; x < head_dim; ++x) out[x] = 0.0;
    for (int64_t t = 0; t < n_keys; ++t) {
        int64_t phys = table_row[t / block_size];
        int64_t off = t % block_size;
        const uint8_t* v = value_cache + ((phys * block_size + off) * num_kv_heads + kv_head) * head_dim;
        const double pt = s[t] / l;
        for (int32_t x = 0; x < head_dim; ++x) out[x] += pt * (oracle_e4m3_decode(v[x]) * v_scale);
    }
}

int oracle_prefill_varlen_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                              const uint8_t* value_cache, const int32_t* query_start_loc,
                              const int32_t* seq_lens, int32_t num_seqs,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, double scale, double k_scale, double v_scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0) return -1;
    int32_t group = num_heads / num_kv_heads;
    int64_t max_len = 0;
    for (int32_t r = 0; r < num_seqs; ++r) if (seq_lens[r] > max_len) max_len = seq_lens[r];
    int failed = 0;
    /* one (request, q head) per iteration, its query rows in order */
#pragma omp parallel num_threads(g_threads) reduction(|| : failed)
    {
        double* s = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        if (!s) {
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (int64_t rh = 0; rh < (int64_t)num_seqs * num_heads; ++rh) {
                int32_t r = (int32_t)(rh / num_heads), h = (int32_t)(rh % num_heads);
                int32_t q_len = query_start_loc[r + 1] - query_start_loc[r];
                int64_t context = (int64_t)seq_lens[r] - q_len;
                for (int32_t i = 0; i < q_len; ++i) {
                    int64_t row = (int64_t)query_start_loc[r] + i;
                    attend_row_fp8(out + (row * num_heads + h) * head_dim,
                                   q + (row * num_heads + h) * head_dim, key_cache, value_cache,
                                   block_tables + (int64_t)r * max_blocks_per_seq, context + 1 + i,
                                   h / group, num_kv_heads, head_dim, block_size, scale, k_scale,
                                   v_scale, s);
                }
            }
            free(s);
        }
    }
    return failed ? -2 : 0;
}

/* ---- The x-split cache layout (page 1 section 3.2.1) --------------------
 * K cache [num_blocks, num_kv_heads, head_dim / x, block_size, x] and
 * V cache [num_blocks, num_kv_heads, head_dim, block_size], with x the
 * number of cache elements in 16 bytes (8 for bf16).  Element d of kv head
 * h of the token in slot s (block s / B, offset s % B) sits at
 *   K: (((block * H + h) * (D / x) + d / x) * B + offset) * x + d % x
 *   V: ((block * H + h) * D + d) * B + offset.                          */
#define ORACLE_XSPLIT_X 8

static int64_t xsplit_k_index(int64_t block, int64_t offset, int32_t h, int32_t d,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
    int64_t chunks = head_dim / ORACLE_XSPLIT_X;
    return (((block * num_kv_heads + h) * chunks + d / ORACLE_XSPLIT_X) * block_size + offset)
               * ORACLE_XSPLIT_X + d % ORACLE_XSPLIT_X;
}

static int64_t xsplit_v_index(int64_t block, int64_t offset, int32_t h, int32_t d,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
    return ((block * num_kv_heads + h) * head_dim + d) * block_size + offset;
}

/* reshape_and_cache into the x-split layout: the same tokens and slots as
 * oracle_reshape_and_cache, each element stored at its x-split position. */
void oracle_reshape_and_cache_xsplit(const uint16_t* key, const uint16_t* value,
                                     int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                     uint16_t* key_cache, uint16_t* value_cache,
                                     int32_t num_blocks, int32_t block_size,
                                     const int64_t* slot_mapping) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
        int64_t block = slot / block_size;
        int64_t in_block = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = i * row + (int64_t)h * head_dim + d;
                key_cache[xsplit_k_index(block, in_block, h, d, num_kv_heads, head_dim, block_size)] =
                    key[src];
                value_cache[xsplit_v_index(block, in_block, h, d, num_kv_heads, head_dim,
                                           block_size)] = value[src];
            }
    }
}

/* Paged decode over x-split caches: exact attention (page 1 section 2.1)
 * with key t of request r read from block block_tables[r][t / B], offset
 * t % B, at the x-split positions above. */
int oracle_decode_xsplit(double* out, const uint16_t* q, const uint16_t* key_cache,
                         const uint16_t* value_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, double scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim % ORACLE_XSPLIT_X != 0)
        return -1;
    int32_t heads_per_kv = num_heads / num_kv_heads;
    for (int32_t r = 0; r < num_seqs; ++r) {
        int64_t n = seq_lens[r];
        double* w = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!w) return -2;
        const int32_t* table = block_tables + (int64_t)r * max_blocks_per_seq;
        for (int32_t h = 0; h < num_heads; ++h) {
            const uint16_t* qh = q + ((int64_t)r * num_heads + h) * head_dim;
            int32_t kvh = h / heads_per_kv;
            double top = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                int64_t block = table[t / block_size], offset = t % block_size;
                double acc = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    acc += bf16_to_double(qh[d]) *
                           bf16_to_double(key_cache[xsplit_k_index(block, offset, kvh, d,
                                                                   num_kv_heads, head_dim,
                                                                   block_size)]);
                w[t] = scale * acc;
                if (w[t] > top) top = w[t];
            }
            double total = 0.0;
            for (int64_t t = 0; t < n; ++t) { w[t] = exp(w[t] - top); total += w[t]; }
            double* o = out + ((int64_t)r * num_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                int64_t block = table[t / block_size], offset = t % block_size;
                double p = w[t] / total;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] += p * bf16_to_double(value_cache[xsplit_v_index(block, offset, kvh, d,
                                                                          num_kv_heads, head_dim,
                                                                          block_size)]);
            }
        }
        free(w);
    }
    return 0;
}

/* ---- The x-split layout with an e4m3 cache ------------------------------
 * x is the number of cache elements in 16 bytes: 16 for one-byte e4m3.
 * K cache [num_blocks, num_kv_heads, head_dim / 16, block_size, 16] and
 * V cache [num_blocks, num_kv_heads, head_dim, block_size] of e4m3 bytes;
 * the values are those of oracle_reshape_and_cache_fp8 at these places. */
#define ORACLE_XSPLIT_X8 16

static int64_t xsplit8_k_index(int64_t block, int64_t offset, int32_t h, int32_t d,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size) {
    int64_t chunks = head_dim / ORACLE_XSPLIT_X8;
    return (((block * num_kv_heads + h) * chunks + d / ORACLE_XSPLIT_X8) * block_size + offset)
               * ORACLE_XSPLIT_X8 + d % ORACLE_XSPLIT_X8;
}

void oracle_reshape_and_cache_xsplit_fp8(const uint16_t* key, const uint16_t* value,
                                         int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, uint8_t* key_cache,
                                         uint8_t* value_cache, int32_t num_blocks,
                                         int32_t block_size, const int64_t* slot_mapping,
                                         float k_scale, float v_scale) {
    int64_t row = (int64_t)num_kv_heads * head_dim;
    for (int32_t i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0 || slot >= (int64_t)num_blocks * block_size) continue;
        int64_t block = slot / block_size;
        int64_t in_block = slot % block_size;
        for (int32_t h = 0; h < num_kv_heads; ++h)
            for (int32_t d = 0; d < head_dim; ++d) {
                int64_t src = i * row + (int64_t)h * head_dim + d;
                float kf = (float)bf16_to_double(key[src]);
                float vf = (float)bf16_to_double(value[src]);
                key_cache[xsplit8_k_index(block, in_block, h, d, num_kv_heads, head_dim,
                                          block_size)] = oracle_e4m3_encode(kf / k_scale);
                value_cache[xsplit_v_index(block, in_block, h, d, num_kv_heads, head_dim,
                                           block_size)] = oracle_e4m3_encode(vf / v_scale);
            }
    }
}

/* Paged decode over e4m3 x-split caches: exact attention with
 * k_t = decoded(K) * k_scale and v_t = decoded(V) * v_scale read at the
 * x-split positions above. */
int oracle_decode_xsplit_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                             const uint8_t* value_cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                             int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, double scale,
                             double k_scale, double v_scale) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads != 0 || head_dim % ORACLE_XSPLIT_X8 != 0)
        return -1;
    int32_t heads_per_kv = num_heads / num_kv_heads;
    for (int32_t r = 0; r < num_seqs; ++r) {
        int64_t n = seq_lens[r];
        double* w = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        if (!w) return -2;
        const int32_t* table = block_tables + (int64_t)r * max_blocks_per_seq;
        for (int32_t h = 0; h < num_heads; ++h) {
            const uint16_t* qh = q + ((int64_t)r * num_heads + h) * head_dim;
            int32_t kvh = h / heads_per_kv;
            double top = -INFINITY;
            for (int64_t t = 0; t < n; ++t) {
                int64_t block = table[t / block_size], offset = t % block_size;
                double acc = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    acc += bf16_to_double(qh[d]) *
                           (oracle_e4m3_decode(key_cache[xsplit8_k_index(
                                block, offset, kvh, d, num_kv_heads, head_dim, block_size)]) *
                            k_scale);
                w[t] = acc * scale;
                if (w[t] > top) top = w[t];
            }
            double total = 0.0;
            for (int64_t t = 0; t < n; ++t) { w[t] = exp(w[t] - top); total += w[t]; }
            double* o = out + ((int64_t)r * num_heads + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
            for (int64_t t = 0; t < n; ++t) {
                int64_t block = table[t / block_size], offset = t % block_size;
                const double pw = w[t] / total;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] += pw * (oracle_e4m3_decode(value_cache[xsplit_v_index(
                                     block, offset, kvh, d, num_kv_heads, head_dim, block_size)]) *
                                 v_scale);
            }
        }
        free(w);
    }
    return 0;
}
