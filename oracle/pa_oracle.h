/*
 * pa_oracle.h -- declarations of the fp64 CPU oracle (test infrastructure
 * only; see pa_oracle.c).  All pointers are host pointers.  bf16 data is
 * passed as its raw 16-bit patterns.  Layouts:
 *   key_cache / value_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *   decode q                 [num_seqs, num_heads, head_dim]
 *   varlen q / out           [total_q, num_heads, head_dim]
 *   block_tables             [num_seqs, max_blocks_per_seq]
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Threads of the attention loops (default 1); results do not depend on it. */
void oracle_set_threads(int32_t n);
/* Processors OpenMP sees (1 when built without OpenMP). */
int32_t oracle_max_threads(void);
int64_t oracle_slot(const int32_t* block_table_row, int32_t block_size, int64_t position);
void oracle_query_start_loc(const int32_t* q_lens, int32_t num_seqs, int32_t* query_start_loc);
void oracle_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* query_start_loc, const int32_t* seq_lens,
                         int32_t num_seqs, int32_t block_size, int64_t* slot_mapping);
void oracle_reshape_and_cache(const uint16_t* key, const uint16_t* value, int32_t num_tokens,
                              int32_t num_kv_heads, int32_t head_dim,
                              uint16_t* key_cache, uint16_t* value_cache,
                              int32_t num_blocks, int32_t block_size,
                              const int64_t* slot_mapping);
int64_t oracle_kv_bytes_per_token(int32_t num_layers, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t elem_bytes);
int oracle_decode(double* out, const uint16_t* q, const uint16_t* key_cache,
                  const uint16_t* value_cache, const int32_t* block_tables,
                  int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t block_size, double scale);
int oracle_prefill_varlen(double* out, const uint16_t* q, const uint16_t* key_cache,
                          const uint16_t* value_cache, const int32_t* query_start_loc,
                          const int32_t* seq_lens, int32_t num_seqs,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, double scale);
void oracle_online_softmax(const double* s, const double* v, int32_t n, int32_t dv,
                           const int32_t* bounds, int32_t num_tiles,
                           double* out, double* m_out, double* l_out);
double oracle_e4m3_decode(uint8_t code);
uint8_t oracle_e4m3_encode(float x);
void oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value, int32_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, uint8_t* key_cache,
                                  uint8_t* value_cache, int32_t num_blocks, int32_t block_size,
                                  const int64_t* slot_mapping, float k_scale, float v_scale);
int oracle_decode_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                      const uint8_t* value_cache, const int32_t* block_tables,
                      int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int32_t block_size, double scale, double k_scale, double v_scale);
int oracle_prefill_varlen_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                              const uint8_t* value_cache, const int32_t* query_start_loc,
                              const int32_t* seq_lens, int32_t num_seqs,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, double scale, double k_scale, double v_scale);
void oracle_reshape_and_cache_xsplit(const uint16_t* key, const uint16_t* value,
                                     int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                     uint16_t* key_cache, uint16_t* value_cache,
                                     int32_t num_blocks, int32_t block_size,
                                     const int64_t* slot_mapping);
int oracle_decode_xsplit(double* out, const uint16_t* q, const uint16_t* key_cache,
                         const uint16_t* value_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                         int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                         int32_t block_size, double scale);
void oracle_reshape_and_cache_xsplit_fp8(const uint16_t* key, const uint16_t* value,
                                         int32_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, uint8_t* key_cache,
                                         uint8_t* value_cache, int32_t num_blocks,
                                         int32_t block_size, const int64_t* slot_mapping,
                                         float k_scale, float v_scale);
int oracle_decode_xsplit_fp8(double* out, const uint16_t* q, const uint8_t* key_cache,
                             const uint8_t* value_cache, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* seq_lens,
                             int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                             int32_t head_dim, int32_t block_size, double scale,
                             double k_scale, double v_scale);
void oracle_map_to_kernel_blocks(const int32_t* ids, int32_t n, int32_t k, int32_t* out);
void oracle_merge_partitions(const double* m_parts, const double* l_parts,
                             const double* o_parts, int32_t num_parts, int32_t dv,
                             double* out);

#ifdef __cplusplus
}
#endif
#endif
