// pa_internal.h -- launch parameters shared by the library's translation
// units (host and device).  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

// The kernels move K/V in tiles of kBlockSize = 16 tokens (the pages'
// default block size).  A cache block of block_size = 16 R tokens (R = 1, 2
// or 4) holds R tiles: tile t of a request is rows 16 (t mod R) .. + 15 of
// block block_table[t / R].
constexpr int kBlockSize = 16;
constexpr int kWorkspaceHeader = 256; // status record + padding at the start of a workspace

// Decode work.  The tiles (request, kv head, block) of all decode rows are
// numbered request-major, then kv head, then block; the W tiles are split
// into num_ctas contiguous, equal ranges, one per CTA of a persistent grid.
// A CTA's range covers whole (request, kv head) pairs, written straight to
// `out`, and at most two pieces of pairs shared with its neighbours, written
// as partials (m, l, O) and merged by whichever contributor finishes last.
struct DecodeArgs {
  __nv_bfloat16* out;               // [rows, num_heads, D]
  const __nv_bfloat16* q;           // [rows, num_heads, D]
  const int32_t* block_tables;      // [num_seqs, max_blocks_per_seq]
  const int32_t* seq_lens;          // [num_seqs]
  const int32_t* query_start_loc;   // nullptr: row r = request r; else only q_len == 1 rows
  unsigned long long* counters;     // [num_seqs * num_kv_heads] (epoch << 32 | contributions)
  float* part_ml;                   // [num_ctas][2][group][2]  (max in log2 units, exp-sum)
  float* part_o;                    // [num_ctas][2][group][D]  normalised partial output
  int32_t* status;                  // device status record (may be null)
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;                 // work units per request (see kv_div)
  int group;                        // q heads per unit: num_heads / num_kv_heads
  int kv_div;                       // units per cache kv head: unit u reads kv head u / kv_div
  int num_ctas;
  int max_seq_len;
  int num_blocks;
  int block_size;                   // tokens per cache block: 16, 32 or 64
  int tile_shift;                   // log2(block_size / 16)
  int total_q;                      // rows of q / out
  unsigned epoch;                   // distinct per call (never 0)
  float scale_log2;                 // softmax scale * log2(e) (* k_scale for an e4m3 cache)
  float v_scale;                    // multiplies O: the e4m3 cache's V scale, else 1
  // 0: wait for the previous kernel in the stream (griddep_wait) before the
  // first global access.  1: this launch follows the prefill tile kernel of
  // the same pa_prefill_varlen call, which only lets it start once the
  // kernels before the call are complete; the decode rows do not read what
  // the tiles write, so the wait moves to the end of the CTA (the launch
  // then completes after the tile kernel, which keeps stream order).
  int defer_griddep;
  // The tile kernel of the same pa_prefill_varlen call works on
  // tile_kernel_sms() of its tile_sms CTAs (one per SM); the decode rows then
  // go to this grid's first num_ctas - ctas_per_sm * that many CTAs, which
  // start on the SMs the tile kernel leaves.  0: no such split.
  int tile_sms;
  int ctas_per_sm;
  int max_query_len;                // of the call (the tile kernel's row checks)
};

// Launch `kernel` on `stream` with programmatic stream serialization: the
// launch may be scheduled while the previous kernel in the stream is still
// running.  Every kernel launched this way calls griddep_wait() before its
// first access to global memory, so only its prologue (shared-memory and
// barrier set-up) overlaps the previous kernel.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launchers (decode.cu).  Return a cudaError_t from the launch.
// kv8: the caches hold e4m3 values (their scales folded into scale_log2
// and v_scale) instead of bf16.  xsplit: bf16 caches in the x-split layout,
// K [blocks, kv heads, head_dim / 8, block, 8] seen through a 5-D map
// {64, block / 8, head_dim / 8, kv heads, blocks} with box {64, 2, head_dim
// / 8, 1, 1}, 128-byte swizzled, and V [blocks, kv heads, head_dim, block]
// through a 4-D map {block, head_dim, kv heads, blocks} with box {16,
// head_dim, 1, 1}, 32-byte swizzled.
cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          int head_dim, bool kv8, bool xsplit, cudaStream_t stream);
// Tensor-core decode (decode_tc.cu): qmap = q as {head_dim, heads, rows}
// with a {64, group, 1} box; kmap, vmap = bf16 caches as {64, 8, head_dim /
// 64, slots / 8, kv heads} with a {64, 8, head_dim / 64, 2, 1} box (one
// block of one kv head per copy), all 128-byte swizzled; kv8: e4m3 caches
// as {head_dim, kv heads, slots} bytes with a {head_dim, 1, 16} box
// (128-byte swizzle at head_dim 128, 64-byte at 64).
cudaError_t launch_decode_tc(const DecodeArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, int head_dim, bool kv8, cudaStream_t stream);
// Smallest group size the decode kernel is instantiated for that covers g.
int decode_gmax(int group);
// CTAs per SM the decode kernel for (head_dim, group) is built for.
int decode_ctas_per_sm(int head_dim, int group);

// Chunked-prefill attention (prefill.cu).  Work unit: 128 query rows of one
// request with q_len > 1 for two q heads of the same kv head (one head when
// the group has no partner left), over all the keys those rows see, in
// 128-key steps.  The steps of all units are numbered (request-major, then
// query tile from the last, then head pair, then key step) and cut into
// num_ctas equal contiguous ranges, one per CTA of a persistent grid; a unit
// cut by a range boundary is finished by merging its pieces' (m, l, O)
// partials, by the contributor that finishes last.
struct PrefillArgs {
  __nv_bfloat16* out;               // [total_q, num_heads, D]
  const __nv_bfloat16* q;           // [total_q, num_heads, D]
  const int32_t* block_tables;      // [num_seqs, max_blocks_per_seq]
  const int32_t* seq_lens;          // [num_seqs]
  const int32_t* query_start_loc;   // [num_seqs + 1]
  int32_t* status;                  // device status record (may be null)
  unsigned long long* counters;     // [max_units] (epoch << 32 | contributions)
  float* part_ml;                   // [num_ctas][2][2 heads][128 rows][2]  (m in log2 units, l)
  float* part_o;                    // [num_ctas][2][2 heads][D / 4][128 rows][4]  normalised partial O
  int max_blocks_per_seq;
  int num_seqs;
  int num_heads;
  int num_kv_heads;
  int group;
  int max_seq_len;
  int max_query_len;
  int num_blocks;
  int block_size;                   // tokens per cache block: 16, 32 or 64
  int tile_shift;                   // log2(block_size / 16)
  int total_q;
  int num_ctas;                     // persistent grid (one CTA per SM)
  long long max_units;              // size of `counters`
  unsigned epoch;                   // distinct per call (never 0)
  float scale_log2;                 // softmax scale (* k_scale for e4m3) * log2(e)
  float o_scale;                    // 1, or v_scale for e4m3
  // 1: the decode rows of the same call follow in the streaming decode
  // kernel, which takes the SMs this grid leaves (tile_kernel_sms()); only
  // that many CTAs work.  0: every CTA works.
  int partition;
};
// Bytes of the prefill partial records (part_ml and part_o) for num_ctas CTAs.
size_t prefill_partials_bytes(int num_ctas, int head_dim);
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& qmap, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int head_dim, bool kv8, cudaStream_t stream);

// Cache writes (cache_write.cu).
cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t key_stride,
                                     int64_t value_stride, void* key_cache, void* value_cache,
                                     const int64_t* slot_mapping, int num_tokens, int row_elems,
                                     int64_t num_slots, int32_t* status, cudaStream_t stream);
// e4m3 cache write: cache = e4m3(x / scale), nearest even, saturated to 448.
cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_stride,
                                         int64_t value_stride, void* key_cache, void* value_cache,
                                         const int64_t* slot_mapping, int num_tokens, int row_elems,
                                         int64_t num_slots, float k_scale, float v_scale,
                                         int32_t* status, cudaStream_t stream);
// x-split cache write: K [blocks, kv heads, head_dim / 8, block, 8],
// V [blocks, kv heads, head_dim, block] (bf16).
cudaError_t launch_reshape_and_cache_xsplit(const void* key, const void* value, int64_t key_stride,
                                            int64_t value_stride, void* key_cache,
                                            void* value_cache, const int64_t* slot_mapping,
                                            int num_tokens, int num_kv_heads, int head_dim,
                                            int block_size, int64_t num_slots, int32_t* status,
                                            cudaStream_t stream);
// x-split e4m3 cache write: K [blocks, kv heads, head_dim / 16, block, 16],
// V [blocks, kv heads, head_dim, block] (bytes), values e4m3(x / scale).
cudaError_t launch_reshape_and_cache_xsplit_fp8(const void* key, const void* value,
                                                int64_t key_stride, int64_t value_stride,
                                                void* key_cache, void* value_cache,
                                                const int64_t* slot_mapping, int num_tokens,
                                                int num_kv_heads, int head_dim, int block_size,
                                                int64_t num_slots, float k_scale, float v_scale,
                                                int32_t* status, cudaStream_t stream);
cudaError_t launch_map_kernel_blocks(int32_t* out, const int32_t* in, int64_t n, int k,
                                     int32_t* status, cudaStream_t stream);
// Slot mapping and token-major cache write of the new tokens in one kernel
// (slot_mapping may be null: the slots are not stored).
cudaError_t launch_append_tokens(const void* key, const void* value, int64_t key_stride,
                                 int64_t value_stride, void* key_cache, void* value_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* query_start_loc, const int32_t* seq_lens,
                                 int num_seqs, int total_tokens, int block_size, int num_blocks,
                                 int row_elems, int64_t* slot_mapping, int32_t* status,
                                 cudaStream_t stream);
cudaError_t launch_slot_mapping(int64_t* slot_mapping, int total_tokens, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* query_start_loc,
                                const int32_t* seq_lens, int num_seqs, int block_size,
                                int num_blocks, int32_t* status, cudaStream_t stream);

}  // namespace pa
