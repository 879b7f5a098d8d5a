// decode_common.cuh -- the split of a decode batch into per-CTA tile ranges
// and the merge of the pieces of a (request, kv head) pair that several
// CTAs share.  Used by both decode kernels.
//
// Every (request, kv head, 16-token block) tile of the decode rows is
// numbered request-major, then kv head, then block; the W tiles are cut into
// num_ctas contiguous ranges of equal size.  A range covers whole pairs,
// written straight to the output, and at most two pieces of pairs shared
// with its neighbours; those are written as partials (m_j, l_j, O_j) and
// merged ("vLLM 深度解析（二）：PagedAttention 核心机制", sections 3.2.7 and
// 3.3: m = max m_j, L = sum l_j e^{m_j - m}, O = sum O_j l_j e^{m_j - m} / L)
// by the contributor that finishes last.
#pragma once

#include "pa_internal.h"
#include "pa_ptx.cuh"
#include "work_split.cuh"

namespace pa {
namespace {

// How a segment's result is written.
constexpr int kWhole = 0;  // the whole (request, kv head): final bf16 output
constexpr int kHead = 1;   // continues a pair begun by an earlier CTA: partial slot 0
constexpr int kTail = 2;   // begins a pair finished by later CTAs: partial slot 1

// 16-token tiles of request r that the decode kernel processes (0 for rows that are
// not decode rows, and for invalid lengths); also its length and q row.
// `len` = seq_lens[r]; q0, q1 = query_start_loc[r], [r + 1] (when present).
__device__ __forceinline__ RowLimits row_limits(const DecodeArgs& a) {
  return RowLimits{a.max_query_len, a.max_seq_len, a.max_blocks_per_seq * a.block_size, a.total_q};
}

__device__ __forceinline__ int blocks_from(const DecodeArgs& a, int r, int len, int q0, int q1,
                                           int* seq_len, int* row) {
  if (a.query_start_loc != nullptr) {  // only decode rows (q_len == 1), at row q0
    const int n = decode_row_tiles(q0, q1, len, row_limits(a));
    if (n > 0) {
      *seq_len = len;
      *row = q0;
    }
    return n;
  }
  if (len < 1 || len > a.max_seq_len || len > a.max_blocks_per_seq * a.block_size) return 0;
  *seq_len = len;
  *row = r;
  return (len + kBlockSize - 1) / kBlockSize;
}

__device__ __forceinline__ int request_blocks(const DecodeArgs& a, int r, int* seq_len, int* row) {
  const int q0 = a.query_start_loc != nullptr ? a.query_start_loc[r] : 0;
  const int q1 = a.query_start_loc != nullptr ? a.query_start_loc[r + 1] : 0;
  return blocks_from(a, r, a.seq_lens[r], q0, q1, seq_len, row);
}

// Sum over the warp of a non-negative per-lane value below 2^31, by two
// 32-bit warp reductions of its 16-bit halves (a reduction is an order of
// magnitude faster than a chain of shuffles here).
__device__ __forceinline__ long long warp_sum_ll(long long v) {
  const unsigned lo = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v) & 0xffffu);
  const unsigned hi = __reduce_add_sync(0xffffffffu, static_cast<unsigned>(v >> 16));
  return (static_cast<long long>(hi) << 16) + lo;
}

// Reports the rows request_blocks() rejects (done once, by CTA 0).
__device__ void report_bad_rows(const DecodeArgs& a, int lane) {
  for (int r = lane; r < a.num_seqs; r += 32) {
    int rw = r;
    if (a.query_start_loc != nullptr) {
      const int q0 = a.query_start_loc[r];
      if (a.query_start_loc[r + 1] - q0 != 1) continue;
      rw = q0;
      if (rw < 0 || rw >= a.total_q) {
        record_error(a.status, PA_DEV_BAD_QUERY_LEN, r, rw);
        continue;
      }
    }
    const int len = a.seq_lens[r];
    if (len < 1 || len > a.max_seq_len || len > a.max_blocks_per_seq * a.block_size)
      record_error(a.status, PA_DEV_BAD_SEQ_LEN, r, len);
  }
}

// First cache row (slot) of 16-token tile `tile` of a request whose tile
// lives in block `block_id`.
__device__ __forceinline__ int tile_row(const DecodeArgs& a, int block_id, int tile) {
  return block_id * a.block_size + (tile & ((1 << a.tile_shift) - 1)) * kBlockSize;
}

}  // namespace
}  // namespace pa
