// cache_write.cu -- the two writes that precede attention in a step:
//
//  * slot mapping ("vLLM 深度解析（二）：PagedAttention 核心机制", section 3.1):
//      logical block = pos / B, offset = pos % B,
//      slot = block_table[r][logical block] * B + offset,
//    for the new tokens of each request, which sit at positions
//    seq_len - q_len .. seq_len - 1 ("分块预填充与混合批处理", section 11.6:
//    seq_lens counts this step's tokens);
//  * reshape_and_cache ("vllm 深度解析：一切从 PagedAttention 谈起",
//    write_to_paged_cache): token i's [kv_heads, head_dim] K and V rows are
//    copied to slot slot_mapping[i] of the [slots, kv_heads, head_dim] cache
//    (also: an e4m3-quantizing variant, and one for the x-split layout).
//
// Both are pure data movement.  The cache write gives each token one warp;
// lanes move 16-byte chunks, so each token's K and V rows (2 KB each at 8 kv
// heads x 128) are read and written with fully coalesced vector accesses.
// Both are launched so that they (and the attention launch after them) may
// be scheduled while the previous kernel in the stream finishes; each waits
// for that kernel before it touches global memory.
#include <algorithm>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kWriteWarps = 8;

__global__ void __launch_bounds__(kWriteWarps * 32)
reshape_and_cache_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                         int64_t key_stride_chunks, int64_t value_stride_chunks,
                         uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                         const int64_t* __restrict__ slot_mapping, int num_tokens,
                         int row_chunks, int64_t num_slots, int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();  // slot_mapping may come from the previous kernel
  const int token = blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (lane == 0) record_error(status, PA_DEV_BAD_SLOT, token, static_cast<int>(slot));
    return;
  }
  const uint4* ks = key + token * key_stride_chunks;
  const uint4* vs = value + token * value_stride_chunks;
  uint4* kd = key_cache + slot * row_chunks;
  uint4* vd = value_cache + slot * row_chunks;
  for (int c = lane; c < row_chunks; c += 32) {
    const uint4 kv = __ldg(ks + c);
    const uint4 vv = __ldg(vs + c);
    kd[c] = kv;
    vd[c] = vv;
  }
}

// Two floats to two e4m3 codes (low byte = lo): nearest even, magnitudes
// beyond 448 saturated, NaN kept.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// The quantizing write of an e4m3 cache ("vLLM 深度解析（二）", section 3.2:
// the FP8 cache is stored quantized with a per-tensor scale): each lane
// turns 8 bf16 values x into e4m3(x / scale) and stores 8 bytes.
__global__ void __launch_bounds__(kWriteWarps * 32)
reshape_and_cache_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                             int64_t key_stride_chunks, int64_t value_stride_chunks,
                             uint2* __restrict__ key_cache, uint2* __restrict__ value_cache,
                             const int64_t* __restrict__ slot_mapping, int num_tokens,
                             int row_chunks, int64_t num_slots, float k_scale, float v_scale,
                             int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();  // slot_mapping may come from the previous kernel
  const int token = blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (lane == 0) record_error(status, PA_DEV_BAD_SLOT, token, static_cast<int>(slot));
    return;
  }
  auto quantize = [](uint4 w, float scale) -> uint2 {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __fdiv_rn(__uint_as_float(ws[e] << 16), scale);
      const float hi = __fdiv_rn(__uint_as_float(ws[e] & 0xffff0000u), scale);
      out[e] = e4m3x2(lo, hi);
    }
    return make_uint2(out[0] | (out[1] << 16), out[2] | (out[3] << 16));
  };
  const uint4* ks = key + token * key_stride_chunks;
  const uint4* vs = value + token * value_stride_chunks;
  uint2* kd = key_cache + slot * row_chunks;
  uint2* vd = value_cache + slot * row_chunks;
  for (int c = lane; c < row_chunks; c += 32) {
    kd[c] = quantize(__ldg(ks + c), k_scale);
    vd[c] = quantize(__ldg(vs + c), v_scale);
  }
}

// The cache write into the x-split layout ("vLLM 深度解析（二）：PagedAttention
// 核心机制", section 3.2.1): chunk c (8 bf16 = 16 bytes) of kv head h of the
// token in slot s goes to K[s / B][h][c][s % B][0..7]; V element d to
// V[s / B][h][d][s % B].  One warp per token, lanes over 16-byte chunks: the
// K chunks are 16-byte stores, the V elements land B elements apart.
__global__ void __launch_bounds__(kWriteWarps * 32)
reshape_and_cache_xsplit_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                int64_t key_stride_chunks, int64_t value_stride_chunks,
                                uint4* __restrict__ key_cache, uint16_t* __restrict__ value_cache,
                                const int64_t* __restrict__ slot_mapping, int num_tokens,
                                int num_kv_heads, int head_dim, int block_size, int64_t num_slots,
                                int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();  // slot_mapping may come from the previous kernel
  const int token = blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (lane == 0) record_error(status, PA_DEV_BAD_SLOT, token, static_cast<int>(slot));
    return;
  }
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot % block_size);
  const int cpr = head_dim / 8;  // 16-byte chunks per kv head
  const uint4* ks = key + token * key_stride_chunks;
  const uint4* vs = value + token * value_stride_chunks;
  for (int c = lane; c < num_kv_heads * cpr; c += 32) {
    const int h = c / cpr, cc = c % cpr;
    const int64_t head_base = blk * num_kv_heads + h;
    const uint4 kv = __ldg(ks + c);
    const uint4 vv = __ldg(vs + c);
    key_cache[(head_base * cpr + cc) * block_size + off] = kv;
    uint16_t* vd = value_cache + (head_base * head_dim + cc * 8) * block_size + off;
    const uint32_t w[4] = {vv.x, vv.y, vv.z, vv.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      vd[(2 * e) * block_size] = static_cast<uint16_t>(w[e] & 0xffffu);
      vd[(2 * e + 1) * block_size] = static_cast<uint16_t>(w[e] >> 16);
    }
  }
}

// The quantizing write into the x-split layout with an e4m3 cache (x = 16
// one-byte elements): chunk c (16 values) of kv head h of the token in slot s
// becomes e4m3(x / k_scale) at K[s / B][h][c][s % B][0..15], one 16-byte
// store; V element d becomes e4m3(x / v_scale) at V[s / B][h][d][s % B].
// One warp per token, lanes over 16-value chunks.
__global__ void __launch_bounds__(kWriteWarps * 32)
reshape_and_cache_xsplit_fp8_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                    int64_t key_stride_chunks, int64_t value_stride_chunks,
                                    uint4* __restrict__ key_cache, uint8_t* __restrict__ value_cache,
                                    const int64_t* __restrict__ slot_mapping, int num_tokens,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int64_t num_slots, float k_scale, float v_scale,
                                    int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();  // slot_mapping may come from the previous kernel
  const int token = blockIdx.x * kWriteWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (token >= num_tokens) return;
  const int64_t slot = slot_mapping[token];
  if (slot < 0) return;  // padding token
  if (slot >= num_slots) {
    if (lane == 0) record_error(status, PA_DEV_BAD_SLOT, token, static_cast<int>(slot));
    return;
  }
  // 8 bf16 values -> 8 e4m3 bytes (in order, as two 32-bit words).
  auto quantize8 = [](uint4 w, float scale, uint32_t* out) {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    uint32_t p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float lo = __fdiv_rn(__uint_as_float(ws[e] << 16), scale);
      const float hi = __fdiv_rn(__uint_as_float(ws[e] & 0xffff0000u), scale);
      p[e] = e4m3x2(lo, hi);
    }
    out[0] = p[0] | (p[1] << 16);
    out[1] = p[2] | (p[3] << 16);
  };
  const int64_t blk = slot / block_size;
  const int off = static_cast<int>(slot % block_size);
  const int cpr = head_dim / 16;  // 16-value chunks per kv head
  const uint4* ks = key + token * key_stride_chunks;
  const uint4* vs = value + token * value_stride_chunks;
  for (int c = lane; c < num_kv_heads * cpr; c += 32) {
    const int h = c / cpr, cc = c % cpr;
    const int64_t head_base = blk * num_kv_heads + h;
    uint32_t kq[4], vq[4];
    quantize8(__ldg(ks + 2 * c), k_scale, kq);
    quantize8(__ldg(ks + 2 * c + 1), k_scale, kq + 2);
    quantize8(__ldg(vs + 2 * c), v_scale, vq);
    quantize8(__ldg(vs + 2 * c + 1), v_scale, vq + 2);
    key_cache[(head_base * cpr + cc) * block_size + off] = make_uint4(kq[0], kq[1], kq[2], kq[3]);
    uint8_t* vd = value_cache + (head_base * head_dim + cc * 16) * block_size + off;
#pragma unroll
    for (int e = 0; e < 16; ++e)
      vd[e * block_size] = static_cast<uint8_t>(vq[e >> 2] >> (8 * (e & 3)));
  }
}

// One CTA per request; its threads cover the request's new tokens.
__global__ void __launch_bounds__(128)
slot_mapping_kernel(int64_t* __restrict__ slot_mapping, int total_tokens,
                    const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
                    const int32_t* __restrict__ query_start_loc,
                    const int32_t* __restrict__ seq_lens, int block_size, int num_blocks,
                    int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int q0 = query_start_loc[r];
  const int q1 = query_start_loc[r + 1];
  const int seq_len = seq_lens[r];
  const int q_len = q1 - q0;
  const int64_t first_pos = static_cast<int64_t>(seq_len) - q_len;
  const int32_t* row = block_tables + static_cast<int64_t>(r) * max_blocks_per_seq;
  for (int i = threadIdx.x; i < q_len; i += blockDim.x) {
    const int64_t flat = static_cast<int64_t>(q0) + i;
    if (flat < 0 || flat >= total_tokens) {
      if (i == 0) record_error(status, PA_DEV_BAD_QUERY_LEN, r, q1);
      continue;
    }
    const int64_t pos = first_pos + i;
    const int64_t logical = pos >= 0 ? pos / block_size : -1;
    int64_t slot = -1;
    if (logical < 0 || logical >= max_blocks_per_seq) {
      record_error(status, PA_DEV_BAD_SEQ_LEN, r, seq_len);
    } else {
      const int32_t phys = row[logical];
      if (phys < 0 || phys >= num_blocks)
        record_error(status, PA_DEV_BAD_BLOCK_ID, r, phys);
      else
        slot = static_cast<int64_t>(phys) * block_size + (pos - logical * block_size);
    }
    slot_mapping[flat] = slot;
  }
}

// Slot mapping and cache write of this step's new tokens in one kernel (one
// launch and one dependent memory round trip fewer than the two kernels
// above in sequence).  CTA (r, y) serves request r; its warps take the
// request's new tokens y * kWriteWarps + warp, then every gridDim.y *
// kWriteWarps-th one after it, so a long chunk is spread over gridDim.y CTAs.
// For each token a warp first loads the token's K and V rows (they depend
// only on its row), then computes its slot exactly as slot_mapping_kernel
// does (optionally storing it) and writes the rows there as
// reshape_and_cache_kernel does.
constexpr int kAppendChunksPerLane = 4;  // 16-byte chunks of a row held per lane per pass
constexpr int kAppendMaxSplit = 16;      // CTAs per request, at most

__global__ void __launch_bounds__(kWriteWarps * 32)
append_tokens_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                     int64_t key_stride_chunks, int64_t value_stride_chunks,
                     uint4* __restrict__ key_cache, uint4* __restrict__ value_cache,
                     const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
                     const int32_t* __restrict__ query_start_loc,
                     const int32_t* __restrict__ seq_lens, int total_tokens, int block_size,
                     int num_blocks, int row_chunks, int64_t* __restrict__ slot_out,
                     int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int q0 = query_start_loc[r];
  const int q1 = query_start_loc[r + 1];
  const int q_len = q1 - q0;
  const int first = static_cast<int>(blockIdx.y) * kWriteWarps + warp;
  if (first >= q_len) return;
  const int seq_len = seq_lens[r];
  const int64_t first_pos = static_cast<int64_t>(seq_len) - q_len;
  const int32_t* row = block_tables + static_cast<int64_t>(r) * max_blocks_per_seq;
  for (int i = first; i < q_len; i += gridDim.y * kWriteWarps) {
    const int64_t flat = static_cast<int64_t>(q0) + i;
    if (flat < 0 || flat >= total_tokens) {
      if (i == 0 && lane == 0) record_error(status, PA_DEV_BAD_QUERY_LEN, r, q1);
      continue;
    }
    const uint4* ks = key + flat * key_stride_chunks;
    const uint4* vs = value + flat * value_stride_chunks;
    // The rows' first pass is loaded before the slot is known.
    uint4 kb[kAppendChunksPerLane], vb[kAppendChunksPerLane];
#pragma unroll
    for (int k = 0; k < kAppendChunksPerLane; ++k) {
      const int c = lane + 32 * k;
      if (c < row_chunks) {
        kb[k] = __ldg(ks + c);
        vb[k] = __ldg(vs + c);
      }
    }
    const int64_t pos = first_pos + i;
    const int64_t logical = pos >= 0 ? pos / block_size : -1;
    int64_t slot = -1;
    if (logical < 0 || logical >= max_blocks_per_seq) {
      if (lane == 0) record_error(status, PA_DEV_BAD_SEQ_LEN, r, seq_len);
    } else {
      const int32_t phys = row[logical];
      if (phys < 0 || phys >= num_blocks) {
        if (lane == 0) record_error(status, PA_DEV_BAD_BLOCK_ID, r, phys);
      } else {
        slot = static_cast<int64_t>(phys) * block_size + (pos - logical * block_size);
      }
    }
    if (slot_out != nullptr && lane == 0) slot_out[flat] = slot;
    if (slot < 0) continue;
    uint4* kd = key_cache + slot * row_chunks;
    uint4* vd = value_cache + slot * row_chunks;
#pragma unroll
    for (int k = 0; k < kAppendChunksPerLane; ++k) {
      const int c = lane + 32 * k;
      if (c < row_chunks) {
        kd[c] = kb[k];
        vd[c] = vb[k];
      }
    }
    for (int c = lane + 32 * kAppendChunksPerLane; c < row_chunks; c += 32) {  // longer rows
      const uint4 kv = __ldg(ks + c);
      const uint4 vv = __ldg(vs + c);
      kd[c] = kv;
      vd[c] = vv;
    }
  }
}

// One thread per manager-block entry writes its k kernel-block ids.
__global__ void __launch_bounds__(256)
map_kernel_blocks_kernel(int32_t* __restrict__ out, const int32_t* __restrict__ in, int64_t n,
                         int k, int32_t* status) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int32_t b = in[i];
  const int64_t first = static_cast<int64_t>(b) * k;
  const bool bad = b >= 0 && first + k - 1 > 0x7fffffffLL;
  if (bad) record_error(status, PA_DEV_BAD_BLOCK_ID, static_cast<int>(i), b);
  for (int j = 0; j < k; ++j)
    out[i * k + j] = (b < 0 || bad) ? -1 : static_cast<int32_t>(first + j);
}

}  // namespace

cudaError_t launch_map_kernel_blocks(int32_t* out, const int32_t* in, int64_t n, int k,
                                     int32_t* status, cudaStream_t stream) {
  const int64_t grid = (n + 255) / 256;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  return launch_overlapped(map_kernel_blocks_kernel, dim3(static_cast<unsigned>(grid)), dim3(256), 0,
                           stream, out, in, n, k, status);
}

cudaError_t launch_reshape_and_cache(const void* key, const void* value, int64_t key_stride,
                                     int64_t value_stride, void* key_cache, void* value_cache,
                                     const int64_t* slot_mapping, int num_tokens, int row_elems,
                                     int64_t num_slots, int32_t* status, cudaStream_t stream) {
  const int grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
  return launch_overlapped(reshape_and_cache_kernel, dim3(grid), dim3(kWriteWarps * 32), 0, stream,
                           static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                           key_stride / 8, value_stride / 8, static_cast<uint4*>(key_cache),
                           static_cast<uint4*>(value_cache), slot_mapping, num_tokens,
                           row_elems / 8, num_slots, status);
}

cudaError_t launch_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_stride,
                                         int64_t value_stride, void* key_cache, void* value_cache,
                                         const int64_t* slot_mapping, int num_tokens, int row_elems,
                                         int64_t num_slots, float k_scale, float v_scale,
                                         int32_t* status, cudaStream_t stream) {
  const int grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
  return launch_overlapped(reshape_and_cache_fp8_kernel, dim3(grid), dim3(kWriteWarps * 32), 0,
                           stream, static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                           key_stride / 8, value_stride / 8, static_cast<uint2*>(key_cache),
                           static_cast<uint2*>(value_cache), slot_mapping, num_tokens,
                           row_elems / 8, num_slots, k_scale, v_scale, status);
}

cudaError_t launch_reshape_and_cache_xsplit(const void* key, const void* value, int64_t key_stride,
                                            int64_t value_stride, void* key_cache,
                                            void* value_cache, const int64_t* slot_mapping,
                                            int num_tokens, int num_kv_heads, int head_dim,
                                            int block_size, int64_t num_slots, int32_t* status,
                                            cudaStream_t stream) {
  const int grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
  return launch_overlapped(reshape_and_cache_xsplit_kernel, dim3(grid), dim3(kWriteWarps * 32), 0,
                           stream, static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                           key_stride / 8, value_stride / 8, static_cast<uint4*>(key_cache),
                           static_cast<uint16_t*>(value_cache), slot_mapping, num_tokens,
                           num_kv_heads, head_dim, block_size, num_slots, status);
}

cudaError_t launch_reshape_and_cache_xsplit_fp8(const void* key, const void* value,
                                                int64_t key_stride, int64_t value_stride,
                                                void* key_cache, void* value_cache,
                                                const int64_t* slot_mapping, int num_tokens,
                                                int num_kv_heads, int head_dim, int block_size,
                                                int64_t num_slots, float k_scale, float v_scale,
                                                int32_t* status, cudaStream_t stream) {
  const int grid = (num_tokens + kWriteWarps - 1) / kWriteWarps;
  return launch_overlapped(reshape_and_cache_xsplit_fp8_kernel, dim3(grid), dim3(kWriteWarps * 32),
                           0, stream, static_cast<const uint4*>(key),
                           static_cast<const uint4*>(value), key_stride / 8, value_stride / 8,
                           static_cast<uint4*>(key_cache), static_cast<uint8_t*>(value_cache),
                           slot_mapping, num_tokens, num_kv_heads, head_dim, block_size, num_slots,
                           k_scale, v_scale, status);
}

cudaError_t launch_append_tokens(const void* key, const void* value, int64_t key_stride,
                                 int64_t value_stride, void* key_cache, void* value_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* query_start_loc, const int32_t* seq_lens,
                                 int num_seqs, int total_tokens, int block_size, int num_blocks,
                                 int row_elems, int64_t* slot_mapping, int32_t* status,
                                 cudaStream_t stream) {
  // Every request has at least one new token in the usual step, so none has
  // more than total_tokens - num_seqs + 1: that many tokens, kWriteWarps per
  // CTA, set the split of a request over CTAs (a longer request is still
  // served, its CTAs looping over it).
  const int64_t longest = std::max<int64_t>(1, static_cast<int64_t>(total_tokens) - num_seqs + 1);
  const int split = static_cast<int>(
      std::min<int64_t>(kAppendMaxSplit, (longest + kWriteWarps - 1) / kWriteWarps));
  return launch_overlapped(append_tokens_kernel, dim3(num_seqs, split), dim3(kWriteWarps * 32), 0,
                           stream,
                           static_cast<const uint4*>(key), static_cast<const uint4*>(value),
                           key_stride / 8, value_stride / 8, static_cast<uint4*>(key_cache),
                           static_cast<uint4*>(value_cache), block_tables, max_blocks_per_seq,
                           query_start_loc, seq_lens, total_tokens, block_size, num_blocks,
                           row_elems / 8, slot_mapping, status);
}

cudaError_t launch_slot_mapping(int64_t* slot_mapping, int total_tokens, const int32_t* block_tables,
                                int max_blocks_per_seq, const int32_t* query_start_loc,
                                const int32_t* seq_lens, int num_seqs, int block_size,
                                int num_blocks, int32_t* status, cudaStream_t stream) {
  return launch_overlapped(slot_mapping_kernel, dim3(num_seqs), dim3(128), 0, stream, slot_mapping,
                           total_tokens, block_tables, max_blocks_per_seq, query_start_loc,
                           seq_lens, block_size, num_blocks, status);
}

}  // namespace pa
