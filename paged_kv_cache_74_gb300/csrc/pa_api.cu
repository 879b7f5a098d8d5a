// pa_api.cu -- the extern "C" entry points declared in include/pa.h:
// host-side validation, TMA tensor-map encoding, the split-KV partition
// choice, workspace carving and kernel dispatch.  No entry point allocates
// device memory or synchronises.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>  // std::call_once

#include "pa_internal.h"

namespace pa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count_current_device() {
  static int counts[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    counts[dev] = n;
  }
  return counts[dev];
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int ceil_div(int64_t a, int64_t b) { return static_cast<int>((a + b - 1) / b); }

// CTAs of the persistent decode grid.  By default as many as fit on the GPU
// at once (never more than one per kMinTilesPerCta tiles of the batch's
// upper bound); with partition_tokens > 0, one CTA per that many tokens of
// the upper bound, resident or not (tests use this to force many splits).
constexpr int64_t kMinTilesPerCta = 4;
constexpr int64_t kMaxDecodeCtas = 1 << 22;

// Which decode kernel runs.  Up to 4 q heads per kv head the CUDA-core
// kernel (3 CTAs per SM, 16-token stages) keeps more bytes in flight than
// the tensor-core one and is faster; from 5 to 16 the q.k and p.v work per
// byte outgrows the CUDA cores and the tensor-core kernel (one CTA per SM)
// takes over.
bool decode_uses_tc(int head_dim, int group) {
  (void)head_dim;
  return group > 4;
}

int64_t decode_num_ctas(int num_seqs, int num_kv_heads, int head_dim, int group, int max_seq_len,
                        int partition_tokens, bool pair = false) {
  const int64_t upper = static_cast<int64_t>(num_kv_heads) * num_seqs *
                        ceil_div(max_seq_len, kBlockSize);  // tiles
  if (partition_tokens > 0) return std::max<int64_t>(1, (upper + partition_tokens / kBlockSize - 1) /
                                                               (partition_tokens / kBlockSize));
  int sms = sm_count_current_device();
  if (sms <= 0) sms = 148;
  // (pair: the streaming decode over units of two kv heads, group = 2 x 4)
  const int64_t resident =
      static_cast<int64_t>(sms) * (pair ? decode_ctas_per_sm(head_dim, group / 2)
                                        : decode_uses_tc(head_dim, group) ? 1
                                                                          : decode_ctas_per_sm(head_dim, group));
  return std::max<int64_t>(1, std::min(resident, (upper + kMinTilesPerCta - 1) / kMinTilesPerCta));
}

// An e4m3 K or V cache as a 3-D tensor [slots][kv_heads][head_dim] (innermost
// first for TMA: {head_dim, kv_heads, slots}); one box is one (block, kv
// head) tile of 16 tokens x head_dim bytes, swizzled (128-byte rows at
// head_dim 128, 64-byte rows at 64) so that the decode's ldmatrix reads of
// 8 token rows are free of bank conflicts; `plain`: rows unswizzled (the
// prefill's converter reads whole rows).
bool make_cache_map_e4m3(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                         int head_dim, bool plain = false, int heads_per_box = 1) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim),
                                 static_cast<cuuint64_t>(num_kv_heads) * head_dim};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(head_dim), static_cast<cuuint32_t>(heads_per_box),
                             static_cast<cuuint32_t>(kBlockSize)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  const int row_bytes = head_dim * heads_per_box;  // contiguous bytes of one token in the box
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             plain ? CU_TENSOR_MAP_SWIZZLE_NONE
                   : (head_dim == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B),
             // A larger L2 promotion than the box's row would fetch the next
             // kv head's row too (a third more DRAM traffic, measured).
             row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                              : (row_bytes == 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                  : CU_TENSOR_MAP_L2_PROMOTION_L2_64B),
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D tiled tensor map with a 128-byte-swizzled box of {64, 1, rows}: the
// operand layout the tcgen05 MMAs read (64 bf16 = one 128-byte row).
bool make_sw128_map(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                    uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box_rows) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {64u, 1u, box_rows};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [rows][heads][head_dim] for the tensor-core decode: box {64, group, 1}
// (one 128-byte row per q head of a kv head).
bool make_q_group_map(CUtensorMap* map, const void* q, int rows, int num_heads, int head_dim,
                      int group) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(num_heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(head_dim) * 2,
                                 static_cast<cuuint64_t>(num_heads) * head_dim * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(group), 1u};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A K or V cache as a 5-D tensor {64, 8, head_dim / 64, slots / 8, kv heads}
// (head_dim low part, token within a group of 8, head_dim half, group of 8
// tokens, kv head) with a box of {64, 8, head_dim / 64, 2, 1}: one copy per
// (block, kv head) lands as [token group][head_dim half][8 tokens][128 B],
// 128-byte swizzled, so the 8-token groups of consecutive blocks sit at one
// uniform stride: the operand layout of both MMAs of the tensor-core decode.
bool make_kv_group_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                       int head_dim) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(num_kv_heads) * head_dim * 2;  // bytes per token
  const cuuint64_t dims[5] = {64u, 8u, static_cast<cuuint64_t>(head_dim / 64),
                              static_cast<cuuint64_t>(num_blocks) * (kBlockSize / 8),
                              static_cast<cuuint64_t>(num_kv_heads)};
  const cuuint64_t strides[4] = {row, 128u, 8 * row, static_cast<cuuint64_t>(head_dim) * 2};
  const cuuint32_t box[5] = {64u, 8u, static_cast<cuuint32_t>(head_dim / 64), kBlockSize / 8, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  // A token's row of one kv head is head_dim * 2 bytes: promote no further
  // than that, or L2 fills fetch the next kv head's row as well.
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             head_dim >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The x-split K cache [blocks, kv heads, head_dim / 8, block, 8] as a 5-D
// tensor {64, block / 8, head_dim / 8, kv heads, blocks} (8 tokens x 8
// elements, token group, 16-byte chunk, kv head, block) with a box of
// {64, 2, head_dim / 8, 1, 1}: one 16-token tile per copy, 128-byte rows,
// 128-byte swizzled.
bool make_xsplit_k_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                       int head_dim, int block_size) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t head = static_cast<cuuint64_t>(head_dim) * block_size * 2;  // bytes
  const cuuint64_t dims[5] = {64u, static_cast<cuuint64_t>(block_size / 8),
                              static_cast<cuuint64_t>(head_dim / 8),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[4] = {128u, static_cast<cuuint64_t>(block_size) * 16, head,
                                 head * num_kv_heads};
  const cuuint32_t box[5] = {64u, 2u, static_cast<cuuint32_t>(head_dim / 8), 1u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The x-split V cache [blocks, kv heads, head_dim, block] as a 4-D tensor
// {block, head_dim, kv heads, blocks} with a box of {16, head_dim, 1, 1}:
// one 16-token tile per copy as [head_dim][16 tokens], 32-byte swizzled.
bool make_xsplit_v_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                       int head_dim, int block_size) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(block_size) * 2;  // bytes per head_dim row
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(block_size),
                              static_cast<cuuint64_t>(head_dim),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {row, row * head_dim, row * head_dim * num_kv_heads};
  const cuuint32_t box[4] = {16u, static_cast<cuuint32_t>(head_dim), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The e4m3 x-split K cache [blocks, kv heads, head_dim / 16, block, 16] as a
// 4-D byte tensor {block * 16, head_dim / 16, kv heads, blocks} with a box of
// {256, head_dim / 16, 1, 1}: one 16-token tile per copy, as head_dim / 16
// runs of 256 contiguous bytes (one 2 KB run at block 16), unswizzled.
bool make_xsplit8_k_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                        int head_dim, int block_size) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t run = static_cast<cuuint64_t>(block_size) * 16;  // bytes of one chunk
  const cuuint64_t head = run * (head_dim / 16);
  const cuuint64_t dims[4] = {run, static_cast<cuuint64_t>(head_dim / 16),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {run, head, head * num_kv_heads};
  const cuuint32_t box[4] = {256u, static_cast<cuuint32_t>(head_dim / 16), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The e4m3 x-split V cache [blocks, kv heads, head_dim, block] as a 4-D byte
// tensor {block, head_dim, kv heads, blocks} with a box of {16, head_dim, 1,
// 1}: one 16-token tile per copy as V^T [head_dim][16 tokens] (one 2 KB run
// at block 16), unswizzled.
bool make_xsplit8_v_map(CUtensorMap* map, const void* cache, int num_blocks, int num_kv_heads,
                        int head_dim, int block_size) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(block_size);  // bytes per head_dim row
  const cuuint64_t dims[4] = {row, static_cast<cuuint64_t>(head_dim),
                              static_cast<cuuint64_t>(num_kv_heads),
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[3] = {row, row * head_dim, row * head_dim * num_kv_heads};
  const cuuint32_t box[4] = {16u, static_cast<cuuint32_t>(head_dim), 1u, 1u};
  const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  std::memset(map, 0, sizeof(*map));
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(cache), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             block_size == 16 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B : CU_TENSOR_MAP_L2_PROMOTION_NONE,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work units per request of the x-split decode: its kernel serves up to 4
// q heads per unit, so a group of g q heads is cut into g / g' units of g'
// heads (g' the largest divisor of g not above 4), each reading its kv
// head's tiles (the units of one kv head are neighbours in the tile order,
// so the repeated reads mostly hit L2).  Units of 8 heads (the 8 columns of
// the kernel's products) measured slower on a batch of many short requests:
// the per-segment hand-off work doubles while the K/V reads mostly hit L2.
int xsplit_heads_per_unit(int group) {
  for (int g = 4; g > 1; --g)
    if (group % g == 0) return g;
  return 1;
}

struct DecodeLayout {
  int64_t num_ctas = 0;
  size_t counters_offset = 0, ml_offset = 0, o_offset = 0, total = 0;
};

// Workspace: status record | per-(request, kv head) counters |
// per-CTA partial (m, l) | per-CTA partial O.
DecodeLayout decode_layout(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                           int max_seq_len, int partition_tokens, bool pair = false) {
  DecodeLayout L;
  const int group = num_heads / num_kv_heads;
  L.num_ctas = decode_num_ctas(num_seqs, num_kv_heads, head_dim, group, max_seq_len,
                               partition_tokens, pair);
  size_t off = kWorkspaceHeader;
  L.counters_offset = off;
  off = align_up(off + static_cast<size_t>(num_seqs) * num_kv_heads * 8, 256);
  L.ml_offset = off;
  off = align_up(off + static_cast<size_t>(L.num_ctas) * 2 * group * 2 * sizeof(float), 256);
  L.o_offset = off;
  off += static_cast<size_t>(L.num_ctas) * 2 * group * head_dim * sizeof(float);
  L.total = align_up(off, 256);
  return L;
}

// The prefill kernel's part of a pa_prefill_varlen workspace, after the
// decode rows' part: one counter per work unit (an upper bound on the units:
// a request of q_len rows has ceil(q_len / 128) query tiles, each with one
// unit per head pair), then the partial records of the persistent grid.
struct PrefillLayout {
  int num_ctas = 0;
  long long max_units = 0;
  size_t counters_offset = 0, ml_offset = 0, o_offset = 0, total = 0;
};

PrefillLayout prefill_layout(size_t base, int num_seqs, int total_q, int num_heads,
                             int num_kv_heads, int head_dim) {
  PrefillLayout P;
  int sms = sm_count_current_device();
  if (sms <= 0) sms = 148;
  P.num_ctas = sms;
  const int group = num_heads / num_kv_heads;
  const long long pairs = static_cast<long long>(num_kv_heads) * ((group + 1) / 2);
  P.max_units = (static_cast<long long>(total_q) / 128 + num_seqs) * pairs;
  size_t off = align_up(base, 256);
  P.counters_offset = off;
  off = align_up(off + static_cast<size_t>(P.max_units) * 8, 256);
  P.ml_offset = off;
  off = align_up(off + static_cast<size_t>(P.num_ctas) * 2 * 2 * 128 * 2 * sizeof(float), 256);
  P.o_offset = off;
  off += prefill_partials_bytes(P.num_ctas, head_dim) -
         static_cast<size_t>(P.num_ctas) * 2 * 2 * 128 * 2 * sizeof(float);
  P.total = align_up(off, 256);
  return P;
}

// A distinct non-zero tag per decode launch (see the pair counters).
unsigned next_epoch() {
  static std::atomic<unsigned> epoch{0};
  unsigned e = ++epoch;
  if (e == 0) e = ++epoch;
  return e;
}

// log2(block_size / 16) for the supported block sizes 16, 32 and 64.
int tile_shift_of(int block_size) { return block_size == 64 ? 2 : block_size == 32 ? 1 : 0; }

// Shared shape checks of the attention entry points.
pa_status check_attention_shape(int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks) {
  if (num_kv_heads < 1 || num_heads < 1 || num_heads % num_kv_heads != 0) return PA_ERR_INVALID;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PA_ERR_UNSUPPORTED;
  if (num_blocks < 1 || static_cast<int64_t>(num_blocks) * block_size > 0x7fffffffLL)
    return PA_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_heads / num_kv_heads > 16) return PA_ERR_UNSUPPORTED;
  if (num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// Validation shared by pa_decode and the decode rows of pa_prefill_varlen.
pa_status check_decode_args(const void* out, const void* q, const void* key_cache,
                            const void* value_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                            int32_t max_seq_len, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int32_t num_blocks, float scale) {
  pa_status st = check_attention_shape(num_heads, num_kv_heads, head_dim, block_size, num_blocks);
  if (st != PA_OK) return st;
  if (num_seqs < 0 || num_seqs > 65535) return num_seqs < 0 ? PA_ERR_INVALID : PA_ERR_UNSUPPORTED;
  if (!out || !q || !key_cache || !value_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(key_cache, 16) || !aligned(value_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PA_ERR_INVALID;
  if (max_blocks_per_seq < 1 || max_seq_len < 1 ||
      static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks_per_seq) * block_size)
    return PA_ERR_INVALID;
  if (!std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID;
  return PA_OK;
}

// Element type and layout of the K/V cache, and its scales.
struct KvFormat {
  bool e4m3 = false;
  bool xsplit = false;  // K [blocks, kv heads, d / 8, block, 8], V [blocks, kv heads, d, block]
  bool pair = false;    // e4m3 streaming decode: work units of two kv heads, one copy for both
  float k_scale = 1.f, v_scale = 1.f;
};

// The e4m3 decode reads two kv heads per copy (4 KB per 16-token tile at
// head_dim 128 instead of 2 KB): a unit is then two kv heads and their 8 q
// heads.  Copies of 2 KB stream at about half the bytes per second of 4 KB
// ones at the same bytes in flight.
bool decode_fp8_pairs(int head_dim, int num_heads, int num_kv_heads) {
  return head_dim == 128 && num_kv_heads % 2 == 0 && num_heads == 4 * num_kv_heads;
}

pa_status launch_decode_rows(void* out, const void* q, const void* key_cache, const void* value_cache,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* query_start_loc,
                             int32_t num_seqs, int32_t total_q, int32_t max_seq_len,
                             int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                             int32_t num_blocks, int32_t block_size, float scale,
                             const DecodeLayout& L, void* workspace, cudaStream_t stream,
                             const KvFormat& kv = KvFormat(), bool after_prefill = false,
                             int tile_sms = 0, int max_query_len = 0) {
  // The TMA views address the cache in 16-token tiles.
  const int num_tiles16 = num_blocks * (block_size / kBlockSize);
  const int group = num_heads / num_kv_heads;
  const bool tc = !kv.xsplit && decode_uses_tc(head_dim, group);
  // x-split: units of up to 4 q heads (see xsplit_heads_per_unit).
  const int unit_heads = kv.xsplit ? xsplit_heads_per_unit(group) : group;
  const int kv_div = group / unit_heads;
  const bool pair = kv.pair && kv.e4m3 && !kv.xsplit && !tc && decode_fp8_pairs(head_dim, num_heads, num_kv_heads);
  if (kv.pair && !pair) return PA_ERR_INVALID;
  CUtensorMap kmap, vmap, qmap;
  if (kv.xsplit && kv.e4m3) {
    if (!make_xsplit8_k_map(&kmap, key_cache, num_blocks, num_kv_heads, head_dim, block_size) ||
        !make_xsplit8_v_map(&vmap, value_cache, num_blocks, num_kv_heads, head_dim, block_size))
      return PA_ERR_CUDA;
  } else if (kv.xsplit) {
    if (!make_xsplit_k_map(&kmap, key_cache, num_blocks, num_kv_heads, head_dim, block_size) ||
        !make_xsplit_v_map(&vmap, value_cache, num_blocks, num_kv_heads, head_dim, block_size))
      return PA_ERR_CUDA;
  } else if (!kv.e4m3) {
    // bf16: the grouped view (both decode kernels read tiles with ldmatrix
    // or as tcgen05 operands).
    if ((tc && !make_q_group_map(&qmap, q, total_q, num_heads, head_dim, group)) ||
        !make_kv_group_map(&kmap, key_cache, num_tiles16, num_kv_heads, head_dim) ||
        !make_kv_group_map(&vmap, value_cache, num_tiles16, num_kv_heads, head_dim))
      return PA_ERR_CUDA;
  } else if ((tc && !make_q_group_map(&qmap, q, total_q, num_heads, head_dim, group)) ||
             !make_cache_map_e4m3(&kmap, key_cache, num_tiles16, num_kv_heads, head_dim, false,
                                  pair ? 2 : 1) ||
             !make_cache_map_e4m3(&vmap, value_cache, num_tiles16, num_kv_heads, head_dim, false,
                                  pair ? 2 : 1)) {
    return PA_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeArgs a;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.query_start_loc = query_start_loc;
  a.counters = reinterpret_cast<unsigned long long*>(ws + L.counters_offset);
  a.part_ml = reinterpret_cast<float*>(ws + L.ml_offset);
  a.part_o = reinterpret_cast<float*>(ws + L.o_offset);
  a.status = reinterpret_cast<int32_t*>(ws);
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_heads = num_heads;
  a.num_kv_heads = pair ? num_kv_heads / 2 : num_kv_heads * kv_div;
  a.group = pair ? 2 * unit_heads : unit_heads;
  a.kv_div = kv_div;
  a.num_ctas = static_cast<int>(L.num_ctas);
  a.max_seq_len = max_seq_len;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.tile_shift = tile_shift_of(block_size);
  a.total_q = total_q;
  a.epoch = next_epoch();
  a.scale_log2 = scale * 1.4426950408889634f * kv.k_scale;
  a.v_scale = kv.v_scale;
  a.defer_griddep = after_prefill ? 1 : 0;
  a.tile_sms = tile_sms;
  a.ctas_per_sm = tile_sms > 0 ? static_cast<int>(L.num_ctas / tile_sms) : 0;
  a.max_query_len = max_query_len;
  const cudaError_t err = tc ? launch_decode_tc(a, qmap, kmap, vmap, head_dim, kv.e4m3, stream)
                            : launch_decode(a, kmap, vmap, head_dim, kv.e4m3, kv.xsplit, stream);
  return err == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: shape not supported by this build";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: the CUDA runtime refused the call";
    default: return "unknown pa_status";
  }
}

int pa_abi_version(void) { return PA_ABI_VERSION; }

pa_status pa_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_stride,
                                   int64_t value_stride, void* key_cache, void* value_cache,
                                   const int64_t* slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                   int32_t num_blocks, float k_scale, float v_scale,
                                   int32_t* device_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1 || block_size < 1) return PA_ERR_INVALID;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID;
  if (head_dim < 16 || head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > (1 << 20)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(slot_mapping, 8) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
    return PA_ERR_INVALID;
  const cudaError_t e = launch_reshape_and_cache_fp8(
      key, value, key_stride, value_stride, key_cache, value_cache, slot_mapping, num_tokens,
      static_cast<int>(row), static_cast<int64_t>(num_blocks) * block_size, k_scale, v_scale,
      device_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_reshape_and_cache(const void* key, const void* value, int64_t key_stride,
                               int64_t value_stride, void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, int32_t* device_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1) return PA_ERR_INVALID;
  if (head_dim < 8 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (block_size < 1) return PA_ERR_INVALID;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > (1 << 20)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(slot_mapping, 8) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
    return PA_ERR_INVALID;
  const cudaError_t e = launch_reshape_and_cache(
      key, value, key_stride, value_stride, key_cache, value_cache, slot_mapping, num_tokens,
      static_cast<int>(row), static_cast<int64_t>(num_blocks) * block_size, device_status,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_compute_slot_mapping(int64_t* slot_mapping, int32_t total_tokens,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* query_start_loc, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t block_size, int32_t num_blocks,
                                  int32_t* device_status, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || block_size < 1 || num_blocks < 1 ||
      max_blocks_per_seq < 1)
    return PA_ERR_INVALID;
  if (num_seqs == 0 || total_tokens == 0) return PA_OK;
  if (!slot_mapping || !block_tables || !query_start_loc || !seq_lens) return PA_ERR_INVALID;
  if (!aligned(slot_mapping, 8) || !aligned(block_tables, 4) || !aligned(query_start_loc, 4) ||
      !aligned(seq_lens, 4) || (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (num_seqs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
  const cudaError_t e = launch_slot_mapping(slot_mapping, total_tokens, block_tables,
                                            max_blocks_per_seq, query_start_loc, seq_lens, num_seqs,
                                            block_size, num_blocks, device_status,
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_append_tokens(const void* key, const void* value, int64_t key_stride,
                           int64_t value_stride, void* key_cache, void* value_cache,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* query_start_loc, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t total_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks,
                           int64_t* slot_mapping, int32_t* device_status, void* stream) {
  if (num_seqs < 0 || total_tokens < 0 || num_kv_heads < 1 || num_blocks < 1 ||
      block_size < 1 || max_blocks_per_seq < 1)
    return PA_ERR_INVALID;
  if (head_dim < 8 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > (1 << 20)) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_tokens == 0) return PA_OK;
  if (num_seqs > 0x7fffffff / 2) return PA_ERR_UNSUPPORTED;
  if (!key || !value || !key_cache || !value_cache || !block_tables || !query_start_loc ||
      !seq_lens)
    return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(block_tables, 4) || !aligned(query_start_loc, 4) ||
      !aligned(seq_lens, 4) || (slot_mapping && !aligned(slot_mapping, 8)) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
    return PA_ERR_INVALID;
  const cudaError_t e = launch_append_tokens(
      key, value, key_stride, value_stride, key_cache, value_cache, block_tables,
      max_blocks_per_seq, query_start_loc, seq_lens, num_seqs, total_tokens, block_size,
      num_blocks, static_cast<int>(row), slot_mapping, device_status,
      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_map_to_kernel_blocks(int32_t* kernel_tables, const int32_t* block_tables,
                                  int32_t num_rows, int32_t max_blocks_per_row,
                                  int32_t blocks_per_kv_block, int32_t* device_status,
                                  void* stream) {
  if (num_rows < 0 || max_blocks_per_row < 0 || blocks_per_kv_block < 1) return PA_ERR_INVALID;
  if (num_rows == 0 || max_blocks_per_row == 0) return PA_OK;
  if (!kernel_tables || !block_tables || !aligned(kernel_tables, 4) || !aligned(block_tables, 4) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  const int64_t n = static_cast<int64_t>(num_rows) * max_blocks_per_row;
  const cudaError_t e = launch_map_kernel_blocks(kernel_tables, block_tables, n, blocks_per_kv_block,
                                                 device_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_seq_len, int32_t partition_tokens) {
  if (num_seqs < 0 || max_seq_len < 1 || num_kv_heads < 1 || num_heads < 1 ||
      num_heads % num_kv_heads != 0 || (head_dim != 64 && head_dim != 128))
    return 0;
  if (partition_tokens < 0 || partition_tokens % kBlockSize != 0) return 0;
  // Enough for either layout: the x-split decode may cut a kv head's q heads
  // into several work units (more pair counters, smaller partials).
  const int units = num_kv_heads * (num_heads / num_kv_heads /
                                    xsplit_heads_per_unit(num_heads / num_kv_heads));
  size_t total = std::max(
      decode_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, partition_tokens)
          .total,
      decode_layout(num_seqs, num_heads, units, head_dim, max_seq_len, partition_tokens).total);
  // ... or the e4m3 decode's units of two kv heads (larger partials).
  if (decode_fp8_pairs(head_dim, num_heads, num_kv_heads))
    total = std::max(total, decode_layout(num_seqs, num_heads, num_kv_heads / 2, head_dim, max_seq_len,
                                          partition_tokens, true)
                                .total);
  return total;
}

pa_status pa_decode(void* out, const void* q, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale,
                    int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                    void* stream) {
  pa_status st = check_decode_args(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads,
                                   head_dim, block_size, num_blocks, scale);
  if (st != PA_OK) return st;
  if (partition_tokens < 0 || partition_tokens % kBlockSize != 0) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  const DecodeLayout L = decode_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len,
                                       partition_tokens);
  if (L.num_ctas > kMaxDecodeCtas) return PA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID;
  return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                            seq_lens, nullptr, num_seqs, num_seqs, max_seq_len, num_heads,
                            num_kv_heads, head_dim, num_blocks, block_size, scale, L, workspace,
                            static_cast<cudaStream_t>(stream));
}

pa_status pa_decode_fp8(void* out, const void* q, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                        int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, float scale, float k_scale,
                        float v_scale, int32_t partition_tokens, void* workspace,
                        size_t workspace_bytes, void* stream) {
  pa_status st = check_decode_args(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads,
                                   head_dim, block_size, num_blocks, scale);
  if (st != PA_OK) return st;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID;
  if (partition_tokens < 0 || partition_tokens % kBlockSize != 0) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  const bool pair = decode_fp8_pairs(head_dim, num_heads, num_kv_heads);
  const DecodeLayout L = decode_layout(num_seqs, num_heads, pair ? num_kv_heads / 2 : num_kv_heads,
                                       head_dim, max_seq_len, partition_tokens, pair);
  if (L.num_ctas > kMaxDecodeCtas) return PA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID;
  KvFormat kv;
  kv.e4m3 = true;
  kv.pair = pair;
  kv.k_scale = k_scale;
  kv.v_scale = v_scale;
  return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                            seq_lens, nullptr, num_seqs, num_seqs, max_seq_len, num_heads,
                            num_kv_heads, head_dim, num_blocks, block_size, scale, L, workspace,
                            static_cast<cudaStream_t>(stream), kv);
}

pa_status pa_reshape_and_cache_xsplit(const void* key, const void* value, int64_t key_stride,
                                      int64_t value_stride, void* key_cache, void* value_cache,
                                      const int64_t* slot_mapping, int32_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int32_t num_blocks, int32_t* device_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1 || block_size < 1) return PA_ERR_INVALID;
  if (head_dim < 8 || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > (1 << 20)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(slot_mapping, 8) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
    return PA_ERR_INVALID;
  const cudaError_t e = launch_reshape_and_cache_xsplit(
      key, value, key_stride, value_stride, key_cache, value_cache, slot_mapping, num_tokens,
      num_kv_heads, head_dim, block_size, static_cast<int64_t>(num_blocks) * block_size,
      device_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_xsplit(void* out, const void* q, const void* key_cache, const void* value_cache,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                           int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t block_size, int32_t num_blocks, float scale,
                           int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                           void* stream) {
  pa_status st = check_decode_args(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads,
                                   head_dim, block_size, num_blocks, scale);
  if (st != PA_OK) return st;
  if (partition_tokens < 0 || partition_tokens % kBlockSize != 0) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  const int group = num_heads / num_kv_heads;
  const int units = num_kv_heads * (group / xsplit_heads_per_unit(group));
  if (units > 65535) return PA_ERR_UNSUPPORTED;
  const DecodeLayout L =
      decode_layout(num_seqs, num_heads, units, head_dim, max_seq_len, partition_tokens);
  if (L.num_ctas > kMaxDecodeCtas) return PA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID;
  KvFormat kv;
  kv.xsplit = true;
  return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                            seq_lens, nullptr, num_seqs, num_seqs, max_seq_len, num_heads,
                            num_kv_heads, head_dim, num_blocks, block_size, scale, L, workspace,
                            static_cast<cudaStream_t>(stream), kv);
}

pa_status pa_reshape_and_cache_xsplit_fp8(const void* key, const void* value,
                                          int64_t key_stride, int64_t value_stride,
                                          void* key_cache, void* value_cache,
                                          const int64_t* slot_mapping, int32_t num_tokens,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          int32_t block_size, int32_t num_blocks, float k_scale,
                                          float v_scale, int32_t* device_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads < 1 || num_blocks < 1 || block_size < 1) return PA_ERR_INVALID;
  if (head_dim < 16 || head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (row > (1 << 20)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(key_cache, 16) ||
      !aligned(value_cache, 16) || !aligned(slot_mapping, 8) ||
      (device_status && !aligned(device_status, 4)))
    return PA_ERR_INVALID;
  if (key_stride < row || value_stride < row || key_stride % 8 != 0 || value_stride % 8 != 0)
    return PA_ERR_INVALID;
  const cudaError_t e = launch_reshape_and_cache_xsplit_fp8(
      key, value, key_stride, value_stride, key_cache, value_cache, slot_mapping, num_tokens,
      num_kv_heads, head_dim, block_size, static_cast<int64_t>(num_blocks) * block_size, k_scale,
      v_scale, device_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_xsplit_fp8(void* out, const void* q, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, float k_scale, float v_scale,
                               int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                               void* stream) {
  pa_status st = check_decode_args(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads,
                                   head_dim, block_size, num_blocks, scale);
  if (st != PA_OK) return st;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID;
  if (num_heads / num_kv_heads > 4) return PA_ERR_UNSUPPORTED;
  if (partition_tokens < 0 || partition_tokens % kBlockSize != 0) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  const DecodeLayout L = decode_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len,
                                       partition_tokens);
  if (L.num_ctas > kMaxDecodeCtas) return PA_ERR_UNSUPPORTED;
  if (!workspace || workspace_bytes < L.total) return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID;
  KvFormat kv;
  kv.e4m3 = true;
  kv.xsplit = true;
  kv.k_scale = k_scale;
  kv.v_scale = v_scale;
  return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                            seq_lens, nullptr, num_seqs, num_seqs, max_seq_len, num_heads,
                            num_kv_heads, head_dim, num_blocks, block_size, scale, L, workspace,
                            static_cast<cudaStream_t>(stream), kv);
}

size_t pa_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len) {
  if (total_q < 0) return 0;
  const size_t dec =
      pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, 0);
  if (dec == 0) return 0;
  return prefill_layout(dec, num_seqs, total_q, num_heads, num_kv_heads, head_dim).total;
}

}  // extern "C"

namespace {

pa_status prefill_varlen_impl(void* out, const void* q, const void* key_cache,
                              const void* value_cache, const int32_t* query_start_loc,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t total_q,
                              int32_t max_query_len, int32_t max_seq_len,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks, float scale,
                              void* workspace, size_t workspace_bytes, void* stream,
                              const KvFormat& kv) {
  pa_status st = check_decode_args(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                                   seq_lens, num_seqs, max_seq_len, num_heads, num_kv_heads,
                                   head_dim, block_size, num_blocks, scale);
  if (st != PA_OK) return st;
  if (!query_start_loc || !aligned(query_start_loc, 4) || total_q < 0 || max_query_len < 0 ||
      max_query_len > max_seq_len)
    return PA_ERR_INVALID;
  if (num_seqs == 0 || total_q == 0) return PA_OK;
  const DecodeLayout L = decode_layout(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len, 0);
  if (L.num_ctas > kMaxDecodeCtas) return PA_ERR_UNSUPPORTED;
  const PrefillLayout PL =
      prefill_layout(L.total, num_seqs, total_q, num_heads, num_kv_heads, head_dim);
  if (!workspace || workspace_bytes < (max_query_len > 1 ? PL.total : L.total))
    return PA_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PA_ERR_INVALID;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (max_query_len > 1) {
    // Rows with q_len > 1: tensor-core tiles.
    CUtensorMap qmap, kmap, vmap;
    const int tiles = num_blocks * (block_size / kBlockSize);
    const bool maps_ok =
        make_sw128_map(&qmap, q, head_dim, num_heads, total_q, head_dim * 2,
                       static_cast<uint64_t>(num_heads) * head_dim * 2, 128) &&
        (kv.e4m3 ? make_cache_map_e4m3(&kmap, key_cache, tiles, num_kv_heads, head_dim, true) &&
                       make_cache_map_e4m3(&vmap, value_cache, tiles, num_kv_heads, head_dim, true)
                 : make_kv_group_map(&kmap, key_cache, tiles, num_kv_heads, head_dim) &&
                       make_kv_group_map(&vmap, value_cache, tiles, num_kv_heads, head_dim));
    if (!maps_ok) return PA_ERR_CUDA;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    PrefillArgs p;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.query_start_loc = query_start_loc;
    p.status = static_cast<int32_t*>(workspace);
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.group = num_heads / num_kv_heads;
    p.max_seq_len = max_seq_len;
    p.max_query_len = max_query_len;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.tile_shift = tile_shift_of(block_size);
    p.total_q = total_q;
    p.num_ctas = PL.num_ctas;  // one CTA per SM
    p.max_units = PL.max_units;
    p.counters = reinterpret_cast<unsigned long long*>(ws + PL.counters_offset);
    p.part_ml = reinterpret_cast<float*>(ws + PL.ml_offset);
    p.part_o = reinterpret_cast<float*>(ws + PL.o_offset);
    p.epoch = next_epoch();
    p.scale_log2 = scale * kv.k_scale * 1.4426950408889634f;
    p.o_scale = kv.v_scale;
    // Decode rows in the streaming decode kernel (head_dim 128), its grid
    // exactly ctas-per-SM CTAs on every SM: the two kernels split the SMs between
    // them (tile_kernel_sms()), so that the decode rows start at once on the
    // SMs the tiles leave instead of after the tile CTAs.
    const int group = num_heads / num_kv_heads;
    const bool split_sms =
        head_dim == 128 && !decode_uses_tc(head_dim, group) &&
        L.num_ctas == static_cast<int64_t>(PL.num_ctas) * decode_ctas_per_sm(head_dim, group);
    p.partition = split_sms ? 1 : 0;
    // Both kernels go on the caller's stream.  The tile kernel lets the
    // decode launch start once the kernels before this call are complete;
    // the decode CTAs then take the SMs the tiles leave free, and the decode
    // launch completes only after the tile kernel.
    if (launch_prefill(p, qmap, kmap, vmap, head_dim, kv.e4m3, cs) != cudaSuccess)
      return PA_ERR_CUDA;
    return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                              seq_lens, query_start_loc, num_seqs, total_q, max_seq_len,
                              num_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, L,
                              workspace, cs, kv, true, split_sms ? PL.num_ctas : 0, max_query_len);
  }
  // Only decode rows: the decode kernel.
  return launch_decode_rows(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq,
                            seq_lens, query_start_loc, num_seqs, total_q, max_seq_len, num_heads,
                            num_kv_heads, head_dim, num_blocks, block_size, scale, L, workspace, cs,
                            kv);
}

}  // namespace

extern "C" {

pa_status pa_prefill_varlen(void* out, const void* q, const void* key_cache,
                            const void* value_cache, const int32_t* query_start_loc,
                            const int32_t* seq_lens, int32_t num_seqs, int32_t total_q,
                            int32_t max_query_len, int32_t max_seq_len,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale,
                            void* workspace, size_t workspace_bytes, void* stream) {
  return prefill_varlen_impl(out, q, key_cache, value_cache, query_start_loc, seq_lens, num_seqs,
                             total_q, max_query_len, max_seq_len, block_tables, max_blocks_per_seq,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             workspace, workspace_bytes, stream, KvFormat());
}

pa_status pa_prefill_varlen_fp8(void* out, const void* q, const void* key_cache,
                                const void* value_cache, const int32_t* query_start_loc,
                                const int32_t* seq_lens, int32_t num_seqs, int32_t total_q,
                                int32_t max_query_len, int32_t max_seq_len,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t num_blocks, float scale,
                                float k_scale, float v_scale, void* workspace,
                                size_t workspace_bytes, void* stream) {
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return PA_ERR_INVALID;
  KvFormat kv;
  kv.e4m3 = true;
  kv.k_scale = k_scale;
  kv.v_scale = v_scale;
  return prefill_varlen_impl(out, q, key_cache, value_cache, query_start_loc, seq_lens, num_seqs,
                             total_q, max_query_len, max_seq_len, block_tables, max_blocks_per_seq,
                             num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                             workspace, workspace_bytes, stream, kv);
}


}  // extern "C"
