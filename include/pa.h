/*
 * pa.h -- C ABI of the paged KV-cache attention library (libpa.so) for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The library implements the hot path that the vLLM PagedAttention pages
 * describe:
 *   - pa_reshape_and_cache   write new K/V tokens into their cache slots
 *                            ("vllm 深度解析：一切从 PagedAttention 谈起",
 *                            write_to_paged_cache -> reshape_and_cache);
 *   - pa_compute_slot_mapping  slot = block_table[r][pos / B] * B + pos % B
 *                            ("vLLM 深度解析（二）：PagedAttention 核心机制",
 *                            section 3.1, BlockTable.compute_slot_mapping);
 *   - pa_decode              paged decode attention with online softmax and
 *                            a split-KV partition + merge pass (same page,
 *                            sections 2.2, 3.2 and 3.3);
 *   - pa_prefill_varlen      mixed chunked-prefill + decode batch driven by
 *                            query_start_loc / seq_lens ("分块预填充与混合批处理",
 *                            section 11.6; first page, section 5.2).
 *
 * Conventions shared by every call
 * --------------------------------
 * Pointers.  Every tensor pointer is a DEVICE pointer owned by the caller.
 *   No call allocates device memory; scratch space is a caller-provided
 *   `workspace` sized by the matching *_workspace_size() call (the one
 *   exception, pa_decode_noalloc, uses a fixed array inside the library).
 *   Tensor pointers must be 16-byte aligned.
 * Element types.  q, key, value, out and the caches are bf16 (IEEE
 *   binary16-brain, stored as 16-bit patterns); block tables, seq_lens and
 *   query_start_loc are int32; slot mappings are int64.
 * Cache layout (NHD).  key_cache and value_cache are each a contiguous
 *   [num_blocks, block_size, num_kv_heads, head_dim] array, i.e. a
 *   [num_blocks * block_size, num_kv_heads, head_dim] array indexed by slot
 *   (the combined [2, num_blocks, block_size, num_kv_heads, head_size]
 *   cache of the page "vllm 深度解析：一切从 PagedAttention 谈起", split
 *   into its K and V halves).  Block 0 is conventionally the null block.
 * GQA.  num_heads must be a multiple of num_kv_heads; q head h reads kv head
 *   h / (num_heads / num_kv_heads).
 * Supported sizes.  head_dim 64 or 128; block_size 16, 32 or 64 for the
 *   attention calls (any positive block_size for the slot helpers); num_heads
 *   / num_kv_heads between 1 and 16; num_seqs up to 65535.
 * Streams.  `stream` is a cudaStream_t passed as void* (NULL = legacy
 *   default stream).  Calls only enqueue work; they never synchronise.
 *   A write through pa_reshape_and_cache must be enqueued before the
 *   attention call that reads it, on the same stream (or ordered by events).
 * Errors.  Arguments are validated on the host before anything is
 *   launched; an invalid call returns a non-zero pa_status and enqueues
 *   nothing.  PA_ERR_CUDA means a launch was refused by the CUDA runtime.
 *   Device data (block ids, slots, lengths) is range-checked inside the
 *   kernels: an out-of-range value is never dereferenced, the affected
 *   output is left unspecified, and an error code is recorded in the
 *   device status word (see pa_device_status below) when one is supplied.
 * Device status word.  The first 16 bytes of every workspace hold an
 *   int32[4] status record: [0] error code (0 = none, else a pa_device_error),
 *   [1] request index, [2] detail (the offending value), [3] reserved.  The
 *   kernels write it only on error (first error wins); the caller zeroes
 *   it (e.g. cudaMemsetAsync) whenever it wants a fresh record.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,      /* null or misaligned pointer, bad size or stride */
    PA_ERR_UNSUPPORTED = 2,  /* valid but not built: head_dim, block_size, group size */
    PA_ERR_WORKSPACE = 3,    /* workspace missing or smaller than *_workspace_size() */
    PA_ERR_CUDA = 4          /* the CUDA runtime refused a launch or query */
} pa_status;

typedef enum pa_device_error {
    PA_DEV_OK = 0,
    PA_DEV_BAD_SLOT = 1,        /* slot >= num_blocks * block_size (write skipped) */
    PA_DEV_BAD_BLOCK_ID = 2,    /* block id outside [0, num_blocks) (tile read as zeros) */
    PA_DEV_BAD_SEQ_LEN = 3,     /* seq_len < 1, > max_seq_len or > max_blocks_per_seq * block_size */
    PA_DEV_BAD_QUERY_LEN = 4,   /* q_len > seq_len, > max_query_len, or rows beyond total_q */
    PA_DEV_WAIT_TIMEOUT = 5     /* a pipeline wait gave up (internal error); the CTA stopped */
} pa_device_error;

/* Human-readable name of a pa_status value (static string, never NULL). */
const char* pa_status_string(int status);

/* ABI version of this header; bumped on any incompatible change. */
#define PA_ABI_VERSION 2
int pa_abi_version(void);

/*
 * pa_reshape_and_cache -- scatter new K/V tokens into the paged cache.
 * ("vllm 深度解析：一切从 PagedAttention 谈起": write_to_paged_cache calls
 * reshape_and_cache, which turns [num_tokens, heads, dim] into
 * [blocks, block_size, heads, dim]; "vLLM 深度解析（二）", section 3.1:
 * slot_mapping decides where each new token's K/V is written.)
 *
 *   key, value    [num_tokens, num_kv_heads, head_dim] bf16; token i starts
 *                 key_stride (value_stride) ELEMENTS after token i-1; the
 *                 heads of one token are contiguous.  Strides must be
 *                 multiples of 8 elements (16 bytes).
 *   key_cache, value_cache   the cache (layout above); written in place.
 *   slot_mapping  [num_tokens] int64: token i goes to slot s =
 *                 slot_mapping[i], i.e. block s / block_size, offset
 *                 s % block_size.  s < 0 skips the token (padding).
 *                 s >= num_blocks * block_size is a device error: skipped
 *                 and recorded in *device_status.
 *   device_status optional int32[4] device status record (NULL = none).
 * Bit-exact copy; num_tokens == 0 is a no-op.  Two tokens with the same
 * slot race (the last writer is unspecified).
 */
pa_status pa_reshape_and_cache(const void* key, const void* value,
                               int64_t key_stride, int64_t value_stride,
                               void* key_cache, void* value_cache,
                               const int64_t* slot_mapping, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int32_t num_blocks,
                               int32_t* device_status, void* stream);

/*
 * pa_reshape_and_cache_fp8 -- pa_reshape_and_cache into an FP8 (e4m3) cache.
 * ("vLLM 深度解析（二）", section 3.2: an FP8 KV cache is stored quantized
 * and converted back with the cache's scale, fp8::scaled_convert; "LLM 推理
 * 基础与 vLLM 内部机制", section 2: FP8 halves the bytes per token.)
 *
 *   key_cache, value_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *                 e4m3 bytes (OCP FP8 E4M3: 1 sign, 4 exponent bits with
 *                 bias 7, 3 mantissa bits, no infinity, 0x7F = NaN)
 *   k_scale, v_scale  per-tensor scales, finite and > 0
 * Each value x becomes e4m3(x / scale): the quotient in binary32, rounded to
 * the nearest e4m3 value (ties to the even mantissa), magnitudes beyond 448
 * saturated to 448, NaN kept.  Other arguments, slots and errors as
 * pa_reshape_and_cache; head_dim a multiple of 16.
 */
pa_status pa_reshape_and_cache_fp8(const void* key, const void* value,
                                   int64_t key_stride, int64_t value_stride,
                                   void* key_cache, void* value_cache,
                                   const int64_t* slot_mapping, int32_t num_tokens,
                                   int32_t num_kv_heads, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks,
                                   float k_scale, float v_scale,
                                   int32_t* device_status, void* stream);

/*
 * pa_compute_slot_mapping -- slots of this step's new tokens.
 * ("vLLM 深度解析（二）", section 3.1: logical_block = pos / B, offset =
 * pos % B, slot = block_table[request][logical_block] * B + offset.)
 * Request r owns flattened tokens query_start_loc[r] .. query_start_loc[r+1]-1;
 * its i-th new token sits at position seq_lens[r] - q_len + i (seq_lens
 * counts this step's tokens).  slot_mapping has total_tokens entries; a
 * token whose position or block id is out of range gets slot -1 and a
 * device error is recorded in *device_status (optional, may be NULL).
 */
pa_status pa_compute_slot_mapping(int64_t* slot_mapping, int32_t total_tokens,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* query_start_loc, const int32_t* seq_lens,
                                  int32_t num_seqs, int32_t block_size, int32_t num_blocks,
                                  int32_t* device_status, void* stream);

/*
 * pa_append_tokens -- pa_compute_slot_mapping and pa_reshape_and_cache of
 * this step's new tokens in one launch (the pages run them as two steps:
 * slot_mapping, then write_to_paged_cache; fused, the cache write does not
 * wait for a separate kernel's slots).
 *
 *   key, value     [total_tokens, num_kv_heads, head_dim] bf16, token rows
 *                  key_stride / value_stride elements apart (multiples of 8)
 *   key_cache, value_cache  [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables, query_start_loc, seq_lens  as pa_compute_slot_mapping
 *   slot_mapping   optional [total_tokens] int64 output (NULL: not stored)
 * Token i of request r goes to the slot pa_compute_slot_mapping gives it
 * and its K and V rows are copied there bit for bit.  Tokens whose position
 * or block id is out of range are skipped (slot -1) and a device error is
 * recorded in *device_status (optional).  num_seqs == 0 or total_tokens == 0
 * is a no-op.
 */
pa_status pa_append_tokens(const void* key, const void* value, int64_t key_stride,
                           int64_t value_stride, void* key_cache, void* value_cache,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* query_start_loc, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t total_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int32_t num_blocks,
                           int64_t* slot_mapping, int32_t* device_status, void* stream);

/*
 * pa_map_to_kernel_blocks -- block tables of KV-manager blocks expanded into
 * block tables of kernel blocks ("vllm 深度解析：一切从 PagedAttention 谈起",
 * BlockTable.map_to_kernel_blocks: when the manager's block holds
 * blocks_per_kv_block kernel blocks, manager block b becomes kernel blocks
 * b * k, b * k + 1, ..., b * k + k - 1 with k = blocks_per_kv_block).
 *
 *   kernel_tables  [num_rows, max_blocks_per_row * k] int32 (written)
 *   block_tables   [num_rows, max_blocks_per_row] int32; an entry < 0
 *                  (padding) becomes k entries of -1
 *   device_status  optional int32[4] status record (NULL = none): an id
 *                  whose kernel ids exceed INT32_MAX is recorded as
 *                  PA_DEV_BAD_BLOCK_ID and written as -1
 * A cache of num_blocks blocks of block_size tokens is the same memory as
 * num_blocks * k blocks of block_size / k tokens, so the attention calls
 * give bit-identical results for (cache viewed with block_size, tables)
 * and (cache viewed with block_size / k, expanded tables).
 * Errors: PA_ERR_INVALID for null or misaligned pointers, negative sizes or
 * k < 1; num_rows == 0 or max_blocks_per_row == 0 is a no-op.
 */
pa_status pa_map_to_kernel_blocks(int32_t* kernel_tables, const int32_t* block_tables,
                                  int32_t num_rows, int32_t max_blocks_per_row,
                                  int32_t blocks_per_kv_block, int32_t* device_status,
                                  void* stream);

/*
 * pa_decode_workspace_size -- bytes of workspace pa_decode needs for these
 * sizes: the status record, one 8-byte counter per (request, work unit) and
 * two partial records (m, l, O) per CTA of the decode grid; the size covers
 * every unit layout the decode entry points use for these sizes (one kv
 * head, a share of one for the x-split layout, two for the e4m3 decode).  The same
 * partition_tokens must be passed to pa_decode, on the same device (the
 * default grid size depends on its SM count).  No part of the workspace
 * needs initialising (the counters carry a per-call tag), and a call leaves
 * its counters at zero, so a call captured in a CUDA graph replays correctly
 * with new inputs.  Returns 0 for arguments pa_decode would reject.
 */
size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                int32_t head_dim, int32_t max_seq_len,
                                int32_t partition_tokens);

/*
 * pa_decode -- paged decode attention, one query row per request.
 * ("vLLM 深度解析（二）", section 2.2 online softmax state (m, l, A);
 * section 3.2 block-table gather, masking of tokens >= seq_len and zeroed
 * out-of-context V; sections 3.2.7, 3.2.9 and 3.3 split-KV partitions and
 * their merge m = max m_j, L = sum l_j e^{m_j - m}, O = sum O_j l_j e^{m_j - m} / L.)
 *
 *   out           [num_seqs, num_heads, head_dim] bf16 (written)
 *   q             [num_seqs, num_heads, head_dim] bf16
 *   block_tables  [num_seqs, max_blocks_per_seq] int32; entries past
 *                 ceil(seq_len / block_size) are never read
 *   seq_lens      [num_seqs] int32, each in [1, max_seq_len]
 *   max_seq_len   host-side upper bound of seq_lens (sizes the grid; no
 *                 device-to-host read happens)
 *   scale         softmax scale applied to q.k (usually 1/sqrt(head_dim));
 *                 finite and > 0 (else PA_ERR_INVALID)
 *   partition_tokens  split-KV granularity.  0 (the default) splits the
 *                 batch's K/V evenly over as many CTAs as the GPU holds at
 *                 once; a positive multiple of block_size instead uses one
 *                 CTA per that many tokens of num_seqs * max_seq_len (more,
 *                 smaller pieces; used to test the merge)
 *   workspace     >= pa_decode_workspace_size(...) bytes, 256-byte aligned;
 *                 calls that overlap on the GPU need separate workspaces
 * out[r, h] = sum_t softmax_t(scale * q[r,h] . k_t) v_t over the
 * seq_lens[r] keys of request r (exact attention, fp32 accumulation,
 * rounded once to bf16).  The products run on the tensor cores (warp-level
 * products up to 4 q heads per kv head, tcgen05 from 5 to 16), and the
 * softmax weights are rounded to bf16 before they multiply V.
 */
pa_status pa_decode(void* out, const void* q, const void* key_cache, const void* value_cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int32_t block_size, int32_t num_blocks, float scale,
                    int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                    void* stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart of this call: it exists for
 * callers such as plugins or backends that a host framework hands only
 * their input and output tensors, programs whose device-memory budget is
 * fixed in advance, and hot paths that must not call cudaMalloc (it can
 * stall the device and is not allowed while a stream is being recorded).
 *
 * Same arguments and result as pa_decode, minus the workspace, plus
 *   device_status  optional int32[4] device pointer (NULL = none).  After
 *                  the call (in stream order) it holds this call's device
 *                  status record: all zero, or the first error a kernel
 *                  recorded (bad block id, bad seq_len, wait timeout; the
 *                  layout of the record at the start of a workspace).
 * Scratch comes from one static device array of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES that the library holds on every GPU that
 * loads it until the process exits.  The call allocates nothing and calls
 * no allocating routine.
 *   - Sizes whose pa_decode_workspace_size(...) exceeds the array return
 *     PA_ERR_WORKSPACE without launching anything (a larger
 *     partition_tokens needs less scratch).
 *   - The first call on a device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.
 *   - Every call on a device shares the array and leaves its contents
 *     behind; each call clears the part that must start at zero.  Calls
 *     whose work overlaps on the GPU (other streams, other host threads)
 *     race on the array and must be serialised by the caller.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)
pa_status pa_decode_noalloc(void* out, const void* q, const void* key_cache,
                            const void* value_cache, const int32_t* block_tables,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int32_t num_blocks, float scale, int32_t partition_tokens,
                            int32_t* device_status, void* stream);

/*
 * pa_decode_fp8 -- pa_decode over an FP8 (e4m3) cache written by
 * pa_reshape_and_cache_fp8: key t contributes decoded(K_t) * k_scale and
 * value t decoded(V_t) * v_scale ("vLLM 深度解析（二）", section 3.2,
 * fp8::scaled_convert inside the K/V load).  Same arguments, workspace
 * (pa_decode_workspace_size), sizes (1 to 16 q heads per kv head) and
 * results as pa_decode otherwise.  The products run on the tensor cores in
 * f16: e4m3 K and V convert to f16 exactly; q and the softmax weights are
 * rounded to f16 (q saturates at +-65504).  Up to 4 q heads per kv head the
 * warp-level products read the e4m3 bytes directly (at head_dim 128 with
 * exactly 4 q heads per kv head and an even num_kv_heads, one work unit
 * takes two kv heads, whose 16-token tiles arrive in one copy); from 5 to
 * 16 the tcgen05 decode converts each landed 128-token chunk (K into
 * tensor memory, V into shared memory) before its MMAs.
 * k_scale and v_scale finite and > 0 (else PA_ERR_INVALID).
 */
pa_status pa_decode_fp8(void* out, const void* q, const void* key_cache, const void* value_cache,
                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                        int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, float scale, float k_scale,
                        float v_scale, int32_t partition_tokens, void* workspace,
                        size_t workspace_bytes, void* stream);

/*
 * The x-split cache layout ("vLLM 深度解析（二）", section 3.2.1: the
 * layout of the pages' own CUDA-core decode kernel), for drop-in use of
 * caches laid out that way:
 *   key_cache    [num_blocks, num_kv_heads, head_dim / 8, block_size, 8] bf16
 *                (x = 16 bytes / 2 = 8 consecutive head_dim elements
 *                innermost)
 *   value_cache  [num_blocks, num_kv_heads, head_dim, block_size] bf16
 * Element d of kv head h of the token in slot s = b * block_size + o sits
 * at key_cache[b][h][d / 8][o][d % 8] and value_cache[b][h][d][o].
 * Only the two calls below (and their FP8 forms after them) read or write
 * this layout; pa_prefill_varlen and the other FP8 calls take the
 * token-major layout.
 *
 * pa_reshape_and_cache_xsplit -- pa_reshape_and_cache into x-split caches.
 * Same arguments, slots, errors and bit-exactness; head_dim a multiple of 8.
 */
pa_status pa_reshape_and_cache_xsplit(const void* key, const void* value,
                                      int64_t key_stride, int64_t value_stride,
                                      void* key_cache, void* value_cache,
                                      const int64_t* slot_mapping, int32_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks,
                                      int32_t* device_status, void* stream);

/*
 * pa_decode_xsplit -- pa_decode over x-split caches.  Same arguments,
 * workspace (pa_decode_workspace_size covers both layouts), sizes (head_dim
 * 64 or 128, block_size 16, 32 or 64, 1 to 16 q heads per kv head) and
 * errors as pa_decode.  Always the warp-level tensor-core decode (weights
 * rounded to bf16): groups of more than 4 q heads are cut into work units of
 * at most 4 (the largest divisor of the group not above 4), each reading its
 * kv head's K/V.
 */
pa_status pa_decode_xsplit(void* out, const void* q, const void* key_cache,
                           const void* value_cache, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* seq_lens,
                           int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int32_t num_blocks, float scale, int32_t partition_tokens,
                           void* workspace, size_t workspace_bytes, void* stream);

/*
 * The x-split layout with an FP8 (e4m3) cache ("vLLM 深度解析（二）",
 * section 3.2.1: x = 16 bytes / element size, 16 for one-byte elements):
 *   key_cache    [num_blocks, num_kv_heads, head_dim / 16, block_size, 16]
 *   value_cache  [num_blocks, num_kv_heads, head_dim, block_size]
 * both e4m3 bytes.  Element d of kv head h of the token in slot
 * s = b * block_size + o sits at key_cache[b][h][d / 16][o][d % 16] and
 * value_cache[b][h][d][o].  At block_size 16 the K (or V) bytes of one
 * (block, kv head) are one contiguous 2 KB run at head_dim 128.
 *
 * pa_reshape_and_cache_xsplit_fp8 -- pa_reshape_and_cache_fp8 into x-split
 * e4m3 caches: the same values e4m3(x / scale) (binary32 quotient, nearest
 * even, saturated to +-448, NaN kept), slots, skips and errors, at the
 * x-split places; head_dim a multiple of 16.
 */
pa_status pa_reshape_and_cache_xsplit_fp8(const void* key, const void* value,
                                          int64_t key_stride, int64_t value_stride,
                                          void* key_cache, void* value_cache,
                                          const int64_t* slot_mapping, int32_t num_tokens,
                                          int32_t num_kv_heads, int32_t head_dim,
                                          int32_t block_size, int32_t num_blocks, float k_scale,
                                          float v_scale, int32_t* device_status, void* stream);

/*
 * pa_decode_xsplit_fp8 -- pa_decode_fp8 over x-split e4m3 caches: key t
 * contributes decoded(K_t) * k_scale and value t decoded(V_t) * v_scale.
 * Same arguments, workspace, limits (1 to 4 q heads per kv head) and
 * results as pa_decode_fp8; the products run on the tensor cores in f16.
 */
pa_status pa_decode_xsplit_fp8(void* out, const void* q, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int32_t num_blocks, float scale, float k_scale, float v_scale,
                               int32_t partition_tokens, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * pa_prefill_workspace_size -- bytes of workspace pa_prefill_varlen needs
 * (status record, decode-row partials).  Returns 0 for invalid arguments.
 */
size_t pa_prefill_workspace_size(int32_t num_seqs, int32_t total_q, int32_t num_heads,
                                 int32_t num_kv_heads, int32_t head_dim, int32_t max_seq_len);

/*
 * pa_prefill_varlen -- attention for a mixed batch of chunked-prefill and
 * decode requests packed by query_start_loc.
 * ("分块预填充与混合批处理", section 11.6: cu_seqlens_q = query_start_loc,
 * seqused_k = seq_lens, which includes this step's tokens, and the block
 * table gives the physical blocks; "vLLM 深度解析（二）", section 5.2:
 * rows with q_len > 1 are prefill, q_len == 1 decode.)
 *
 *   out, q          [total_q, num_heads, head_dim] bf16
 *   query_start_loc [num_seqs + 1] int32, non-decreasing, [0] = 0,
 *                   [num_seqs] = total_q
 *   seq_lens        [num_seqs] int32 K/V lengths (>= q_len of the request)
 *   max_query_len, max_seq_len  host-side upper bounds
 * Query i (0 <= i < q_len) of request r sits at position
 * seq_lens[r] - q_len + i and attends keys 0 .. that position (causal,
 * aligned to the end of the context).  Rows with q_len > 1 run on the
 * tcgen05 tensor-core prefill tile; rows with q_len == 1 run the decode
 * kernel; requests with q_len == 0 produce no rows.  K/V of this step's
 * tokens must already be in the cache (pa_reshape_and_cache first).
 * Both kernels are enqueued on `stream` and nowhere else (the library
 * creates no stream or event).  When max_query_len > 1 the tile kernel goes
 * first; the decode kernel is a programmatic dependent launch that may start
 * once every kernel enqueued before this call has completed, so its CTAs
 * fill the SMs the tiles leave free, and it completes only after the tile
 * kernel: work enqueued on `stream` after this call sees both results, as
 * for a single kernel.  When the tile work is small (up to about 150 us of
 * one SM's time per SM) and the decode rows run in the streaming decode
 * kernel (up to 4 q heads per kv head) on every SM, the two kernels split
 * the SMs from the batch's own sums: only as many tile CTAs as the tile
 * work's share of the estimated SM time work, the others exit at once, and
 * the decode rows go to the decode CTAs that start on the freed SMs.  The
 * split depends only on the batch, so results stay the same from call to
 * call.
 */
pa_status pa_prefill_varlen(void* out, const void* q, const void* key_cache,
                            const void* value_cache, const int32_t* query_start_loc,
                            const int32_t* seq_lens, int32_t num_seqs, int32_t total_q,
                            int32_t max_query_len, int32_t max_seq_len,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, float scale,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill_varlen_fp8 -- pa_prefill_varlen over FP8 (e4m3) caches written
 * by pa_reshape_and_cache_fp8: key t contributes decoded(K_t) * k_scale and
 * value t decoded(V_t) * v_scale ("vLLM 深度解析（二）", section 3.2,
 * fp8::scaled_convert inside the K/V load; "分块预填充与混合批处理",
 * section 11.6, for the varlen batch).  Same arguments, layouts (one byte
 * per cache element), workspace (pa_prefill_workspace_size), ordering on
 * `stream` and results as pa_prefill_varlen otherwise.  The prefill rows'
 * products run on the tensor cores in f16: each landed e4m3 K/V step is
 * converted exactly to f16 in shared memory, q is rounded to f16 (saturating
 * at +-65504) and the softmax weights to f16; the decode rows run as in
 * pa_decode_fp8.  k_scale and v_scale finite and > 0 (else PA_ERR_INVALID).
 */
pa_status pa_prefill_varlen_fp8(void* out, const void* q, const void* key_cache,
                                const void* value_cache, const int32_t* query_start_loc,
                                const int32_t* seq_lens, int32_t num_seqs, int32_t total_q,
                                int32_t max_query_len, int32_t max_seq_len,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                                int32_t block_size, int32_t num_blocks, float scale,
                                float k_scale, float v_scale, void* workspace,
                                size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */
