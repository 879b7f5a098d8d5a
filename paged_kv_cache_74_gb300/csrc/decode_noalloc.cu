// decode_noalloc.cu -- pa_decode_noalloc: paged decode attention for callers
// that cannot allocate device memory.
//
// pa_decode needs a scratch workspace for its split-KV partials, and asks the
// caller to provide it.  Some callers have no way to do that: code that runs
// inside a host framework which hands it only its input and output tensors
// (a plugin or backend interface with no allocator in its execute path),
// code whose memory budget is fixed up front by someone else, and code that
// must not call cudaMalloc on its hot path because that call can stall the
// device or is not allowed while a stream is being recorded.  For them this
// entry point takes the partials from a fixed-size array that lives in the
// library's own device memory.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, not a device address, so the device address is looked
// up once per device (cudaGetSymbolAddress, with that device current) and
// passed to the kernels.
#include <mutex>

#include "pa_internal.h"

namespace {

__device__ __align__(256) static unsigned char g_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (looked up on
// first use per device).  Returns nullptr if the lookup fails.
void* scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* key_cache,
                                       const void* value_cache, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                       int32_t num_seqs, int32_t max_seq_len, int32_t num_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t num_blocks, float scale, int32_t partition_tokens,
                                       int32_t* device_status, void* stream) {
  // Argument checks only: with no workspace, pa_decode validates everything
  // else and then answers PA_ERR_WORKSPACE without launching anything.
  const pa_status check =
      pa_decode(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                num_seqs, max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                scale, partition_tokens, nullptr, 0, stream);
  if (check != PA_ERR_WORKSPACE) return check;  // invalid arguments, or nothing to do
  if (device_status != nullptr && reinterpret_cast<uintptr_t>(device_status) % 4 != 0)
    return PA_ERR_INVALID;
  const size_t need = pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                               max_seq_len, partition_tokens);
  if (need == 0 || need > PA_DECODE_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = scratch_on_current_device();
  if (scratch == nullptr) return PA_ERR_CUDA;
  // The device status record at the start of the scratch must start at
  // zero; the split-KV partials are always written before they are read.
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 16, cs) != cudaSuccess) return PA_ERR_CUDA;
  const pa_status st =
      pa_decode(out, q, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens,
                num_seqs, max_seq_len, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                scale, partition_tokens, scratch, PA_DECODE_NOALLOC_SCRATCH_BYTES, stream);
  if (st != PA_OK || device_status == nullptr) return st;
  // The record lives in the shared scratch, which the caller cannot see:
  // hand this call's record over, in stream order.
  return cudaMemcpyAsync(device_status, scratch, 16, cudaMemcpyDeviceToDevice, cs) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}
