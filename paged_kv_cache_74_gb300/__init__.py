"""Paged KV-cache attention for one NVIDIA GB300 (sm_103a).

The compute path is libpa.so (hand-written CUDA behind a C ABI, see
include/pa.h); this package holds its build script, a thin ctypes binding
with the same names, and the seeded synthetic workload generator used by
the tests and the benchmark.
"""
from ._binding import (ABI_SYMBOLS, DEVICE_ERRORS, PAError, append_tokens, compute_slot_mapping, decode,
                       decode_fp8, decode_noalloc, decode_workspace_size, decode_xsplit,
                       decode_xsplit_fp8, device_status, library_path, load_library, map_to_kernel_blocks,
                       new_workspace, prefill_varlen, prefill_varlen_fp8, prefill_workspace_size, reshape_and_cache,
                       reshape_and_cache_fp8, reshape_and_cache_xsplit,
                       reshape_and_cache_xsplit_fp8)
from .builder import build

__all__ = ["ABI_SYMBOLS", "DEVICE_ERRORS", "PAError", "append_tokens", "build", "compute_slot_mapping", "decode",
           "decode_fp8", "decode_noalloc", "decode_workspace_size", "decode_xsplit",
           "decode_xsplit_fp8", "device_status", "library_path", "load_library", "map_to_kernel_blocks",
           "new_workspace", "prefill_varlen", "prefill_varlen_fp8", "prefill_workspace_size", "reshape_and_cache",
           "reshape_and_cache_fp8", "reshape_and_cache_xsplit", "reshape_and_cache_xsplit_fp8"]
