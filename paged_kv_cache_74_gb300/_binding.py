"""ctypes binding of libpa.so -- argument marshalling only.

Every step of the path runs in the library's CUDA kernels; these wrappers
only check tensor dtypes and shapes, turn torch tensors into device
pointers, pass torch's current CUDA stream, and raise on a non-zero
pa_status.  There is no fallback: if the library is missing, or a call is
made on tensors that are not on a CUDA device, they raise.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import builder as _build

_lock = threading.Lock()
_lib = None

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_WORKSPACE, PA_ERR_CUDA = range(5)
DEVICE_ERRORS = {0: "ok", 1: "bad slot", 2: "bad block id", 3: "bad seq_len",
                 4: "bad query length", 5: "wait timeout"}
ABI_SYMBOLS = ("pa_status_string", "pa_abi_version", "pa_reshape_and_cache",
               "pa_compute_slot_mapping", "pa_decode_workspace_size", "pa_decode",
               "pa_prefill_workspace_size", "pa_prefill_varlen", "pa_decode_noalloc",
               "pa_map_to_kernel_blocks", "pa_reshape_and_cache_fp8", "pa_decode_fp8",
               "pa_reshape_and_cache_xsplit", "pa_decode_xsplit", "pa_append_tokens",
               "pa_reshape_and_cache_xsplit_fp8", "pa_decode_xsplit_fp8", "pa_prefill_varlen_fp8")


class PAError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn} failed: {msg}")
        self.status = status


_i32, _i64, _sz, _vp, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


def _declare(lib):
    lib.pa_status_string.restype = ctypes.c_char_p
    lib.pa_status_string.argtypes = [ctypes.c_int]
    lib.pa_abi_version.restype = ctypes.c_int
    lib.pa_abi_version.argtypes = []
    lib.pa_reshape_and_cache.restype = ctypes.c_int
    lib.pa_reshape_and_cache.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _i32, _i32,
                                         _i32, _i32, _vp, _vp]
    lib.pa_compute_slot_mapping.restype = ctypes.c_int
    lib.pa_compute_slot_mapping.argtypes = [_vp, _i32, _vp, _i32, _vp, _vp, _i32, _i32, _i32,
                                            _vp, _vp]
    lib.pa_reshape_and_cache_fp8.restype = ctypes.c_int
    lib.pa_reshape_and_cache_fp8.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _i32,
                                             _i32, _i32, _i32, _f32, _f32, _vp, _vp]
    lib.pa_decode_fp8.restype = ctypes.c_int
    lib.pa_decode_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                  _i32, _i32, _i32, _f32, _f32, _f32, _i32, _vp, _sz, _vp]
    lib.pa_reshape_and_cache_xsplit.restype = ctypes.c_int
    lib.pa_reshape_and_cache_xsplit.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _i32,
                                                _i32, _i32, _i32, _vp, _vp]
    lib.pa_decode_xsplit.restype = ctypes.c_int
    lib.pa_decode_xsplit.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                     _i32, _i32, _i32, _f32, _i32, _vp, _sz, _vp]
    lib.pa_reshape_and_cache_xsplit_fp8.restype = ctypes.c_int
    lib.pa_reshape_and_cache_xsplit_fp8.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _i32,
                                                    _i32, _i32, _i32, _f32, _f32, _vp, _vp]
    lib.pa_decode_xsplit_fp8.restype = ctypes.c_int
    lib.pa_decode_xsplit_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32,
                                         _i32, _i32, _i32, _i32, _f32, _f32, _f32, _i32, _vp, _sz,
                                         _vp]
    lib.pa_append_tokens.restype = ctypes.c_int
    lib.pa_append_tokens.argtypes = [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _vp, _vp, _i32,
                                     _i32, _i32, _i32, _i32, _i32, _vp, _vp, _vp]
    lib.pa_map_to_kernel_blocks.restype = ctypes.c_int
    lib.pa_map_to_kernel_blocks.argtypes = [_vp, _vp, _i32, _i32, _i32, _vp, _vp]
    lib.pa_decode_workspace_size.restype = _sz
    lib.pa_decode_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    lib.pa_decode.restype = ctypes.c_int
    lib.pa_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32, _i32,
                              _i32, _i32, _f32, _i32, _vp, _sz, _vp]
    lib.pa_decode_noalloc.restype = ctypes.c_int
    lib.pa_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i32, _vp, _i32, _i32, _i32, _i32,
                                      _i32, _i32, _i32, _f32, _i32, _vp, _vp]
    lib.pa_prefill_workspace_size.restype = _sz
    lib.pa_prefill_workspace_size.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
    lib.pa_prefill_varlen.restype = ctypes.c_int
    lib.pa_prefill_varlen.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp,
                                      _i32, _i32, _i32, _i32, _i32, _i32, _f32, _vp, _sz, _vp]
    lib.pa_prefill_varlen_fp8.restype = ctypes.c_int
    lib.pa_prefill_varlen_fp8.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _vp,
                                          _i32, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32, _vp,
                                          _sz, _vp]
    return lib


def library_path() -> str:
    return _build.LIB


def load_library(path: str | None = None):
    """Load libpa.so (built by paged_kv_cache_74_gb300.build()).  Raises if absent."""
    global _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or _build.LIB
            if not os.path.exists(p):
                raise RuntimeError(f"libpa.so not built at {p}; run paged_kv_cache_74_gb300.build()")
            lib = _declare(ctypes.CDLL(p))
            if path is not None:
                return lib
            _lib = lib
        return _lib


def _check(fn, status):
    if status != PA_OK:
        raise PAError(fn, status, load_library().pa_status_string(status).decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(name, t, dtype):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def _contig(name, t, dtype):
    _cuda(name, t, dtype)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def reshape_and_cache(key, value, key_cache, value_cache, slot_mapping, status=None):
    """Write key/value [T, Hkv, d] (token stride may exceed Hkv*d) into the
    caches at slot_mapping[T] (int64; negative = skip)."""
    _cuda("key", key, torch.bfloat16)
    _cuda("value", value, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("slot_mapping", slot_mapping, torch.int64)
    nb, bs, hkv, d = key_cache.shape
    T = slot_mapping.shape[0]
    for name, t in (("key", key), ("value", value)):
        if tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, {hkv}, {d}] with contiguous heads")
    lib = load_library()
    _check("pa_reshape_and_cache", lib.pa_reshape_and_cache(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache),
        _ptr(value_cache), _ptr(slot_mapping), T, hkv, d, bs, nb, _ptr(status), _stream()))


def reshape_and_cache_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale, v_scale,
                          status=None):
    """Quantizing write into e4m3 caches (uint8 [nb, bs, Hkv, d]): e4m3(x / scale)."""
    _cuda("key", key, torch.bfloat16)
    _cuda("value", value, torch.bfloat16)
    _contig("key_cache", key_cache, torch.uint8)
    _contig("value_cache", value_cache, torch.uint8)
    _contig("slot_mapping", slot_mapping, torch.int64)
    nb, bs, hkv, d = key_cache.shape
    T = slot_mapping.shape[0]
    for name, t in (("key", key), ("value", value)):
        if tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, {hkv}, {d}] with contiguous heads")
    lib = load_library()
    _check("pa_reshape_and_cache_fp8", lib.pa_reshape_and_cache_fp8(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache),
        _ptr(value_cache), _ptr(slot_mapping), T, hkv, d, bs, nb, float(k_scale), float(v_scale),
        _ptr(status), _stream()))


def _xsplit_shape(key_cache, value_cache):
    """(num_blocks, block_size, num_kv_heads, head_dim) of x-split caches:
    key [nb, Hkv, d / 8, bs, 8], value [nb, Hkv, d, bs]."""
    if key_cache.dim() != 5 or key_cache.shape[4] != 8:
        raise ValueError("x-split key_cache must be [num_blocks, kv_heads, head_dim / 8, block, 8]")
    nb, hkv, dx, bs, _ = key_cache.shape
    d = dx * 8
    if tuple(value_cache.shape) != (nb, hkv, d, bs):
        raise ValueError("x-split value_cache must be [num_blocks, kv_heads, head_dim, block]")
    return nb, bs, hkv, d


def reshape_and_cache_xsplit(key, value, key_cache, value_cache, slot_mapping, status=None):
    """reshape_and_cache into x-split caches (key [nb, Hkv, d / 8, bs, 8],
    value [nb, Hkv, d, bs], bf16)."""
    _cuda("key", key, torch.bfloat16)
    _cuda("value", value, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("slot_mapping", slot_mapping, torch.int64)
    nb, bs, hkv, d = _xsplit_shape(key_cache, value_cache)
    T = slot_mapping.shape[0]
    for name, t in (("key", key), ("value", value)):
        if tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, {hkv}, {d}] with contiguous heads")
    lib = load_library()
    _check("pa_reshape_and_cache_xsplit", lib.pa_reshape_and_cache_xsplit(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache),
        _ptr(value_cache), _ptr(slot_mapping), T, hkv, d, bs, nb, _ptr(status), _stream()))


def _xsplit8_shape(key_cache, value_cache):
    """(num_blocks, block_size, num_kv_heads, head_dim) of e4m3 x-split caches:
    key [nb, Hkv, d / 16, bs, 16], value [nb, Hkv, d, bs] (uint8)."""
    if key_cache.dim() != 5 or key_cache.shape[4] != 16:
        raise ValueError("e4m3 x-split key_cache must be [num_blocks, kv_heads, head_dim / 16, block, 16]")
    nb, hkv, dx, bs, _ = key_cache.shape
    d = dx * 16
    if tuple(value_cache.shape) != (nb, hkv, d, bs):
        raise ValueError("e4m3 x-split value_cache must be [num_blocks, kv_heads, head_dim, block]")
    return nb, bs, hkv, d


def reshape_and_cache_xsplit_fp8(key, value, key_cache, value_cache, slot_mapping, k_scale,
                                 v_scale, status=None):
    """reshape_and_cache_fp8 into e4m3 x-split caches (key [nb, Hkv, d / 16,
    bs, 16], value [nb, Hkv, d, bs], uint8)."""
    _cuda("key", key, torch.bfloat16)
    _cuda("value", value, torch.bfloat16)
    _contig("key_cache", key_cache, torch.uint8)
    _contig("value_cache", value_cache, torch.uint8)
    _contig("slot_mapping", slot_mapping, torch.int64)
    nb, bs, hkv, d = _xsplit8_shape(key_cache, value_cache)
    T = slot_mapping.shape[0]
    for name, t in (("key", key), ("value", value)):
        if tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, {hkv}, {d}] with contiguous heads")
    lib = load_library()
    _check("pa_reshape_and_cache_xsplit_fp8", lib.pa_reshape_and_cache_xsplit_fp8(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache),
        _ptr(value_cache), _ptr(slot_mapping), T, hkv, d, bs, nb, float(k_scale), float(v_scale),
        _ptr(status), _stream()))


def compute_slot_mapping(block_tables, query_start_loc, seq_lens, block_size, num_blocks,
                         total_tokens, out=None, status=None):
    _contig("block_tables", block_tables, torch.int32)
    _contig("query_start_loc", query_start_loc, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    if out is None:
        out = torch.empty(total_tokens, dtype=torch.int64, device=block_tables.device)
    _contig("slot_mapping", out, torch.int64)
    lib = load_library()
    _check("pa_compute_slot_mapping", lib.pa_compute_slot_mapping(
        _ptr(out), total_tokens, _ptr(block_tables), block_tables.shape[1], _ptr(query_start_loc),
        _ptr(seq_lens), seq_lens.shape[0], block_size, num_blocks, _ptr(status), _stream()))
    return out


def append_tokens(key, value, key_cache, value_cache, block_tables, query_start_loc, seq_lens,
                  slot_mapping=None, status=None):
    """Slot mapping and cache write of the new tokens in one launch: token i of
    request r goes to the slot compute_slot_mapping gives it (slots stored in
    slot_mapping if given)."""
    _cuda("key", key, torch.bfloat16)
    _cuda("value", value, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("block_tables", block_tables, torch.int32)
    _contig("query_start_loc", query_start_loc, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    nb, bs, hkv, d = key_cache.shape
    T = key.shape[0]
    for name, t in (("key", key), ("value", value)):
        if tuple(t.shape) != (T, hkv, d) or t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError(f"{name} must be [T, {hkv}, {d}] with contiguous heads")
    if slot_mapping is not None:
        _contig("slot_mapping", slot_mapping, torch.int64)
    lib = load_library()
    _check("pa_append_tokens", lib.pa_append_tokens(
        _ptr(key), _ptr(value), key.stride(0), value.stride(0), _ptr(key_cache), _ptr(value_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(query_start_loc), _ptr(seq_lens),
        seq_lens.shape[0], T, hkv, d, bs, nb, _ptr(slot_mapping), _ptr(status), _stream()))
    return slot_mapping


def map_to_kernel_blocks(block_tables, blocks_per_kv_block, out=None, status=None):
    """Block tables of manager blocks -> tables of kernel blocks (k per manager block)."""
    _contig("block_tables", block_tables, torch.int32)
    rows, cols = block_tables.shape
    k = int(blocks_per_kv_block)
    if out is None:
        out = torch.empty((rows, cols * k), dtype=torch.int32, device=block_tables.device)
    _contig("kernel_tables", out, torch.int32)
    lib = load_library()
    _check("pa_map_to_kernel_blocks", lib.pa_map_to_kernel_blocks(
        _ptr(out), _ptr(block_tables), rows, cols, k, _ptr(status), _stream()))
    return out


def decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim, max_seq_len,
                          partition_tokens=0):
    return int(load_library().pa_decode_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                       max_seq_len, partition_tokens))


def new_workspace(nbytes, device):
    """A zeroed workspace (the status record starts clean)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def decode(q, key_cache, value_cache, block_tables, seq_lens, max_seq_len, scale, out=None,
           workspace=None, partition_tokens=0):
    """Paged decode attention; q [S, Hq, d] -> out [S, Hq, d] (bf16)."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("block_tables", block_tables, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    S, hq, d = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    if d2 != d or value_cache.shape != key_cache.shape:
        raise ValueError("cache shapes do not match q")
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(S, hq, hkv, d, max_seq_len, partition_tokens),
                                  q.device)
    lib = load_library()
    _check("pa_decode", lib.pa_decode(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, int(max_seq_len), hq, hkv, d, bs, nb,
        float(scale), int(partition_tokens), _ptr(workspace), workspace.numel(), _stream()))
    return out


def decode_fp8(q, key_cache, value_cache, block_tables, seq_lens, max_seq_len, scale, k_scale,
               v_scale, out=None, workspace=None, partition_tokens=0):
    """Paged decode over e4m3 caches (uint8 [nb, bs, Hkv, d]); q, out bf16."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.uint8)
    _contig("value_cache", value_cache, torch.uint8)
    _contig("block_tables", block_tables, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    S, hq, d = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    if d2 != d or value_cache.shape != key_cache.shape:
        raise ValueError("cache shapes do not match q")
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(S, hq, hkv, d, max_seq_len, partition_tokens),
                                  q.device)
    lib = load_library()
    _check("pa_decode_fp8", lib.pa_decode_fp8(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, int(max_seq_len), hq, hkv, d, bs, nb,
        float(scale), float(k_scale), float(v_scale), int(partition_tokens), _ptr(workspace),
        workspace.numel(), _stream()))
    return out


def decode_xsplit(q, key_cache, value_cache, block_tables, seq_lens, max_seq_len, scale,
                  out=None, workspace=None, partition_tokens=0):
    """Paged decode over x-split caches (see reshape_and_cache_xsplit)."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("block_tables", block_tables, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    S, hq, d = q.shape
    nb, bs, hkv, d2 = _xsplit_shape(key_cache, value_cache)
    if d2 != d:
        raise ValueError("cache shapes do not match q")
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(S, hq, hkv, d, max_seq_len, partition_tokens),
                                  q.device)
    lib = load_library()
    _check("pa_decode_xsplit", lib.pa_decode_xsplit(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, int(max_seq_len), hq, hkv, d, bs, nb,
        float(scale), int(partition_tokens), _ptr(workspace), workspace.numel(), _stream()))
    return out


def decode_xsplit_fp8(q, key_cache, value_cache, block_tables, seq_lens, max_seq_len, scale,
                      k_scale, v_scale, out=None, workspace=None, partition_tokens=0):
    """Paged decode over e4m3 x-split caches (see reshape_and_cache_xsplit_fp8)."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.uint8)
    _contig("value_cache", value_cache, torch.uint8)
    _contig("block_tables", block_tables, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    S, hq, d = q.shape
    nb, bs, hkv, d2 = _xsplit8_shape(key_cache, value_cache)
    if d2 != d:
        raise ValueError("cache shapes do not match q")
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(decode_workspace_size(S, hq, hkv, d, max_seq_len, partition_tokens),
                                  q.device)
    lib = load_library()
    _check("pa_decode_xsplit_fp8", lib.pa_decode_xsplit_fp8(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, int(max_seq_len), hq, hkv, d, bs, nb,
        float(scale), float(k_scale), float(v_scale), int(partition_tokens), _ptr(workspace),
        workspace.numel(), _stream()))
    return out


def decode_noalloc(q, key_cache, value_cache, block_tables, seq_lens, max_seq_len, scale,
                   out=None, partition_tokens=0, status=None):
    """pa_decode without a workspace: for callers that cannot allocate device
    memory.  Scratch comes from a fixed-size array inside the library (see
    include/pa.h); calls that overlap on the GPU must be serialised.  status:
    optional int32[4] CUDA tensor that receives the call's device status
    record."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("block_tables", block_tables, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    S, hq, d = q.shape
    nb, bs, hkv, _ = key_cache.shape
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    lib = load_library()
    _check("pa_decode_noalloc", lib.pa_decode_noalloc(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), S, int(max_seq_len), hq, hkv, d, bs, nb,
        float(scale), int(partition_tokens), _ptr(status), _stream()))
    return out


def prefill_workspace_size(num_seqs, total_q, num_heads, num_kv_heads, head_dim, max_seq_len):
    return int(load_library().pa_prefill_workspace_size(num_seqs, total_q, num_heads, num_kv_heads,
                                                        head_dim, max_seq_len))


def prefill_varlen(q, key_cache, value_cache, query_start_loc, seq_lens, block_tables,
                   max_query_len, max_seq_len, scale, out=None, workspace=None):
    """Mixed chunked-prefill + decode attention; q [total_q, Hq, d]."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.bfloat16)
    _contig("value_cache", value_cache, torch.bfloat16)
    _contig("query_start_loc", query_start_loc, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    _contig("block_tables", block_tables, torch.int32)
    tq, hq, d = q.shape
    nb, bs, hkv, _ = key_cache.shape
    S = seq_lens.shape[0]
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(prefill_workspace_size(S, tq, hq, hkv, d, max_seq_len), q.device)
    lib = load_library()
    _check("pa_prefill_varlen", lib.pa_prefill_varlen(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(query_start_loc),
        _ptr(seq_lens), S, tq, int(max_query_len), int(max_seq_len), _ptr(block_tables),
        block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), _ptr(workspace),
        workspace.numel(), _stream()))
    return out


def prefill_varlen_fp8(q, key_cache, value_cache, query_start_loc, seq_lens, block_tables,
                       max_query_len, max_seq_len, scale, k_scale, v_scale, out=None, workspace=None):
    """prefill_varlen over e4m3 caches (uint8 [nb, bs, Hkv, d]) with their scales."""
    _contig("q", q, torch.bfloat16)
    _contig("key_cache", key_cache, torch.uint8)
    _contig("value_cache", value_cache, torch.uint8)
    _contig("query_start_loc", query_start_loc, torch.int32)
    _contig("seq_lens", seq_lens, torch.int32)
    _contig("block_tables", block_tables, torch.int32)
    tq, hq, d = q.shape
    nb, bs, hkv, d2 = key_cache.shape
    if d2 != d or value_cache.shape != key_cache.shape:
        raise ValueError("cache shapes do not match q")
    S = seq_lens.shape[0]
    if out is None:
        out = torch.empty_like(q)
    _contig("out", out, torch.bfloat16)
    if workspace is None:
        workspace = new_workspace(prefill_workspace_size(S, tq, hq, hkv, d, max_seq_len), q.device)
    lib = load_library()
    _check("pa_prefill_varlen_fp8", lib.pa_prefill_varlen_fp8(
        _ptr(out), _ptr(q), _ptr(key_cache), _ptr(value_cache), _ptr(query_start_loc),
        _ptr(seq_lens), S, tq, int(max_query_len), int(max_seq_len), _ptr(block_tables),
        block_tables.shape[1], hq, hkv, d, bs, nb, float(scale), float(k_scale), float(v_scale),
        _ptr(workspace), workspace.numel(), _stream()))
    return out


def device_status(workspace_or_status):
    """Read the int32[4] device status record (synchronises the stream)."""
    t = workspace_or_status
    rec = t[:16].view(torch.int32) if t.dtype == torch.uint8 else t[:4]
    return [int(x) for x in rec.cpu()]
