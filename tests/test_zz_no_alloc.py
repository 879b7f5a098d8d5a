"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers get only their input and output tensors from a host framework
and have no allocator on their execute path, or must not call cudaMalloc
there.  pa_decode_noalloc serves them from a fixed scratch array inside the
library.  These tests call it through the C ABI (ctypes, no Python wrapper)
and compare it with pa_decode, which uses a caller-provided workspace, on
two calls in a row with different batches, so a call that picked up the
previous call's leftovers would show.  This file is collected last.
"""
import ctypes

import pytest
import torch

from helpers import MAX_ABS, MEAN_ABS
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE = 3


def _noalloc(lib, w, t, out, partition_tokens, status=None, block_tables=None):
    vp = ctypes.c_void_p
    bt = t.block_tables if block_tables is None else block_tables
    return lib.pa_decode_noalloc(
        vp(out.data_ptr()), vp(t.q.data_ptr()), vp(t.key_cache.data_ptr()),
        vp(t.value_cache.data_ptr()), vp(bt.data_ptr()), w.max_blocks_per_seq,
        vp(t.seq_lens.data_ptr()), w.num_seqs, w.max_seq_len, w.num_heads, w.num_kv_heads,
        w.head_dim, w.block_size, w.num_blocks, ctypes.c_float(w.scale), partition_tokens,
        vp(status.data_ptr() if status is not None else 0),
        vp(torch.cuda.current_stream().cuda_stream))


def _case(seed, max_len):
    w = wl.random_workload(seed, num_seqs=12, max_len=max_len, min_len=max_len // 3,
                           num_heads=32, num_kv_heads=8, head_dim=128)
    return w, wl.make_tensors(w, device="cuda", poison=True)


def test_noalloc_matches_workspace_decode_on_consecutive_calls(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    for w, t, pt in [(*_case(71, 3000), 128), (*_case(72, 1700), 256)]:
        need = pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim,
                                        w.max_seq_len, pt)
        assert need > 1 << 20  # several partitions per request: the scratch is really used
        ref = pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens,
                        w.max_seq_len, w.scale, partition_tokens=pt)
        out = torch.full_like(t.q, float("nan"))
        status = torch.full((4,), -7, dtype=torch.int32, device="cuda")
        assert _noalloc(lib, w, t, out, pt, status) == 0
        torch.cuda.synchronize()
        assert status.tolist() == [0, 0, 0, 0]  # this call's record: no device error
        err = (out.double() - ref.double()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS
        assert torch.equal(out, ref)  # same kernels, same partitions


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    pa = cuda_lib
    lib = pa.load_library()
    w, t = _case(73, 600)
    # 64 requests of 32K tokens in 16-token partitions need far more than the array
    need = pa.decode_workspace_size(64, 32, 8, 128, 32768, 16)
    assert need > 32 << 20
    vp = ctypes.c_void_p
    rc = lib.pa_decode_noalloc(vp(t.q.data_ptr()), vp(t.q.data_ptr()), vp(t.key_cache.data_ptr()),
                               vp(t.value_cache.data_ptr()), vp(t.block_tables.data_ptr()),
                               32768 // 16, vp(t.seq_lens.data_ptr()), 64, 32768, 32,
                               8, 128, 16, w.num_blocks, ctypes.c_float(0.1), 16, vp(0),
                               vp(torch.cuda.current_stream().cuda_stream))
    assert rc == PA_ERR_WORKSPACE


def test_noalloc_reports_device_errors_through_device_status(cuda_lib):
    """The kernels' status record lives in the library's scratch array; the
    call hands it to the caller's device_status.  A block id outside the pool
    is range-checked in the kernel (never dereferenced: the tile reads as
    zeros) and must come back as PA_DEV_BAD_BLOCK_ID with its request and
    value; the next clean call must report a clean record again."""
    pa = cuda_lib
    lib = pa.load_library()
    w, t = _case(74, 900)
    bad = t.block_tables.clone()
    bad_row = 5
    bad[bad_row, 0] = w.num_blocks + 3  # outside the pool
    out = torch.empty_like(t.q)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    assert _noalloc(lib, w, t, out, 128, status, block_tables=bad) == 0
    torch.cuda.synchronize()
    rec = status.tolist()
    assert rec[0] == 2 and rec[1] == bad_row and rec[2] == w.num_blocks + 3, rec
    assert _noalloc(lib, w, t, out, 128, status) == 0
    torch.cuda.synchronize()
    assert status.tolist() == [0, 0, 0, 0]
