"""GPU parity of the slot mapping and the reshape_and_cache write: both are
integer / byte work and must match the oracle bit for bit (whole pool)."""
import numpy as np
import pytest
import torch

from helpers import bits
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _slot_case(name):
    if name == "random_varlen":
        return wl.random_workload(31, num_seqs=23, max_len=300, num_heads=4, num_kv_heads=2,
                                  head_dim=64, max_q_len=70, prefill_fraction=0.5)
    return wl.NAMED[name]()


@pytest.mark.parametrize("name", ["tiny_decode", "mixed_chunked_prefill", "random_varlen",
                                  "prefix_shared_decode_b256"])
def test_slot_mapping_bit_exact(cuda_lib, oracle, name):
    pa = cuda_lib
    w = _slot_case(name)
    dev = torch.device("cuda")
    bt = torch.from_numpy(w.block_tables).to(dev)
    qsl = torch.from_numpy(w.query_start_loc).to(dev)
    sl = torch.from_numpy(w.seq_lens).to(dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    got = pa.compute_slot_mapping(bt, qsl, sl, w.block_size, w.num_blocks, w.total_q, status=status)
    ref = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, w.block_size)
    np.testing.assert_array_equal(got.cpu().numpy(), ref)
    assert pa.device_status(status)[0] == 0


@pytest.mark.parametrize("name", ["tiny_decode", "mixed_chunked_prefill"])
def test_reshape_and_cache_whole_pool_bit_exact(cuda_lib, oracle, name):
    pa = cuda_lib
    w = wl.NAMED[name]()
    t = wl.make_tensors(w, device="cuda")
    slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, w.block_size)
    slots[::7] = -1  # padding tokens are skipped
    kc0, vc0 = bits(t.key_cache), bits(t.value_cache)
    ref_k, ref_v = oracle.reshape_and_cache(bits(t.key), bits(t.value), kc0, vc0, slots)
    del kc0, vc0
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache,
                         torch.from_numpy(slots).cuda(), status=status)
    np.testing.assert_array_equal(bits(t.key_cache), ref_k)
    np.testing.assert_array_equal(bits(t.value_cache), ref_v)
    assert pa.device_status(status)[0] == 0


def test_reshape_and_cache_strided_source(cuda_lib, oracle):
    """K and V taken as views of a fused [T, 3, Hkv, d]-like buffer (token
    stride larger than one row) are written the same as contiguous ones."""
    pa = cuda_lib
    w = wl.tiny_decode()
    t = wl.make_tensors(w, device="cuda")
    T, hkv, d = t.key.shape
    fused = torch.zeros((T, 3, hkv, d), dtype=torch.bfloat16, device="cuda")
    fused[:, 1] = t.key
    fused[:, 2] = t.value
    k_view, v_view = fused[:, 1], fused[:, 2]
    assert k_view.stride(0) == 3 * hkv * d
    slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, w.block_size)
    ref_k, ref_v = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                            bits(t.value_cache), slots)
    pa.reshape_and_cache(k_view, v_view, t.key_cache, t.value_cache, torch.from_numpy(slots).cuda())
    np.testing.assert_array_equal(bits(t.key_cache), ref_k)
    np.testing.assert_array_equal(bits(t.value_cache), ref_v)


def test_reshape_and_cache_out_of_range_slot_is_reported_and_skipped(cuda_lib, oracle):
    pa = cuda_lib
    w = wl.tiny_decode()
    t = wl.make_tensors(w, device="cuda")
    num_slots = w.num_blocks * w.block_size
    slots = np.array([5, num_slots, 17, num_slots + 1000], np.int64)
    ref_k, _ = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                        bits(t.value_cache), np.where(slots < num_slots, slots, -1))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache,
                         torch.from_numpy(slots).cuda(), status=status)
    np.testing.assert_array_equal(bits(t.key_cache), ref_k)
    st = pa.device_status(status)
    assert st[0] == 1 and st[1] in (1, 3)


def test_slot_mapping_reports_bad_block_id(cuda_lib):
    pa = cuda_lib
    w = wl.tiny_decode()
    bt = w.block_tables.copy()
    bt[2, 2] = w.num_blocks + 5  # the last block of request 2 (37 tokens) is bogus
    dev = torch.device("cuda")
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    got = pa.compute_slot_mapping(torch.from_numpy(bt).to(dev),
                                  torch.from_numpy(w.query_start_loc).to(dev),
                                  torch.from_numpy(w.seq_lens).to(dev), 16, w.num_blocks, w.total_q,
                                  status=status)
    assert int(got[2]) == -1
    st = pa.device_status(status)
    assert st[0] == 2 and st[1] == 2 and st[2] == w.num_blocks + 5


@pytest.mark.parametrize("k", [1, 2, 4])
def test_map_to_kernel_blocks_bit_exact(cuda_lib, oracle, k):
    pa = cuda_lib
    rng = np.random.default_rng(70 + k)
    tables = rng.integers(0, 5000, size=(37, 23)).astype(np.int32)
    tables[rng.random(tables.shape) < 0.2] = -1  # padding
    got = pa.map_to_kernel_blocks(torch.from_numpy(tables).cuda(), k)
    np.testing.assert_array_equal(got.cpu().numpy(), oracle.map_to_kernel_blocks(tables, k))


@pytest.mark.parametrize("B", [32, 64])
def test_slot_write_with_larger_blocks(cuda_lib, oracle, B):
    """Slot mapping and the cache write with 32- and 64-token blocks."""
    pa = cuda_lib
    w = wl.random_workload(80 + B, num_seqs=6, max_len=500, num_heads=8, num_kv_heads=2,
                           head_dim=128, block_size=B, max_q_len=70, prefill_fraction=0.5)
    t = wl.make_tensors(w, device="cuda", poison=True)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, B,
                                    w.num_blocks, w.total_q)
    ref_slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, B)
    np.testing.assert_array_equal(slots.cpu().numpy(), ref_slots)
    kc, vc = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                      bits(t.value_cache), ref_slots)
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache, slots)
    np.testing.assert_array_equal(bits(t.key_cache), kc)
    np.testing.assert_array_equal(bits(t.value_cache), vc)


@pytest.mark.parametrize("name", ["tiny_decode", "mixed_chunked_prefill", "random_varlen",
                                  "llama8b_decode_b64"])
def test_append_tokens_equals_slot_mapping_then_write(cuda_lib, oracle, name):
    """The fused launch gives the oracle's slots and the oracle's whole pool
    after its slot mapping and cache write, bit for bit."""
    pa = cuda_lib
    w = _slot_case(name)
    t = wl.make_tensors(w, device="cuda")
    ref_slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, w.block_size)
    kc, vc = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                      bits(t.value_cache), ref_slots)
    slots = torch.full((w.total_q,), -7, dtype=torch.int64, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pa.append_tokens(t.key, t.value, t.key_cache, t.value_cache, t.block_tables,
                     t.query_start_loc, t.seq_lens, slot_mapping=slots, status=status)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(slots.cpu().numpy(), ref_slots)
    np.testing.assert_array_equal(bits(t.key_cache), kc)
    np.testing.assert_array_equal(bits(t.value_cache), vc)
    assert pa.device_status(status)[0] == 0


def test_append_tokens_without_slot_output_and_bad_block(cuda_lib, oracle):
    """No slot output requested; a request whose block id is out of range is
    reported and its token skipped, the others are written."""
    pa = cuda_lib
    w = wl.tiny_decode()
    t = wl.make_tensors(w, device="cuda")
    bt = t.block_tables.clone()
    L = int(w.seq_lens[2])
    bt[2, (L - 1) // 16] = w.num_blocks + 9  # the block of request 2's new token
    good = w.block_tables.copy()
    ref_slots = oracle.slot_mapping(good, w.query_start_loc, w.seq_lens, 16)
    ref_slots[2] = -1
    kc, vc = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                      bits(t.value_cache), ref_slots)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pa.append_tokens(t.key, t.value, t.key_cache, t.value_cache, bt, t.query_start_loc,
                     t.seq_lens, status=status)
    st = pa.device_status(status)
    assert st[0] == 2 and st[1] == 2 and st[2] == w.num_blocks + 9
    np.testing.assert_array_equal(bits(t.key_cache), kc)
    np.testing.assert_array_equal(bits(t.value_cache), vc)
