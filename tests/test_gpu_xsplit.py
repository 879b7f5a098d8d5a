"""GPU parity of the x-split cache layout (K [blocks, kv heads, d / 8, block,
8], V [blocks, kv heads, d, block]): the cache write is bit-exact against
the oracle's x-split writer, and pa_decode_xsplit matches the oracle's
x-split decode (max abs <= 1e-2, mean abs <= 1e-3).  Up to 4 q heads per kv
head the x-split decode runs the same arithmetic as the token-major decode,
so the two outputs must agree bit for bit."""
import numpy as np
import pytest
import torch

from helpers import assert_close_to_oracle, bits
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def to_xsplit(key_cache, value_cache):
    """Token-major [nb, B, H, d] caches -> the x-split tensors (same device)."""
    nb, B, H, d = key_cache.shape
    kx = key_cache.view(nb, B, H, d // 8, 8).permute(0, 2, 3, 1, 4).contiguous()
    vx = value_cache.view(nb, B, H, d).permute(0, 2, 3, 1).contiguous()
    return kx, vx


def run_xsplit(pa, w, t, kx, vx, partition_tokens=0, workspace=None):
    return pa.decode_xsplit(t.q, kx, vx, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                            partition_tokens=partition_tokens, workspace=workspace)


def oracle_xsplit(oracle, w, t, kx, vx, rows=None):
    q, bt, sl = bits(t.q), w.block_tables, w.seq_lens
    if rows is not None:
        q, bt, sl = q[rows], bt[rows], sl[rows]
    return oracle.decode_xsplit(q, bits(kx), bits(vx), bt, sl, w.scale)


@pytest.mark.parametrize("hkv,d,B", [(2, 64, 16), (8, 128, 16), (4, 128, 32), (1, 64, 64)])
def test_xsplit_write_is_bit_exact(cuda_lib, oracle, hkv, d, B):
    """Random pools, random distinct slots (some negative): the whole pool
    after the GPU write equals the oracle's x-split write."""
    pa = cuda_lib
    nb, n = 40, 45
    gen = torch.Generator(device="cuda").manual_seed(300 + B + d)
    rnd = lambda *s: torch.randn(s, generator=gen, device="cuda").to(torch.bfloat16)
    kx, vx = rnd(nb, hkv, d // 8, B, 8), rnd(nb, hkv, d, B)
    key, value = rnd(n, hkv, d), rnd(n, hkv, d)
    rng = np.random.default_rng(300 + B)
    slots = rng.choice(nb * B, size=n, replace=False).astype(np.int64)
    slots[::7] = -1
    ref_k, ref_v = oracle.reshape_and_cache_xsplit(bits(key), bits(value), bits(kx), bits(vx),
                                                   slots)
    pa.reshape_and_cache_xsplit(key, value, kx, vx, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(kx), ref_k)
    np.testing.assert_array_equal(bits(vx), ref_v)


def test_xsplit_write_with_strided_rows(cuda_lib, oracle):
    """key/value rows taken from a wider fused [T, 3, Hkv, d] buffer."""
    pa = cuda_lib
    hkv, d, B, nb, n = 4, 128, 16, 16, 20
    gen = torch.Generator(device="cuda").manual_seed(310)
    fused = torch.randn((n, 3, hkv, d), generator=gen, device="cuda").to(torch.bfloat16)
    key, value = fused[:, 1], fused[:, 2]
    kx = torch.zeros((nb, hkv, d // 8, B, 8), dtype=torch.bfloat16, device="cuda")
    vx = torch.zeros((nb, hkv, d, B), dtype=torch.bfloat16, device="cuda")
    slots = np.random.default_rng(310).choice(nb * B, size=n, replace=False).astype(np.int64)
    ref_k, ref_v = oracle.reshape_and_cache_xsplit(bits(key), bits(value), bits(kx), bits(vx),
                                                   slots)
    pa.reshape_and_cache_xsplit(key, value, kx, vx, torch.from_numpy(slots).cuda())
    torch.cuda.synchronize()
    np.testing.assert_array_equal(bits(kx), ref_k)
    np.testing.assert_array_equal(bits(vx), ref_v)


def test_xsplit_tiny_decode_after_slot_write(cuda_lib, oracle):
    """Slot mapping, x-split write of each request's last token, x-split
    decode; the oracle does the same steps on its own x-split pools."""
    pa = cuda_lib
    w = wl.tiny_decode()
    t = wl.make_tensors(w, device="cuda", poison=True)
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    ref_slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, 16)
    ok, ov = oracle.reshape_and_cache_xsplit(bits(t.key), bits(t.value), bits(kx), bits(vx),
                                             ref_slots)
    pa.reshape_and_cache_xsplit(t.key, t.value, kx, vx, slots)
    ref = oracle.decode_xsplit(bits(t.q), ok, ov, w.block_tables, w.seq_lens, w.scale)
    out = run_xsplit(pa, w, t, kx, vx)
    assert_close_to_oracle(out, ref, what="tiny x-split")


SWEEP = [
    # (head_dim, q heads, kv heads, max_len, num_seqs, block_size, seed)
    (64, 4, 2, 200, 9, 16, 401), (128, 32, 8, 600, 6, 16, 402), (128, 8, 8, 40, 11, 16, 403),
    (64, 3, 3, 33, 8, 16, 404), (128, 16, 8, 500, 5, 32, 405), (64, 8, 4, 300, 6, 64, 406),
    (128, 7, 1, 257, 4, 16, 407), (128, 64, 8, 700, 3, 16, 408), (128, 6, 2, 513, 5, 32, 409),
    (64, 16, 1, 260, 6, 16, 410), (128, 80, 8, 150, 3, 64, 411), (64, 1, 1, 17, 4, 16, 412),
    (128, 24, 2, 333, 4, 16, 413),
]


@pytest.mark.parametrize("d,hq,hkv,max_len,ns,B,seed", SWEEP)
def test_xsplit_decode_random_shapes(cuda_lib, oracle, d, hq, hkv, max_len, ns, B, seed):
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, block_size=B)
    t = wl.make_tensors(w, device="cuda", poison=True)
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    out = run_xsplit(pa, w, t, kx, vx)
    ref = oracle_xsplit(oracle, w, t, kx, vx)
    assert_close_to_oracle(out, ref, what=f"x-split d{d} hq{hq} hkv{hkv} B{B}")


def test_xsplit_decode_split_partitions(cuda_lib, oracle):
    """Lengths around block boundaries with forced split-KV pieces of
    several sizes (the partial merge path)."""
    pa = cuda_lib
    lens = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1025, 2048]
    w = wl.build_workload("edges", lens, [1] * len(lens), num_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16,
                          num_blocks=1 + sum(-(-x // 16) for x in lens) + 3, seed=17)
    t = wl.make_tensors(w, device="cuda", poison=True)
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    ref = oracle_xsplit(oracle, w, t, kx, vx)
    for pt in (0, 16, 48, 512):
        out = run_xsplit(pa, w, t, kx, vx, partition_tokens=pt)
        assert_close_to_oracle(out, ref, what=f"x-split partition {pt}")


@pytest.mark.parametrize("d,hq,hkv,B", [(128, 32, 8, 16), (64, 8, 4, 32), (128, 16, 8, 64),
                                        (128, 8, 8, 16)])
def test_xsplit_decode_equals_token_major_decode(cuda_lib, d, hq, hkv, B):
    """Up to 4 q heads per kv head both layouts run the same arithmetic in
    the same order: bit-identical outputs."""
    pa = cuda_lib
    w = wl.random_workload(420 + B, num_seqs=24, max_len=1500, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, block_size=B)
    t = wl.make_tensors(w, device="cuda", poison=True)
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    a = pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens, w.max_seq_len,
                  w.scale)
    b = run_xsplit(pa, w, t, kx, vx)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_xsplit_llama8b_full_size(cuda_lib, oracle):
    """The 8B-shaped batch (64 requests, U[512, 4096]) at full size: bit-
    identical to the token-major decode, and sampled rows against the oracle."""
    pa = cuda_lib
    w = wl.llama8b_decode()
    t = wl.make_tensors(w, device="cuda")
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    a = pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens, w.max_seq_len,
                  w.scale)
    b = run_xsplit(pa, w, t, kx, vx)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    rows = np.array([0, 17, 40, 63])
    ref = oracle_xsplit(oracle, w, t, kx, vx, rows)
    assert_close_to_oracle(b, ref, rows=rows, what="llama8b x-split rows")


def test_xsplit_prefix_shared_full_size_sampled(cuda_lib, oracle):
    """The 70B-shaped shared-prefix batch (8 q heads per kv head: two work
    units per kv head) at full size, sampled rows against the oracle."""
    pa = cuda_lib
    w = wl.prefix_shared_decode()
    t = wl.make_tensors(w, device="cuda")
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    out = run_xsplit(pa, w, t, kx, vx)
    order = np.argsort(w.seq_lens)
    rows = np.array([order[0], order[len(order) // 2], order[-1]])
    ref = oracle_xsplit(oracle, w, t, kx, vx, rows)
    assert_close_to_oracle(out, ref, rows=rows, what="prefix-shared x-split rows")


def test_xsplit_bad_block_id_is_reported(cuda_lib, oracle):
    """A block id outside the pool is recorded in the status word and its
    tile reads as zeros; requests that do not use it are unaffected."""
    pa = cuda_lib
    w = wl.random_workload(430, num_seqs=4, max_len=200, num_heads=8, num_kv_heads=2,
                           head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    kx, vx = to_xsplit(t.key_cache, t.value_cache)
    bt = t.block_tables.clone()
    bt[1, 0] = w.num_blocks + 123
    ws = pa.new_workspace(pa.decode_workspace_size(4, 8, 2, 128, w.max_seq_len), "cuda")
    out = pa.decode_xsplit(t.q, kx, vx, bt, t.seq_lens, w.max_seq_len, w.scale, workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 2 and st[1] == 1 and st[2] == w.num_blocks + 123
    ref = oracle_xsplit(oracle, w, t, kx, vx)
    assert_close_to_oracle(out[[0, 2, 3]], ref[[0, 2, 3]], what="other rows")
