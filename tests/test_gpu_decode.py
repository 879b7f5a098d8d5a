"""GPU parity of pa_decode (and of the decode rows of pa_prefill_varlen)
against the fp64 oracle: max abs <= 1e-2 and mean abs <= 1e-3 on N(0,1)
inputs, plus bit-exact invariances (NaN poison, block relocation, shared
prefix, determinism) and device-side error reporting."""
import numpy as np
import pytest
import torch

from helpers import assert_close_to_oracle, bits, oracle_decode_rows
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_decode(pa, w, t, partition_tokens=0, workspace=None):
    return pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens, w.max_seq_len,
                     w.scale, partition_tokens=partition_tokens, workspace=workspace)


def test_tiny_decode_after_slot_write(cuda_lib, oracle):
    """The tiny workload end to end: slot mapping, write of each request's
    last token, decode; compared with the oracle doing the same steps."""
    pa = cuda_lib
    w = wl.tiny_decode()
    t = wl.make_tensors(w, device="cuda", poison=True)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    ref_slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, 16)
    np.testing.assert_array_equal(slots.cpu().numpy(), ref_slots)
    kc, vc = oracle.reshape_and_cache(bits(t.key), bits(t.value), bits(t.key_cache),
                                      bits(t.value_cache), ref_slots)
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache, slots)
    ref = oracle.decode(bits(t.q), kc, vc, w.block_tables, w.seq_lens, w.scale)
    out = run_decode(pa, w, t)
    assert_close_to_oracle(out, ref, what="tiny")


SWEEP = [
    # (head_dim, q heads, kv heads, max_len, num_seqs, seed)
    (64, 4, 2, 200, 9, 101), (64, 8, 8, 70, 5, 102), (64, 8, 1, 300, 6, 103),
    (64, 16, 4, 129, 7, 104), (128, 32, 8, 600, 6, 105), (128, 8, 8, 40, 11, 106),
    (128, 16, 2, 1100, 3, 107), (128, 7, 1, 257, 4, 108), (128, 6, 2, 513, 5, 109),
    (64, 3, 3, 33, 8, 110), (128, 64, 8, 700, 3, 111), (64, 1, 1, 17, 4, 112),
    # 9 to 16 q heads per kv head (tensor-core decode only)
    (128, 32, 2, 900, 5, 113), (64, 16, 1, 260, 6, 114), (128, 24, 2, 333, 4, 115),
    (128, 80, 8, 150, 3, 116),
]


@pytest.mark.parametrize("d,hq,hkv,max_len,ns,seed", SWEEP)
def test_decode_random_shapes(cuda_lib, oracle, d, hq, hkv, max_len, ns, seed):
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out = run_decode(pa, w, t)
    ref = oracle.decode(bits(t.q), bits(t.key_cache), bits(t.value_cache), w.block_tables,
                        w.seq_lens, w.scale)
    assert_close_to_oracle(out, ref, what=f"d{d} hq{hq} hkv{hkv}")


def test_decode_edge_lengths(cuda_lib, oracle):
    """Lengths at and around block and partition boundaries, and 1."""
    pa = cuda_lib
    lens = [1, 15, 16, 17, 31, 32, 33, 511, 512, 513, 1023, 1024, 1025, 2048]
    w = wl.build_workload("edges", lens, [1] * len(lens), num_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16, num_blocks=1 + sum(-(-x // 16) for x in lens) + 3,
                          seed=7)
    t = wl.make_tensors(w, device="cuda", poison=True)
    ref = oracle.decode(bits(t.q), bits(t.key_cache), bits(t.value_cache), w.block_tables,
                        w.seq_lens, w.scale)
    for pt in (0, 16, 48, 128, 512, 4096):
        out = run_decode(pa, w, t, partition_tokens=pt)
        assert_close_to_oracle(out, ref, what=f"partition {pt}")


def test_decode_single_token_is_exact_value(cuda_lib):
    pa = cuda_lib
    w = wl.build_workload("one", [1, 1, 1], [1, 1, 1], num_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, num_blocks=8, seed=9)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out = run_decode(pa, w, t)
    for r in range(3):
        v0 = t.value_cache[int(w.block_tables[r, 0]), 0]  # [Hkv, d]
        torch.testing.assert_close(out[r], v0.repeat_interleave(4, dim=0), rtol=0, atol=0)


def test_nan_poison_does_not_change_output(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(41, num_seqs=12, max_len=700, num_heads=32, num_kv_heads=8,
                           head_dim=128, spare_blocks=20)
    clean = wl.make_tensors(w, device="cuda")
    dirty = wl.make_tensors(w, device="cuda", poison=True)
    a = run_decode(pa, w, clean, partition_tokens=128)
    b = run_decode(pa, w, dirty, partition_tokens=128)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)


def test_block_relocation_is_bit_invariant(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(42, num_seqs=10, max_len=900, num_heads=32, num_kv_heads=8,
                           head_dim=128, spare_blocks=10)
    t = wl.make_tensors(w, device="cuda")
    a = run_decode(pa, w, t)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(w.num_blocks)).cuda()
    kc2 = torch.empty_like(t.key_cache)
    vc2 = torch.empty_like(t.value_cache)
    kc2[perm] = t.key_cache
    vc2[perm] = t.value_cache
    bt2 = perm[t.block_tables.long()].to(torch.int32)
    b = pa.decode(t.q, kc2, vc2, bt2, t.seq_lens, w.max_seq_len, w.scale)
    assert torch.equal(a, b)


def test_shared_prefix_equals_private_copy(cuda_lib):
    """Requests reading one shared set of prefix blocks get the same bits as
    requests that each hold a private copy of those blocks."""
    pa = cuda_lib
    lens = [1500, 700, 1024, 90, 2000]
    ws = wl.build_workload("shared", lens, [1] * 5, num_heads=16, num_kv_heads=2, head_dim=128,
                           block_size=16, num_blocks=400, seed=5, shared_prefix_blocks=64)
    t = wl.make_tensors(ws, device="cuda")
    a = run_decode(pa, ws, t)
    # give each request its own copy of the shared blocks
    bt = ws.block_tables.copy()
    kc, vc = t.key_cache.clone(), t.value_cache.clone()
    used = set(int(x) for x in ws.used_blocks())
    free = [b for b in range(1, ws.num_blocks) if b not in used]
    for r in range(len(lens)):
        nb = -(-lens[r] // 16)
        for j in range(min(nb, 64)):
            dst = free.pop()
            kc[dst] = t.key_cache[bt[r, j]]
            vc[dst] = t.value_cache[bt[r, j]]
            bt[r, j] = dst
    b = pa.decode(t.q, kc, vc, torch.from_numpy(bt).cuda(), t.seq_lens, ws.max_seq_len, ws.scale)
    assert torch.equal(a, b)


def test_decode_is_deterministic(cuda_lib):
    pa = cuda_lib
    w = wl.long_context_decode()
    w = wl.build_workload("det", w.seq_lens[:2] // 4, [1, 1], num_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16, num_blocks=1100, seed=8)
    t = wl.make_tensors(w, device="cuda")
    a = run_decode(pa, w, t)
    b = run_decode(pa, w, t)
    assert torch.equal(a, b)


def test_varlen_decode_rows_match_decode(cuda_lib):
    """pa_prefill_varlen on a batch of q_len == 1 rows runs the decode kernel
    on rows query_start_loc[r]; outputs equal pa_decode bit for bit."""
    pa = cuda_lib
    w = wl.random_workload(43, num_seqs=9, max_len=1300, num_heads=32, num_kv_heads=8, head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    a = run_decode(pa, w, t)
    b = pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens,
                          t.block_tables, 1, w.max_seq_len, w.scale)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name,sample", [("llama8b_decode_b64", None),
                                         ("long_ctx_decode_8x32k", None),
                                         ("prefix_shared_decode_b256", None)])
def test_full_size_workloads(cuda_lib, oracle, name, sample):
    """Full-size workloads in the benchmark's launch configuration; the
    oracle checks every request (or a seeded sample of them)."""
    pa = cuda_lib
    w = wl.NAMED[name]()
    t = wl.make_tensors(w, device="cuda", poison=True)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), "cuda")
    out = run_decode(pa, w, t, workspace=ws)
    assert pa.device_status(ws)[0] == 0
    rows = np.arange(w.num_seqs)
    if sample:
        rows = np.sort(np.random.default_rng(99).choice(w.num_seqs, sample, replace=False))
    ref = oracle_decode_rows(oracle, w, t, rows)
    assert_close_to_oracle(out[torch.from_numpy(rows).cuda()], ref, what=name)


@pytest.mark.parametrize("hq,hkv,d", [(32, 4, 128), (64, 4, 64)])
def test_many_short_requests_tensor_core_decode(cuda_lib, oracle, hq, hkv, d):
    """600 short requests of uneven length, 8 or 16 q heads per kv head: the
    tensor-core decode splits its chunks over the CTAs by cost (segment
    starts weigh as chunks do), so CTA ranges hold many segments and end
    wherever the cost falls; every request is checked against the oracle."""
    pa = cuda_lib
    w = wl.random_workload(48 + hkv, num_seqs=600, max_len=300, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d)
    t = wl.make_tensors(w, device="cuda", poison=True)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, hq, hkv, d, w.max_seq_len), "cuda")
    out = run_decode(pa, w, t, workspace=ws)
    assert pa.device_status(ws)[0] == 0
    ref = oracle_decode_rows(oracle, w, t, np.arange(w.num_seqs))
    assert_close_to_oracle(out, ref, what=f"600 short requests, {hq // hkv} q heads per kv head")


def test_bad_block_id_is_reported_not_dereferenced(cuda_lib, oracle):
    pa = cuda_lib
    w = wl.random_workload(44, num_seqs=4, max_len=200, num_heads=8, num_kv_heads=2, head_dim=64)
    t = wl.make_tensors(w, device="cuda")
    bt = t.block_tables.clone()
    bt[1, 0] = w.num_blocks + 123
    ws = pa.new_workspace(pa.decode_workspace_size(4, 8, 2, 64, w.max_seq_len), "cuda")
    out = pa.decode(t.q, t.key_cache, t.value_cache, bt, t.seq_lens, w.max_seq_len, w.scale,
                    workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 2 and st[1] == 1 and st[2] == w.num_blocks + 123
    # requests that do not use the bad entry are unaffected
    ref = oracle.decode(bits(t.q), bits(t.key_cache), bits(t.value_cache), w.block_tables,
                        w.seq_lens, w.scale)
    assert_close_to_oracle(out[[0, 2, 3]], ref[[0, 2, 3]], what="other rows")


def test_seq_len_beyond_bound_is_reported(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(45, num_seqs=3, max_len=100, num_heads=8, num_kv_heads=2, head_dim=64)
    t = wl.make_tensors(w, device="cuda")
    sl = t.seq_lens.clone()
    sl[2] = w.max_seq_len + 1  # larger than the max_seq_len the host passes
    ws = pa.new_workspace(pa.decode_workspace_size(3, 8, 2, 64, w.max_seq_len), "cuda")
    pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, sl, w.max_seq_len, w.scale,
              workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 3 and st[1] == 2


@pytest.mark.parametrize("hq,hkv", [(32, 8), (64, 8)])
def test_cuda_graph_replays_with_new_inputs(cuda_lib, hq, hkv):
    """A captured decode replays correctly with new query values each time:
    every replay equals an eager call on the same data (the pair counters of
    the split requests start clean on every launch, also on a replay, which
    reuses the launch's arguments)."""
    pa = cuda_lib
    w = wl.random_workload(47, num_seqs=16, max_len=3000, num_heads=hq, num_kv_heads=hkv,
                           head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    ws = pa.new_workspace(pa.decode_workspace_size(16, hq, hkv, 128, w.max_seq_len), "cuda")
    out = torch.empty_like(t.q)
    q = t.q.clone()
    call = lambda: pa.decode(q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens,
                             w.max_seq_len, w.scale, out=out, workspace=ws)
    call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    gen = torch.Generator(device="cuda").manual_seed(48)
    for rep in range(3):
        q.copy_(torch.randn(q.shape, generator=gen, device="cuda").to(torch.bfloat16))
        g.replay()
        torch.cuda.synchronize()
        ref = pa.decode(q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens, w.max_seq_len,
                        w.scale)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"replay {rep}"


def test_decode_step_in_a_cuda_graph(cuda_lib):
    """A decode step captured in a CUDA graph replays to the eager result."""
    pa = cuda_lib
    w = wl.random_workload(46, num_seqs=16, max_len=2000, num_heads=32, num_kv_heads=8,
                           head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    ws = pa.new_workspace(pa.decode_workspace_size(16, 32, 8, 128, w.max_seq_len), "cuda")
    out = torch.empty_like(t.q)
    call = lambda: pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens,
                             w.max_seq_len, w.scale, out=out, workspace=ws)
    call()
    torch.cuda.synchronize()
    eager = out.clone()
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            call()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("B,hq,hkv,d", [(32, 32, 8, 128), (64, 16, 4, 64), (32, 64, 8, 128),
                                        (64, 24, 2, 128)])
def test_decode_larger_blocks(cuda_lib, oracle, B, hq, hkv, d):
    """Cache blocks of 32 and 64 tokens, both decode kernels (4 and 8-12 q heads per kv head)."""
    pa = cuda_lib
    w = wl.random_workload(120 + B + hq, num_seqs=7, max_len=900, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, block_size=B)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out = run_decode(pa, w, t)
    ref = oracle.decode(bits(t.q), bits(t.key_cache), bits(t.value_cache), w.block_tables,
                        w.seq_lens, w.scale)
    assert_close_to_oracle(out, ref, what=f"block {B} hq{hq} hkv{hkv}")


@pytest.mark.parametrize("B,k,hq", [(32, 2, 32), (64, 4, 64), (64, 2, 32)])
def test_decode_through_kernel_blocks_is_bit_identical(cuda_lib, B, k, hq):
    """Blocks of B tokens and the same memory as blocks of B / k tokens with
    the tables expanded by pa_map_to_kernel_blocks give identical bits."""
    pa = cuda_lib
    w = wl.random_workload(130 + B + k, num_seqs=9, max_len=1200, num_heads=hq, num_kv_heads=8,
                           head_dim=128, block_size=B)
    t = wl.make_tensors(w, device="cuda", poison=True)
    a = run_decode(pa, w, t)
    small = (w.num_blocks * k, B // k, w.num_kv_heads, w.head_dim)
    tables = pa.map_to_kernel_blocks(t.block_tables, k)
    b = pa.decode(t.q, t.key_cache.view(small), t.value_cache.view(small), tables, t.seq_lens,
                  w.max_seq_len, w.scale)
    assert torch.equal(a, b)
