"""GPU parity of pa_prefill_varlen (tcgen05 prefill tiles + decode rows)
against the fp64 oracle: max abs <= 1e-2, mean abs <= 1e-3 on N(0,1) inputs.

Rows are compared one by one.  For a sample of rows of a long chunk, the
oracle's reference for query i of a request with context ctx is its decode
of the same block table cut to length ctx + i + 1: by the definition of the
bottom-right causal mask that row attends exactly keys 0 .. ctx + i.
"""
import numpy as np
import pytest
import torch

from helpers import assert_close_to_oracle, bits
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def run_prefill(pa, w, t):
    ws = pa.new_workspace(pa.prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads,
                                                    w.num_kv_heads, w.head_dim, w.max_seq_len),
                          "cuda")
    out = pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens,
                            t.block_tables, w.max_query_len, w.max_seq_len, w.scale, workspace=ws)
    return out, ws


def oracle_rows(oracle, w, t, rows_per_req):
    """Oracle outputs of selected rows: {flat row: [Hq, d]}."""
    res = {}
    q = bits(t.q)
    kc, vc = bits(t.key_cache), bits(t.value_cache)
    for r, rows in rows_per_req.items():
        q0 = int(w.query_start_loc[r])
        ql = int(w.q_lens[r])
        ctx = int(w.seq_lens[r]) - ql
        sel = np.asarray(rows)
        lens = (ctx + sel + 1).astype(np.int32)
        tables = np.repeat(w.block_tables[r:r + 1], len(sel), axis=0)
        out = oracle.decode(q[q0 + sel], kc, vc, tables, lens, w.scale)
        for k, i in enumerate(sel):
            res[q0 + int(i)] = out[k]
    return res


MIXES = [
    # (seed, num_seqs, max_len, max_q_len, head_dim, q heads, kv heads)
    (201, 5, 300, 200, 128, 8, 2),
    (202, 6, 700, 260, 128, 32, 8),
    (203, 4, 150, 150, 64, 4, 2),
    (204, 7, 520, 300, 128, 16, 16),
    (205, 3, 400, 400, 128, 8, 1),
    (206, 5, 290, 130, 64, 16, 2),
    (209, 4, 400, 200, 128, 32, 2),
]


@pytest.mark.parametrize("seed,ns,max_len,max_q,d,hq,hkv", MIXES)
def test_prefill_varlen_random_mixes(cuda_lib, oracle, seed, ns, max_len, max_q, d, hq, hkv):
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, max_q_len=max_q, prefill_fraction=0.7)
    assert w.max_query_len > 1
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what=f"mix {seed}")


@pytest.mark.parametrize("q_len,ctx", [(2, 0), (2, 37), (127, 0), (128, 0), (129, 5), (256, 16),
                                       (300, 1000), (16, 15), (17, 2047)])
def test_prefill_tile_edges(cuda_lib, oracle, q_len, ctx):
    """Chunks at and around the 128-row tile and 16-token block edges, with
    and without cached context, next to a decode row."""
    pa = cuda_lib
    lens = [ctx + q_len, 77]
    w = wl.build_workload("edge", lens, [q_len, 1], num_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, num_blocks=1 + sum(-(-x // 16) for x in lens) + 4, seed=q_len)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what=f"q_len {q_len} ctx {ctx}")


def test_prefill_nan_poison_does_not_change_output(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(207, num_seqs=4, max_len=400, num_heads=8, num_kv_heads=2,
                           head_dim=128, max_q_len=200, prefill_fraction=1.0, spare_blocks=12)
    clean = wl.make_tensors(w, device="cuda")
    dirty = wl.make_tensors(w, device="cuda", poison=True)
    a, _ = run_prefill(pa, w, clean)
    b, _ = run_prefill(pa, w, dirty)
    assert torch.isfinite(b.float()).all()
    assert torch.equal(a, b)


def test_mixed_chunked_prefill_full_size(cuda_lib, oracle):
    """The 512-token chunk at context 3584 plus 63 decode rows: write all 575
    new tokens through the slot mapping, then attend; compare every decode
    row and a sample of the chunk's rows (all heads) with the oracle."""
    pa = cuda_lib
    w = wl.mixed_chunked_prefill()
    t = wl.make_tensors(w, device="cuda", poison=True)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache, slots)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    chunk_rows = sorted(set([0, 1, 2, 15, 16, 127, 128, 129, 255, 256, 383, 384, 510, 511]) |
                        set(range(3, 512, 37)))
    rows = {0: chunk_rows}
    for r in range(1, w.num_seqs):
        rows[r] = [0]
    ref = oracle_rows(oracle, w, t, rows)
    flat = sorted(ref)
    got = out[torch.tensor(flat, device="cuda")]
    assert_close_to_oracle(got, np.stack([ref[k] for k in flat]), what="mixed chunked prefill")


def test_prefill_without_context_is_causal_self_attention(cuda_lib, oracle):
    """q_len == seq_len: a whole prompt attends to itself causally."""
    pa = cuda_lib
    w = wl.build_workload("prompt", [333], [333], num_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=16, num_blocks=30, seed=9)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, _ = run_prefill(pa, w, t)
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what="prompt")


def test_prefill_is_deterministic(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(208, num_seqs=5, max_len=600, num_heads=32, num_kv_heads=8,
                           head_dim=128, max_q_len=300, prefill_fraction=0.6)
    t = wl.make_tensors(w, device="cuda")
    a, _ = run_prefill(pa, w, t)
    b, _ = run_prefill(pa, w, t)
    assert torch.equal(a, b)


def test_prefill_zero_length_requests_produce_nothing(cuda_lib, oracle):
    """Requests with q_len == 0 own no rows; the others are unaffected."""
    pa = cuda_lib
    lens, qls = [50, 90, 33, 200], [0, 40, 0, 1]
    w = wl.build_workload("zero", lens, qls, num_heads=8, num_kv_heads=2, head_dim=64,
                          block_size=16, num_blocks=40, seed=3)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what="zero-length requests")


def test_prefill_bad_block_id_is_reported_not_dereferenced(cuda_lib, oracle):
    pa = cuda_lib
    lens, qls = [300, 120, 77], [200, 1, 60]
    w = wl.build_workload("badblk", lens, qls, num_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, num_blocks=40, seed=4)
    t = wl.make_tensors(w, device="cuda")
    bt = t.block_tables.clone()
    bt[0, 3] = w.num_blocks + 77  # a block the chunk of request 0 reads
    ws = pa.new_workspace(pa.prefill_workspace_size(3, w.total_q, 8, 2, 128, w.max_seq_len), "cuda")
    out = pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens, bt,
                            w.max_query_len, w.max_seq_len, w.scale, workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 2 and st[1] == 0 and st[2] == w.num_blocks + 77
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    rows = slice(int(w.query_start_loc[1]), int(w.query_start_loc[3]))  # requests 1 and 2
    assert_close_to_oracle(out[rows], ref[rows], what="other requests")


def test_prefill_query_longer_than_context_is_reported(cuda_lib):
    pa = cuda_lib
    w = wl.build_workload("qlong", [64, 40], [30, 1], num_heads=4, num_kv_heads=2, head_dim=64,
                          block_size=16, num_blocks=12, seed=5)
    t = wl.make_tensors(w, device="cuda")
    sl = t.seq_lens.clone()
    sl[0] = 20  # fewer keys than the request's 30 new queries
    ws = pa.new_workspace(pa.prefill_workspace_size(2, w.total_q, 4, 2, 64, w.max_seq_len), "cuda")
    pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, sl, t.block_tables,
                      w.max_query_len, w.max_seq_len, w.scale, workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 4 and st[1] == 0


def test_mixed_step_in_a_cuda_graph(cuda_lib):
    """Slot mapping, cache write and pa_prefill_varlen captured in one CUDA
    graph (after an eager warm-up) replay to the eager result."""
    pa = cuda_lib
    w = wl.random_workload(209, num_seqs=6, max_len=500, num_heads=32, num_kv_heads=8,
                           head_dim=128, max_q_len=200, prefill_fraction=0.5)
    t = wl.make_tensors(w, device="cuda")
    kc0, vc0 = t.key_cache.clone(), t.value_cache.clone()
    ws = pa.new_workspace(pa.prefill_workspace_size(w.num_seqs, w.total_q, 32, 8, 128,
                                                    w.max_seq_len), "cuda")
    out = torch.empty_like(t.q)
    slots = torch.empty(w.total_q, dtype=torch.int64, device="cuda")

    def step():
        pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16, w.num_blocks,
                                w.total_q, out=slots)
        pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache, slots)
        pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens,
                          t.block_tables, w.max_query_len, w.max_seq_len, w.scale, out=out,
                          workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    t.key_cache.copy_(kc0)
    t.value_cache.copy_(vc0)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            step()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("B,seed", [(32, 211), (64, 212)])
def test_prefill_larger_blocks(cuda_lib, oracle, B, seed):
    """Chunked prefill and decode rows over 32- and 64-token cache blocks."""
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=6, max_len=700, num_heads=16, num_kv_heads=4,
                           head_dim=128, block_size=B, max_q_len=300, prefill_fraction=0.6)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what=f"prefill block {B}")


def test_multi_chunk_prefill_full_size(cuda_lib, oracle):
    """Four long chunks (1344 query tiles, several per CTA of the persistent
    grid) plus decode rows; every decode row and a sample of each chunk's
    rows against the oracle."""
    pa = cuda_lib
    w = wl.multi_chunk_prefill()
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    rows = {}
    for r in range(w.num_seqs):
        ql = int(w.q_lens[r])
        rows[r] = sorted({0, 1, 127, 128, ql // 2, ql - 2, ql - 1}) if ql > 1 else [0]
    ref = oracle_rows(oracle, w, t, rows)
    flat = sorted(ref)
    got = out[torch.tensor(flat, device="cuda")]
    assert_close_to_oracle(got, np.stack([ref[k] for k in flat]), what="multi-chunk prefill")
