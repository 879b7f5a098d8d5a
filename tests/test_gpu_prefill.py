"""GPU parity of pa_prefill_varlen (tcgen05 prefill tiles + decode rows)
against the fp64 oracle: max abs <= 1e-2, mean abs <= 1e-3 on N(0,1) inputs.

Every row and head is compared, the full-size batches included (the oracle
runs its independent rows on all host cores).
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


@pytest.mark.parametrize("seed,n_pref,n_dec,dec_len", [
    (241, 1, 120, 3000),  # decode rows dominate: the tiles keep a few SMs
    (242, 6, 2, 64),      # tiles dominate: the decode rows go to one CTA
    (243, 3, 40, 1500),   # in between
])
def test_mixed_batches_split_the_sms(cuda_lib, oracle, seed, n_pref, n_dec, dec_len):
    """Mixed batches large enough for the decode grid to fill every SM, so
    that the tile and decode kernels split the SMs between them, at several
    ratios of tile to decode work; prefill chunks and decode rows
    interleaved; every row against the oracle."""
    pa = cuda_lib
    rng = np.random.default_rng(seed)
    pq = [int(x) for x in rng.integers(130, 300, n_pref)]
    lens = [int(c) + q for c, q in zip(rng.integers(0, 900, n_pref), pq)]
    lens += [int(x) for x in rng.integers(dec_len // 2, dec_len, n_dec)]
    q_lens = pq + [1] * n_dec
    order = rng.permutation(len(lens))
    lens = [lens[i] for i in order]
    q_lens = [q_lens[i] for i in order]
    w = wl.build_workload("split", lens, q_lens, num_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, num_blocks=sum(-(-x // 16) for x in lens) + 8, seed=seed)
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what=f"split {seed}")
    again, _ = run_prefill(pa, w, t)
    assert torch.equal(out, again)


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
    new tokens through the slot mapping, then attend; compare every row and
    head with the oracle."""
    pa = cuda_lib
    w = wl.mixed_chunked_prefill()
    t = wl.make_tensors(w, device="cuda", poison=True)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    pa.reshape_and_cache(t.key, t.value, t.key_cache, t.value_cache, slots)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what="mixed chunked prefill (every row)")


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
    grid) plus decode rows; every row and head against the oracle."""
    pa = cuda_lib
    w = wl.multi_chunk_prefill()
    t = wl.make_tensors(w, device="cuda", poison=True)
    out, ws = run_prefill(pa, w, t)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what="multi-chunk prefill (every row)")


def _mixed_case(seed):
    w = wl.random_workload(seed, num_seqs=7, max_len=900, num_heads=32, num_kv_heads=8,
                           head_dim=128, max_q_len=400, prefill_fraction=0.5)
    assert w.max_query_len > 1 and (w.q_lens == 1).any()
    return w, wl.make_tensors(w, device="cuda", poison=True)


def test_two_mixed_calls_run_concurrently_on_two_caller_streams(cuda_lib, oracle):
    """pa_prefill_varlen enqueues on the caller's stream only: two calls on
    two streams, each with its own workspace and output, may run at the same
    time, and each equals the oracle.  The calls are enqueued alternately,
    several times, with no ordering between the streams."""
    pa = cuda_lib
    cases = [_mixed_case(231), _mixed_case(232)]
    refs = [oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                  w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
            for w, t in cases]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss, outs = [], []
    for w, t in cases:
        wss.append(pa.new_workspace(pa.prefill_workspace_size(
            w.num_seqs, w.total_q, w.num_heads, w.num_kv_heads, w.head_dim, w.max_seq_len),
            "cuda"))
        outs.append(torch.full_like(t.q, float("nan")))
    torch.cuda.synchronize()
    for _ in range(4):
        for (w, t), s, ws, out in zip(cases, streams, wss, outs):
            with torch.cuda.stream(s):
                pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens,
                                  t.block_tables, w.max_query_len, w.max_seq_len, w.scale, out=out,
                                  workspace=ws)
    torch.cuda.synchronize()
    for k, ((w, t), ws, out, ref) in enumerate(zip(cases, wss, outs, refs)):
        assert pa.device_status(ws)[0] == 0
        assert_close_to_oracle(out, ref, what=f"stream {k}")


def test_batch_order_does_not_change_a_requests_rows(cuda_lib, oracle):
    """The same requests in another order (block tables, lengths and query
    rows permuted together; the cache unchanged) give every request the same
    rows up to rounding.  Both kernels split the batch's work over the CTAs
    by position in the whole batch, so where a request's keys are cut into
    merged pieces moves with the order: each order is compared with the
    oracle, and the two orders with each other, within the bf16 tolerance."""
    pa = cuda_lib
    w, t = _mixed_case(233)
    out_a, ws = run_prefill(pa, w, t)
    perm = np.array([4, 0, 6, 2, 5, 1, 3])
    qls = w.q_lens[perm]
    qsl = np.concatenate([[0], np.cumsum(qls)]).astype(np.int32)
    rows = np.concatenate([np.arange(w.query_start_loc[r], w.query_start_loc[r + 1]) for r in perm])
    wp = wl.Workload(w.name + "_perm", w.seq_lens[perm], qls, qsl, w.block_tables[perm],
                     w.num_heads, w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.scale,
                     w.seed, w.shared_blocks)
    tp = wl.Tensors(q=t.q[torch.from_numpy(rows).cuda()].contiguous(), key=t.key, value=t.value,
                    key_cache=t.key_cache, value_cache=t.value_cache,
                    block_tables=t.block_tables[torch.from_numpy(perm).cuda()].contiguous(),
                    seq_lens=t.seq_lens[torch.from_numpy(perm).cuda()].contiguous(),
                    query_start_loc=torch.from_numpy(qsl).cuda())
    out_b, ws_b = run_prefill(pa, wp, tp)
    assert pa.device_status(ws)[0] == 0 and pa.device_status(ws_b)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    for k, r in enumerate(perm):
        a = out_a[int(w.query_start_loc[r]):int(w.query_start_loc[r + 1])]
        b = out_b[int(qsl[k]):int(qsl[k + 1])]
        rr = ref[int(w.query_start_loc[r]):int(w.query_start_loc[r + 1])]
        assert_close_to_oracle(a, rr, what=f"request {r}, batch order")
        assert_close_to_oracle(b, rr, what=f"request {r}, permuted order")
        assert_close_to_oracle(b, a.double().cpu().numpy(), what=f"request {r}, the two orders")


@pytest.mark.parametrize("q_len,ctx,hq,hkv,d", [(256, 2000, 2, 1, 128), (200, 3000, 3, 1, 64),
                                                (130, 700, 4, 2, 128), (2, 5000, 2, 2, 128)])
def test_prefill_unit_split_over_many_ctas(cuda_lib, oracle, q_len, ctx, hq, hkv, d):
    """A batch with few key steps against a grid of one CTA per SM: each
    128-row unit is cut into pieces of one or two steps held by many CTAs,
    whose partials the last contributor merges (directly from tensor memory
    when every other piece has already counted, else from the published
    partials); an odd group leaves a single-head unit."""
    pa = cuda_lib
    lens = [ctx + q_len, 90]
    w = wl.build_workload("split", lens, [q_len, 1], num_heads=hq, num_kv_heads=hkv, head_dim=d,
                          block_size=16, num_blocks=1 + sum(-(-x // 16) for x in lens) + 4,
                          seed=q_len + ctx)
    t = wl.make_tensors(w, device="cuda", poison=True)
    for _ in range(2):  # the second call reuses the workspace (counters left at zero)
        out, ws = run_prefill(pa, w, t)
        assert pa.device_status(ws)[0] == 0
    ref = oracle.prefill_varlen(bits(t.q), bits(t.key_cache), bits(t.value_cache),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    assert_close_to_oracle(out, ref, what=f"split q_len {q_len} ctx {ctx} heads {hq}/{hkv}")
