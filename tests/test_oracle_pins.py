"""Pins of the fp64 oracle against what the pages and the mathematics fix.

Nothing here touches the CUDA library.  Each check compares the oracle with
something other than itself: a value printed on the pages (tests/golden/),
a library routine (scipy's softmax, torch's fp64 scaled_dot_product_attention
on the CPU), a closed form, or an invariance the definition implies.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

from conftest import read_golden
from paged_kv_cache_74_gb300 import workloads as wl


def _ints(s):
    return [int(x) for x in s.split()]


# --------------------------------------------------------------- addressing

def test_slot_examples_printed_on_pages(oracle):
    rows = read_golden("slot_examples.txt")
    assert len(rows) >= 2
    for bs, table, pos, slot, _src in rows:
        assert oracle.slot(_ints(table), int(bs), int(pos)) == int(slot)


def test_query_start_loc_printed_on_pages(oracle):
    for q_lens, qsl, _src in read_golden("query_start_loc.txt"):
        assert oracle.query_start_loc(_ints(q_lens)).tolist() == _ints(qsl)


def test_varlen_positions_of_mixed_batch(oracle):
    """With an identity block table a slot equals its token position, so the
    slot mapping exposes which positions the oracle gives the new tokens."""
    rows = read_golden("varlen_positions.txt")
    q_lens = [int(r[1]) for r in rows]
    seq_lens = np.array([int(r[2]) for r in rows], np.int32)
    qsl = oracle.query_start_loc(q_lens)
    B = 16
    nb = -(-int(seq_lens.max()) // B)
    table = np.tile(np.arange(nb, dtype=np.int32), (len(rows), 1))
    slots = oracle.slot_mapping(table, qsl, seq_lens, B)
    for r, row in enumerate(rows):
        got = slots[qsl[r]:qsl[r + 1]]
        assert got[0] == int(row[3]) and got[-1] == int(row[4])
        assert np.all(np.diff(got) == 1)


def test_slot_mapping_matches_printed_walkthrough(oracle):
    """Req1 (25 tokens in P3, P7) and Req2 (12 tokens in P1), one new token
    each: their slots are 7*16+8 and 1*16+11."""
    table = np.array([[3, 7], [1, 0]], np.int32)
    qsl = oracle.query_start_loc([1, 1])
    slots = oracle.slot_mapping(table, qsl, np.array([25, 12], np.int32), 16)
    assert slots.tolist() == [120, 27]


def test_kv_bytes_formula_printed_on_pages(oracle):
    for shape, per_tok, tokens, total, _src in read_golden("kv_bytes.txt"):
        L, hkv, d, b = _ints(shape)
        got = oracle.kv_bytes_per_token(L, hkv, d, b)
        assert got == int(per_tok)
        assert got * int(tokens) == int(total)


# ----------------------------------------------------------- softmax algebra

def _direct(s, v):
    return scipy.special.softmax(s) @ v


@pytest.mark.parametrize("split", ["one", "block16", "part512", "random", "whole"])
def test_online_softmax_equals_direct(oracle, split):
    rng = np.random.default_rng(11)
    n, dv = 1500, 64
    s = rng.standard_normal(n) * 3.0
    s[700] = 40.0  # a late large score forces a rescale of the running state
    v = rng.standard_normal((n, dv))
    if split == "one":
        bounds = np.arange(n + 1)
    elif split == "block16":
        bounds = np.append(np.arange(0, n, 16), n)
    elif split == "part512":
        bounds = np.append(np.arange(0, n, 512), n)
    elif split == "random":
        cuts = np.sort(rng.choice(np.arange(1, n), size=37, replace=False))
        bounds = np.concatenate([[0], cuts, [n]])
    else:
        bounds = np.array([0, n])
    out, m, l = oracle.online_softmax(s, v, bounds)
    np.testing.assert_allclose(out, _direct(s, v), rtol=0, atol=1e-12)
    assert m == s.max()
    np.testing.assert_allclose(l, np.exp(s - s.max()).sum(), rtol=1e-13)


def test_partition_merge_equals_global_softmax(oracle):
    rng = np.random.default_rng(12)
    n, dv, P = 2000, 32, 512
    s = rng.standard_normal(n) * 4.0
    v = rng.standard_normal((n, dv))
    ms, ls, os_ = [], [], []
    for lo in range(0, n, P):
        sp, vp = s[lo:lo + P], v[lo:lo + P]
        ms.append(sp.max())
        ls.append(np.exp(sp - sp.max()).sum())
        os_.append(_direct(sp, vp))
    out = oracle.merge_partitions(np.array(ms), np.array(ls), np.array(os_))
    np.testing.assert_allclose(out, _direct(s, v), rtol=0, atol=1e-12)


def test_partition_merge_single_partition_is_identity(oracle):
    o = np.arange(8.0)[None, :]
    out = oracle.merge_partitions(np.array([3.0]), np.array([2.5]), o)
    np.testing.assert_array_equal(out, o[0])


# --------------------------------------------------------------- attention

def _contiguous_workload(seq_lens, hq, hkv, d, seed, q_lens=None, B=16):
    """Each request owns consecutive physical blocks, so its keys form one
    contiguous range of the pool viewed as [slots, kv_heads, d]."""
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.ones_like(seq_lens) if q_lens is None else np.asarray(q_lens, np.int32)
    need = -(-seq_lens // B)
    tables = np.zeros((len(seq_lens), int(need.max())), np.int32)
    starts = np.concatenate([[1], 1 + np.cumsum(need)[:-1]])
    for r in range(len(seq_lens)):
        tables[r, :need[r]] = np.arange(starts[r], starts[r] + need[r])
    w = wl.build_workload("contig", seq_lens, q_lens, num_heads=hq, num_kv_heads=hkv,
                          head_dim=d, block_size=B, num_blocks=1 + int(need.sum()), seed=seed)
    w.block_tables = tables
    return w, starts * B


def _sdpa(q, k, v, scale, mask=None):
    """torch fp64 CPU attention; q [Hq, n_q, d], k/v [Hkv, n_k, d] (GQA by
    repeating each kv head for its group of consecutive q heads)."""
    g = q.shape[0] // k.shape[0]
    k = k.repeat_interleave(g, dim=0)
    v = v.repeat_interleave(g, dim=0)
    return torch.nn.functional.scaled_dot_product_attention(
        q[None], k[None], v[None], attn_mask=mask, scale=scale)[0]


@pytest.mark.parametrize("hq,hkv,d,lens,B", [(4, 2, 64, [25, 12, 37, 20], 16),
                                             (8, 1, 128, [1, 16, 17, 100], 16),
                                             (6, 6, 64, [3, 48], 16),
                                             (16, 2, 128, [129, 33], 16),
                                             (8, 2, 64, [31, 64, 70], 32),
                                             (4, 4, 128, [1, 65, 200], 64)])
def test_decode_matches_torch_sdpa(oracle, hq, hkv, d, lens, B):
    w, first_slot = _contiguous_workload(lens, hq, hkv, d, seed=21, B=B)
    t = wl.make_tensors(w)
    out = oracle.decode(t.q.view(torch.int16).numpy(), t.key_cache.view(torch.int16).numpy(),
                        t.value_cache.view(torch.int16).numpy(), w.block_tables, w.seq_lens,
                        w.scale)
    kf = t.key_cache.double().reshape(-1, hkv, d)
    vf = t.value_cache.double().reshape(-1, hkv, d)
    for r, L in enumerate(lens):
        k = kf[first_slot[r]:first_slot[r] + L].permute(1, 0, 2)
        v = vf[first_slot[r]:first_slot[r] + L].permute(1, 0, 2)
        ref = _sdpa(t.q[r].double()[:, None, :], k, v, w.scale)[:, 0, :]
        np.testing.assert_allclose(out[r], ref.numpy(), rtol=0, atol=1e-12)


def test_decode_single_token_returns_its_value(oracle):
    w, first = _contiguous_workload([1, 1], 4, 2, 64, seed=22)
    t = wl.make_tensors(w)
    out = oracle.decode(t.q.view(torch.int16).numpy(), t.key_cache.view(torch.int16).numpy(),
                        t.value_cache.view(torch.int16).numpy(), w.block_tables, w.seq_lens,
                        w.scale)
    for r in range(2):
        v0 = t.value_cache.double().reshape(-1, 2, 64)[first[r]]
        np.testing.assert_array_equal(out[r], v0.repeat_interleave(2, dim=0).numpy())


def test_decode_identical_keys_average_values(oracle):
    w, first = _contiguous_workload([37], 2, 1, 64, seed=23)
    t = wl.make_tensors(w)
    kc = t.key_cache.clone()
    kc[:] = kc[1, 0]  # every key equal -> uniform weights
    out = oracle.decode(t.q.view(torch.int16).numpy(), kc.view(torch.int16).numpy(),
                        t.value_cache.view(torch.int16).numpy(), w.block_tables, w.seq_lens,
                        w.scale)
    vals = t.value_cache.double().reshape(-1, 1, 64)[first[0]:first[0] + 37, 0]
    np.testing.assert_allclose(out[0, 0], vals.mean(0).numpy(), rtol=0, atol=1e-13)


def test_decode_relocation_invariance(oracle):
    """Moving physical blocks (and their contents) leaves outputs unchanged."""
    w = wl.tiny_decode()
    t = wl.make_tensors(w)
    args = lambda kc, vc, bt: oracle.decode(t.q.view(torch.int16).numpy(),
                                           kc.view(torch.int16).numpy(),
                                           vc.view(torch.int16).numpy(), bt, w.seq_lens, w.scale)
    base = args(t.key_cache, t.value_cache, w.block_tables)
    perm = np.random.default_rng(5).permutation(w.num_blocks)  # new id of each block
    kc2 = torch.empty_like(t.key_cache)
    vc2 = torch.empty_like(t.value_cache)
    kc2[torch.from_numpy(perm)] = t.key_cache
    vc2[torch.from_numpy(perm)] = t.value_cache
    moved = args(kc2, vc2, perm[w.block_tables].astype(np.int32))
    np.testing.assert_array_equal(base, moved)


def test_prefill_matches_torch_sdpa_bottom_right_causal(oracle):
    lens, qls = [40, 33, 16, 70], [7, 1, 16, 70]
    hq, hkv, d = 4, 2, 64
    w, first = _contiguous_workload(lens, hq, hkv, d, seed=24, q_lens=qls)
    t = wl.make_tensors(w)
    out = oracle.prefill_varlen(t.q.view(torch.int16).numpy(),
                                t.key_cache.view(torch.int16).numpy(),
                                t.value_cache.view(torch.int16).numpy(), w.query_start_loc,
                                w.seq_lens, w.block_tables, w.scale)
    kf = t.key_cache.double().reshape(-1, hkv, d)
    vf = t.value_cache.double().reshape(-1, hkv, d)
    for r, (L, ql) in enumerate(zip(lens, qls)):
        k = kf[first[r]:first[r] + L].permute(1, 0, 2)
        v = vf[first[r]:first[r] + L].permute(1, 0, 2)
        q = t.q[w.query_start_loc[r]:w.query_start_loc[r + 1]].double().permute(1, 0, 2)
        # bottom-right causal: query i (of ql) may see keys j <= L - ql + i
        i = torch.arange(ql)[:, None]
        j = torch.arange(L)[None, :]
        mask = j <= (L - ql) + i
        ref = _sdpa(q, k, v, w.scale, mask=mask).permute(1, 0, 2)
        np.testing.assert_allclose(out[w.query_start_loc[r]:w.query_start_loc[r + 1]],
                                   ref.numpy(), rtol=0, atol=1e-12)


def test_prefill_square_chunk_is_plain_causal(oracle):
    """With no cached context (q_len == seq_len) the mask is the usual
    top-left causal one, which torch builds itself with is_causal."""
    w, first = _contiguous_workload([48], 2, 2, 64, seed=25, q_lens=[48])
    t = wl.make_tensors(w)
    out = oracle.prefill_varlen(t.q.view(torch.int16).numpy(),
                                t.key_cache.view(torch.int16).numpy(),
                                t.value_cache.view(torch.int16).numpy(), w.query_start_loc,
                                w.seq_lens, w.block_tables, w.scale)
    k = t.key_cache.double().reshape(-1, 2, 64)[first[0]:first[0] + 48].permute(1, 0, 2)
    v = t.value_cache.double().reshape(-1, 2, 64)[first[0]:first[0] + 48].permute(1, 0, 2)
    q = t.q.double().permute(1, 0, 2)
    ref = torch.nn.functional.scaled_dot_product_attention(q[None], k[None], v[None],
                                                           is_causal=True, scale=w.scale)[0]
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_prefill_decode_rows_equal_decode(oracle):
    w = wl.tiny_decode()
    t = wl.make_tensors(w)
    a = oracle.decode(t.q.view(torch.int16).numpy(), t.key_cache.view(torch.int16).numpy(),
                      t.value_cache.view(torch.int16).numpy(), w.block_tables, w.seq_lens,
                      w.scale)
    b = oracle.prefill_varlen(t.q.view(torch.int16).numpy(),
                              t.key_cache.view(torch.int16).numpy(),
                              t.value_cache.view(torch.int16).numpy(), w.query_start_loc,
                              w.seq_lens, w.block_tables, w.scale)
    np.testing.assert_array_equal(a, b)


def test_decode_ignores_nan_outside_context(oracle):
    """Out-of-context slots, the null block and free blocks may hold NaN."""
    w = wl.tiny_decode()
    clean = wl.make_tensors(w)
    dirty = wl.make_tensors(w, poison=True)
    assert torch.isnan(dirty.key_cache.float()).any()
    run = lambda t: oracle.decode(t.q.view(torch.int16).numpy(),
                                  t.key_cache.view(torch.int16).numpy(),
                                  t.value_cache.view(torch.int16).numpy(), w.block_tables,
                                  w.seq_lens, w.scale)
    np.testing.assert_array_equal(run(clean), run(dirty))


# ------------------------------------------------------------ slot writer

def test_reshape_and_cache_scatter(oracle):
    """Identity tables make slot == position, so token i must land in row
    slot of the pool viewed as [num_blocks * block_size, kv_heads, d]; all
    other rows, and tokens with a negative slot, leave the pool untouched."""
    w = wl.tiny_decode()
    t = wl.make_tensors(w)
    n = 6
    gen = torch.Generator().manual_seed(3)
    key = torch.randn((n, 2, 64), generator=gen).to(torch.bfloat16)
    val = torch.randn((n, 2, 64), generator=gen).to(torch.bfloat16)
    slots = np.array([5, 100, -1, 511, 17, -3], np.int64)
    kc, vc = oracle.reshape_and_cache(key.view(torch.int16).numpy(), val.view(torch.int16).numpy(),
                                      t.key_cache.view(torch.int16).numpy(),
                                      t.value_cache.view(torch.int16).numpy(), slots)
    kc0 = t.key_cache.view(torch.int16).numpy().view(np.uint16).reshape(-1, 2, 64)
    vc0 = t.value_cache.view(torch.int16).numpy().view(np.uint16).reshape(-1, 2, 64)
    kc, vc = kc.reshape(-1, 2, 64), vc.reshape(-1, 2, 64)
    written = {int(s): i for i, s in enumerate(slots) if s >= 0}
    for s in range(kc.shape[0]):
        if s in written:
            i = written[s]
            np.testing.assert_array_equal(kc[s], key[i].view(torch.int16).numpy().view(np.uint16))
            np.testing.assert_array_equal(vc[s], val[i].view(torch.int16).numpy().view(np.uint16))
        else:
            np.testing.assert_array_equal(kc[s], kc0[s])
            np.testing.assert_array_equal(vc[s], vc0[s])


def test_reshape_and_cache_skips_slots_past_the_pool(oracle):
    """A slot at or past num_blocks * block_size names no cache row: the
    writer must leave every byte alone, including memory just past the pool
    (the C function is handed a larger buffer and told the pool is smaller,
    so a missing check writes into the spare rows instead of out of bounds)."""
    import ctypes
    nb_real, nb_told, B, H, d = 6, 4, 16, 2, 8
    gen = np.random.default_rng(11)
    key = gen.integers(0, 1 << 16, (4, H, d), dtype=np.uint16)
    val = gen.integers(0, 1 << 16, (4, H, d), dtype=np.uint16)
    kc = gen.integers(0, 1 << 16, (nb_real, B, H, d), dtype=np.uint16)
    vc = gen.integers(0, 1 << 16, (nb_real, B, H, d), dtype=np.uint16)
    kc0, vc0 = kc.copy(), vc.copy()
    slots = np.array([nb_told * B, nb_told * B + 17, 3, nb_told * B - 1], np.int64)
    u16 = ctypes.POINTER(ctypes.c_uint16)
    i64 = ctypes.POINTER(ctypes.c_int64)
    oracle.lib.oracle_reshape_and_cache(key.ctypes.data_as(u16), val.ctypes.data_as(u16), 4, H, d,
                                        kc.ctypes.data_as(u16), vc.ctypes.data_as(u16), nb_told, B,
                                        slots.ctypes.data_as(i64))
    kf, vf, kf0, vf0 = (a.reshape(-1, H, d) for a in (kc, vc, kc0, vc0))
    for s in range(nb_real * B):
        if s == 3 or s == nb_told * B - 1:
            i = 2 if s == 3 else 3
            np.testing.assert_array_equal(kf[s], key[i])
            np.testing.assert_array_equal(vf[s], val[i])
        else:
            np.testing.assert_array_equal(kf[s], kf0[s])
            np.testing.assert_array_equal(vf[s], vf0[s])


def test_reshape_then_slot_mapping_places_token_where_decode_reads_it(oracle):
    """Writing each request's last token through the slot mapping and then
    decoding is the same as decoding a pool that already held those keys."""
    w = wl.tiny_decode()
    t = wl.make_tensors(w)
    slots = oracle.slot_mapping(w.block_tables, w.query_start_loc, w.seq_lens, w.block_size)
    kc, vc = oracle.reshape_and_cache(t.key.view(torch.int16).numpy(),
                                      t.value.view(torch.int16).numpy(),
                                      t.key_cache.view(torch.int16).numpy(),
                                      t.value_cache.view(torch.int16).numpy(), slots)
    for r in range(w.num_seqs):
        L = int(w.seq_lens[r])
        phys = w.block_tables[r, (L - 1) // 16]
        np.testing.assert_array_equal(kc[phys, (L - 1) % 16],
                                      t.key[r].view(torch.int16).numpy().view(np.uint16))


# ------------------------------------------------------- kernel block ids

def test_kernel_blocks_printed_on_pages(oracle):
    for ids, k, expect, _src in read_golden("kernel_blocks.txt"):
        got = oracle.map_to_kernel_blocks(np.array([int(x) for x in ids.split(",")]), int(k))
        np.testing.assert_array_equal(got, [int(x) for x in expect.split(",")])


def test_kernel_blocks_identity_and_padding(oracle):
    ids = np.array([[7, 3, -1, -1], [0, 12, 5, -1]], np.int32)
    np.testing.assert_array_equal(oracle.map_to_kernel_blocks(ids, 1), ids)
    got = oracle.map_to_kernel_blocks(ids, 4)
    assert got.shape == (2, 16)
    np.testing.assert_array_equal(got[0, :8], [28, 29, 30, 31, 12, 13, 14, 15])
    assert (got[0, 8:] == -1).all() and (got[1, 12:] == -1).all()
    # each kernel id names a distinct 1/k of its manager block
    np.testing.assert_array_equal(got[1, :12] // 4, np.repeat([0, 12, 5], 4))
    np.testing.assert_array_equal(got[1, :12] % 4, np.tile(np.arange(4), 3))


@pytest.mark.parametrize("B,k", [(32, 2), (64, 4), (64, 2)])
def test_block_size_views_agree(oracle, B, k):
    """A cache of nb blocks of B tokens is the memory of nb * k blocks of
    B / k tokens; attention through the expanded tables must match exactly."""
    w = wl.random_workload(31 + B + k, num_seqs=5, max_len=300, num_heads=8, num_kv_heads=2,
                           head_dim=64, block_size=B, max_q_len=40, prefill_fraction=0.6)
    t = wl.make_tensors(w)
    q = t.q.view(torch.int16).numpy()
    kc = t.key_cache.view(torch.int16).numpy()
    vc = t.value_cache.view(torch.int16).numpy()
    small = (w.num_blocks * k, B // k, w.num_kv_heads, w.head_dim)
    tables_k = oracle.map_to_kernel_blocks(w.block_tables, k)
    dec = oracle.decode(q[w.query_start_loc[1:] - 1], kc, vc, w.block_tables, w.seq_lens, w.scale)
    dec_k = oracle.decode(q[w.query_start_loc[1:] - 1], kc.reshape(small), vc.reshape(small),
                          tables_k, w.seq_lens, w.scale)
    np.testing.assert_array_equal(dec, dec_k)
    pre = oracle.prefill_varlen(q, kc, vc, w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    pre_k = oracle.prefill_varlen(q, kc.reshape(small), vc.reshape(small), w.query_start_loc,
                                  w.seq_lens, tables_k, w.scale)
    np.testing.assert_array_equal(pre, pre_k)


# ------------------------------------------------------------ FP8 (e4m3)

def test_e4m3_codes_decode_like_torch(oracle):
    codes = np.arange(256, dtype=np.uint8)
    mine = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(np.isnan(mine), np.isnan(ref))
    np.testing.assert_array_equal(mine[~np.isnan(mine)], ref[~np.isnan(ref)])
    assert np.nanmax(mine) == 448.0 and mine[0x01] == 2.0 ** -9 and mine[0x08] == 2.0 ** -6


def test_e4m3_encode_matches_torch_in_range(oracle):
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    finite = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = (finite[1:] + finite[:-1]) / 2  # every tie between neighbours
    rng = np.random.default_rng(8)
    probe = np.concatenate([finite, mids, rng.uniform(-463.9, 463.9, 4000),
                            rng.standard_normal(2000) * 1e-2]).astype(np.float32)
    probe = probe[np.abs(probe) < 464]
    ref = torch.from_numpy(probe).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle.e4m3_encode(probe), ref)


def test_e4m3_encode_saturates_and_keeps_nan(oracle):
    got = oracle.e4m3_encode(np.array([464.0, 1e6, np.inf, -464.0, -3e38, np.nan], np.float32))
    np.testing.assert_array_equal(got, [0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F])


def test_e4m3_encode_inverts_decode(oracle):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    np.testing.assert_array_equal(oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32)),
                                  codes)


def _fp8_workload(seed):
    w = wl.random_workload(seed, num_seqs=5, max_len=180, num_heads=8, num_kv_heads=2, head_dim=64)
    t = wl.make_tensors(w)
    rng = np.random.default_rng(seed)
    kc8 = rng.integers(0, 256, size=t.key_cache.shape, dtype=np.uint8)
    vc8 = rng.integers(0, 256, size=t.value_cache.shape, dtype=np.uint8)
    for c in (kc8, vc8):  # no NaN codes
        c[(c & 0x7F) == 0x7F] = 0x3C
    return w, t, kc8, vc8


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.25, 4.0), (2.0 ** -7, 2.0 ** 5)])
def test_decode_fp8_equals_decode_of_dequantized_cache(oracle, k_scale, v_scale):
    """With power-of-two scales every dequantized value is a bf16 value, so
    the FP8 decode must equal the (separately pinned) bf16 decode exactly."""
    w, t, kc8, vc8 = _fp8_workload(61)
    deq = lambda c, s: torch.from_numpy(oracle.e4m3_decode(c) * s).to(torch.bfloat16)
    kb, vb = deq(kc8, k_scale), deq(vc8, v_scale)
    assert torch.equal(kb.double(), torch.from_numpy(oracle.e4m3_decode(kc8) * k_scale))
    q = t.q.view(torch.int16).numpy()
    ref = oracle.decode(q, kb.view(torch.int16).numpy(), vb.view(torch.int16).numpy(),
                        w.block_tables, w.seq_lens, w.scale)
    got = oracle.decode_fp8(q, kc8, vc8, w.block_tables, w.seq_lens, w.scale, k_scale, v_scale)
    np.testing.assert_array_equal(got, ref)


def _fp8_prefill_workload(seed):
    """A mixed varlen batch (prefill chunks with context, decode rows, an
    empty request) over random e4m3 caches without NaN codes."""
    w = wl.build_workload("fp8mix", [90, 33, 140, 20, 5], [30, 1, 140, 1, 0], num_heads=6,
                          num_kv_heads=2, head_dim=64, block_size=16, num_blocks=40, seed=seed)
    t = wl.make_tensors(w)
    rng = np.random.default_rng(seed)
    kc8 = rng.integers(0, 256, size=t.key_cache.shape, dtype=np.uint8)
    vc8 = rng.integers(0, 256, size=t.value_cache.shape, dtype=np.uint8)
    for c in (kc8, vc8):
        c[(c & 0x7F) == 0x7F] = 0x3C
    return w, t, kc8, vc8


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 8.0), (2.0 ** -6, 2.0 ** 4)])
def test_prefill_fp8_equals_prefill_of_dequantized_cache(oracle, k_scale, v_scale):
    """Power-of-two scales keep every dequantized value a bf16 value: the FP8
    varlen prefill must equal the (separately pinned) bf16 one exactly, rows
    of every kind included."""
    w, t, kc8, vc8 = _fp8_prefill_workload(63)
    deq = lambda c, s: torch.from_numpy(oracle.e4m3_decode(c) * s).to(torch.bfloat16)
    kb, vb = deq(kc8, k_scale), deq(vc8, v_scale)
    assert torch.equal(vb.double(), torch.from_numpy(oracle.e4m3_decode(vc8) * v_scale))
    q = t.q.view(torch.int16).numpy()
    ref = oracle.prefill_varlen(q, kb.view(torch.int16).numpy(), vb.view(torch.int16).numpy(),
                                w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    got = oracle.prefill_varlen_fp8(q, kc8, vc8, w.query_start_loc, w.seq_lens, w.block_tables,
                                    w.scale, k_scale, v_scale)
    np.testing.assert_array_equal(got, ref)


def test_prefill_fp8_decode_rows_equal_decode_fp8(oracle):
    """A q_len == 1 row of the FP8 varlen prefill is the FP8 decode of its
    request (non-power-of-two scales)."""
    w, t, kc8, vc8 = _fp8_prefill_workload(64)
    got = oracle.prefill_varlen_fp8(t.q.view(torch.int16).numpy(), kc8, vc8, w.query_start_loc,
                                    w.seq_lens, w.block_tables, w.scale, 0.37, 1.9)
    for r in (1, 3):
        row = int(w.query_start_loc[r])
        q1 = t.q[row:row + 1].view(torch.int16).numpy()
        ref = oracle.decode_fp8(q1, kc8, vc8, w.block_tables[r:r + 1], w.seq_lens[r:r + 1],
                                w.scale, 0.37, 1.9)
        np.testing.assert_array_equal(got[row], ref[0])


def test_reshape_and_cache_fp8_scatter(oracle):
    w, t, kc8, vc8 = _fp8_workload(62)
    rng = np.random.default_rng(62)
    n = 11
    gen = torch.Generator().manual_seed(62)
    shape = (n, w.num_kv_heads, w.head_dim)
    key = (torch.randn(shape, generator=gen) * 20).to(torch.bfloat16).view(torch.int16).numpy()
    value = torch.randn(shape, generator=gen).to(torch.bfloat16).view(torch.int16).numpy()
    slots = rng.choice(w.num_blocks * w.block_size, size=n, replace=False).astype(np.int64)
    slots[3] = -1
    kn, vn = oracle.reshape_and_cache_fp8(key, value, kc8, vc8, slots, 0.5, 0.125)
    flat = lambda c: c.reshape(-1, w.num_kv_heads, w.head_dim)
    kf = torch.from_numpy(key).view(torch.bfloat16).float().numpy()
    vf = torch.from_numpy(value).view(torch.bfloat16).float().numpy()
    touched = np.zeros(w.num_blocks * w.block_size, bool)
    for i, s in enumerate(slots):
        if s < 0:
            continue
        touched[s] = True
        np.testing.assert_array_equal(flat(kn)[s], oracle.e4m3_encode(kf[i] / np.float32(0.5)))
        np.testing.assert_array_equal(flat(vn)[s], oracle.e4m3_encode(vf[i] / np.float32(0.125)))
    np.testing.assert_array_equal(flat(kn)[~touched], flat(kc8)[~touched])
    np.testing.assert_array_equal(flat(vn)[~touched], flat(vc8)[~touched])


# ------------------------------------------------------ x-split cache layout

def _to_xsplit(key_cache, value_cache):
    """[nb, B, H, d] caches -> the x-split shapes of the pages (numpy's own
    reshape and transpose: K [nb, H, d / 8, B, 8], V [nb, H, d, B])."""
    nb, B, H, d = key_cache.shape
    kx = np.ascontiguousarray(key_cache.reshape(nb, B, H, d // 8, 8).transpose(0, 2, 3, 1, 4))
    vx = np.ascontiguousarray(value_cache.reshape(nb, B, H, d).transpose(0, 2, 3, 1))
    return kx, vx


@pytest.mark.parametrize("hkv,d,B", [(2, 64, 16), (8, 128, 32), (1, 128, 64)])
def test_xsplit_writer_places_elements_at_the_pages_shape(oracle, hkv, d, B):
    """Token i with slot s must appear at K[s // B, h, d // 8, s % B, d % 8]
    and V[s // B, h, d, s % B] (x = 16 bytes / 2 bytes = 8); every other
    element, and tokens with a negative slot, leave the pool untouched."""
    nb, n = 6, 9
    rng = np.random.default_rng(71 + B)
    key = rng.integers(0, 1 << 16, size=(n, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(n, hkv, d), dtype=np.uint16)
    kx0 = rng.integers(0, 1 << 16, size=(nb, hkv, d // 8, B, 8), dtype=np.uint16)
    vx0 = rng.integers(0, 1 << 16, size=(nb, hkv, d, B), dtype=np.uint16)
    slots = rng.choice(nb * B, size=n, replace=False).astype(np.int64)
    slots[4] = -1
    kx, vx = oracle.reshape_and_cache_xsplit(key, val, kx0, vx0, slots)
    k_seen, v_seen = kx0.copy(), vx0.copy()
    for i, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), B)
        for h in range(hkv):
            for e in range(d):
                assert kx[blk, h, e // 8, off, e % 8] == key[i, h, e]
                assert vx[blk, h, e, off] == val[i, h, e]
        k_seen[blk, :, :, off, :] = kx[blk, :, :, off, :]
        v_seen[blk, :, :, off] = vx[blk, :, :, off]
    np.testing.assert_array_equal(kx, k_seen)
    np.testing.assert_array_equal(vx, v_seen)


def test_xsplit_writer_is_a_permutation_of_the_token_major_writer(oracle):
    """The same tokens written by both writers give caches that numpy's
    reshape + transpose carries into one another."""
    w = wl.tiny_decode()
    t = wl.make_tensors(w)
    n = 12
    gen = torch.Generator().manual_seed(72)
    key = torch.randn((n, 2, 64), generator=gen).to(torch.bfloat16).view(torch.int16).numpy()
    val = torch.randn((n, 2, 64), generator=gen).to(torch.bfloat16).view(torch.int16).numpy()
    slots = np.random.default_rng(72).choice(w.num_blocks * 16, size=n, replace=False)
    kc0 = t.key_cache.view(torch.int16).numpy()
    vc0 = t.value_cache.view(torch.int16).numpy()
    kn, vn = oracle.reshape_and_cache(key, val, kc0, vc0, slots.astype(np.int64))
    kx0, vx0 = _to_xsplit(kc0.view(np.uint16), vc0.view(np.uint16))
    kx, vx = oracle.reshape_and_cache_xsplit(key, val, kx0, vx0, slots.astype(np.int64))
    kref, vref = _to_xsplit(kn, vn)
    np.testing.assert_array_equal(kx, kref)
    np.testing.assert_array_equal(vx, vref)


@pytest.mark.parametrize("hq,hkv,d,lens,B", [(4, 2, 64, [25, 12, 37, 20], 16),
                                             (8, 2, 128, [1, 31, 64, 70], 32),
                                             (16, 2, 128, [129, 33], 64)])
def test_decode_xsplit_equals_decode_of_the_same_cache(oracle, hq, hkv, d, lens, B):
    """Decoding the x-split form of a cache must give exactly the (pinned)
    decode of the token-major form: same keys, same arithmetic."""
    w, _ = _contiguous_workload(lens, hq, hkv, d, seed=73, B=B)
    need = -(-np.asarray(lens) // B)
    for r, n in enumerate(need):  # blocks in reverse order: table lookups matter
        w.block_tables[r, :n] = w.block_tables[r, :n][::-1].copy()
    t = wl.make_tensors(w)
    kc = t.key_cache.view(torch.int16).numpy().view(np.uint16)
    vc = t.value_cache.view(torch.int16).numpy().view(np.uint16)
    q = t.q.view(torch.int16).numpy()
    ref = oracle.decode(q, kc, vc, w.block_tables, w.seq_lens, w.scale)
    kx, vx = _to_xsplit(kc, vc)
    got = oracle.decode_xsplit(q, kx, vx, w.block_tables, w.seq_lens, w.scale)
    np.testing.assert_array_equal(got, ref)


def _to_xsplit8(key_cache, value_cache):
    """e4m3 [nb, B, H, d] caches -> the x-split shapes with x = 16 one-byte
    elements (numpy's own reshape and transpose: K [nb, H, d / 16, B, 16],
    V [nb, H, d, B])."""
    nb, B, H, d = key_cache.shape
    kx = np.ascontiguousarray(key_cache.reshape(nb, B, H, d // 16, 16).transpose(0, 2, 3, 1, 4))
    vx = np.ascontiguousarray(value_cache.reshape(nb, B, H, d).transpose(0, 2, 3, 1))
    return kx, vx


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.013, 7.7)])
def test_xsplit_fp8_writer_is_a_permutation_of_the_token_major_fp8_writer(oracle, k_scale,
                                                                         v_scale):
    """The e4m3 x-split writer stores exactly the bytes of the (pinned)
    token-major e4m3 writer, at K[s // B, h, d // 16, s % B, d % 16] and
    V[s // B, h, d, s % B]; tokens with a negative slot write nothing."""
    nb, B, hkv, d, n = 7, 16, 2, 64, 11
    rng = np.random.default_rng(74)
    gen = torch.Generator().manual_seed(74)
    key = torch.randn((n, hkv, d), generator=gen).to(torch.bfloat16).view(torch.int16).numpy()
    val = torch.randn((n, hkv, d), generator=gen).to(torch.bfloat16).view(torch.int16).numpy()
    kc0 = rng.integers(0, 256, size=(nb, B, hkv, d), dtype=np.uint8)
    vc0 = rng.integers(0, 256, size=(nb, B, hkv, d), dtype=np.uint8)
    slots = rng.choice(nb * B, size=n, replace=False).astype(np.int64)
    slots[3] = -1
    kn, vn = oracle.reshape_and_cache_fp8(key, val, kc0, vc0, slots, k_scale, v_scale)
    kx0, vx0 = _to_xsplit8(kc0, vc0)
    kx, vx = oracle.reshape_and_cache_xsplit_fp8(key, val, kx0, vx0, slots, k_scale, v_scale)
    kref, vref = _to_xsplit8(kn, vn)
    np.testing.assert_array_equal(kx, kref)
    np.testing.assert_array_equal(vx, vref)
    i = 5
    blk, off = divmod(int(slots[i]), B)
    for e in range(d):
        assert kx[blk, 1, e // 16, off, e % 16] == kn[blk, off, 1, e]
        assert vx[blk, 1, e, off] == vn[blk, off, 1, e]


@pytest.mark.parametrize("hq,hkv,d,lens,B", [(4, 2, 64, [25, 12, 37, 20], 16),
                                             (8, 2, 128, [1, 31, 64, 70], 32)])
def test_decode_xsplit_fp8_equals_decode_fp8_of_the_same_cache(oracle, hq, hkv, d, lens, B):
    """Decoding the e4m3 x-split form of a cache gives exactly the (pinned)
    e4m3 decode of the token-major form."""
    w, _ = _contiguous_workload(lens, hq, hkv, d, seed=75, B=B)
    need = -(-np.asarray(lens) // B)
    for r, n in enumerate(need):
        w.block_tables[r, :n] = w.block_tables[r, :n][::-1].copy()
    t = wl.make_tensors(w)
    rng = np.random.default_rng(75)
    kc8 = rng.integers(0, 127, size=t.key_cache.shape, dtype=np.uint8)
    vc8 = rng.integers(0, 127, size=t.value_cache.shape, dtype=np.uint8)
    kc8[rng.random(kc8.shape) < 0.5] |= 0x80
    vc8[rng.random(vc8.shape) < 0.5] |= 0x80
    q = t.q.view(torch.int16).numpy()
    ref = oracle.decode_fp8(q, kc8, vc8, w.block_tables, w.seq_lens, w.scale, 0.5, 0.125)
    kx, vx = _to_xsplit8(kc8, vc8)
    got = oracle.decode_xsplit_fp8(q, kx, vx, w.block_tables, w.seq_lens, w.scale, 0.5, 0.125)
    np.testing.assert_array_equal(got, ref)


def test_thread_count_does_not_change_results(oracle):
    """The OpenMP loops only spread independent output rows: decode, e4m3
    decode and varlen prefill on several threads give the single-thread
    doubles bit for bit (the all-core CPU baseline times the same arithmetic)."""
    w = wl.random_workload(21, num_seqs=5, max_len=300, min_len=20, num_heads=8, num_kv_heads=2,
                           head_dim=64, max_q_len=40, prefill_fraction=0.6)
    t = wl.make_tensors(w)
    b = lambda x: x.contiguous().view(torch.int16).numpy().view(np.uint16)
    runs = []
    for n in (1, 4):
        oracle.set_threads(n)
        try:
            runs.append((oracle.decode(b(t.q)[:w.num_seqs], b(t.key_cache), b(t.value_cache),
                                       w.block_tables, w.seq_lens, w.scale),
                         oracle.prefill_varlen(b(t.q), b(t.key_cache), b(t.value_cache),
                                               w.query_start_loc, w.seq_lens, w.block_tables,
                                               w.scale)))
        finally:
            oracle.set_threads(1)
    np.testing.assert_array_equal(runs[0][0], runs[1][0])
    np.testing.assert_array_equal(runs[0][1], runs[1][1])
    codes = np.random.default_rng(22).integers(0, 127, t.key_cache.shape, dtype=np.uint8)
    fp8 = []
    for n in (1, 4):
        oracle.set_threads(n)
        try:
            fp8.append(oracle.decode_fp8(b(t.q)[:w.num_seqs], codes, codes[::-1].copy(),
                                         w.block_tables, w.seq_lens, w.scale, 0.03, 0.07))
        finally:
            oracle.set_threads(1)
    np.testing.assert_array_equal(fp8[0], fp8[1])
