"""GPU parity of the FP8 (e4m3) KV cache: the quantizing cache write is
bit-exact against the oracle (round to nearest even, saturating, scales that
are not powers of two included), and pa_decode_fp8 matches the fp64 oracle's
FP8 decode within max abs 1e-2, mean abs 1e-3."""
import numpy as np
import pytest
import torch

from helpers import assert_close_to_oracle, bits
from paged_kv_cache_74_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

NAN_E4M3 = 0x7F


def fp8_caches(w, t, k_scale, v_scale, seed):
    """e4m3 caches holding N(0, 1) values (codes of x / scale), NaN codes in
    every slot outside a request's context."""
    gen = torch.Generator(device="cuda").manual_seed(seed)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    k = torch.randn(shape, generator=gen, device="cuda")
    v = torch.randn(shape, generator=gen, device="cuda")
    kc = (k / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (v / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    used = torch.zeros(w.num_blocks * w.block_size, dtype=torch.bool)
    for r in range(w.num_seqs):
        L = int(w.seq_lens[r])
        for tok in range(L):
            used[int(w.block_tables[r, tok // w.block_size]) * w.block_size + tok % w.block_size] = True
    unused = (~used).cuda().view(w.num_blocks, w.block_size)
    kc[unused] = NAN_E4M3
    vc[unused] = NAN_E4M3
    return kc.contiguous(), vc.contiguous()


@pytest.mark.parametrize("k_scale,v_scale", [(1.0, 1.0), (0.5, 0.125), (0.013, 7.7), (3e-4, 0.021)])
def test_fp8_write_bit_exact(cuda_lib, oracle, k_scale, v_scale):
    pa = cuda_lib
    w = wl.random_workload(301, num_seqs=6, max_len=400, num_heads=8, num_kv_heads=2,
                           head_dim=128, max_q_len=50, prefill_fraction=0.5)
    t = wl.make_tensors(w, device="cuda")
    key = (t.key.float() * 8).to(torch.bfloat16)  # some values saturate at the small scales
    value = t.value
    kc = torch.randint(0, 127, (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim),
                       dtype=torch.uint8, device="cuda")
    vc = kc.flip(0).contiguous()
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    ref_k, ref_v = oracle.reshape_and_cache_fp8(bits(key), bits(value), kc.cpu().numpy(),
                                                vc.cpu().numpy(), slots.cpu().numpy(), k_scale, v_scale)
    pa.reshape_and_cache_fp8(key, value, kc, vc, slots, k_scale, v_scale)
    np.testing.assert_array_equal(kc.cpu().numpy(), ref_k)
    np.testing.assert_array_equal(vc.cpu().numpy(), ref_v)


FP8_SWEEP = [
    # (head_dim, q heads, kv heads, max_len, num_seqs, block size, seed)
    (128, 32, 8, 900, 7, 16, 311), (128, 8, 8, 300, 9, 16, 312), (128, 16, 8, 1500, 4, 32, 313),
    (64, 8, 2, 700, 6, 16, 314), (64, 4, 4, 120, 10, 64, 315), (64, 2, 2, 2000, 3, 16, 316),
    (128, 4, 1, 257, 5, 16, 317),
    # 4 q heads per kv head, an even number of kv heads: units of two kv heads
    (128, 8, 2, 700, 5, 64, 319), (128, 16, 4, 450, 6, 32, 322),
    # 5 to 16 q heads per kv head: the tensor-core decode with converted K/V
    (128, 64, 8, 1100, 6, 16, 340), (128, 16, 1, 700, 5, 32, 341), (64, 40, 8, 900, 4, 16, 342),
    (128, 48, 4, 400, 9, 64, 343), (64, 16, 2, 130, 7, 16, 344),
]


@pytest.mark.parametrize("d,hq,hkv,max_len,ns,B,seed", FP8_SWEEP)
def test_decode_fp8_matches_oracle(cuda_lib, oracle, d, hq, hkv, max_len, ns, B, seed):
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, block_size=B)
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 2.0 ** -5, 0.03
    kc, vc = fp8_caches(w, t, k_scale, v_scale, seed)
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                        k_scale, v_scale)
    ref = oracle.decode_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(), w.block_tables,
                            w.seq_lens, w.scale, k_scale, v_scale)
    assert torch.isfinite(out.float()).all()
    assert_close_to_oracle(out, ref, what=f"fp8 d{d} hq{hq} hkv{hkv} B{B}")


def test_decode_fp8_forced_splits(cuda_lib, oracle):
    """16-token partitions: many partial pieces merged in the kernel."""
    pa = cuda_lib
    w = wl.random_workload(318, num_seqs=5, max_len=600, num_heads=32, num_kv_heads=8, head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.05, 0.05, 318)
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale, 0.05,
                        0.05, partition_tokens=16)
    ref = oracle.decode_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(), w.block_tables,
                            w.seq_lens, w.scale, 0.05, 0.05)
    assert_close_to_oracle(out, ref, what="fp8 forced splits")


def test_fp8_write_then_decode(cuda_lib, oracle):
    """Slot mapping, quantizing write of each request's new token, decode."""
    pa = cuda_lib
    w = wl.random_workload(319, num_seqs=8, max_len=800, num_heads=32, num_kv_heads=8, head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 0.04, 0.06
    kc, vc = fp8_caches(w, t, k_scale, v_scale, 319)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    ref_k, ref_v = oracle.reshape_and_cache_fp8(bits(t.key), bits(t.value), kc.cpu().numpy(),
                                                vc.cpu().numpy(), slots.cpu().numpy(), k_scale, v_scale)
    pa.reshape_and_cache_fp8(t.key, t.value, kc, vc, slots, k_scale, v_scale)
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale, k_scale,
                        v_scale)
    ref = oracle.decode_fp8(bits(t.q), ref_k, ref_v, w.block_tables, w.seq_lens, w.scale,
                            k_scale, v_scale)
    assert_close_to_oracle(out, ref, what="fp8 write then decode")


def test_decode_fp8_full_size_8b(cuda_lib, oracle):
    """The 8B-shaped batch (64 requests, U[512, 4096]) in the benchmark's launch configuration."""
    pa = cuda_lib
    w = wl.llama8b_decode()
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 2.0 ** -5, 2.0 ** -5, 320)
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                        2.0 ** -5, 2.0 ** -5)
    rows = np.sort(np.random.default_rng(320).choice(w.num_seqs, 16, replace=False))
    ref = oracle.decode_fp8(bits(t.q)[rows], kc.cpu().numpy(), vc.cpu().numpy(),
                            w.block_tables[rows], w.seq_lens[rows], w.scale, 2.0 ** -5, 2.0 ** -5)
    assert_close_to_oracle(out[torch.from_numpy(rows).cuda()], ref, what="fp8 8B batch")


@pytest.mark.parametrize("pt", [128, 256])
def test_decode_fp8_large_group_forced_splits(cuda_lib, oracle, pt):
    """8 q heads per kv head (the tensor-core decode) cut into pieces of one
    or two 128-token chunks, merged in the kernel, over NaN-coded unused slots."""
    pa = cuda_lib
    w = wl.random_workload(321, num_seqs=5, max_len=1300, min_len=200, num_heads=64,
                           num_kv_heads=8, head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.05, 0.02, 321)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, 64, 8, 128, w.max_seq_len, pt), "cuda")
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale, 0.05,
                        0.02, workspace=ws, partition_tokens=pt)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.decode_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(), w.block_tables,
                            w.seq_lens, w.scale, 0.05, 0.02)
    assert_close_to_oracle(out, ref, what=f"fp8 group 8, {pt}-token pieces")


def test_decode_fp8_full_size_70b_prefix_shared(cuda_lib, oracle):
    """The 70B-shaped prefix-shared batch (256 requests, 64 q / 8 kv heads,
    a shared 1024-token prefix) over an e4m3 copy of its cache, in the
    benchmark's launch configuration; every row against the oracle."""
    pa = cuda_lib
    w = wl.prefix_shared_decode()
    t = wl.make_tensors(w, device="cuda")
    k_scale = float(t.key_cache.float().abs().max()) / 448.0
    v_scale = float(t.value_cache.float().abs().max()) / 448.0
    kc = (t.key_cache.float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (t.value_cache.float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), "cuda")
    out = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                        k_scale, v_scale, workspace=ws)
    assert pa.device_status(ws)[0] == 0
    ref = oracle.decode_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(), w.block_tables,
                            w.seq_lens, w.scale, k_scale, v_scale)
    assert_close_to_oracle(out, ref, what="fp8 70B prefix-shared batch (every row)")


# ---- the x-split layout with an e4m3 cache (x = 16 one-byte elements)

def to_xsplit8(kc, vc):
    """e4m3 [nb, B, H, d] caches -> K [nb, H, d / 16, B, 16], V [nb, H, d, B]."""
    nb, B, H, d = kc.shape
    kx = kc.view(nb, B, H, d // 16, 16).permute(0, 2, 3, 1, 4).contiguous()
    vx = vc.view(nb, B, H, d).permute(0, 2, 3, 1).contiguous()
    return kx, vx


@pytest.mark.parametrize("k_scale,v_scale,d,B", [(0.013, 7.7, 128, 16), (1.0, 1.0, 64, 32),
                                                 (2.0 ** -5, 0.03, 128, 64)])
def test_xsplit_fp8_write_bit_exact(cuda_lib, oracle, k_scale, v_scale, d, B):
    """The e4m3 x-split writer against the oracle's, over the whole pool."""
    pa = cuda_lib
    w = wl.random_workload(330 + B, num_seqs=9, max_len=300, num_heads=16, num_kv_heads=4,
                           head_dim=d, block_size=B, max_q_len=40, prefill_fraction=0.5)
    t = wl.make_tensors(w, device="cuda")
    gen = torch.Generator(device="cuda").manual_seed(330)
    kx = torch.randint(0, 256, (w.num_blocks, 4, d // 16, B, 16), generator=gen, device="cuda",
                       dtype=torch.uint8)
    vx = torch.randint(0, 256, (w.num_blocks, 4, d, B), generator=gen, device="cuda",
                       dtype=torch.uint8)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, B,
                                    w.num_blocks, w.total_q)
    slots[3] = -1
    ref_k, ref_v = oracle.reshape_and_cache_xsplit_fp8(bits(t.key), bits(t.value), kx.cpu().numpy(),
                                                       vx.cpu().numpy(), slots.cpu().numpy(),
                                                       k_scale, v_scale)
    pa.reshape_and_cache_xsplit_fp8(t.key, t.value, kx, vx, slots, k_scale, v_scale)
    torch.cuda.synchronize()
    assert np.array_equal(kx.cpu().numpy(), ref_k)
    assert np.array_equal(vx.cpu().numpy(), ref_v)


XS8_SWEEP = [
    # (head_dim, q heads, kv heads, max_len, num_seqs, block size, seed)
    (128, 32, 8, 900, 7, 16, 341), (128, 8, 8, 300, 9, 16, 342), (128, 16, 8, 1500, 4, 32, 343),
    (64, 8, 2, 700, 6, 16, 344), (64, 4, 4, 120, 10, 64, 345), (64, 2, 2, 2000, 3, 16, 346),
    (128, 12, 4, 257, 5, 16, 347),
]


@pytest.mark.parametrize("d,hq,hkv,max_len,ns,B,seed", XS8_SWEEP)
def test_decode_xsplit_fp8_matches_oracle(cuda_lib, oracle, d, hq, hkv, max_len, ns, B, seed):
    """Decode over e4m3 x-split caches (NaN codes in every unused slot)
    against the oracle's x-split e4m3 decode."""
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, block_size=B)
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 2.0 ** -5, 0.03
    kc, vc = fp8_caches(w, t, k_scale, v_scale, seed)
    kx, vx = to_xsplit8(kc, vc)
    out = pa.decode_xsplit_fp8(t.q, kx, vx, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                               k_scale, v_scale)
    ref = oracle.decode_xsplit_fp8(bits(t.q), kx.cpu().numpy(), vx.cpu().numpy(), w.block_tables,
                                   w.seq_lens, w.scale, k_scale, v_scale)
    assert torch.isfinite(out.float()).all()
    assert_close_to_oracle(out, ref, what=f"x-split fp8 d{d} hq{hq} hkv{hkv} B{B}")


def test_decode_xsplit_fp8_forced_splits_and_write(cuda_lib, oracle):
    """Write each request's new token into e4m3 x-split caches, then decode
    with 16-token partitions (many pieces merged in the kernel)."""
    pa = cuda_lib
    w = wl.random_workload(348, num_seqs=6, max_len=700, num_heads=32, num_kv_heads=8, head_dim=128)
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 0.04, 0.06
    kc, vc = fp8_caches(w, t, k_scale, v_scale, 348)
    kx, vx = to_xsplit8(kc, vc)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    ref_k, ref_v = oracle.reshape_and_cache_xsplit_fp8(bits(t.key), bits(t.value), kx.cpu().numpy(),
                                                       vx.cpu().numpy(), slots.cpu().numpy(),
                                                       k_scale, v_scale)
    pa.reshape_and_cache_xsplit_fp8(t.key, t.value, kx, vx, slots, k_scale, v_scale)
    out = pa.decode_xsplit_fp8(t.q, kx, vx, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                               k_scale, v_scale, partition_tokens=16)
    ref = oracle.decode_xsplit_fp8(bits(t.q), ref_k, ref_v, w.block_tables, w.seq_lens, w.scale,
                                   k_scale, v_scale)
    assert_close_to_oracle(out, ref, what="x-split fp8 write + forced splits")


def test_decode_xsplit_fp8_full_size_8b(cuda_lib, oracle):
    """The 8B-shaped batch over e4m3 x-split caches in the benchmark's launch
    configuration, against the oracle on a seeded sample of requests and
    against the token-major e4m3 decode of the same values on all of them."""
    pa = cuda_lib
    w = wl.llama8b_decode()
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 2.0 ** -5, 2.0 ** -5, 349)
    kx, vx = to_xsplit8(kc, vc)
    out = pa.decode_xsplit_fp8(t.q, kx, vx, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                               2.0 ** -5, 2.0 ** -5)
    tm = pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len, w.scale,
                       2.0 ** -5, 2.0 ** -5)
    err = (out.float() - tm.float()).abs()
    assert torch.isfinite(out.float()).all() and err.max().item() <= 2e-2 and err.mean().item() <= 2e-3
    rows = np.sort(np.random.default_rng(349).choice(w.num_seqs, 12, replace=False))
    ref = oracle.decode_xsplit_fp8(bits(t.q)[rows], kx.cpu().numpy(), vx.cpu().numpy(),
                                   w.block_tables[rows], w.seq_lens[rows], w.scale, 2.0 ** -5,
                                   2.0 ** -5)
    assert_close_to_oracle(out[torch.from_numpy(rows).cuda()], ref, what="x-split fp8 8B batch")


# ---- pa_prefill_varlen_fp8: the prefill tiles over e4m3 caches (each landed
# step converted to f16 in shared memory) plus the FP8 decode rows.

def run_prefill_fp8(pa, w, t, kc, vc, k_scale, v_scale):
    ws = pa.new_workspace(pa.prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads,
                                                    w.num_kv_heads, w.head_dim, w.max_seq_len),
                          "cuda")
    out = pa.prefill_varlen_fp8(t.q, kc, vc, t.query_start_loc, t.seq_lens, t.block_tables,
                                w.max_query_len, w.max_seq_len, w.scale, k_scale, v_scale,
                                workspace=ws)
    return out, ws


def prefill_fp8_ref(oracle, w, t, kc, vc, k_scale, v_scale):
    return oracle.prefill_varlen_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(),
                                     w.query_start_loc, w.seq_lens, w.block_tables, w.scale,
                                     k_scale, v_scale)


FP8_PREFILL_MIXES = [
    # (seed, num_seqs, max_len, max_q_len, head_dim, q heads, kv heads, block size)
    (351, 5, 300, 200, 128, 8, 2, 16),
    (352, 6, 700, 260, 128, 32, 8, 16),
    (353, 4, 150, 150, 64, 4, 2, 16),
    (354, 5, 520, 300, 128, 16, 16, 32),
    (355, 3, 400, 400, 128, 8, 1, 64),
    (356, 5, 290, 130, 64, 16, 2, 16),
    (357, 4, 400, 200, 128, 64, 8, 16),
]


@pytest.mark.parametrize("seed,ns,max_len,max_q,d,hq,hkv,B", FP8_PREFILL_MIXES)
def test_prefill_fp8_random_mixes(cuda_lib, oracle, seed, ns, max_len, max_q, d, hq, hkv, B):
    """Random prefill chunks with context next to decode rows, NaN codes in
    every slot outside a request's context, scales that are not powers of two."""
    pa = cuda_lib
    w = wl.random_workload(seed, num_seqs=ns, max_len=max_len, num_heads=hq, num_kv_heads=hkv,
                           head_dim=d, max_q_len=max_q, prefill_fraction=0.7, block_size=B)
    assert w.max_query_len > 1
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 0.037, 0.0213
    kc, vc = fp8_caches(w, t, k_scale, v_scale, seed)
    out, ws = run_prefill_fp8(pa, w, t, kc, vc, k_scale, v_scale)
    assert pa.device_status(ws)[0] == 0
    assert torch.isfinite(out.float()).all()
    ref = prefill_fp8_ref(oracle, w, t, kc, vc, k_scale, v_scale)
    assert_close_to_oracle(out, ref, what=f"fp8 prefill mix {seed}")


@pytest.mark.parametrize("q_len,ctx,d", [(2, 0, 128), (2, 37, 64), (127, 0, 128), (128, 0, 64),
                                         (129, 5, 128), (256, 16, 128), (300, 1000, 64),
                                         (17, 2047, 128)])
def test_prefill_fp8_tile_edges(cuda_lib, oracle, q_len, ctx, d):
    """Chunks at and around the 128-row tile and 16-token block edges (steps
    with fewer than 8 landed blocks), next to a decode row."""
    pa = cuda_lib
    lens = [ctx + q_len, 77]
    w = wl.build_workload("edge8", lens, [q_len, 1], num_heads=8, num_kv_heads=2, head_dim=d,
                          block_size=16, num_blocks=1 + sum(-(-x // 16) for x in lens) + 4,
                          seed=q_len + 7)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.05, 0.04, q_len)
    out, ws = run_prefill_fp8(pa, w, t, kc, vc, 0.05, 0.04)
    assert pa.device_status(ws)[0] == 0
    ref = prefill_fp8_ref(oracle, w, t, kc, vc, 0.05, 0.04)
    assert_close_to_oracle(out, ref, what=f"fp8 q_len {q_len} ctx {ctx} d {d}")


@pytest.mark.parametrize("q_len,ctx,hq,hkv", [(256, 2000, 2, 1), (130, 700, 4, 2), (2, 5000, 2, 2)])
def test_prefill_fp8_unit_split_over_many_ctas(cuda_lib, oracle, q_len, ctx, hq, hkv):
    """Few key steps over a grid of one CTA per SM: units cut into pieces that
    are merged in the kernel (the v_scale of each piece included)."""
    pa = cuda_lib
    lens = [ctx + q_len, 90]
    w = wl.build_workload("split8", lens, [q_len, 1], num_heads=hq, num_kv_heads=hkv, head_dim=128,
                          block_size=16, num_blocks=1 + sum(-(-x // 16) for x in lens) + 4,
                          seed=q_len + ctx)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.03, 0.3, q_len + ctx)
    for _ in range(2):
        out, ws = run_prefill_fp8(pa, w, t, kc, vc, 0.03, 0.3)
        assert pa.device_status(ws)[0] == 0
    ref = prefill_fp8_ref(oracle, w, t, kc, vc, 0.03, 0.3)
    assert_close_to_oracle(out, ref, what=f"fp8 split q_len {q_len} ctx {ctx}")


def test_prefill_fp8_write_then_attend_full_size(cuda_lib, oracle):
    """The 512-token chunk at context 3584 plus 63 decode rows over e4m3
    caches: quantize all 575 new tokens through the slot mapping, then
    attend; every row and head compared with the oracle."""
    pa = cuda_lib
    w = wl.mixed_chunked_prefill()
    t = wl.make_tensors(w, device="cuda")
    k_scale, v_scale = 2.0 ** -5, 0.0371
    kc, vc = fp8_caches(w, t, k_scale, v_scale, 358)
    slots = pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16,
                                    w.num_blocks, w.total_q)
    pa.reshape_and_cache_fp8(t.key, t.value, kc, vc, slots, k_scale, v_scale)
    out, ws = run_prefill_fp8(pa, w, t, kc, vc, k_scale, v_scale)
    assert pa.device_status(ws)[0] == 0
    ref = prefill_fp8_ref(oracle, w, t, kc, vc, k_scale, v_scale)
    assert_close_to_oracle(out, ref, what="fp8 mixed chunked prefill (every row)")


def test_prefill_fp8_is_deterministic_and_rejects_bad_scales(cuda_lib):
    pa = cuda_lib
    w = wl.random_workload(359, num_seqs=5, max_len=600, num_heads=32, num_kv_heads=8,
                           head_dim=128, max_q_len=300, prefill_fraction=0.6)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.05, 0.05, 359)
    a, _ = run_prefill_fp8(pa, w, t, kc, vc, 0.05, 0.05)
    b, _ = run_prefill_fp8(pa, w, t, kc, vc, 0.05, 0.05)
    assert torch.equal(a, b)
    for ks, vs in ((0.0, 1.0), (1.0, float("nan")), (-1.0, 1.0)):
        with pytest.raises(pa.PAError):
            run_prefill_fp8(pa, w, t, kc, vc, ks, vs)


def test_prefill_fp8_mixed_step_in_a_cuda_graph(cuda_lib):
    """Slot mapping, the quantizing cache write and pa_prefill_varlen_fp8
    captured in one CUDA graph (after an eager warm-up) replay to the eager
    result bit for bit."""
    pa = cuda_lib
    w = wl.random_workload(360, num_seqs=6, max_len=500, num_heads=32, num_kv_heads=8,
                           head_dim=128, max_q_len=200, prefill_fraction=0.5)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.04, 0.05, 360)
    kc0, vc0 = kc.clone(), vc.clone()
    ws = pa.new_workspace(pa.prefill_workspace_size(w.num_seqs, w.total_q, 32, 8, 128,
                                                    w.max_seq_len), "cuda")
    out = torch.empty_like(t.q)
    slots = torch.empty(w.total_q, dtype=torch.int64, device="cuda")

    def step():
        pa.compute_slot_mapping(t.block_tables, t.query_start_loc, t.seq_lens, 16, w.num_blocks,
                                w.total_q, out=slots)
        pa.reshape_and_cache_fp8(t.key, t.value, kc, vc, slots, 0.04, 0.05)
        pa.prefill_varlen_fp8(t.q, kc, vc, t.query_start_loc, t.seq_lens, t.block_tables,
                              w.max_query_len, w.max_seq_len, w.scale, 0.04, 0.05, out=out,
                              workspace=ws)

    step()
    torch.cuda.synchronize()
    eager = out.clone()
    kc.copy_(kc0)
    vc.copy_(vc0)
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


def test_prefill_fp8_bad_block_id_is_reported_not_dereferenced(cuda_lib, oracle):
    """An out-of-range block id of one prefill chunk is reported in the status
    record and read as zeros; the other requests' rows stay exact."""
    pa = cuda_lib
    w = wl.build_workload("bad8", [300, 90, 40], [200, 1, 30], num_heads=8, num_kv_heads=2,
                          head_dim=128, block_size=16, num_blocks=40, seed=361)
    t = wl.make_tensors(w, device="cuda")
    kc, vc = fp8_caches(w, t, 0.05, 0.05, 361)
    bt = t.block_tables.clone()
    bt[0, 3] = w.num_blocks + 77
    ws = pa.new_workspace(pa.prefill_workspace_size(3, w.total_q, 8, 2, 128, w.max_seq_len), "cuda")
    out = pa.prefill_varlen_fp8(t.q, kc, vc, t.query_start_loc, t.seq_lens, bt, w.max_query_len,
                                w.max_seq_len, w.scale, 0.05, 0.05, workspace=ws)
    st = pa.device_status(ws)
    assert st[0] == 2 and st[2] == w.num_blocks + 77
    ref = oracle.prefill_varlen_fp8(bits(t.q), kc.cpu().numpy(), vc.cpu().numpy(),
                                    w.query_start_loc, w.seq_lens, w.block_tables, w.scale,
                                    0.05, 0.05)
    rows = slice(int(w.query_start_loc[1]), int(w.query_start_loc[3]))
    assert_close_to_oracle(out[rows], ref[rows], what="fp8: other requests")
