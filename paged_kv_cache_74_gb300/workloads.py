"""Seeded synthetic inputs for the paged KV-cache path.

This module is shared by the tests, the benchmark and the oracle checks, and
it holds none of the method's arithmetic: it draws sequence and query
lengths, hands out physical blocks the way a block allocator would (a seeded
permutation of the free blocks, block 0 kept back as the null block), packs
the varlen query ranges, and fills tensors with N(0, 1) bf16 values.  Slot
numbers and attention results are never computed here; the oracle and the
CUDA library each compute those on their own.

Workload shapes follow the pages' examples (vLLM PagedAttention pages:
16-token blocks, GQA with Llama-3-8B/70B head shapes, contexts up to 32K,
a shared 1024-token prefix, a mixed chunked-prefill + decode batch).  The
pages measure on ShareGPT/Alpaca traces with trained models; these seeded
synthetic inputs stand in for them.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


@dataclass
class Workload:
    """Host-side description of one batch (all arrays are numpy, int32).

    seq_lens[r]     K/V length of request r after this step's tokens are
                    written (the varlen ``seqused_k``).
    q_lens[r]       number of new query tokens of request r in this step
                    (1 for a decode row).
    query_start_loc cumulative q_lens with a leading 0, length num_seqs + 1.
    block_tables    [num_seqs, max_blocks_per_seq] physical block ids; entries
                    past a request's last block hold 0 (the null block).
    shared_blocks   physical ids used by more than one request (read-only).
    """

    name: str
    seq_lens: np.ndarray
    q_lens: np.ndarray
    query_start_loc: np.ndarray
    block_tables: np.ndarray
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    seed: int
    shared_blocks: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_seqs else 0

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.num_seqs else 0

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    def used_blocks(self) -> np.ndarray:
        """Distinct physical blocks that hold at least one live token."""
        ids = []
        for r in range(self.num_seqs):
            nb = -(-int(self.seq_lens[r]) // self.block_size)
            ids.append(self.block_tables[r, :nb])
        if not ids:
            return np.zeros(0, np.int32)
        return np.unique(np.concatenate(ids))


def _pack_query_start_loc(q_lens: np.ndarray) -> np.ndarray:
    qsl = np.zeros(q_lens.shape[0] + 1, np.int64)
    np.cumsum(q_lens, out=qsl[1:])
    return qsl.astype(np.int32)


def build_workload(name: str, seq_lens, q_lens, *, num_heads: int, num_kv_heads: int,
                   head_dim: int, block_size: int, num_blocks: int, seed: int,
                   shared_prefix_blocks: int = 0, max_blocks_per_seq: int | None = None,
                   rng: np.random.Generator | None = None,
                   permutation: np.ndarray | None = None) -> Workload:
    """Lay out block tables for the given lengths.

    Physical blocks are handed out from a seeded permutation of blocks
    1..num_blocks-1 (block 0 is the null block and is never handed out).
    With ``shared_prefix_blocks = P`` the first P logical blocks of every
    request map to the same physical blocks 1..P (a shared prefix); a request
    shorter than the prefix uses only the leading blocks it needs.
    """
    seq_lens = np.asarray(seq_lens, np.int32).copy()
    q_lens = np.asarray(q_lens, np.int32).copy()
    assert seq_lens.shape == q_lens.shape
    assert np.all(q_lens <= seq_lens) and np.all(q_lens >= 0) and np.all(seq_lens >= 1)
    B = block_size
    need = -(-seq_lens.astype(np.int64) // B)
    mb = int(need.max()) if need.size else 1
    if max_blocks_per_seq is None:
        max_blocks_per_seq = max(mb, 1)
    assert max_blocks_per_seq >= mb
    if rng is None:
        rng = np.random.default_rng(seed)
    P = shared_prefix_blocks
    shared = np.arange(1, P + 1, dtype=np.int32)
    if permutation is None:
        permutation = rng.permutation(np.arange(P + 1, num_blocks, dtype=np.int32))
    private_need = np.maximum(need - P, 0)
    if int(private_need.sum()) > permutation.shape[0]:
        raise ValueError(f"{name}: pool of {num_blocks} blocks too small")
    tables = np.zeros((seq_lens.shape[0], max_blocks_per_seq), np.int32)
    cur = 0
    for r in range(seq_lens.shape[0]):
        n_sh = int(min(need[r], P))
        tables[r, :n_sh] = shared[:n_sh]
        k = int(private_need[r])
        tables[r, n_sh:n_sh + k] = permutation[cur:cur + k]
        cur += k
    return Workload(name=name, seq_lens=seq_lens, q_lens=q_lens,
                    query_start_loc=_pack_query_start_loc(q_lens),
                    block_tables=tables, num_heads=num_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, block_size=B, num_blocks=num_blocks,
                    scale=1.0 / math.sqrt(head_dim), seed=seed,
                    shared_blocks=shared if P > 0 else np.zeros(0, np.int32))


# ---------------------------------------------------------------------------
# The five named workloads.
# ---------------------------------------------------------------------------

def tiny_decode() -> Workload:
    """4 seqs of lengths 25, 12, 37, 20; 4 q heads / 2 kv heads; d = 64;
    16-token blocks; a 32-block pool whose block 0 is the null block; block
    tables sliced in order from a seeded permutation of blocks 1..31."""
    rng = np.random.default_rng(1)
    perm = rng.permutation(np.arange(1, 32, dtype=np.int32))
    return build_workload("tiny_decode", [25, 12, 37, 20], [1, 1, 1, 1], num_heads=4,
                          num_kv_heads=2, head_dim=64, block_size=16, num_blocks=32, seed=1,
                          permutation=perm)


def llama8b_decode() -> Workload:
    """Llama-3-8B-shaped decode layer: 64 seqs with lengths uniform in
    [512, 4096]; 32 q heads / 8 kv heads; d = 128; 20000-block pool."""
    rng = np.random.default_rng(2)
    lens = rng.integers(512, 4096, size=64, endpoint=True)
    return build_workload("llama8b_decode_b64", lens, np.ones(64, np.int32), num_heads=32,
                          num_kv_heads=8, head_dim=128, block_size=16, num_blocks=20000,
                          seed=2, rng=rng)


def long_context_decode() -> Workload:
    """8 seqs of 32768 tokens each; 32 q heads / 8 kv heads; d = 128;
    randomly scattered physical blocks in a 20000-block pool."""
    rng = np.random.default_rng(3)
    return build_workload("long_ctx_decode_8x32k", np.full(8, 32768), np.ones(8, np.int32),
                          num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                          num_blocks=20000, seed=3, rng=rng)


def prefix_shared_decode() -> Workload:
    """70B-shaped decode: 256 seqs, lengths log-normal with median 1000
    (sigma 1 in log space), rounded and clipped to [16, 8192]; 64 q heads /
    8 kv heads; d = 128; the first 64 logical blocks of every seq map to
    the same 64 physical blocks; the pool has 25 % free holes."""
    rng = np.random.default_rng(4)
    z = rng.standard_normal(256)
    lens = np.clip(np.rint(np.exp(math.log(1000.0) + z)), 16, 8192).astype(np.int32)
    need = -(-lens.astype(np.int64) // 16)
    private = int(np.maximum(need - 64, 0).sum())
    num_blocks = 1 + 64 + private + (private + 3) // 4
    return build_workload("prefix_shared_decode_b256", lens, np.ones(256, np.int32),
                          num_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                          num_blocks=num_blocks, seed=4, shared_prefix_blocks=64, rng=rng)


def mixed_chunked_prefill() -> Workload:
    """One 512-token query chunk at context offset 3584 (K/V length 4096)
    plus 63 single-token decode rows with K/V lengths uniform in
    [256, 8192]; 32 q heads / 8 kv heads; d = 128; 40000-block pool."""
    rng = np.random.default_rng(5)
    dec = rng.integers(256, 8192, size=63, endpoint=True)
    lens = np.concatenate([[4096], dec]).astype(np.int32)
    qls = np.concatenate([[512], np.ones(63, np.int64)]).astype(np.int32)
    return build_workload("mixed_chunked_prefill", lens, qls, num_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16, num_blocks=40000, seed=5, rng=rng)


def multi_chunk_prefill() -> Workload:
    """Four long query chunks (q_len, context) = (2048, 0), (1024, 3072),
    (1536, 6656), (768, 12032) plus 28 single-token decode rows with K/V
    lengths uniform in [256, 8192]; 32 q heads / 8 kv heads; d = 128;
    12000-block pool.  1344 query tiles: several per SM."""
    rng = np.random.default_rng(6)
    chunks = [(2048, 0), (1024, 3072), (1536, 6656), (768, 12032)]
    dec = rng.integers(256, 8192, size=28, endpoint=True)
    lens = np.concatenate([[q + c for q, c in chunks], dec]).astype(np.int32)
    qls = np.concatenate([[q for q, _ in chunks], np.ones(28, np.int64)]).astype(np.int32)
    return build_workload("multi_chunk_prefill", lens, qls, num_heads=32, num_kv_heads=8,
                          head_dim=128, block_size=16, num_blocks=12000, seed=6, rng=rng)


NAMED = {
    "tiny_decode": tiny_decode,
    "llama8b_decode_b64": llama8b_decode,
    "long_ctx_decode_8x32k": long_context_decode,
    "prefix_shared_decode_b256": prefix_shared_decode,
    "mixed_chunked_prefill": mixed_chunked_prefill,
    "multi_chunk_prefill": multi_chunk_prefill,
}


def random_workload(seed: int, *, num_seqs: int, max_len: int, num_heads: int,
                    num_kv_heads: int, head_dim: int, block_size: int = 16,
                    max_q_len: int = 1, min_len: int = 1, spare_blocks: int = 8,
                    prefill_fraction: float = 0.0) -> Workload:
    """Small seeded case for parity sweeps: lengths uniform in
    [min_len, max_len]; a fraction of rows get q_len uniform in
    [2, max_q_len] (capped by their length), the rest q_len 1."""
    rng = np.random.default_rng(seed)
    lens = rng.integers(min_len, max_len, size=num_seqs, endpoint=True).astype(np.int32)
    qls = np.ones(num_seqs, np.int32)
    if max_q_len > 1:
        pre = rng.random(num_seqs) < prefill_fraction
        for r in np.nonzero(pre)[0]:
            hi = int(min(max_q_len, lens[r]))
            if hi >= 2:
                qls[r] = int(rng.integers(2, hi, endpoint=True))
    need = int((-(-lens.astype(np.int64) // block_size)).sum())
    return build_workload(f"random_{seed}", lens, qls, num_heads=num_heads,
                          num_kv_heads=num_kv_heads, head_dim=head_dim,
                          block_size=block_size, num_blocks=1 + need + spare_blocks,
                          seed=seed, rng=rng)


# ---------------------------------------------------------------------------
# Tensors.
# ---------------------------------------------------------------------------

@dataclass
class Tensors:
    """Device (or CPU) tensors of one workload.

    key_cache / value_cache  [num_blocks, block_size, num_kv_heads, head_dim] bf16
    q                        [total_q, num_heads, head_dim] bf16
    key / value              [total_q, num_kv_heads, head_dim] bf16 (new tokens)
    block_tables             [num_seqs, max_blocks_per_seq] int32
    seq_lens                 [num_seqs] int32
    query_start_loc          [num_seqs + 1] int32
    """

    key_cache: torch.Tensor
    value_cache: torch.Tensor
    q: torch.Tensor
    key: torch.Tensor
    value: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor


def _randn_bf16(shape, gen: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_tensors(w: Workload, device="cpu", poison: bool = False,
                 data_seed: int | None = None) -> Tensors:
    """Fill the pool, queries and new K/V with seeded N(0, 1) bf16 values.

    With ``poison=True`` every slot that no request may read holds NaN:
    the null block 0, every block no request uses, and the slots past each
    request's length in its last block (unless that block is shared, in
    which case its later slots are live tokens of a longer request).
    """
    device = torch.device(device)
    seed = w.seed if data_seed is None else data_seed
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    kc = _randn_bf16(shape, gen, device)
    vc = _randn_bf16(shape, gen, device)
    q = _randn_bf16((w.total_q, w.num_heads, w.head_dim), gen, device)
    k = _randn_bf16((w.total_q, w.num_kv_heads, w.head_dim), gen, device)
    v = _randn_bf16((w.total_q, w.num_kv_heads, w.head_dim), gen, device)
    if poison:
        poison_unused(w, kc, vc)
    return Tensors(kc, vc, q, k, v,
                   torch.from_numpy(w.block_tables).to(device),
                   torch.from_numpy(w.seq_lens).to(device),
                   torch.from_numpy(w.query_start_loc).to(device))


def poison_unused(w: Workload, key_cache: torch.Tensor, value_cache: torch.Tensor) -> None:
    """Write NaN into every slot no request may read (see make_tensors)."""
    nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16).view(torch.bfloat16).item()
    used = np.zeros(w.num_blocks, bool)
    used[w.used_blocks()] = True
    unused = torch.from_numpy(np.nonzero(~used)[0]).to(key_cache.device)
    key_cache[unused] = nan
    value_cache[unused] = nan
    shared = set(int(b) for b in w.shared_blocks)
    for r in range(w.num_seqs):
        L = int(w.seq_lens[r])
        nb = -(-L // w.block_size)
        last = int(w.block_tables[r, nb - 1])
        off = L - (nb - 1) * w.block_size
        if off < w.block_size and last not in shared:
            key_cache[last, off:] = nan
            value_cache[last, off:] = nan


def flush_l2(buf: torch.Tensor) -> None:
    """Overwrite a buffer larger than L2 so the next kernel starts cold."""
    buf.add_(1)
