#!/usr/bin/env python3
"""Benchmark of the paged decode step on one GB300 (or N independent replicas).

One step = the whole hot path for one decode batch: the slot mapping of
the batch's new tokens, their reshape_and_cache write, and paged decode
attention (split-KV partitions + merge).  Inputs are seeded synthetic
tensors of the named workload, resident in HBM; L2 is flushed before every
step, outside the timed events: a 512 MiB write, then a 256 MiB read that
writes the flush's dirty lines back to HBM, so that L2 holds clean,
unrelated lines when the step starts (the decode's time with the dirty
lines of the write alone is reported beside it).

Prints ONE JSON line (rank 0).  `value` is KV GB/s: the step's algorithmic
bytes (each distinct K/V token the attention must read once, plus q, out,
the block-table entries, and the new tokens' K/V read and written) over
the device time of the step.  `--impl reference` times the fp64 CPU oracle
on the same workload instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_74_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attention KV GB/s & µs/call vs 8 TB/s HBM roofline (1×GB300)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# dram__bytes_read.sum + dram__bytes_write.sum of one launch of the named
# workload's dominant kernel, from an ncu capture of the full workload; valid
# only while that kernel's source is unchanged (sha256 prefix of its .cu file
# when the counters were taken), else reported as null.
PROFILED_TRAFFIC: dict = {
    # 636.340736 MB read + 3.247616 MB written
    "llama8b_decode_b64": {"bytes": 639588352, "src": "decode.cu",
                           "src_sha": "28bbfc5e29ee225b"},
    # 940.190720 MB read + 5.581824 MB written
    "prefix_shared_decode_b256": {"bytes": 945772544, "src": "decode_tc.cu",
                                  "src_sha": "77528aa33e5a5c65"},
    # prefill rows of the four-chunk batch: 877.759744 MB read + 14.742016 MB written
    "multi_chunk_prefill": {"bytes": 892501760, "src": "prefill.cu",
                            "src_sha": "02e57917f8ebd2f1"},
}


# ----------------------------------------------------------------- helpers

def decode_src_sha(src: str = "decode.cu") -> str:
    p = os.path.join(ROOT, "paged_kv_cache_74_gb300", "csrc", src)
    return hashlib.sha256(open(p, "rb").read()).hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def measured_bf16_tflops():
    """Burst bf16 tensor peak (a kernel timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def profiled_traffic(name):
    prof = PROFILED_TRAFFIC.get(name)
    return prof["bytes"] if prof and prof.get("src_sha") == decode_src_sha(prof["src"]) else None


def hbm_roofline(kernel, algo_bytes, seconds, traffic=None):
    peak, src = measured_peaks()
    achieved = algo_bytes / seconds / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(achieved, 2), "peak": peak,
            "peak_source": src, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "algorithmic_bytes_per_launch": int(algo_bytes),
            "us_per_launch": round(seconds * 1e6, 2)}


def tensor_roofline(kernel, flops, seconds, traffic=None):
    peak, src = measured_bf16_tflops()
    achieved = flops / seconds / 1e12
    return {"bound": "tensor", "kernel": kernel, "achieved": round(achieved, 2), "peak": peak,
            "peak_source": src, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "algorithmic_flops_per_launch": int(flops),
            "us_per_launch": round(seconds * 1e6, 2)}


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def algorithmic_bytes(w: wl.Workload) -> dict:
    """Bytes the decode step must move at least once.

    KV: every distinct (physical block, offset) token slot read by some
    request, times 2 (K and V) * kv_heads * head_dim * 2 bytes; a prefix
    shared by several requests counts once.  Plus q read, out written,
    block-table entries and seq_lens read, and the write of the new tokens
    (read K/V rows, write them, read the slots).
    """
    per_tok = 2 * w.num_kv_heads * w.head_dim * 2
    slots = set()
    logical = 0
    table_entries = 0
    for r in range(w.num_seqs):
        L = int(w.seq_lens[r])
        logical += L
        nb = -(-L // w.block_size)
        table_entries += nb
        for j in range(nb):
            phys = int(w.block_tables[r, j])
            n = min(w.block_size, L - j * w.block_size)
            slots.add((phys, n))
    # distinct tokens: per physical block the largest prefix any request reads
    best = {}
    for phys, n in slots:
        best[phys] = max(best.get(phys, 0), n)
    unique = sum(best.values())
    kv = unique * per_tok
    qo = 2 * w.total_q * w.num_heads * w.head_dim * 2
    meta = table_entries * 4 + w.num_seqs * 4 * 2
    write = w.total_q * (2 * per_tok + 8) + w.num_seqs * 4 * 2
    return {"kv_unique_tokens": unique, "kv_logical_tokens": logical, "kv_bytes": kv,
            "decode_bytes": kv + qo + meta, "step_bytes": kv + qo + meta + write,
            "kv_bytes_per_token": per_tok}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *self.sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        self.proc.wait()
        rows = [l.split(",") for l in open(self.path).read().strip().splitlines() if l.strip()]
        os.unlink(self.path)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1].split()[0]))
                smax.append(float(r[2].split()[0]))
            except (ValueError, IndexError):
                continue
            for name, v in zip(names, r[5:9]):
                if "Active" in v and "Not" not in v:
                    reasons.add(name)
        load = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_info():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate_over_ranks(local_seconds: float, local_bytes: float, world: int) -> tuple:
    """Max of the per-rank times and sum of the per-rank bytes (whole job)."""
    if world == 1:
        return local_seconds, local_bytes
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([local_seconds], dtype=torch.float64, device=dev)
    b = torch.tensor([local_bytes], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class L2Flush:
    """Evicts the timed inputs from L2 between steps.

    A 512 MiB write (four times the 129 MB L2), then a 256 MiB read of
    another buffer.  The write alone leaves L2 full of dirty lines whose
    write-back the next kernel would pay for inside its timed region; after
    the read L2 holds clean lines of unrelated data.  `dirty=True` skips
    the read (the write-only flush)."""

    def __init__(self, dev):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self.dirty = False

    def __call__(self):
        self.w.add_(1)
        if not self.dirty:
            torch.sum(self.r, dim=0, out=self.sink)


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import paged_kv_cache_74_gb300 as pa
    pa.load_library()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.NAMED[args.workload]()
    t = wl.make_tensors(w, device=dev)
    ab = algorithmic_bytes(w)
    stream = torch.cuda.current_stream(dev)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), dev)
    out = torch.empty_like(t.q)
    slots = torch.empty(w.total_q, dtype=torch.int64, device=dev)
    flush = L2Flush(dev)

    def step():  # slot mapping and cache write of the new tokens, one launch
        pa.append_tokens(t.key, t.value, t.key_cache, t.value_cache, t.block_tables,
                         t.query_start_loc, t.seq_lens, slot_mapping=slots)

    def attend():
        pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens, w.max_seq_len,
                  w.scale, out=out, workspace=ws)

    for _ in range(args.warmup):
        flush()
        step()
        attend()
    torch.cuda.synchronize(dev)

    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.perf_counter()
    for i in range(K):
        flush()
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
        attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_ms = [a.elapsed_time(c) for a, b, c in ev]
    dec_ms = [b.elapsed_time(c) for a, b, c in ev]
    local_s = sum(step_ms) / 1e3
    tot_s, tot_bytes = aggregate_over_ranks(local_s, ab["step_bytes"] * K, world)
    value = tot_bytes / tot_s / 1e9
    dec_avg_s = statistics.mean(dec_ms) / 1e3
    n_launch = 2  # append_tokens (slot mapping + cache write), decode (one persistent kernel)

    # e2e through the public API with pinned host buffers (H2D inputs, D2H out)
    e2e = run_e2e(pa, w, t, dev, stream, flush, args, ab, world)
    # The decode call after the write-only flush (L2 full of dirty lines).
    flush.dirty = True
    dirty_s = _time(attend, flush, min(K, 100))
    flush.dirty = False

    traffic = profiled_traffic(w.name)
    res = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(tot_s / K * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, seeded block permutations)",
        "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_heads": w.num_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "block_size": w.block_size, "num_blocks": w.num_blocks,
                   "max_seq_len": w.max_seq_len, "kv_unique_tokens": ab["kv_unique_tokens"],
                   "step": "append_tokens (slot mapping + cache write, one launch) + decode",
                   "l2": ("flushed before every step, outside the timed events: 512 MiB "
                          "write, then a 256 MiB read that writes its dirty lines back"),
                   "parallelism": f"replicas x{world}"},
        "us_per_call": round(dec_avg_s * 1e6, 2),
        "us_per_call_dirty_l2": round(dirty_s * 1e6, 2),
        "decode_kv_gbs": round(ab["kv_bytes"] / dec_avg_s / 1e9, 2),
        "wall_ms_per_step": round(wall / K * 1e3, 4),
        "roofline": hbm_roofline(decode_kernel_name(w), ab["decode_bytes"], dec_avg_s, traffic),
        "e2e": e2e,
        "gpu_launches": n_launch * K,
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_baseline(w, t, ab)
    if args.extra and rank == 0:
        res["extra"] = {name: extra_decode(pa, name, dev, flush, cpu=not args.no_cpu_baseline)
                        for name in args.extra}
        # Every target configuration's own roofline, beside the headline one.
        res["rooflines"] = {w.name: res["roofline"]}
        for name, e in res["extra"].items():
            for k, v in e.items():
                if k == "roofline" or k.startswith("roofline_"):
                    res["rooflines"][name + k[len("roofline"):]] = v
    return res, rank


def decode_kernel_name(w) -> str:
    return ("paged_decode_tc_kernel (pa_decode)" if w.num_heads // w.num_kv_heads > 4
            else "paged_decode_kernel (pa_decode)")


def run_e2e(pa, w, t, dev, stream, flush, args, ab, world):
    """The step through the public API with host inputs: the step's inputs
    (q, new K/V, block tables, seq_lens, query_start_loc) sit in one pinned
    staging buffer, as a serving loop would assemble them, and reach the GPU
    in one copy; the result comes back in one copy."""
    src = {"q": t.q, "key": t.key, "value": t.value, "bt": t.block_tables,
           "sl": t.seq_lens, "qsl": t.query_start_loc}
    offs, total = {}, 0
    for k, v in src.items():
        offs[k] = total
        total += -(-(v.numel() * v.element_size()) // 256) * 256
    stage_h = torch.empty(total, dtype=torch.uint8).pin_memory()
    stage_d = torch.empty(total, dtype=torch.uint8, device=dev)
    d = {}
    for k, v in src.items():
        n = v.numel() * v.element_size()
        stage_h[offs[k]:offs[k] + n].copy_(v.contiguous().view(-1).view(torch.uint8).cpu())
        d[k] = stage_d[offs[k]:offs[k] + n].view(v.dtype).view(v.shape)
    out_h = torch.empty(t.q.shape, dtype=torch.bfloat16).pin_memory()
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), dev)
    out = torch.empty_like(t.q)
    slots = torch.empty(w.total_q, dtype=torch.int64, device=dev)
    h2d = total
    d2h = out_h.numel() * out_h.element_size()

    def once():
        stage_d.copy_(stage_h, non_blocking=True)
        pa.append_tokens(d["key"], d["value"], t.key_cache, t.value_cache, d["bt"], d["qsl"],
                         d["sl"], slot_mapping=slots)
        pa.decode(d["q"], t.key_cache, t.value_cache, d["bt"], d["sl"], w.max_seq_len, w.scale,
                  out=out, workspace=ws)
        out_h.copy_(out, non_blocking=True)

    for _ in range(3):
        flush()
        once()
    torch.cuda.synchronize(dev)
    K = max(1, args.steps // 2)
    ts = []
    for _ in range(K):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        once()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b) / 1e3)
    tot_s, tot_bytes = aggregate_over_ranks(sum(ts), ab["step_bytes"] * K, world)
    return {"value": round(tot_bytes / tot_s / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(tot_s / K * 1e3, 5), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h}


def causal_pairs(w: wl.Workload) -> int:
    """(query, key) pairs the prefill rows (q_len > 1) attend."""
    n = 0
    for r in range(w.num_seqs):
        ql, L = int(w.q_lens[r]), int(w.seq_lens[r])
        if ql > 1:
            ctx = L - ql
            n += ql * ctx + ql * (ql + 1) // 2
    return n


def _time(call, flush, reps):
    """Median device time of `call` over `reps` calls, each after an L2
    flush, events on the launching stream.  The calls are enqueued back to
    back (one synchronisation at the end), so a call's events measure the
    GPU's work, not the host's time to enqueue it (the flush before each
    call gives the host ample lead)."""
    for _ in range(3):
        flush()
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for a, b in ev:
        flush()
        a.record()
        call()
        b.record()
    torch.cuda.synchronize()
    return statistics.median([a.elapsed_time(b) for a, b in ev]) / 1e3


def extra_mixed(pa, name, dev, flush, reps=20, cpu=True):
    """The mixed chunked-prefill batch: slot mapping + write of every new
    token + pa_prefill_varlen, and the prefill tiles alone (the chunk's
    request by itself) as tensor-core FLOP/s."""
    w = wl.NAMED[name]()
    t = wl.make_tensors(w, device=dev)
    ab = algorithmic_bytes(w)
    ws = pa.new_workspace(pa.prefill_workspace_size(w.num_seqs, w.total_q, w.num_heads,
                                                    w.num_kv_heads, w.head_dim, w.max_seq_len), dev)
    out = torch.empty_like(t.q)
    slots = torch.empty(w.total_q, dtype=torch.int64, device=dev)

    def step():
        pa.append_tokens(t.key, t.value, t.key_cache, t.value_cache, t.block_tables,
                         t.query_start_loc, t.seq_lens, slot_mapping=slots)
        pa.prefill_varlen(t.q, t.key_cache, t.value_cache, t.query_start_loc, t.seq_lens,
                          t.block_tables, w.max_query_len, w.max_seq_len, w.scale, out=out,
                          workspace=ws)
    s_step = _time(step, flush, reps)
    # prefill rows alone
    pre = [r for r in range(w.num_seqs) if w.q_lens[r] > 1]
    qsl = torch.tensor([0] + list(np.cumsum(w.q_lens[pre])), dtype=torch.int32, device=dev)
    rows = torch.cat([torch.arange(int(w.query_start_loc[r]), int(w.query_start_loc[r + 1]))
                      for r in pre]).to(dev)
    q_p = t.q[rows].contiguous()
    bt_p = t.block_tables[pre].contiguous()
    sl_p = t.seq_lens[pre].contiguous()
    out_p = torch.empty_like(q_p)
    mql = int(w.q_lens[pre].max())
    msl = int(w.seq_lens[pre].max())
    ws_p = pa.new_workspace(pa.prefill_workspace_size(len(pre), q_p.shape[0], w.num_heads,
                                                      w.num_kv_heads, w.head_dim, msl), dev)
    pcall = lambda: pa.prefill_varlen(q_p, t.key_cache, t.value_cache, qsl, sl_p, bt_p, mql, msl,
                                      w.scale, out=out_p, workspace=ws_p)
    s_pre = _time(pcall, flush, reps)
    flops = 4.0 * causal_pairs(w) * w.num_heads * w.head_dim
    # The same prefill rows over an e4m3 copy of the cache (per-tensor scales amax / 448).
    k_scale = float(t.key_cache.float().abs().max()) / 448.0
    v_scale = float(t.value_cache.float().abs().max()) / 448.0
    kc8 = (t.key_cache.float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vc8 = (t.value_cache.float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    pcall8 = lambda: pa.prefill_varlen_fp8(q_p, kc8, vc8, qsl, sl_p, bt_p, mql, msl, w.scale,
                                           k_scale, v_scale, out=out_p, workspace=ws_p)
    s_pre8 = _time(pcall8, flush, reps)
    # The whole step over the e4m3 copy: quantizing write of the new tokens
    # (at the slots the bf16 step computed) + pa_prefill_varlen_fp8.
    out8 = torch.empty_like(t.q)

    def step8():
        pa.reshape_and_cache_fp8(t.key, t.value, kc8, vc8, slots, k_scale, v_scale)
        pa.prefill_varlen_fp8(t.q, kc8, vc8, t.query_start_loc, t.seq_lens, t.block_tables,
                              w.max_query_len, w.max_seq_len, w.scale, k_scale, v_scale, out=out8,
                              workspace=ws)
    s_step8 = _time(step8, flush, reps)
    del kc8, vc8, out8
    res = {"us_per_step": round(s_step * 1e6, 2),
           "step": "append_tokens (all new tokens) + prefill_varlen",
           "step_kv_gbs": round(ab["step_bytes"] / s_step / 1e9, 2),
           "prefill_only_us": round(s_pre * 1e6, 2),
           "prefill_tflops": round(flops / s_pre / 1e12, 2),
           "prefill_gflop": round(flops / 1e9, 3),
           "us_per_step_fp8": round(s_step8 * 1e6, 2),
           "prefill_fp8_only_us": round(s_pre8 * 1e6, 2),
           "prefill_fp8_tflops": round(flops / s_pre8 / 1e12, 2),
           "roofline": tensor_roofline("prefill_kernel (pa_prefill_varlen, prefill rows alone)",
                                       flops, s_pre, profiled_traffic(w.name)),
           "roofline_step": hbm_roofline("append_tokens + pa_prefill_varlen (whole step)",
                                         ab["step_bytes"], s_step)}
    if cpu:
        res["cpu_baseline"] = cpu_baseline_prefill(w, t)
    del t
    torch.cuda.empty_cache()
    return res


def extra_decode_fp8(pa, name, dev, flush, reps=20, xsplit=False):
    """Decode-only timing of a named workload over an e4m3 copy of its cache
    (per-tensor scales amax / 448), token-major or in the x-split layout
    (K [blocks, kv heads, d / 16, block, 16], V [blocks, kv heads, d, block]);
    bytes counted at 1 per element."""
    w = wl.NAMED[name]()
    t = wl.make_tensors(w, device=dev)
    ab = algorithmic_bytes(w)
    k_scale = float(t.key_cache.float().abs().max()) / 448.0
    v_scale = float(t.value_cache.float().abs().max()) / 448.0
    kc = (t.key_cache.float() / k_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    vc = (t.value_cache.float() / v_scale).to(torch.float8_e4m3fn).view(torch.uint8)
    del t.key_cache, t.value_cache
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), dev)
    out = torch.empty_like(t.q)
    if xsplit:
        nb, B, H, d = kc.shape
        kc = kc.view(nb, B, H, d // 16, 16).permute(0, 2, 3, 1, 4).contiguous()
        vc = vc.view(nb, B, H, d).permute(0, 2, 3, 1).contiguous()
        call = lambda: pa.decode_xsplit_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len,
                                            w.scale, k_scale, v_scale, out=out, workspace=ws)
    else:
        call = lambda: pa.decode_fp8(t.q, kc, vc, t.block_tables, t.seq_lens, w.max_seq_len,
                                     w.scale, k_scale, v_scale, out=out, workspace=ws)
    s = _time(call, flush, reps)
    kv8 = ab["kv_bytes"] // 2
    dec8 = ab["decode_bytes"] - ab["kv_bytes"] + kv8
    rl = hbm_roofline(("pa_decode_xsplit_fp8" if xsplit else "pa_decode_fp8") + " (e4m3 cache, " +
                      ("tcgen05 decode)" if w.num_heads // w.num_kv_heads > 4 and not xsplit
                       else "warp-level products)"), dec8, s)
    res = {"kv_dtype": "e4m3", "kv_layout": "x-split" if xsplit else "token-major",
           "us_per_call": round(s * 1e6, 2), "kv_gbs": round(kv8 / s / 1e9, 2),
           "decode_gbs": round(dec8 / s / 1e9, 2),
           "frac_of_measured_peak": rl["frac"],
           "kv_tokens_per_us": round(ab["kv_unique_tokens"] / (s * 1e6), 1), "roofline": rl}
    del kc, vc
    torch.cuda.empty_cache()
    return res


def extra_decode(pa, name, dev, flush, reps=20, cpu=True):
    """Decode-only timing of another named workload, with its own roofline
    block (and, for token-major bf16 caches, the oracle on the host cores).
    Suffix _fp8: over an e4m3 copy of the cache; _xsplit: over the x-split
    layout (K [blocks, kv heads, d / 8, block, 8], V [blocks, kv heads, d,
    block]) of the same cache."""
    if name.endswith("_fp8_xsplit"):
        return extra_decode_fp8(pa, name[:-len("_fp8_xsplit")], dev, flush, reps, xsplit=True)
    if name.endswith("_fp8"):
        return extra_decode_fp8(pa, name[:-len("_fp8")], dev, flush, reps)
    xsplit = name.endswith("_xsplit")
    if xsplit:
        name = name[:-len("_xsplit")]
    if wl.NAMED[name]().max_query_len > 1:
        return extra_mixed(pa, name, dev, flush, reps, cpu=cpu)
    w = wl.NAMED[name]()
    t = wl.make_tensors(w, device=dev)
    ab = algorithmic_bytes(w)
    ws = pa.new_workspace(pa.decode_workspace_size(w.num_seqs, w.num_heads, w.num_kv_heads,
                                                   w.head_dim, w.max_seq_len), dev)
    out = torch.empty_like(t.q)
    if xsplit:
        nb, B, H, d = t.key_cache.shape
        kx = t.key_cache.view(nb, B, H, d // 8, 8).permute(0, 2, 3, 1, 4).contiguous()
        vx = t.value_cache.view(nb, B, H, d).permute(0, 2, 3, 1).contiguous()
        call = lambda: pa.decode_xsplit(t.q, kx, vx, t.block_tables, t.seq_lens, w.max_seq_len,
                                        w.scale, out=out, workspace=ws)
    else:
        call = lambda: pa.decode(t.q, t.key_cache, t.value_cache, t.block_tables, t.seq_lens,
                                 w.max_seq_len, w.scale, out=out, workspace=ws)
    s = _time(call, flush, reps)
    kernel = "paged_decode_kernel (pa_decode_xsplit)" if xsplit else decode_kernel_name(w)
    rl = hbm_roofline(kernel, ab["decode_bytes"], s, None if xsplit else profiled_traffic(w.name))
    res = {"kv_layout": "x-split" if xsplit else "token-major",
           "us_per_call": round(s * 1e6, 2), "kv_gbs": round(ab["kv_bytes"] / s / 1e9, 2),
           "decode_gbs": round(ab["decode_bytes"] / s / 1e9, 2),
           "frac_of_measured_peak": rl["frac"],
           "kv_unique_tokens": ab["kv_unique_tokens"], "kv_logical_tokens": ab["kv_logical_tokens"],
           "roofline": rl}
    if cpu and not xsplit:
        res["cpu_baseline"] = cpu_baseline(w, t, ab, single_core=False)
    if xsplit:
        del kx, vx
    del t, call
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU baseline

def _bits(x):
    return x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle(threads):
    from oracle import Oracle
    o = Oracle()
    o.set_threads(threads)
    return o


def _oracle_sample(w, kc, vc, q, rows, threads=1):
    o = _oracle(threads)
    t0 = time.perf_counter()
    o.decode(q[rows], kc, vc, w.block_tables[rows], w.seq_lens[rows], w.scale)
    return time.perf_counter() - t0


def _sample_bytes(w, rows):
    sub = wl.Workload(w.name, w.seq_lens[rows], w.q_lens[rows],
                      np.concatenate([[0], np.cumsum(w.q_lens[rows])]).astype(np.int32),
                      w.block_tables[rows], w.num_heads, w.num_kv_heads, w.head_dim,
                      w.block_size, w.num_blocks, w.scale, w.seed, w.shared_blocks)
    return algorithmic_bytes(sub)["decode_bytes"]


def cpu_baseline(w, t, ab, single_core=True):
    """The oracle, as it stands, timed on the host: one decode of the whole
    batch on every core (OpenMP over independent (request, head) rows; the
    same arithmetic as on one core), and, as context, a bounded sample of
    the batch on one core."""
    kc, vc, q = _bits(t.key_cache), _bits(t.value_cache), _bits(t.q)
    cores = min(host_cores(), _oracle(1).max_threads())
    rows = np.arange(w.num_seqs)
    secs = _oracle_sample(w, kc, vc, q, rows, threads=cores)
    b = _sample_bytes(w, rows)
    res = {"value": round(b / secs / 1e9, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": f"oracle decode of all {w.num_seqs} requests of {w.name} (fp64, "
                     f"{cores} threads over (request, head) rows), {secs:.2f} s"}
    if single_core:
        rows1 = _rows_for_fraction(w, 0.25)
        secs1 = _oracle_sample(w, kc, vc, q, rows1, threads=1)
        res["single_core"] = {
            "value": round(_sample_bytes(w, rows1) / secs1 / 1e9, 4), "unit": "GB/s", "cores": 1,
            "sample": f"oracle decode of requests 0..{rows1[-1]} ({len(rows1)} of {w.num_seqs}), "
                      f"fp64, one thread, {secs1:.2f} s"}
    return res


def cpu_baseline_prefill(w, t):
    """The oracle's varlen prefill of the whole mixed batch on every core,
    as causal-pair FLOP/s of the prefill rows (the tensor-core kernel's
    unit) and KV GB/s of the batch."""
    cores = min(host_cores(), _oracle(1).max_threads())
    o = _oracle(cores)
    kc, vc, q = _bits(t.key_cache), _bits(t.value_cache), _bits(t.q)
    t0 = time.perf_counter()
    o.prefill_varlen(q, kc, vc, w.query_start_loc, w.seq_lens, w.block_tables, w.scale)
    secs = time.perf_counter() - t0
    flops = 4.0 * causal_pairs(w) * w.num_heads * w.head_dim
    ab = algorithmic_bytes(w)
    return {"value": round(ab["decode_bytes"] / secs / 1e9, 4), "unit": "GB/s",
            "prefill_gflops": round(flops / secs / 1e9, 3), "cores": cores, "kind": "oracle",
            "sample": f"oracle varlen attention of the whole {w.name} batch (fp64, {cores} "
                      f"threads), {secs:.2f} s"}


def _rows_for_fraction(w, frac):
    lens = w.seq_lens.astype(np.int64)
    c = np.cumsum(lens)
    n = int(np.searchsorted(c, frac * c[-1])) + 1
    return np.arange(min(max(n, 1), w.num_seqs))


# --------------------------------------------------------- reference arm

def run_reference(args, world, rank):
    """The oracle, as it stands, on every host core: each step is one decode
    of the whole workload when the --steps K --warmup W run fits in about
    two minutes that way, else of its first requests, sized to fit."""
    if rank != 0:
        return None, rank
    w = wl.NAMED[args.workload]()
    t = wl.make_tensors(w, device="cpu")
    kc, vc, q = _bits(t.key_cache), _bits(t.value_cache), _bits(t.q)
    cores = min(host_cores(), _oracle(1).max_threads())
    rows = np.arange(w.num_seqs)
    probe = _oracle_sample(w, kc, vc, q, rows, threads=cores)
    budget = 120.0
    if probe * (args.steps + args.warmup) > budget:
        frac = max(budget / (args.steps + args.warmup) / probe, 0.01)
        rows = _rows_for_fraction(w, frac)
    b = _sample_bytes(w, rows)
    for _ in range(args.warmup):
        _oracle_sample(w, kc, vc, q, rows, threads=cores)
    secs = [_oracle_sample(w, kc, vc, q, rows, threads=cores) for _ in range(args.steps)]
    tot = sum(secs)
    v = b * args.steps / tot / 1e9
    whole = len(rows) == w.num_seqs
    sample = (f"oracle decode of {'all' if whole else 'the first'} {len(rows)} of {w.num_seqs} "
              f"requests of {w.name} per step (fp64, {cores} threads over (request, head) rows)")
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(tot / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "sample_rows": len(rows), "num_seqs": w.num_seqs},
            "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}, rank


# -------------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama8b_decode_b64", choices=sorted(wl.NAMED))
    ap.add_argument("--extra", nargs="*", default=["long_ctx_decode_8x32k",
                                                    "prefix_shared_decode_b256",
                                                    "mixed_chunked_prefill",
                                                    "multi_chunk_prefill",
                                                    "llama8b_decode_b64_fp8",
                                                    "prefix_shared_decode_b256_fp8",
                                                    "llama8b_decode_b64_fp8_xsplit",
                                                    "llama8b_decode_b64_xsplit",
                                                    "prefix_shared_decode_b256_xsplit"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        res, rank = run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py: no CUDA device (the library has no CPU path)")
        res, rank = run_ours(args, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
