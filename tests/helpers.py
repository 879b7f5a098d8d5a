"""Shared helpers of the GPU parity tests."""
import numpy as np
import torch

# Tolerances for bf16 attention outputs against the fp64 oracle (N(0,1) inputs).
MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a bf16 tensor as a host numpy uint16 array."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_close_to_oracle(got: torch.Tensor, ref: np.ndarray, rows=None, what=""):
    g = got.double().cpu().numpy()
    if rows is not None:
        g = g[rows]
        ref = ref[rows] if ref.shape[0] == got.shape[0] else ref
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    err = np.abs(g - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3e}, mean abs {mean:.3e}"
    return mx, mean


def oracle_decode_rows(oracle, w, t, rows):
    """Oracle decode output for a subset of requests (their rows only)."""
    rows = np.asarray(rows)
    return oracle.decode(bits(t.q)[rows], bits(t.key_cache), bits(t.value_cache),
                         w.block_tables[rows], w.seq_lens[rows], w.scale)
