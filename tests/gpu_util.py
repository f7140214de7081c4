"""Helpers shared by the GPU tests: moving bf16 bit patterns to and from the
device, and comparing GPU rows with the oracle."""

import numpy as np

from bitwise_aligned_causal_gb300.inputs import bf16_bits_to_f32

# Tolerance of a bf16 output row against the fp64 oracle.
MAX_ABS_TOL = 2e-2
MEAN_ABS_TOL = 2e-3


def to_dev(bits):
    import torch

    a = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()


def from_dev(t):
    import torch

    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def compare(gpu_bits, oracle_vals):
    """(max_abs, mean_abs) of bf16 GPU rows against float64 oracle rows."""
    g = bf16_bits_to_f32(gpu_bits).astype(np.float64)
    d = np.abs(g - np.asarray(oracle_vals, dtype=np.float64))
    return float(d.max()), float(d.mean())


def assert_close_to_oracle(gpu_bits, oracle_vals, what=""):
    mx, mean = compare(gpu_bits, oracle_vals)
    assert np.all(np.isfinite(bf16_bits_to_f32(gpu_bits))), f"{what}: non-finite output"
    assert mx <= MAX_ABS_TOL and mean <= MEAN_ABS_TOL, f"{what}: max-abs {mx:.3e} mean-abs {mean:.3e}"
    return mx, mean


def gather_rows(bits_bhld, rows):
    """Select (b, h, i) rows from a [B, H, L, D] array."""
    r = np.asarray(rows)
    return bits_bhld[r[:, 0], r[:, 1], r[:, 2]]
