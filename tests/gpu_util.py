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


# --------------------------------------------------------------- rescale coverage
#
# The contract's row function moves a row's reference max m only when a later
# key tile's max t exceeds it by more than 64 raw score units (t - m > 64, in
# fp32 scores q . k), and only then rescales the row's O accumulator.  A
# bitwise test exercises that branch only if its rows really take it.  The
# helper below replays the decision on the host in float64 and keeps only
# decisions that no fp32 rounding of the scores can flip: a score summed from
# 128 exact bf16 products in any fp32 order is within 128 * 2^-24 * sum|q_i k_i|
# of the exact value.

def rescale_after_first_tile(q_bits, k_bits, positions, tile=128, threshold=64.0):
    """For query rows q_bits [n, D] at absolute `positions` against keys
    k_bits [S, D] (bf16 bits), return a bool array: True where the row's
    reference max certainly moves on some key tile after tile 0."""
    from bitwise_aligned_causal_gb300.inputs import bf16_bits_to_f32

    q = bf16_bits_to_f32(q_bits).astype(np.float64)
    k = bf16_bits_to_f32(k_bits).astype(np.float64)
    pos = np.asarray(positions)
    s = q @ k.T
    bound = 128.0 * 2.0 ** -24 * (np.abs(q) @ np.abs(k).T)
    cols = np.arange(k.shape[0])
    s = np.where(cols[None, :] <= pos[:, None], s, -np.inf)
    n_tiles = (k.shape[0] + tile - 1) // tile
    pad = n_tiles * tile - k.shape[0]
    sp = np.pad(s, ((0, 0), (0, pad)), constant_values=-np.inf).reshape(len(pos), n_tiles, tile)
    bp = np.pad(bound, ((0, 0), (0, pad))).reshape(len(pos), n_tiles, tile)
    tmax = sp.max(axis=2)
    tbound = bp.max(axis=2)
    m = tmax[:, 0].copy()
    mb = tbound[:, 0].copy()
    moved = np.zeros(len(pos), bool)
    sure = np.ones(len(pos), bool)
    for j in range(1, n_tiles):
        live = j <= pos // tile
        d = tmax[:, j] - m
        margin = np.abs(d - threshold) > 2.0 * (tbound[:, j] + mb)
        sure &= ~live | margin
        mv = live & (d > threshold)
        moved |= mv & sure
        m = np.where(mv, tmax[:, j], m)
        mb = np.where(mv, tbound[:, j], mb)
    return moved & sure


def rescale_fraction(x, rows, tile=128):
    """Fraction of (b, h, i) rows of an input set (inputs.QKV, query row i at
    position i) whose reference max certainly moves after key tile 0."""
    rows = np.asarray(rows)
    hits = 0
    for b in np.unique(rows[:, 0]):
        for h in np.unique(rows[rows[:, 0] == b][:, 1]):
            sel = rows[(rows[:, 0] == b) & (rows[:, 1] == h)]
            g = h * x.k.shape[1] // x.q.shape[1]
            hits += int(rescale_after_first_tile(x.q[b, h, sel[:, 2]], x.k[b, g], sel[:, 2], tile).sum())
    return hits / len(rows)
