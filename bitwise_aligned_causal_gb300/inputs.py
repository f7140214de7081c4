"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no attention arithmetic: it only draws numbers and rounds
them to bf16.  Both the CUDA path and the CPU oracle are fed the same bytes
from here, so the two never depend on each other.

Recipe (shapes and distributions of the KernelBraid README "Features" grid):
* numpy ``default_rng(seed)`` draws float32 normals; q, k, v are drawn in that
  order (so a tensor's bytes depend only on the seed and the shapes).
* Each float32 is rounded to bf16 with round-to-nearest-even by integer bit
  arithmetic (``f32_to_bf16_bits``).
* The stress recipe draws q, k from N(0, 8^2), then scales exactly
  round(0.01 * rows) key rows per (batch, kv-head), picked without
  replacement, by 32 before the bf16 rounding; v stays N(0, 1).
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

HEAD_DIM = 128
N_Q_HEADS = 32
N_KV_HEADS = 8


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); return uint16 bits."""
    a = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(a)):
        raise ValueError("inputs must be finite")
    u = a.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(rng: np.random.Generator, shape, sigma: float = 1.0, chunk: int = 1 << 26) -> np.ndarray:
    """Draw N(0, sigma^2) float32 in chunks and round to bf16 bits."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = rng.standard_normal(e - s, dtype=np.float32)
        if sigma != 1.0:
            x *= np.float32(sigma)
        out[s:e] = f32_to_bf16_bits(x)
    return out.reshape(shape)


@dataclass
class QKV:
    """bf16 bit patterns: q [B,Hq,Lq,D], k and v [B,Hkv,cap,D]."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray


def make_qkv(B: int, S: int, seed: int, *, Hq: int = N_Q_HEADS, Hkv: int = N_KV_HEADS,
             D: int = HEAD_DIM, Lq: int | None = None) -> QKV:
    """iid N(0, 1) q, k, v rounded to bf16, drawn in the order q, k, v.

    k and v hold S key rows; q holds Lq rows (default S).
    """
    rng = np.random.default_rng(seed)
    Lq = S if Lq is None else Lq
    q = _normal_bf16(rng, (B, Hq, Lq, D))
    k = _normal_bf16(rng, (B, Hkv, S, D))
    v = _normal_bf16(rng, (B, Hkv, S, D))
    return QKV(q, k, v)


def make_stress_qkv(B: int, S: int, seed: int, *, Hq: int = N_Q_HEADS, Hkv: int = N_KV_HEADS,
                    D: int = HEAD_DIM, sigma_qk: float = 8.0, frac_peaked: float = 0.01,
                    peak_scale: float = 32.0) -> QKV:
    """Peaked-softmax recipe: q, k ~ N(0, 8^2), 1% of key rows scaled x32, v ~ N(0,1)."""
    rng = np.random.default_rng(seed)
    q = _normal_bf16(rng, (B, Hq, S, D), sigma_qk)
    n_peak = int(round(frac_peaked * S))
    k = np.empty((B, Hkv, S, D), dtype=np.uint16)
    for b in range(B):
        for g in range(Hkv):
            x = rng.standard_normal((S, D), dtype=np.float32) * np.float32(sigma_qk)
            idx = rng.choice(S, size=n_peak, replace=False)
            x[idx] *= np.float32(peak_scale)
            k[b, g] = f32_to_bf16_bits(x)
    v = _normal_bf16(rng, (B, Hkv, S, D), 1.0)
    return QKV(q, k, v)


def chunk_lengths(total: int, seed: int, lo: int = 1, hi: int = 2048) -> list[int]:
    """Seeded chunk lengths, uniform in [lo, hi], summing to ``total``.

    Draws until the running sum reaches ``total``; the last chunk is cut short.
    """
    rng = np.random.default_rng(seed)
    out: list[int] = []
    acc = 0
    while acc < total:
        n = int(rng.integers(lo, hi + 1))
        n = min(n, total - acc)
        out.append(n)
        acc += n
    return out


def sample_rows(B: int, Hq: int, L: int, per_bh: int, seed: int) -> np.ndarray:
    """(b, h, i) triples: per (b, h) rows 0 and L-1 plus others drawn without replacement."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        for h in range(Hq):
            if L <= per_bh:
                idx = np.arange(L)
            else:
                mid = rng.choice(np.arange(1, L - 1), size=per_bh - 2, replace=False)
                idx = np.concatenate([[0, L - 1], np.sort(mid)])
            for i in idx:
                rows.append((b, h, int(i)))
    return np.asarray(rows, dtype=np.int32)


# Seeds of the five workloads.  The prefill and decode sweeps use one seed
# per (S or ctx, B) cell.
SEED_CONFIG1 = 0


def seed_prefill_sweep(S: int, B: int) -> int:
    return 1_000_000 + 1000 * (S // 1024) + B


def seed_decode_sweep(ctx: int, B: int) -> int:
    return 2_000_000 + 10 * ctx + B


SEED_PARTITIONED = 3_000_000
SEED_PARTITIONED_CHUNKS = 3_000_001
SEED_STRESS_PREFILL = 5_000_000
SEED_STRESS_DECODE = 5_000_001
