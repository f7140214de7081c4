"""The seeded input generator: bf16 rounding, determinism and the workload recipes."""

import numpy as np
import torch

from bitwise_aligned_causal_gb300 import inputs


def test_bf16_rounding_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100_000).astype(np.float32) * np.float32(37.0),
        # exact ties: the halfway bit set, below it zero -> ties go to even
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x3F80C000, 0x3F807FFF], dtype=np.uint32).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -3e-39, 3.3e38], dtype=np.float32),
    ])
    ours = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_widening_is_exact():
    b = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    b = b[(b & 0x7F80) != 0x7F80]              # drop inf / NaN
    f = inputs.bf16_bits_to_f32(b)
    assert np.array_equal(inputs.f32_to_bf16_bits(f), b)


def test_generator_is_deterministic_and_ordered():
    a = inputs.make_qkv(1, 64, seed=5)
    b = inputs.make_qkv(1, 64, seed=5)
    assert np.array_equal(a.q, b.q) and np.array_equal(a.k, b.k) and np.array_equal(a.v, b.v)
    c = inputs.make_qkv(1, 64, seed=6)
    assert not np.array_equal(a.q, c.q)
    # q is drawn first: its bytes do not depend on the key length
    d = inputs.make_qkv(1, 64, seed=5, Lq=64)
    assert np.array_equal(a.q, d.q)
    x = inputs.bf16_bits_to_f32(inputs.make_qkv(2, 512, seed=1).q)
    assert abs(float(x.mean())) < 0.01 and abs(float(x.std()) - 1.0) < 0.01


def test_stress_recipe_scales_one_percent_of_key_rows():
    s = inputs.make_stress_qkv(1, 1000, seed=3, Hkv=2, Hq=8)
    k = inputs.bf16_bits_to_f32(s.k).astype(np.float64)
    norms = np.linalg.norm(k, axis=-1)         # ~ 8*sqrt(128) = 90, peaked ~ 2900
    for g in range(2):
        assert int(np.sum(norms[0, g] > 1000)) == 10
    v = inputs.bf16_bits_to_f32(s.v)
    assert abs(float(v.std()) - 1.0) < 0.02


def test_chunk_lengths():
    for seed in range(20):
        c = inputs.chunk_lengths(8192, seed)
        assert sum(c) == 8192
        assert all(1 <= n <= 2048 for n in c)


def test_sample_rows_include_ends():
    r = inputs.sample_rows(2, 4, 1000, 64, seed=1)
    assert r.shape == (2 * 4 * 64, 3)
    for b in range(2):
        for h in range(4):
            sel = r[(r[:, 0] == b) & (r[:, 1] == h), 2]
            assert 0 in sel and 999 in sel and len(set(sel.tolist())) == 64
