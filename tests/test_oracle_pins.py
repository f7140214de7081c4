"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

The attention computed is plain causal GQA attention (KernelBraid README,
"Features": BF16, causal, [batch, heads, sequence, head_dim], 32 query heads,
8 KV heads, head_dim 128; "Usage": prefill and one-token decode over the same
KV context).  Each test below would fail for a plausible slip in the oracle:
a dropped 1/sqrt(D) scale, an off-by-one causal boundary, a wrong GQA group
map, a wrong sign, a transposed operand or a wrong KV stride.
"""

import math

import numpy as np
import pytest

from bitwise_aligned_causal_gb300.inputs import bf16_bits_to_f32, f32_to_bf16_bits, make_qkv

D = 128


def bits(x):
    """float array -> bf16 bits; the values used in these pins are exact in bf16."""
    a = np.asarray(x, dtype=np.float32)
    b = f32_to_bf16_bits(a)
    assert np.array_equal(bf16_bits_to_f32(b), a), "pin values must be exact in bf16"
    return b


def small_qkv(B, Hq, Hkv, S, seed, scale=1.0, cap=None):
    rng = np.random.default_rng(seed)
    cap = S if cap is None else cap
    q = f32_to_bf16_bits(rng.standard_normal((B, Hq, S, D)).astype(np.float32) * np.float32(scale))
    k = f32_to_bf16_bits(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32) * np.float32(scale))
    v = f32_to_bf16_bits(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32))
    return q, k, v


# ---------------------------------------------------------------- closed forms

def test_first_row_is_v0_exactly(oracle_mod):
    """A causal row at position 0 sees one key: softmax weight 1, output V[0]."""
    q, k, v = small_qkv(2, 32, 8, 5, seed=1)
    out = oracle_mod.attention_full(q, k, v)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    for h in range(32):
        assert np.array_equal(out[:, h, 0, :], vf[:, h // 4, 0, :])


def test_decode_context_one_is_v0(oracle_mod):
    q, k, v = small_qkv(1, 32, 8, 1, seed=2, cap=7)
    out = oracle_mod.attention_rows(q, k, v, [(0, h, 0) for h in range(32)], start=0)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    for h in range(32):
        assert np.array_equal(out[h], vf[0, h // 4, 0])


def test_identical_keys_give_cumulative_mean(oracle_mod):
    """All keys equal -> uniform softmax -> row p is the mean of V[0..p]."""
    S = 40
    q, k, v = small_qkv(1, 4, 1, S, seed=3)
    k[:] = k[:, :, :1, :]
    out = oracle_mod.attention_full(q, k, v)
    vf = bf16_bits_to_f32(v).astype(np.float64)[0, 0]
    for p in range(S):
        want = np.array([math.fsum(vf[: p + 1, d]) / (p + 1) for d in range(D)])
        for h in range(4):
            np.testing.assert_allclose(out[0, h, p], want, rtol=0, atol=1e-13)


def test_zero_query_gives_cumulative_mean(oracle_mod):
    S = 33
    q, k, v = small_qkv(1, 4, 1, S, seed=4)
    q[:] = 0
    out = oracle_mod.attention_full(q, k, v)
    vf = bf16_bits_to_f32(v).astype(np.float64)[0, 0]
    want = np.cumsum(vf, axis=0) / np.arange(1, S + 1)[:, None]
    np.testing.assert_allclose(out[0, 2], want, rtol=0, atol=1e-13)


def test_dominant_key_selects_its_value_row(oracle_mod):
    """One key with a score margin above 60 takes all the weight (e^-60 ~ 1e-26)."""
    S = 24
    star = 9
    qf = np.zeros((1, 4, S, D), np.float32)
    qf[..., 0] = 8.0
    kf = np.zeros((1, 1, S, D), np.float32)
    kf[0, 0, star, 0] = 128.0            # score 8*128/sqrt(128) = 90.5 vs 0
    rng = np.random.default_rng(5)
    kf[0, 0, :, 1:] = np.round(rng.standard_normal((S, D - 1)) * 4) / 4   # q is 0 there
    vf = (np.round(rng.standard_normal((1, 1, S, D)) * 8) / 8).astype(np.float32)
    out = oracle_mod.attention_full(bits(qf), bits(kf), bits(vf))
    for p in range(star, S):
        np.testing.assert_allclose(out[0, 1, p], vf[0, 0, star], rtol=0, atol=1e-20)
    # before the dominant key is visible the scores are all 0: cumulative mean
    for p in range(star):
        np.testing.assert_allclose(out[0, 1, p], vf[0, 0, : p + 1].astype(np.float64).mean(axis=0), rtol=0, atol=1e-13)


def test_negative_dominant_key_is_suppressed(oracle_mod):
    """The sign matters: a key with score -90 gets weight ~e^-90."""
    S = 6
    qf = np.zeros((1, 4, S, D), np.float32)
    qf[..., 0] = 8.0
    kf = np.zeros((1, 1, S, D), np.float32)
    kf[0, 0, 2, 0] = -128.0
    vf = np.zeros((1, 1, S, D), np.float32)
    vf[0, 0, :, 0] = [1, 2, 1000, 3, 4, 5]
    out = oracle_mod.attention_full(bits(qf), bits(kf), bits(vf))
    for p in range(3, S):
        visible = [x for j, x in enumerate([1, 2, 1000, 3, 4, 5][: p + 1]) if j != 2]
        assert abs(out[0, 0, p, 0] - sum(visible) / len(visible)) < 1e-20 * 1000 + 1e-13


def test_two_keys_closed_form_fixes_the_scale(oracle_mod):
    """Row 1 sees keys 0 and 1: o = v0 + (v1 - v0) * logistic((s1 - s0)), s = q.k / sqrt(128)."""
    qf = np.zeros((1, 4, 2, D), np.float32)
    kf = np.zeros((1, 1, 2, D), np.float32)
    vf = np.zeros((1, 1, 2, D), np.float32)
    qf[0, :, 1, 0] = 3.0
    qf[0, :, 1, 1] = -1.5
    kf[0, 0, 0, 0] = 0.5
    kf[0, 0, 0, 1] = 2.0
    kf[0, 0, 1, 0] = 2.0
    kf[0, 0, 1, 1] = 0.25
    vf[0, 0, 0, :] = np.linspace(-2, 2, D, dtype=np.float32).round(2)
    vf[0, 0, 1, :] = np.linspace(3, -1, D, dtype=np.float32).round(2)
    qb, kb, vb = bits(qf), bits(kf), f32_to_bf16_bits(vf)
    out = oracle_mod.attention_full(qb, kb, vb)
    v0 = bf16_bits_to_f32(vb)[0, 0, 0].astype(np.float64)
    v1 = bf16_bits_to_f32(vb)[0, 0, 1].astype(np.float64)
    s0 = (3.0 * 0.5 + -1.5 * 2.0) / math.sqrt(128.0)
    s1 = (3.0 * 2.0 + -1.5 * 0.25) / math.sqrt(128.0)
    w1 = 1.0 / (1.0 + math.exp(-(s1 - s0)))
    np.testing.assert_allclose(out[0, 3, 1], v0 + (v1 - v0) * w1, rtol=0, atol=1e-14)
    # the unscaled variant would differ by far more than the tolerance
    w1_unscaled = 1.0 / (1.0 + math.exp(-(s1 - s0) * math.sqrt(128.0)))
    assert np.max(np.abs((v0 + (v1 - v0) * w1_unscaled) - out[0, 3, 1])) > 1e-2


def test_constant_value_column_passes_through(oracle_mod):
    q, k, v = small_qkv(1, 8, 2, 50, seed=6)
    v[..., 17] = f32_to_bf16_bits(np.float32(-0.3125))
    out = oracle_mod.attention_full(q, k, v)
    np.testing.assert_allclose(out[..., 17], -0.3125, rtol=0, atol=1e-15)


def test_outputs_lie_in_convex_hull_of_visible_values(oracle_mod):
    q, k, v = small_qkv(1, 4, 1, 30, seed=7, scale=2.0)
    out = oracle_mod.attention_full(q, k, v)
    vf = bf16_bits_to_f32(v).astype(np.float64)[0, 0]
    for p in range(30):
        lo = vf[: p + 1].min(axis=0) - 1e-12
        hi = vf[: p + 1].max(axis=0) + 1e-12
        assert np.all(out[0, :, p] >= lo) and np.all(out[0, :, p] <= hi)


# ------------------------------------------------------------------ invariants

def test_common_score_shift_leaves_rows_unchanged(oracle_mod):
    """A shared key component c shifts every score of a row by q_0 * c / sqrt(D)."""
    q, k, v = small_qkv(1, 4, 1, 20, seed=8)
    k[..., 0] = f32_to_bf16_bits(np.float32(4.0))
    q2 = q.copy()
    q2[..., 0] = f32_to_bf16_bits(np.float32(6.0))
    a = oracle_mod.attention_full(q, k, v)
    b = oracle_mod.attention_full(q2, k, v)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


def test_gqa_groups_are_contiguous(oracle_mod):
    """Query head h reads KV head h // (Hq/Hkv): changing KV head g moves heads 4g..4g+3 only."""
    q, k, v = small_qkv(1, 32, 8, 12, seed=9)
    base = oracle_mod.attention_full(q, k, v)
    for g in (0, 3, 7):
        k2, v2 = k.copy(), v.copy()
        rng = np.random.default_rng(100 + g)
        v2[0, g] = f32_to_bf16_bits(rng.standard_normal((12, D)).astype(np.float32))
        k2[0, g] = f32_to_bf16_bits(rng.standard_normal((12, D)).astype(np.float32))
        out = oracle_mod.attention_full(q, k2, v2)
        changed = [h for h in range(32) if not np.array_equal(out[0, h], base[0, h])]
        assert changed == [4 * g, 4 * g + 1, 4 * g + 2, 4 * g + 3]


def test_future_keys_do_not_matter(oracle_mod):
    """Causality: rows 0..p ignore keys and values after p, bit for bit."""
    S, p = 40, 17
    q, k, v = small_qkv(1, 8, 2, S, seed=10)
    base = oracle_mod.attention_full(q, k, v)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, p + 1:] ^= np.uint16(0x1234)
    v2[:, :, p + 1:] ^= np.uint16(0x0F0F)
    out = oracle_mod.attention_full(q, k2, v2)
    assert np.array_equal(out[:, :, : p + 1], base[:, :, : p + 1])
    assert not np.array_equal(out[:, :, p + 1:], base[:, :, p + 1:])


def test_chunk_and_decode_rows_equal_full_rows(oracle_mod):
    """A query block at offset `start`, and a one-row decode block, index the same rows."""
    S = 70
    q, k, v = small_qkv(2, 8, 2, S, seed=11)
    full = oracle_mod.attention_full(q, k, v)
    start, L = 23, 31
    chunk = oracle_mod.attention_full(q[:, :, start:start + L], k, v, start=start)
    assert np.array_equal(chunk, full[:, :, start:start + L])
    dec = oracle_mod.attention_full(q[:, :, S - 1:], k, v, start=S - 1)
    assert np.array_equal(dec[:, :, 0], full[:, :, S - 1])


def test_kv_capacity_stride(oracle_mod):
    """k, v with capacity > context: rows beyond the context are never read."""
    S, cap = 20, 64
    q, k, v = small_qkv(2, 8, 2, S, seed=12)
    kc = np.zeros((2, 2, cap, D), np.uint16)
    vc = np.zeros((2, 2, cap, D), np.uint16)
    kc[:, :, :S] = k
    vc[:, :, :S] = v
    kc[:, :, S:] = 0x7FC0   # NaN bits in the unused tail
    vc[:, :, S:] = 0x7FC0
    a = oracle_mod.attention_full(q, k, v)
    b = oracle_mod.attention_full(q, kc, vc)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------- brute force

def brute_force(qb, kb, vb, Hq, Hkv):
    """Independent tiny-shape attention: direct exp(s) / sum exp(s), fsum, no max trick."""
    q = bf16_bits_to_f32(qb).astype(np.float64)
    k = bf16_bits_to_f32(kb).astype(np.float64)
    v = bf16_bits_to_f32(vb).astype(np.float64)
    B, _, S, Dd = q.shape
    out = np.zeros_like(q)
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for p in range(S):
                e = []
                for j in range(p + 1):
                    s = math.fsum(float(q[b, h, p, d]) * float(k[b, g, j, d]) for d in range(Dd))
                    e.append(math.exp(s / math.sqrt(Dd)))
                z = math.fsum(e)
                for d in range(Dd):
                    out[b, h, p, d] = math.fsum(e[j] * float(v[b, g, j, d]) for j in range(p + 1)) / z
    return out


@pytest.mark.parametrize("B,Hq,Hkv,S,seed", [(2, 4, 1, 9, 20), (1, 8, 2, 16, 21), (1, 32, 8, 3, 22)])
def test_brute_force_agreement(oracle_mod, B, Hq, Hkv, S, seed):
    q, k, v = small_qkv(B, Hq, Hkv, S, seed=seed, scale=0.5)
    want = brute_force(q, k, v, Hq, Hkv)
    got = oracle_mod.attention_full(q, k, v)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-13)


def test_threads_do_not_change_bits(oracle_mod):
    x = make_qkv(1, 96, seed=13)
    a = oracle_mod.attention_full(x.q, x.k, x.v, n_threads=1)
    b = oracle_mod.attention_full(x.q, x.k, x.v, n_threads=7)
    assert np.array_equal(a, b)


def test_bad_rows_are_rejected(oracle_mod):
    q, k, v = small_qkv(1, 4, 1, 4, seed=14)
    with pytest.raises(ValueError):
        oracle_mod.attention_rows(q, k, v, [(0, 4, 0)])
    with pytest.raises(ValueError):
        oracle_mod.attention_rows(q, k, v, [(0, 0, 0)], start=4)   # context 5 > cap 4
