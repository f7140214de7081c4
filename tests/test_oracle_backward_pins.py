"""Pins of the backward oracle (dq, dk, dv of causal GQA attention).

The gradient has no printed worked example on the pages, so it is pinned
to things other than its own formulas (KernelBraid README, "Motivation":
the policy update of RL training differentiates this attention):

* central finite differences of the forward oracle, itself pinned by
  closed forms and brute force in test_oracle_pins.py;
* float64 autograd of an attention expression written with PyTorch ops;
* closed forms: one visible key gives dq = 0; sum_j dv_j = sum of dO over
  the group's rows; sum_j dk_j = 0 (softmax rows sum to one);
* invariants: adding one vector to every key leaves dq unchanged; dO of
  one query head moves only its own dq and its group's dk, dv;
* the row statistics (lse, delta) against the forward oracle.
"""

import math

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs

D = 128


def grid_bits(rng, shape, step=2.0 ** -8, bound=0.99):
    """bf16 bits of values on a 2^-8 grid in (-bound, bound): exact in bf16,
    and x +- 2^-8 stays exact, so finite differences move one input only."""
    x = np.round(rng.uniform(-bound, bound, size=shape) / step) * step
    return inputs.f32_to_bf16_bits(x.astype(np.float32)), x


def bits_to_f64(bits):
    u = (np.asarray(bits, dtype=np.uint32) << 16).astype(np.uint32)
    return u.view(np.float32).astype(np.float64)


def make_small_case():
    rng = np.random.default_rng(4242)
    B, Hq, Hkv, S = 1, 8, 2, 7
    q, _ = grid_bits(rng, (B, Hq, S, D))
    k, _ = grid_bits(rng, (B, Hkv, S, D))
    v, _ = grid_bits(rng, (B, Hkv, S, D))
    do, _ = grid_bits(rng, (B, Hq, S, D))
    return q, k, v, do


@pytest.fixture(scope="module")
def small_case():
    return make_small_case()


def loss(oracle_mod, q, k, v, do):
    """L = sum(dO * O) with O from the forward oracle."""
    o = oracle_mod.attention_full(q, k, v)
    return float(np.sum(o * bits_to_f64(do)))


def test_finite_differences(oracle_mod, small_case):
    q, k, v, do = small_case
    dq, dk, dv = oracle_mod.backward(q, k, v, do)
    rng = np.random.default_rng(7)
    h = 2.0 ** -8
    for name, arr, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in arr.shape)
            x0 = bits_to_f64(arr[idx])
            plus, minus = arr.copy(), arr.copy()
            plus[idx] = inputs.f32_to_bf16_bits(np.array([x0 + h], dtype=np.float32))[0]
            minus[idx] = inputs.f32_to_bf16_bits(np.array([x0 - h], dtype=np.float32))[0]
            assert bits_to_f64(plus[idx]) == x0 + h and bits_to_f64(minus[idx]) == x0 - h
            args = {"q": (q, k, v), "k": (q, k, v), "v": (q, k, v)}[name]
            lp = loss(oracle_mod, *[plus if a is arr else a for a in args], do)
            lm = loss(oracle_mod, *[minus if a is arr else a for a in args], do)
            fd = (lp - lm) / (2 * h)
            scale = max(1e-3, float(np.abs(grad).max()))
            assert abs(fd - grad[idx]) <= 2e-4 * scale, (name, idx, fd, grad[idx])


def test_against_float64_autograd(oracle_mod):
    torch = pytest.importorskip("torch")
    x = inputs.make_qkv(2, 23, seed=4243, Hq=8, Hkv=2)
    do = inputs.make_qkv(2, 23, seed=4244, Hq=8, Hkv=2).q
    dq, dk, dv = oracle_mod.backward(x.q, x.k, x.v, do)

    q = torch.tensor(bits_to_f64(x.q), requires_grad=True)
    k = torch.tensor(bits_to_f64(x.k), requires_grad=True)
    v = torch.tensor(bits_to_f64(x.v), requires_grad=True)
    g = torch.tensor(bits_to_f64(do))
    group = q.shape[1] // k.shape[1]
    kk = k.repeat_interleave(group, dim=1)
    vv = v.repeat_interleave(group, dim=1)
    S = q.shape[2]
    scores = torch.matmul(q, kk.transpose(-1, -2)) / math.sqrt(D)
    future = torch.triu(torch.ones(S, S, dtype=torch.bool), diagonal=1)
    scores = scores.masked_fill(future, float("-inf"))
    o = torch.matmul(torch.softmax(scores, dim=-1), vv)
    gq, gk, gv = torch.autograd.grad((o * g).sum(), (q, k, v))
    for mine, ref in ((dq, gq), (dk, gk), (dv, gv)):
        ref = ref.numpy()
        assert np.abs(mine - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())


def test_one_visible_key(oracle_mod):
    """S = 1: P = 1, so dS = 0 (dq = dk = 0) and dv_0 = sum of dO over the group's heads."""
    rng = np.random.default_rng(4245)
    q, _ = grid_bits(rng, (2, 8, 1, D))
    k, _ = grid_bits(rng, (2, 2, 1, D))
    v, _ = grid_bits(rng, (2, 2, 1, D))
    do, dof = grid_bits(rng, (2, 8, 1, D))
    dq, dk, dv = oracle_mod.backward(q, k, v, do)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    want = dof.reshape(2, 2, 4, 1, D).sum(axis=2)
    assert np.array_equal(dv, want)


def test_row_zero_and_sum_rules(oracle_mod):
    x = inputs.make_qkv(2, 40, seed=4246, Hq=8, Hkv=2)
    do = inputs.make_qkv(2, 40, seed=4247, Hq=8, Hkv=2).q
    dq, dk, dv = oracle_mod.backward(x.q, x.k, x.v, do)
    assert np.all(dq[:, :, 0] == 0.0)                                   # row 0 sees one key
    scale = np.abs(dk).max()
    assert np.abs(dk.sum(axis=2)).max() <= 1e-12 * scale * 40           # rows of dS sum to zero
    want = bits_to_f64(do).reshape(2, 2, 4, 40, D).sum(axis=(2, 3))   # P rows sum to one
    assert np.abs(dv.sum(axis=2) - want).max() <= 1e-12 * np.abs(want).max() * 40


def test_key_shift_leaves_dq(oracle_mod):
    """Adding one vector to every key shifts a row's scores by a constant."""
    rng = np.random.default_rng(4248)
    q, _ = grid_bits(rng, (1, 4, 12, D), step=2.0 ** -6, bound=0.45)
    k, kf = grid_bits(rng, (1, 1, 12, D), step=2.0 ** -6, bound=0.45)
    v, _ = grid_bits(rng, (1, 1, 12, D))
    do, _ = grid_bits(rng, (1, 4, 12, D))
    shift = np.where(rng.random(D) < 0.5, 0.25, -0.25)
    k2 = inputs.f32_to_bf16_bits((kf + shift).astype(np.float32))
    assert np.array_equal(bits_to_f64(k2), kf + shift)
    dq1, _, _ = oracle_mod.backward(q, k, v, do)
    dq2, _, _ = oracle_mod.backward(q, k2, v, do)
    assert np.abs(dq1 - dq2).max() <= 1e-12 * np.abs(dq1).max()


def test_gqa_locality(oracle_mod):
    """dO of head 5 (group 1 of 2) moves dq of head 5 and dk, dv of group 1 only."""
    x = inputs.make_qkv(1, 16, seed=4249, Hq=8, Hkv=2)
    do = inputs.make_qkv(1, 16, seed=4250, Hq=8, Hkv=2).q
    do2 = do.copy()
    do2[0, 5] = inputs.make_qkv(1, 16, seed=4251, Hq=8, Hkv=2).q[0, 5]
    a = oracle_mod.backward(x.q, x.k, x.v, do)
    b = oracle_mod.backward(x.q, x.k, x.v, do2)
    changed_q = [h for h in range(8) if not np.array_equal(a[0][0, h], b[0][0, h])]
    assert changed_q == [5]
    assert np.array_equal(a[1][0, 0], b[1][0, 0]) and np.array_equal(a[2][0, 0], b[2][0, 0])
    assert not np.array_equal(a[1][0, 1], b[1][0, 1]) and not np.array_equal(a[2][0, 1], b[2][0, 1])


def test_row_statistics_against_forward(oracle_mod):
    """dq_rows agrees with the full backward; its lse reproduces the forward
    oracle's output through sum_j exp(s_ij - lse_i) v_j, and delta = dO_i . o_i."""
    x = inputs.make_qkv(2, 50, seed=4252, Hq=8, Hkv=2)
    do = inputs.make_qkv(2, 50, seed=4253, Hq=8, Hkv=2).q
    dq, _, _ = oracle_mod.backward(x.q, x.k, x.v, do)
    rows = [(0, 0, 0), (0, 3, 17), (1, 7, 49), (1, 4, 1), (0, 6, 33)]
    dqr, lse, delta = oracle_mod.dq_rows(x.q, x.k, x.v, do, rows)
    o = oracle_mod.attention_rows(x.q, x.k, x.v, rows)
    qf, kf, vf, dof = (bits_to_f64(a) for a in (x.q, x.k, x.v, do))
    for r, (b, h, i) in enumerate(rows):
        assert np.abs(dqr[r] - dq[b, h, i]).max() <= 1e-13 * max(1.0, np.abs(dq[b, h, i]).max())
        g = h // 4
        s = kf[b, g, :i + 1] @ qf[b, h, i] / math.sqrt(D)
        o_from_lse = np.exp(s - lse[r]) @ vf[b, g, :i + 1]
        assert np.abs(o_from_lse - o[r]).max() <= 1e-12
        assert abs(delta[r] - float(dof[b, h, i] @ o[r])) <= 1e-12 * max(1.0, abs(delta[r]))
