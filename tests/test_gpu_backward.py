"""Backward of the causal GQA attention on the GPU against the fp64 oracle.

The training forward (kb_attn_prefill_lse) must give prefill's bits plus the
row log-sum-exp; the backward (kb_attn_backward) must give dq, dk, dv within
the tolerance below of the oracle's exact gradient, the same bits on every
run (no atomics), and, at sizes where the full oracle is too slow, the sum
rules of the gradient and sampled dq rows (KernelBraid README, "Motivation":
the RL policy update differentiates the same attention).

Tolerance (derived from the arithmetic): P and dS are rounded to bf16
(relative 2^-9) before their products, the forward output o that delta
uses is bf16, and the gradients are stored as bf16 (relative 2^-9).  Sums
of many such terms with independent rounding stay within a few 2^-9 of the
result's scale, so each tensor must satisfy
    max |g - ref| <= 1e-2 * max |ref| + 1e-5   and   mean |g - ref| <= 1e-2 * mean |ref| + 1e-6,
the small absolute terms covering gradients that are exactly zero (one
visible key), where rounding leaves values of order 1e-7.  Measured: 2-5e-3
(max) and 2.3e-3 (mean) of the scale.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu

D = 128
REL_MAX = 1e-2
REL_MEAN = 1e-2


@pytest.fixture(scope="module")
def kb():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bitwise_aligned_causal_gb300 import build

    build.build()
    from bitwise_aligned_causal_gb300 import kb_attn

    yield kb_attn
    assert kb_attn.kb_attn_check_device_status(None) == kb_attn.KB_OK


def f64(bits):
    return inputs.bf16_bits_to_f32(bits).astype(np.float64)


def assert_grad_close(got_bits, ref, what):
    g = f64(got_bits)
    assert np.all(np.isfinite(g)), f"{what}: non-finite gradient"
    err = np.abs(g - ref)
    scale_max, scale_mean = float(np.abs(ref).max()), float(np.abs(ref).mean())
    assert err.max() <= REL_MAX * scale_max + 1e-5, f"{what}: max-abs {err.max():.3e} vs scale {scale_max:.3e}"
    assert err.mean() <= REL_MEAN * scale_mean + 1e-6, f"{what}: mean-abs {err.mean():.3e} vs scale {scale_mean:.3e}"


def run(kb, B, Hkv, S, seed):
    x = inputs.make_qkv(B, S, seed=seed, Hq=4 * Hkv, Hkv=Hkv)
    do_bits = inputs.make_qkv(B, S, seed=seed + 1, Hq=4 * Hkv, Hkv=Hkv).q
    q, k, v, do = to_dev(x.q), to_dev(x.k), to_dev(x.v), to_dev(do_bits)
    o, lse = kb.prefill_lse(q, k, v)
    dq, dk, dv, delta = kb.backward(q, k, v, o, do, lse)
    kb.check_device_status()
    return x, do_bits, (q, k, v, do, o, lse), (dq, dk, dv, delta)


def test_prefill_lse_bits_and_values(kb, oracle_mod):
    B, Hkv, S = 2, 8, 300
    x = inputs.make_qkv(B, S, seed=60_000)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    o, lse = kb.prefill_lse(q, k, v)
    pre = kb.prefill(q, k, v)
    kb.check_device_status()
    assert np.array_equal(from_dev(o), from_dev(pre))
    rows = [(b, h, i) for b in range(B) for h in range(0, 32, 3) for i in range(S)]
    _, lse_ref, _ = oracle_mod.dq_rows(x.q, x.k, x.v, x.q, rows)
    got = lse.cpu().numpy()[tuple(np.asarray(rows).T)]
    assert np.abs(got - lse_ref).max() <= 2e-5 * max(1.0, np.abs(lse_ref).max())


@pytest.mark.parametrize("B,Hkv,S", [(1, 2, 1), (1, 2, 5), (2, 8, 127), (1, 8, 128), (1, 2, 129), (1, 8, 300),
                                     (2, 2, 520)])
def test_backward_against_oracle(kb, oracle_mod, B, Hkv, S):
    x, do_bits, dev, (dq, dk, dv, delta) = run(kb, B, Hkv, S, seed=61_000 + S)
    rq, rk, rv = oracle_mod.backward(x.q, x.k, x.v, do_bits)
    assert_grad_close(from_dev(dq), rq, "dq")
    assert_grad_close(from_dev(dk), rk, "dk")
    assert_grad_close(from_dev(dv), rv, "dv")
    # delta = dO . o with the kernel's own bf16 o, against the exact row's P . dP
    rows = [(b, h, i) for b in range(B) for h in range(4 * Hkv) for i in range(S)]
    _, _, dref = oracle_mod.dq_rows(x.q, x.k, x.v, do_bits, rows)
    got = delta.cpu().numpy().reshape(-1)
    assert np.abs(got - dref).max() <= 1e-2 * max(1.0, np.abs(dref).max())


def test_backward_is_deterministic(kb):
    _, _, (q, k, v, do, o, lse), (dq, dk, dv, delta) = run(kb, 2, 8, 777, seed=62_000)
    for _ in range(3):
        dq2, dk2, dv2, delta2 = kb.backward(q, k, v, o, do, lse)
        kb.check_device_status()
        for a, b_ in ((dq, dq2), (dk, dk2), (dv, dv2)):
            assert np.array_equal(from_dev(a), from_dev(b_))
        assert np.array_equal(delta.cpu().numpy(), delta2.cpu().numpy())


def test_backward_S2048_full_dk_dv_and_sampled_dq(kb, oracle_mod):
    B, Hkv, S = 1, 8, 2048
    x, do_bits, dev, (dq, dk, dv, delta) = run(kb, B, Hkv, S, seed=63_000)
    _, rk, rv = oracle_mod.backward(x.q, x.k, x.v, do_bits)
    assert_grad_close(from_dev(dk), rk, "dk")
    assert_grad_close(from_dev(dv), rv, "dv")
    rows = inputs.sample_rows(B, 32, S, 96, seed=63_001)
    rq, _, _ = oracle_mod.dq_rows(x.q, x.k, x.v, do_bits, rows)
    got = from_dev(dq)[tuple(np.asarray(rows).T)]
    assert_grad_close(got, rq, "dq rows")


def sum_rules(dk_bits, dv_bits, do_bits, B, Hkv, S):
    """|sum_j dk_j| against sum_j |dk_j| (exactly 0 in exact arithmetic) and
    sum_j dv_j against the sum of dO over the group's rows (exact identity)."""
    dk, dv, do = f64(dk_bits), f64(dv_bits), f64(do_bits)
    skew = np.abs(dk.sum(axis=2)) / np.maximum(np.abs(dk).sum(axis=2), 1e-30)
    want = do.reshape(B, Hkv, 4, S, D).sum(axis=(2, 3))
    dv_err = np.abs(dv.sum(axis=2) - want).max() / max(1.0, np.abs(want).max())
    return float(skew.max()), float(dv_err)


def test_backward_bench_size_properties(kb, oracle_mod):
    """B=4, S=16384 (the bench size): sum rules on every (b, kv head) and
    sampled dq rows against the oracle."""
    B, Hkv, S = 4, 8, 16384
    x, do_bits, dev, (dq, dk, dv, delta) = run(kb, B, Hkv, S, seed=64_000)
    skew, dv_err = sum_rules(from_dev(dk), from_dev(dv), do_bits, B, Hkv, S)
    assert skew <= 1e-2 and dv_err <= 1e-2, (skew, dv_err)
    rows = inputs.sample_rows(B, 32, S, 48, seed=64_001)
    rq, _, _ = oracle_mod.dq_rows(x.q, x.k, x.v, do_bits, rows)
    got = from_dev(dq)[tuple(np.asarray(rows).T)]
    assert_grad_close(got, rq, "dq rows")


def test_backward_S8192_one_unit_elementwise(kb, oracle_mod):
    """S=8192 with all eight KV heads in the launch: dq, dk and dv of one
    (b, kv head) unit element by element against the oracle.  dk and dv sum
    over the group's four query heads, so the oracle runs each head alone
    (a group of one) and the four results are added; the four calls run in
    threads, since ctypes releases the GIL during a foreign call."""
    from concurrent.futures import ThreadPoolExecutor

    B, Hkv, S, g = 1, 8, 8192, 5
    x, do_bits, dev, (dq, dk, dv, delta) = run(kb, B, Hkv, S, seed=65_000)
    heads = range(4 * g, 4 * g + 4)

    def one_head(h):
        return oracle_mod.backward(x.q[:, h:h + 1], x.k[:, g:g + 1], x.v[:, g:g + 1], do_bits[:, h:h + 1],
                                   n_threads=1)

    with ThreadPoolExecutor(max_workers=4) as ex:
        parts = list(ex.map(one_head, heads))
    rk = sum(p[1] for p in parts)[0, 0]
    rv = sum(p[2] for p in parts)[0, 0]
    assert_grad_close(from_dev(dk)[0, g], rk, "dk")
    assert_grad_close(from_dev(dv)[0, g], rv, "dv")
    got_dq = from_dev(dq)[0, 4 * g:4 * g + 4]
    for i, p in enumerate(parts):
        assert_grad_close(got_dq[i], p[0][0, 0], f"dq head {4 * g + i}")
