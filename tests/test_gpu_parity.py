"""GPU path against the fp64 oracle, and the three entry points against each other.

Workloads follow the KernelBraid README grid ("Features": Hq=32, Hkv=8,
D=128, prefill 1K-16K, decode contexts 128-8K, batches 1-16; "Usage": decode
of the last token equals the prefill row bit for bit, compared as int16).
The oracle bar is max-abs <= 2e-2 and mean-abs <= 2e-3 on the bf16 output;
the bar between entry points is bit equality.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import assert_close_to_oracle, from_dev, gather_rows, to_dev

pytestmark = pytest.mark.gpu

HQ, HKV, D = 32, 8, 128


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


def run_prefill(kb, x):
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    o = kb.prefill(q, k, v)
    kb.check_device_status()
    return from_dev(o)


# ------------------------------------------------------------ config 1

def test_config1_prefill_all_rows_and_decode_bitwise(kb, oracle_mod):
    """B=1, S=1024, seed 0: every prefill row vs the oracle; decode of
    positions 896..1023 (ctx = pos+1, same cache) bit-equal to prefill."""
    import torch

    x = inputs.make_qkv(1, 1024, inputs.SEED_CONFIG1)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    o = kb.prefill(q, k, v)
    kb.check_device_status()
    pre = from_dev(o)
    want = oracle_mod.attention_full(x.q, x.k, x.v)
    assert_close_to_oracle(pre, want, "config1 prefill")
    outs = []
    for pos in range(896, 1024):
        qd = q[:, :, pos:pos + 1].contiguous()
        outs.append(kb.decode(qd, k, v, pos + 1))
    kb.check_device_status()
    dec = np.stack([from_dev(t)[:, :, 0] for t in outs], axis=2)      # [1, 32, 128, D]
    assert np.array_equal(dec, pre[:, :, 896:1024]), "decode rows differ from prefill rows"
    torch.cuda.synchronize()


# --------------------------------------------------------- small / ragged edge cases

@pytest.mark.parametrize("B,S,Hkv", [(1, 1, 8), (1, 5, 8), (2, 127, 8), (1, 128, 8), (1, 129, 8),
                                     (3, 300, 8), (1, 256, 1), (2, 513, 16), (1, 777, 2)])
def test_prefill_small_shapes_vs_oracle(kb, oracle_mod, B, S, Hkv):
    x = inputs.make_qkv(B, S, seed=10_000 + S + B, Hq=4 * Hkv, Hkv=Hkv)
    pre = run_prefill(kb, x)
    want = oracle_mod.attention_full(x.q, x.k, x.v)
    assert_close_to_oracle(pre, want, f"prefill B={B} S={S}")
    # position 0 sees one key: its row is V[0] rounded to bf16, exactly
    for h in range(4 * Hkv):
        assert np.array_equal(pre[:, h, 0], x.v[:, h // 4, 0])


@pytest.mark.parametrize("ctx,cap", [(1, 1), (1, 64), (2, 300), (127, 127), (128, 200), (129, 129), (1000, 1500)])
def test_decode_small_contexts_bitwise_and_oracle(kb, oracle_mod, ctx, cap):
    B = 2
    x = inputs.make_qkv(B, cap, seed=20_000 + ctx)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    o = kb.chunk(q[:, :, :ctx].contiguous(), k, v, 0)
    pre = from_dev(o)
    d = kb.decode(q[:, :, ctx - 1:ctx].contiguous(), k, v, ctx)
    kb.check_device_status()
    dec = from_dev(d)
    assert np.array_equal(dec[:, :, 0], pre[:, :, ctx - 1])
    want = oracle_mod.attention_rows(x.q, x.k, x.v, [(b, h, ctx - 1) for b in range(B) for h in range(HQ)])
    assert_close_to_oracle(dec[:, :, 0].reshape(-1, D), want, f"decode ctx={ctx}")


def test_cache_rows_beyond_context_are_ignored(kb):
    """Rows of the KV cache after the context hold NaN bit patterns; outputs do not change."""
    import torch

    S, cap = 300, 512
    x = inputs.make_qkv(1, S, seed=30_000)
    kc = np.full((1, HKV, cap, D), 0x7FC1, np.uint16)
    vc = np.full((1, HKV, cap, D), 0xFFC3, np.uint16)
    kc[:, :, :S] = x.k
    vc[:, :, :S] = x.v
    q = to_dev(x.q)
    a = from_dev(kb.chunk(q, to_dev(x.k), to_dev(x.v), 0))
    b = from_dev(kb.chunk(q, to_dev(kc), to_dev(vc), 0))
    c = from_dev(kb.decode(q[:, :, S - 1:].contiguous(), to_dev(kc), to_dev(vc), S))
    kb.check_device_status()
    torch.cuda.synchronize()
    assert np.array_equal(a, b)
    assert np.array_equal(c[:, :, 0], a[:, :, S - 1])


@pytest.mark.parametrize("S", [700, 1300])
def test_cta_shapes_give_identical_bits(kb, S):
    """The tile kernel launched one CTA per query tile or persistent (CTAs
    walking pairs of query tiles, or single tiles dealt back and forth), and
    short chunks on the packed kernel: same contract, same bits."""
    x = inputs.make_qkv(2, S, seed=40_000 + S)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    c = from_dev(kb.chunk(q, k, v, 0, q_tiles_per_cta=3))
    d = from_dev(kb.chunk(q, k, v, 0, q_tiles_per_cta=4))          # persistent launch forced
    s = from_dev(kb.chunk(q, k, v, 0, q_tiles_per_cta=5))          # the snake schedule forced
    kb.check_device_status()
    assert np.array_equal(c, d)
    assert np.array_equal(c, s)
    for start in (0, 130, S - 32):
        e = from_dev(kb.chunk(q[:, :, start:start + 32].contiguous(), k, v, start, q_tiles_per_cta=0))
        assert np.array_equal(e, c[:, :, start:start + 32]), start


def test_repeat_runs_are_identical(kb):
    """Eight back-to-back runs give the same bits (no order- or timing-dependent arithmetic)."""
    import torch

    x = inputs.make_qkv(2, 4100, seed=41_000)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    outs = [kb.prefill(q, k, v) for _ in range(8)]
    kb.check_device_status()
    ref = outs[0].view(torch.int16)
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), ref)


@pytest.mark.parametrize("start,L", [(0, 1), (1, 1), (127, 1), (128, 1), (5, 300), (130, 126), (256, 128),
                                     (1000, 24)])
def test_chunks_bitwise_equal_prefill(kb, start, L):
    S = 1024
    x = inputs.make_qkv(2, S, seed=50_000)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = from_dev(kb.prefill(q, k, v))
    ch = from_dev(kb.chunk(q[:, :, start:start + L].contiguous(), k, v, start))
    kb.check_device_status()
    assert np.array_equal(ch, pre[:, :, start:start + L])


# ----------------------------------------------------------- config 4: partitioned

def test_partitioned_forward_bitwise_equals_prefill(kb):
    """B=4, S=8192 split into seeded chunk lengths in [1, 2048]; the cache is
    filled chunk by chunk (unfilled rows hold NaN bits); every row bit-equal
    to single-pass prefill."""
    import torch

    B, S = 4, 8192
    x = inputs.make_qkv(B, S, inputs.SEED_PARTITIONED)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = kb.prefill(q, k, v)
    kc = torch.full_like(k, float("nan"))
    vc = torch.full_like(v, float("nan"))
    out = torch.empty_like(q)
    start = 0
    lens = inputs.chunk_lengths(S, inputs.SEED_PARTITIONED_CHUNKS)
    for L in lens:
        kc[:, :, start:start + L] = k[:, :, start:start + L]
        vc[:, :, start:start + L] = v[:, :, start:start + L]
        o = kb.chunk(q[:, :, start:start + L].contiguous(), kc, vc, start)
        out[:, :, start:start + L] = o
        start += L
    kb.check_device_status()
    assert len(lens) > 3
    assert torch.equal(out.view(torch.int16), pre.view(torch.int16))


# ------------------------------------------------------------ config 2: prefill sweep

@pytest.mark.parametrize("S", [1024, 4096, 8192, 16384])
@pytest.mark.parametrize("B", [1, 4, 8, 16])
def test_prefill_sweep_sampled_rows(kb, oracle_mod, S, B):
    x = inputs.make_qkv(B, S, inputs.seed_prefill_sweep(S, B))
    pre = run_prefill(kb, x)
    rows = inputs.sample_rows(B, HQ, S, 64, seed=inputs.seed_prefill_sweep(S, B) + 7)
    want = oracle_mod.attention_rows(x.q, x.k, x.v, rows)
    assert_close_to_oracle(gather_rows(pre, rows), want, f"prefill S={S} B={B}")


# ------------------------------------------------------------- config 3: decode sweep

@pytest.mark.parametrize("ctx", [128, 1024, 4096, 8192])
@pytest.mark.parametrize("B", [1, 4, 8, 16])
def test_decode_sweep_bitwise_and_oracle(kb, oracle_mod, ctx, B):
    x = inputs.make_qkv(B, ctx, inputs.seed_decode_sweep(ctx, B))
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = from_dev(kb.prefill(q, k, v))
    dec = from_dev(kb.decode(q[:, :, ctx - 1:].contiguous(), k, v, ctx))
    kb.check_device_status()
    assert np.array_equal(dec[:, :, 0], pre[:, :, ctx - 1])
    want = oracle_mod.attention_rows(x.q, x.k, x.v, [(b, h, ctx - 1) for b in range(B) for h in range(HQ)])
    assert_close_to_oracle(dec[:, :, 0].reshape(-1, D), want, f"decode ctx={ctx} B={B}")


# ------------------------------------------------------------------ config 5: stress

def test_stress_prefill_and_decode(kb, oracle_mod):
    """q, k ~ N(0, 8^2) with 1% of key rows x32 (peaked softmax), v ~ N(0, 1)."""
    x = inputs.make_stress_qkv(4, 16384, inputs.SEED_STRESS_PREFILL)
    pre = run_prefill(kb, x)
    rows = inputs.sample_rows(4, HQ, 16384, 64, seed=inputs.SEED_STRESS_PREFILL + 7)
    want = oracle_mod.attention_rows(x.q, x.k, x.v, rows)
    assert_close_to_oracle(gather_rows(pre, rows), want, "stress prefill")

    y = inputs.make_stress_qkv(16, 8192, inputs.SEED_STRESS_DECODE)
    q, k, v = to_dev(y.q), to_dev(y.k), to_dev(y.v)
    pre = from_dev(kb.prefill(q, k, v))
    dec = from_dev(kb.decode(q[:, :, 8191:].contiguous(), k, v, 8192))
    kb.check_device_status()
    assert np.array_equal(dec[:, :, 0], pre[:, :, 8191])
    want = oracle_mod.attention_rows(y.q, y.k, y.v, [(b, h, 8191) for b in range(16) for h in range(HQ)])
    assert_close_to_oracle(dec[:, :, 0].reshape(-1, D), want, "stress decode")
