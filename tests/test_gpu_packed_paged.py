"""Packed small chunks and paged decode keep the prefill row bits.

Chunks of at most 32 query rows run with the four heads of a GQA group and
the chunk's rows packed into one MMA tile (README "Method": partitioned
forward execution; "Usage": prompt/answer splits).  Decode over a paged KV
cache reads keys and values through a page table.  Both must reproduce the
prefill rows bit for bit, and the fp64 oracle within tolerance.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import assert_close_to_oracle, from_dev, to_dev

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


@pytest.fixture(scope="module")
def seq(kb):
    S = 1100
    x = inputs.make_qkv(3, S, seed=70_000)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = from_dev(kb.prefill(q, k, v))
    kb.check_device_status()
    return x, q, k, v, pre


@pytest.mark.parametrize("start,L", [(0, 1), (0, 2), (0, 3), (0, 32), (5, 17), (100, 32), (120, 9), (127, 2),
                                     (127, 32), (128, 32), (255, 1), (1000, 31), (1068, 32), (1099, 1)])
def test_small_chunks_bitwise_equal_prefill(kb, seq, start, L):
    x, q, k, v, pre = seq
    qc = q[:, :, start:start + L].contiguous()
    packed = from_dev(kb.chunk(qc, k, v, start))                       # L <= 32: packed kernel
    two_s = from_dev(kb.chunk(qc, k, v, start, q_tiles_per_cta=3))     # the tile kernel, three S buffers
    persist = from_dev(kb.chunk(qc, k, v, start, q_tiles_per_cta=4))   # the same, persistent launch
    kb.check_device_status()
    assert np.array_equal(persist, packed)
    assert np.array_equal(packed, pre[:, :, start:start + L])
    assert np.array_equal(two_s, packed)


def test_small_chunk_with_short_cache(kb, oracle_mod):
    """The cache holds exactly start + L rows; rows past them are never read."""
    S, start, L = 300, 270, 30
    x = inputs.make_qkv(2, S, seed=71_000)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    out = from_dev(kb.chunk(q[:, :, start:].contiguous(), k, v, start))
    kb.check_device_status()
    rows = [(b, h, i) for b in range(2) for h in range(HQ) for i in range(L)]
    want = oracle_mod.attention_rows(x.q[:, :, start:], x.k, x.v, rows, start=start)
    got = np.stack([out[b, h, i] for b, h, i in rows])
    assert_close_to_oracle(got, want, "packed chunk")


def _paged(k, v, ctx_lens, page_size, seed, spare_pages=5):
    """Scatter contiguous caches into shuffled page pools; unused rows hold NaN."""
    import torch

    B, Hkv, S, _ = k.shape
    per_seq = (S + page_size - 1) // page_size
    n_pages = B * per_seq + spare_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(n_pages)[: B * per_seq].reshape(B, per_seq)
    kp = torch.full((n_pages, Hkv, page_size, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    vp = torch.full_like(kp, float("nan"))
    for b in range(B):
        for pi in range(per_seq):
            lo = pi * page_size
            hi = min(S, lo + page_size, int(ctx_lens[b]))
            if hi <= lo:
                continue
            kp[perm[b, pi], :, : hi - lo] = k[b, :, lo:hi]
            vp[perm[b, pi], :, : hi - lo] = v[b, :, lo:hi]
    table = torch.tensor(perm, dtype=torch.int32, device="cuda")
    return kp, vp, table


@pytest.mark.parametrize("page_size", [128, 256])
def test_paged_decode_bitwise_equals_contiguous_and_prefill(kb, seq, page_size):
    import torch

    x, q, k, v, pre = seq
    ctx = np.array([1100, 129, 1], dtype=np.int32)
    kp, vp, table = _paged(k, v, ctx, page_size, seed=72_000 + page_size)
    qd = torch.stack([q[b, :, int(c) - 1] for b, c in enumerate(ctx)])[:, :, None, :].contiguous()
    lens = torch.tensor(ctx, device="cuda")
    out = from_dev(kb.decode_paged(qd, kp, vp, table, lens))
    kb.check_device_status()
    for b, c in enumerate(ctx):
        assert np.array_equal(out[b, :, 0], pre[b, :, int(c) - 1]), f"batch {b} ctx {c}"
        cont = from_dev(kb.decode(qd[b:b + 1], k[b:b + 1], v[b:b + 1], int(c)))
        assert np.array_equal(out[b:b + 1], cont)
    kb.check_device_status()


def test_paged_decode_full_size(kb, oracle_mod):
    """B=16, ctx 8192, page 128: bits equal contiguous decode; oracle within tolerance."""
    import torch

    B, S = 16, 8192
    x = inputs.make_qkv(B, S, seed=73_000, Lq=1)
    k, v = to_dev(x.k), to_dev(x.v)
    qd = to_dev(x.q)
    ctx = np.full(B, S, dtype=np.int32)
    ctx[1], ctx[5] = 4097, 8000
    kp, vp, table = _paged(k, v, ctx, 128, seed=73_001)
    out = from_dev(kb.decode_paged(qd, kp, vp, table, torch.tensor(ctx, device="cuda")))
    kb.check_device_status()
    for b in (0, 1, 5, 15):
        cont = from_dev(kb.decode(qd[b:b + 1], k[b:b + 1], v[b:b + 1], int(ctx[b])))
        assert np.array_equal(out[b:b + 1], cont)
    rows = [(b, h, 0) for b in (0, 1, 5) for h in range(HQ)]
    got = np.stack([out[b, h, 0] for b, h, _ in rows])
    for b in (0, 1, 5):
        want = oracle_mod.attention_rows(x.q[b:b + 1], x.k[b:b + 1, :, : ctx[b]], x.v[b:b + 1, :, : ctx[b]],
                                         [(0, h, 0) for h in range(HQ)], start=int(ctx[b]) - 1)
        assert_close_to_oracle(got[[i for i, r in enumerate(rows) if r[0] == b]], want, f"paged b={b}")


def test_paged_decode_bad_device_arguments_are_reported(kb):
    import torch

    x = inputs.make_qkv(2, 256, seed=74_000, Lq=1)
    qd = to_dev(x.q)
    kp = torch.zeros(4, HKV, 128, D, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    table = torch.tensor([[0, 1], [2, 7]], dtype=torch.int32, device="cuda")     # page 7 does not exist
    kb.decode_paged(qd, kp, vp, table, torch.tensor([200, 256], dtype=torch.int32, device="cuda"))
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
    table = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device="cuda")
    kb.decode_paged(qd, kp, vp, table, torch.tensor([300, 0], dtype=torch.int32, device="cuda"))  # > capacity, 0
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
    kb.decode_paged(qd, kp, vp, table, torch.tensor([256, 1], dtype=torch.int32, device="cuda"))
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK


def test_paged_decode_long_contexts_over_a_cluster(kb):
    """B=2 with 20000 and 9000 keys: the segments of each sequence spread over a
    cluster whose partials overflow the first CTA's slots (they are gathered into
    its K/V rings); bits equal the contiguous decode of each sequence alone.  A
    context length beyond the pool is then reported, and the next call is clean."""
    import torch

    B, S = 2, 20000
    x = inputs.make_qkv(B, S, seed=75_000, Lq=1)
    k, v = to_dev(x.k), to_dev(x.v)
    qd = to_dev(x.q)
    ctx = np.array([20000, 9000], dtype=np.int32)
    kp, vp, table = _paged(k, v, ctx, 128, seed=75_001)
    out = from_dev(kb.decode_paged(qd, kp, vp, table, torch.tensor(ctx, device="cuda")))
    kb.check_device_status()
    for b in range(B):
        cont = from_dev(kb.decode(qd[b:b + 1], k[b:b + 1], v[b:b + 1], int(ctx[b])))
        assert np.array_equal(out[b:b + 1], cont), f"batch {b}"
    bad = torch.tensor([20000, 30000], dtype=torch.int32, device="cuda")      # beyond the pages of sequence 1
    kb.decode_paged(qd, kp, vp, table, bad)
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
    again = from_dev(kb.decode_paged(qd, kp, vp, table, torch.tensor(ctx, device="cuda")))
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK
    assert np.array_equal(again, out)


@pytest.mark.parametrize("page_size", [128, 384])
@pytest.mark.parametrize("start,L", [(0, 1100), (0, 33), (200, 300), (1000, 100), (1099, 1), (64, 32), (500, 17)])
def test_paged_chunks_bitwise_equal_prefill(kb, seq, page_size, start, L):
    """Chunks against a shuffled paged pool (unused rows NaN) give the prefill bits."""
    import torch

    x, q, k, v, pre = seq
    B = q.shape[0]
    filled = np.full(B, start + L, dtype=np.int32)
    kp, vp, table = _paged(k, v, filled, page_size, seed=75_000 + start + L)
    out = from_dev(kb.chunk_paged(q[:, :, start:start + L].contiguous(), kp, vp, table, start))
    kb.check_device_status()
    assert np.array_equal(out, pre[:, :, start:start + L])


def test_paged_chunk_bad_page_is_reported(kb):
    import torch

    x = inputs.make_qkv(1, 256, seed=76_000)
    q = to_dev(x.q)
    kp = torch.zeros(2, HKV, 128, D, dtype=torch.bfloat16, device="cuda")
    table = torch.tensor([[0, 9]], dtype=torch.int32, device="cuda")
    kb.chunk_paged(q, kp, kp, table, 0)
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
