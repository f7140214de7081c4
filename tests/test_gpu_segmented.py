"""Explicit segment lengths (contract C5 with seg_tiles tiles instead of the
contract's 8): a fixed split of each row's key tiles, folded left to right.

For one segment length every entry point must give the same bits for a row
(KernelBraid README, "Method" and "Advantages": one contract for prefill,
partitioned forward and decode); the contract's own length (8 tiles) must
give the default entry points' bits; a row that fits in one segment is the
unsplit online softmax; and results must match the fp64 oracle within the
forward tolerance.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import assert_close_to_oracle, from_dev, gather_rows, to_dev

pytestmark = pytest.mark.gpu


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
    S = 1500
    x = inputs.make_qkv(2, S, seed=95_000)
    return x, to_dev(x.q), to_dev(x.k), to_dev(x.v)


@pytest.mark.parametrize("seg", [1, 2, 5])
def test_prefill_seg_against_oracle(kb, oracle_mod, seq, seg):
    x, q, k, v = seq
    out = from_dev(kb.prefill_seg(q, k, v, seg))
    kb.check_device_status()
    rows = inputs.sample_rows(2, 32, x.q.shape[2], 40, seed=95_001 + seg)
    want = oracle_mod.attention_rows(x.q, x.k, x.v, rows)
    assert_close_to_oracle(gather_rows(out, rows), want, f"prefill_seg seg={seg}")


def test_contract_segment_length_is_the_default_mode(kb, seq):
    """seg_tiles = 8 is the contract's own split: prefill_seg, decode_seg and
    chunk_seg at 8 (the workspace fold path) give the default entry points'
    bits, and a row whose keys fit in one segment is the unsplit online
    softmax whatever the segment length."""
    x, q, k, v = seq
    S = x.q.shape[2]
    n_tiles = (S + 127) // 128
    default = from_dev(kb.prefill(q, k, v))
    a = from_dev(kb.prefill_seg(q, k, v, 8))
    kb.check_device_status()
    assert np.array_equal(a, default)
    unsplit = from_dev(kb.prefill_seg(q, k, v, n_tiles))
    assert np.array_equal(unsplit[:, :, :1024], default[:, :, :1024])     # rows of one 8-tile segment
    c = from_dev(kb.prefill_seg(q, k, v, 3))
    assert np.array_equal(c[:, :, :384], unsplit[:, :, :384])             # rows of one 3-tile segment
    for pos in (0, 127, 1023, 1024, 1499):
        d = from_dev(kb.decode_seg(q[:, :, pos:pos + 1].contiguous(), k, v, pos + 1, 8))
        e = from_dev(kb.decode(q[:, :, pos:pos + 1].contiguous(), k, v, pos + 1))
        assert np.array_equal(d[:, :, 0], default[:, :, pos]), pos
        assert np.array_equal(e[:, :, 0], default[:, :, pos]), pos
        f = from_dev(kb.decode_seg(q[:, :, pos:pos + 1].contiguous(), k, v, pos + 1, n_tiles))
        assert np.array_equal(f[:, :, 0], unsplit[:, :, pos]), pos
    kb.check_device_status()


@pytest.mark.parametrize("seg", [1, 3])
def test_decode_seg_equals_prefill_seg_rows(kb, seq, seg):
    x, q, k, v = seq
    pre = from_dev(kb.prefill_seg(q, k, v, seg))
    # positions at, just before and just after segment and tile boundaries
    edge = [seg * 128 * m + d for m in range(1, 5) for d in (-2, -1, 0, 1)]
    for pos in sorted({p for p in edge + [0, 1, 700, 1499] if 0 <= p < 1500}):
        d = from_dev(kb.decode_seg(q[:, :, pos:pos + 1].contiguous(), k, v, pos + 1, seg))
        assert np.array_equal(d[:, :, 0], pre[:, :, pos]), f"seg={seg} pos={pos}"
    kb.check_device_status()


@pytest.mark.parametrize("seg", [2, 4])
def test_chunk_seg_equals_prefill_seg_rows(kb, seq, seg):
    """A random partition into chunks of 1..400 rows (packed and tile kernels),
    the cache holding NaN past each chunk, gives prefill_seg's bits."""
    import torch

    x, q, k, v = seq
    pre = kb.prefill_seg(q, k, v, seg)
    rng = np.random.default_rng(95_100 + seg)
    kc = torch.full_like(k, float("nan"))
    vc = torch.full_like(v, float("nan"))
    out = torch.empty_like(q)
    pos, S = 0, q.shape[2]
    while pos < S:
        n = int(rng.choice([rng.integers(1, 33), rng.integers(33, 400)]))
        n = min(n, S - pos)
        kc[:, :, pos:pos + n] = k[:, :, pos:pos + n]
        vc[:, :, pos:pos + n] = v[:, :, pos:pos + n]
        out[:, :, pos:pos + n] = kb.chunk_seg(q[:, :, pos:pos + n].contiguous(), kc, vc, pos, seg)
        pos += n
    kb.check_device_status()
    assert torch.equal(out.view(torch.int16), pre.view(torch.int16))


def test_decode_seg_long_context(kb, oracle_mod):
    """B=1 and B=16 at ctx 8192 (64 key tiles), segments of 8 tiles: oracle and
    prefill_seg bits."""
    for B in (1, 16):
        ctx = 8192
        x = inputs.make_qkv(B, ctx, seed=96_000 + B)
        q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
        d = from_dev(kb.decode_seg(q[:, :, ctx - 1:].contiguous(), k, v, ctx, 8))
        kb.check_device_status()
        rows = [(b, h, ctx - 1) for b in range(B) for h in range(32)]
        want = oracle_mod.attention_rows(x.q, x.k, x.v, rows)
        assert_close_to_oracle(d.reshape(-1, 128), want, f"decode_seg B={B}")
        if B == 1:
            pre = from_dev(kb.prefill_seg(q, k, v, 8))
            assert np.array_equal(d[:, :, 0], pre[:, :, ctx - 1])


def test_workspace_too_small_is_rejected(kb, seq):
    import torch

    x, q, k, v = seq
    need = kb.kb_attn_seg_workspace_bytes(2, 32, 1, 1499, 2)
    assert need == 2 * 32 * 1 * 6 * 132 * 4
    ws = torch.empty(need - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(kb.KBError):
        kb.decode_seg(q[:, :, 1499:].contiguous(), k, v, 1500, 2, workspace=ws)
