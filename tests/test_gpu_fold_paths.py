"""The contract's segment split at long contexts, through every fold path.

Contract version 3 cuts each row's keys into segments of 1024 keys (8 tiles
of 128), runs each from the fresh softmax state and folds them left to right
(KernelBraid README, "Method": one numerical contract for prefill,
partitioned forward and decode).  The kernels fold in four places:
  - prefill and long chunks: in the softmax threads' registers;
  - a decode of a small batch: over a cluster of up to 8 CTAs, the first of
    which folds the others' partials in its shared memory: pushed there as
    they finish (up to ~15 partials), copied into its K/V rings once it has
    streamed its last tile (B=1 ctx 32768, B=2 ctx 20000, two-row chunks),
    or read from the others' shared memory (the longest contexts);
  - a decode of a large batch, or one whose segments exceed the cluster's
    shared-memory slots: one CTA, in registers;
  - chunks of 3-32 rows: one CTA, in TMEM;
and the explicit-length entry points (decode_seg with 8 tiles) fold a
workspace in a second kernel.  Every path must give the prefill rows' bits,
and the rows must match the fp64 oracle.
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


@pytest.mark.parametrize("B,ctx", [(1, 1025), (1, 8192), (2, 20000), (3, 8192), (1, 32768)])
def test_decode_equals_prefill_and_workspace_fold(kb, oracle_mod, B, ctx):
    """B=1..3: 8, 8, 4.. CTAs per (sequence, KV head) in a cluster."""
    x = inputs.make_qkv(B, ctx, seed=110_000 + ctx + B)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = from_dev(kb.prefill(q, k, v))
    qd = q[:, :, ctx - 1:].contiguous()
    dec = from_dev(kb.decode(qd, k, v, ctx))
    ws = from_dev(kb.decode_seg(qd, k, v, ctx, 8))
    kb.check_device_status()
    assert np.array_equal(dec[:, :, 0], pre[:, :, ctx - 1])
    assert np.array_equal(ws, dec)
    want = oracle_mod.attention_rows(x.q, x.k, x.v, [(b, h, ctx - 1) for b in range(B) for h in range(HQ)])
    assert_close_to_oracle(dec[:, :, 0].reshape(-1, D), want, f"decode B={B} ctx={ctx}")


@pytest.mark.parametrize("ctx", [122_880, 131_072])
def test_very_long_decode(kb, oracle_mod, ctx):
    """120 segments fill a cluster of 8 CTAs' shared-memory slots exactly (too
    many for the first CTA's rings, so it reads them remotely); 128 segments do
    not, and the decode folds them all in one CTA instead."""
    x = inputs.make_qkv(1, ctx, seed=111_000 + ctx, Lq=1)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    dec = from_dev(kb.decode(q, k, v, ctx))
    ws = from_dev(kb.decode_seg(q, k, v, ctx, 8))
    kb.check_device_status()
    assert np.array_equal(ws, dec)
    want = oracle_mod.attention_rows(x.q, x.k, x.v, [(0, h, 0) for h in range(HQ)], start=ctx - 1)
    assert_close_to_oracle(dec[:, :, 0].reshape(-1, D), want, f"decode ctx={ctx}")


@pytest.mark.parametrize("start,L", [(8191, 1), (8191, 2), (8190, 3), (9000, 17), (9950, 32), (8150, 32),
                                     (1020, 9), (4000, 2)])
def test_short_chunks_at_long_positions(kb, start, L):
    """Narrow chunks (a cluster per sub-chunk; L=2 at 8191 crosses a tile
    boundary) and wide chunks (segments folded in TMEM) against prefill rows."""
    q, k, v, pre = _shared_sequence()
    out = from_dev(kb.chunk(q[:, :, start:start + L].contiguous(), k, v, start))
    kb.check_device_status()
    assert np.array_equal(out, pre[:, :, start:start + L])


_SEQ = {}


def _shared_sequence():
    if "x" not in _SEQ:
        from bitwise_aligned_causal_gb300 import kb_attn

        x = inputs.make_qkv(2, 10_000, seed=112_000)
        q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
        _SEQ["x"] = (q, k, v, from_dev(kb_attn.prefill(q, k, v)))
    return _SEQ["x"]


def test_paged_decode_with_mixed_lengths(kb):
    """One launch, sequences of 10 and 1 segments: the cluster is sized for
    the longer one, and the shorter leaves CTAs of its cluster idle."""
    import torch

    from tests.test_gpu_packed_paged import _paged

    q, k, v, pre = _shared_sequence()
    ctx = np.array([10_000, 300], dtype=np.int32)
    kp, vp, table = _paged(k, v, ctx, 256, seed=112_500)
    qd = torch.stack([q[b, :, int(c) - 1] for b, c in enumerate(ctx)])[:, :, None, :].contiguous()
    dp = from_dev(kb.decode_paged(qd, kp, vp, table, torch.tensor(ctx, device="cuda")))
    kb.check_device_status()
    for b, c in enumerate(ctx):
        assert np.array_equal(dp[b, :, 0], pre[b, :, int(c) - 1]), b
