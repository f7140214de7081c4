"""Ragged batches: every sequence with its own start and row count.

Each sequence of a ragged call must give exactly the bits of a call on that
sequence alone (and hence of its prefill rows), whatever the other sequences
hold; padding rows of q and cache rows past a sequence are NaN here.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import from_dev, to_dev

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


def ragged_case(starts, lens, L_max, cap, seed):
    """q [B,Hq,L_max,D] with NaN padding rows; caches [B,Hkv,cap,D] with NaN past each sequence."""
    import torch

    B = len(starts)
    x = inputs.make_qkv(B, cap, seed=seed, Lq=L_max)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    for b in range(B):
        q[b, :, lens[b]:] = float("nan")
        k[b, :, starts[b] + lens[b]:] = float("nan")
        v[b, :, starts[b] + lens[b]:] = float("nan")
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, k, v, st, ln


def solo(kb, q, k, v, starts, lens, b):
    """Reference: sequence b alone through kb_attn_chunk, its cache cut to its keys."""
    e = starts[b] + lens[b]
    return from_dev(kb.chunk(q[b:b + 1, :, :lens[b]].contiguous(), k[b:b + 1, :, :e].contiguous(),
                             v[b:b + 1, :, :e].contiguous(), starts[b]))


@pytest.mark.parametrize("starts,lens,L_max,cap", [
    ([0, 0, 0, 0, 0], [1, 127, 300, 1024, 0], 1024, 1024),    # ragged prefill, one empty sequence
    ([5, 0, 700, 130], [20, 1, 32, 17], 32, 1024),             # short continuations: packed kernel
    ([0, 129, 900, 3], [300, 200, 124, 1], 300, 1100),         # tile kernel
    ([1023, 0, 511], [1, 1, 1], 1, 1024),                      # ragged one-token decode
])
def test_ragged_equals_each_sequence_alone(kb, starts, lens, L_max, cap):
    import torch

    q, k, v, st, ln = ragged_case(starts, lens, L_max, cap, seed=80_000 + L_max)
    o = torch.full_like(q, 7.0)
    kb.chunk_varlen(q, k, v, st, ln, out=o)
    kb.check_device_status()
    out = from_dev(o)
    for b in range(len(starts)):
        if lens[b] == 0:
            assert np.all(out[b] == from_dev(torch.full((1,), 7.0, dtype=torch.bfloat16, device="cuda"))[0])
            continue
        assert np.array_equal(out[b:b + 1, :, :lens[b]], solo(kb, q, k, v, starts, lens, b)), f"sequence {b}"
        # rows past the sequence are untouched
        assert np.all(out[b, :, lens[b]:] == out[b, 0, L_max - 1, 0] if lens[b] < L_max else True)


def test_ragged_persistent_launch(kb):
    """With 8 query heads the default kernel's persistent launch (CTAs walking
    pairs of query tiles) runs this ragged batch, whose shorter sequences
    leave holes in the pair schedule; each sequence must still give the bits
    of the tile kernel launched one CTA per query tile, run on it alone."""
    import torch

    starts, lens, L_max, cap = [0, 129, 700, 3], [300, 200, 124, 1], 300, 1000
    B, Hkv = len(starts), 2
    x = inputs.make_qkv(B, cap, seed=80_500, Hq=4 * Hkv, Hkv=Hkv, Lq=L_max)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    for b in range(B):
        q[b, :, lens[b]:] = float("nan")
        k[b, :, starts[b] + lens[b]:] = float("nan")
        v[b, :, starts[b] + lens[b]:] = float("nan")
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = from_dev(kb.chunk_varlen(q, k, v, st, ln))
    for b in range(B):
        e = starts[b] + lens[b]
        ref = from_dev(kb.chunk(q[b:b + 1, :, :lens[b]].contiguous(), k[b:b + 1, :, :e].contiguous(),
                                v[b:b + 1, :, :e].contiguous(), starts[b], q_tiles_per_cta=3))
        assert np.array_equal(out[b:b + 1, :, :lens[b]], ref), b
    kb.check_device_status()


def test_ragged_paged(kb):
    import torch

    from tests.test_gpu_packed_paged import _paged

    starts, lens, L_max, cap = [0, 40, 300], [700, 33, 1], 700, 1024
    q, k, v, st, ln = ragged_case(starts, lens, L_max, cap, seed=81_000)
    filled = np.array([s + n for s, n in zip(starts, lens)], dtype=np.int32)
    kp, vp, table = _paged(k, v, filled, 256, seed=81_001)
    out = from_dev(kb.chunk_varlen(q, kp, vp, st, ln, block_table=table))
    kb.check_device_status()
    for b in range(3):
        assert np.array_equal(out[b:b + 1, :, :lens[b]], solo(kb, q, k, v, starts, lens, b)), f"sequence {b}"


def test_ragged_bad_lengths_are_reported(kb):
    import torch

    q, k, v, st, ln = ragged_case([0, 0], [10, 10], 16, 64, seed=82_000)
    kb.chunk_varlen(q, k, v, st, torch.tensor([10, 17], dtype=torch.int32, device="cuda"))   # 17 > L_max
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
    kb.chunk_varlen(q, k, v, torch.tensor([0, 60], dtype=torch.int32, device="cuda"), ln)    # 60 + 10 > cap
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_INVALID_ARG
    kb.chunk_varlen(q, k, v, st, ln)
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK
