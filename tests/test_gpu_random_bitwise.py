"""Randomised bit-equality of the entry points (seeded).

For random shapes, random partitions of the sequence into chunks (small ones
take the packed kernel, large ones the tile kernel), decodes at random
positions, and the same data through a ragged call and a paged pool, every
output row must equal the full prefill row bit for bit (KernelBraid README,
"Advantages": prefill and incremental decode give bitwise-identical outputs;
"Usage": prompt/answer splits).
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu

D = 128


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


def random_partition(rng, S):
    cuts, pos = [], 0
    while pos < S:
        n = int(rng.choice([rng.integers(1, 33), rng.integers(33, 400)]))
        n = min(n, S - pos)
        cuts.append((pos, n))
        pos += n
    return cuts


@pytest.mark.parametrize("case", range(10))
def test_random_partitions_decodes_ragged_and_paged(kb, case):
    import torch

    from tests.test_gpu_packed_paged import _paged

    rng = np.random.default_rng(90_000 + case)
    B = int(rng.integers(1, 4))
    Hkv = int(rng.choice([1, 2, 8]))
    Hq = 4 * Hkv
    S = int(rng.integers(1, 1400))
    x = inputs.make_qkv(B, S, seed=90_100 + case, Hq=Hq, Hkv=Hkv)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    pre = kb.prefill(q, k, v)

    # chunked forward over a random partition, cache filled as we go
    kc = torch.full_like(k, float("nan"))
    vc = torch.full_like(v, float("nan"))
    out = torch.empty_like(q)
    for start, n in random_partition(rng, S):
        kc[:, :, start:start + n] = k[:, :, start:start + n]
        vc[:, :, start:start + n] = v[:, :, start:start + n]
        out[:, :, start:start + n] = kb.chunk(q[:, :, start:start + n].contiguous(), kc, vc, start)
    assert torch.equal(out.view(torch.int16), pre.view(torch.int16)), "chunked"

    # decodes at random positions
    for pos in rng.integers(0, S, size=4):
        pos = int(pos)
        d = kb.decode(q[:, :, pos:pos + 1].contiguous(), k, v, pos + 1)
        assert torch.equal(d[:, :, 0].view(torch.int16), pre[:, :, pos].view(torch.int16)), f"decode {pos}"

    # ragged: each sequence takes a random window [start, start + n)
    starts = [int(rng.integers(0, S)) for _ in range(B)]
    lens = [int(rng.integers(0, S - s + 1)) for s in starts]
    L_max = max(1, max(lens))
    qr = torch.full((B, Hq, L_max, D), float("nan"), dtype=torch.bfloat16, device="cuda")
    for b in range(B):
        qr[b, :, :lens[b]] = q[b, :, starts[b]:starts[b] + lens[b]]
    st = torch.tensor(starts, dtype=torch.int32, device="cuda")
    ln = torch.tensor(lens, dtype=torch.int32, device="cuda")
    rag = kb.chunk_varlen(qr, k, v, st, ln)
    for b in range(B):
        got = rag[b, :, :lens[b]].view(torch.int16)
        want = pre[b, :, starts[b]:starts[b] + lens[b]].view(torch.int16)
        assert torch.equal(got, want), f"ragged sequence {b}"

    # the same decodes through a shuffled paged pool
    page = int(rng.choice([128, 256]))
    ctx = np.array([int(rng.integers(1, S + 1)) for _ in range(B)], dtype=np.int32)
    kp, vp, table = _paged(k, v, ctx, page, seed=90_200 + case)
    qd = torch.stack([q[b, :, int(c) - 1] for b, c in enumerate(ctx)])[:, :, None, :].contiguous()
    dp = kb.decode_paged(qd, kp, vp, table, torch.tensor(ctx, device="cuda"))
    for b, c in enumerate(ctx):
        assert torch.equal(dp[b, :, 0].view(torch.int16), pre[b, :, int(c) - 1].view(torch.int16)), f"paged {b}"
    kb.check_device_status()
