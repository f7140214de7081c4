"""kb_attn_decode_seg_static: the segmented decode with the library's own
scratch array instead of a caller workspace.

It must give kb_attn_decode_seg's bits, allocate no device memory on any
call, and refuse requests larger than its 4 MiB scratch before launching
anything.
"""

import numpy as np
import pytest

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import from_dev, to_dev

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


@pytest.mark.parametrize("B,ctx,seg", [(1, 1, 1), (1, 300, 1), (2, 1500, 3), (1, 8192, 4), (4, 8192, 8),
                                       (1, 32768, 16)])
def test_same_bits_as_caller_workspace(kb, B, ctx, seg):
    x = inputs.make_qkv(B, ctx, seed=97_000 + ctx)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    qd = q[:, :, ctx - 1:].contiguous()
    a = from_dev(kb.decode_seg(qd, k, v, ctx, seg))
    b = from_dev(kb.decode_seg_static(qd, k, v, ctx, seg))
    kb.check_device_status()
    assert np.array_equal(a, b)


def test_allocates_nothing(kb):
    import torch

    B, ctx, seg = 2, 4096, 2
    x = inputs.make_qkv(B, ctx, seed=97_100)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    qd = q[:, :, ctx - 1:].contiguous()
    o = torch.empty_like(qd)
    kb.decode_seg_static(qd, k, v, ctx, seg, out=o)          # first call loads nothing new either way
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    held0 = torch.cuda.memory_allocated()
    for _ in range(20):
        kb.decode_seg_static(qd, k, v, ctx, seg, out=o)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert torch.cuda.memory_allocated() == held0
    assert free1 == free0
    kb.check_device_status()


def test_too_large_is_refused(kb):
    import torch

    # 64 x 32 rows x 64 segments x 528 bytes = 69 MB of partials > 4 MiB
    B, ctx = 64, 8192
    q = torch.zeros((B, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, 8, ctx, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kb.KBError) as e:
        kb.decode_seg_static(q, k, k, ctx, 1)
    assert e.value.status == kb.KB_ERR_UNSUPPORTED


def test_just_under_the_limit(kb):
    """31 x 32 rows x 8 segments x 528 bytes = 4,190,208 bytes of partials, just
    under the 4 MiB scratch: bits equal the caller-workspace call, and the
    device status stays clean (nothing was written past the scratch)."""
    B, ctx, seg = 31, 1024, 1
    assert kb.kb_attn_seg_workspace_bytes(B, 32, 1, ctx - 1, seg) == 4_190_208 <= 4 << 20
    x = inputs.make_qkv(B, ctx, seed=97_200)
    q, k, v = to_dev(x.q), to_dev(x.k), to_dev(x.v)
    qd = q[:, :, ctx - 1:].contiguous()
    for _ in range(2):
        a = from_dev(kb.decode_seg(qd, k, v, ctx, seg))
        b = from_dev(kb.decode_seg_static(qd, k, v, ctx, seg))
        assert kb.kb_attn_check_device_status(None) == kb.KB_OK
        assert np.array_equal(a, b)


def test_one_segment_over_the_limit_is_refused(kb):
    import torch

    # ctx 1025 needs a ninth segment: 31 x 32 x 9 x 528 = 4,713,984 bytes > 4 MiB
    B, ctx = 31, 1025
    assert kb.kb_attn_seg_workspace_bytes(B, 32, 1, ctx - 1, 1) > 4 << 20
    q = torch.zeros((B, 32, 1, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((B, 8, ctx, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(kb.KBError) as e:
        kb.decode_seg_static(q, k, k, ctx, 1)
    assert e.value.status == kb.KB_ERR_UNSUPPORTED
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK
