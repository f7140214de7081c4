"""The torch binding refuses mismatched tensors before any kernel is enqueued.

The C ABI receives only pointers and sizes; a key cache shorter than the
sequence or an output smaller than the query would be read or written past
its end.  The binding compares every tensor's shape with the others first
(KernelBraid README, "Usage": a checked interface whose inputs share one
device), so such a call raises ValueError and leaves the output untouched.
"""

import pytest

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


def test_mismatches_raise_and_write_nothing(kb):
    import torch

    B, S = 2, 256
    q = torch.randn(B, 32, S, 128, device="cuda").to(torch.bfloat16)
    k = torch.randn(B, 8, S, 128, device="cuda").to(torch.bfloat16)
    short = k[:, :, : S - 1].contiguous()
    out = torch.full_like(q, 3.0)
    small_out = torch.full((B, 32, S - 1, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    cases = [
        lambda: kb.prefill(q, short, short, out=out),            # cache shorter than the sequence
        lambda: kb.prefill(q, k, short, out=out),                # v differs from k
        lambda: kb.prefill(q, k, k, out=small_out),              # output smaller than q
        lambda: kb.prefill(q, k[:1].contiguous(), k[:1].contiguous(), out=out),   # batch differs
        lambda: kb.chunk(q[:, :, :10].contiguous(), k, k, S - 5),                 # chunk past the cache
        lambda: kb.decode(q[:, :, :2].contiguous(), k, k, S),                     # two query rows
        lambda: kb.decode(q[:, :, :1].contiguous(), k, k, S + 1),                 # context past the cache
    ]
    for call in cases:
        with pytest.raises(ValueError):
            call()
    torch.cuda.synchronize()
    assert bool((out == 3.0).all()) and bool((small_out == 3.0).all())
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK
    # the same tensors, consistent, run
    o = kb.prefill(q, k, k, out=out, check=True)
    assert not bool((o == 3.0).all())
