"""Failure detection on the GPU without faulting it: a bounded device-side
wait that runs out sets the library's error word and returns; the host reads
KB_ERR_TIMEOUT, the context stays usable, and later calls work."""

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

    return kb_attn


def test_wait_that_runs_out_reports_timeout(kb):
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK
    assert kb.kb_attn_debug_wait_timeout(20_000) == kb.KB_OK          # 20 ms, nothing will signal
    assert kb.kb_attn_check_device_status(None) == kb.KB_ERR_TIMEOUT
    assert kb.kb_attn_check_device_status(None) == kb.KB_OK           # the word was cleared
    x = inputs.make_qkv(1, 200, seed=60_000)
    o = from_dev(kb.prefill(to_dev(x.q), to_dev(x.k), to_dev(x.v)))
    kb.check_device_status()
    assert np.array_equal(o[:, :, 0], x.v[:, np.arange(32) // 4, 0])


def test_host_memory_is_rejected(kb):
    import torch

    x = torch.zeros(1, 32, 16, 128, dtype=torch.bfloat16).pin_memory()
    d = torch.zeros(1, 8, 16, 128, dtype=torch.bfloat16, device="cuda")
    st = kb.kb_attn_prefill(x.data_ptr(), d.data_ptr(), d.data_ptr(), d.data_ptr(), 1, 32, 8, 16, None)
    assert st == kb.KB_ERR_INVALID_ARG
