"""The C ABI: the library loads on a machine without a GPU, exports every
symbol include/kb_attn.h declares, and rejects bad arguments before it makes
any CUDA call."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kb_attn.h")


@pytest.fixture(scope="module")
def kb():
    from bitwise_aligned_causal_gb300 import build

    build.build()
    from bitwise_aligned_causal_gb300 import kb_attn

    return kb_attn


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kb_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("kb_attn_prefill", "kb_attn_chunk", "kb_attn_decode", "kb_attn_check_device_status",
              "kb_status_string", "kb_contract_version"):
        assert n in names


def test_library_exports_every_declared_symbol(kb):
    lib = ctypes.CDLL(kb.LIB_PATH)
    for n in declared_functions():
        assert hasattr(lib, n), f"{n} declared in kb_attn.h but not exported"
    assert set(declared_functions()) == set(kb.EXPORTED)


def test_status_strings_and_version(kb):
    assert kb.kb_status_string(0) == "ok"
    assert "timed out" in kb.kb_status_string(4)
    assert kb.kb_status_string(99) == "unknown status"
    assert kb.kb_contract_version() == 3


FAKE = 0x1000_0000     # aligned, non-null; never dereferenced by the host checks below


def test_null_and_misaligned_pointers_rejected(kb):
    assert kb.kb_attn_prefill(None, FAKE, FAKE, FAKE, 1, 32, 8, 16) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_prefill(FAKE + 2, FAKE, FAKE, FAKE, 1, 32, 8, 16) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode(FAKE, FAKE, FAKE, None, 1, 32, 8, 1, 1) == kb.KB_ERR_INVALID_ARG


def test_shapes_outside_the_contract_rejected(kb):
    assert kb.kb_attn_prefill(FAKE, FAKE, FAKE, FAKE, 1, 32, 4, 16) == kb.KB_ERR_UNSUPPORTED
    assert kb.kb_attn_prefill(FAKE, FAKE, FAKE, FAKE, 1, 30, 8, 16) == kb.KB_ERR_UNSUPPORTED
    assert kb.kb_attn_decode(FAKE, FAKE, FAKE, FAKE, 1, 8, 8, 4, 4) == kb.KB_ERR_UNSUPPORTED
    assert kb.kb_attn_chunk(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 16, 0, 1 << 23) == kb.KB_ERR_UNSUPPORTED


def test_bad_sizes_rejected(kb):
    for args in [(0, 32, 8, 16), (1, 32, 8, 0), (-1, 32, 8, 4), (1, 0, 0, 4)]:
        assert kb.kb_attn_prefill(FAKE, FAKE, FAKE, FAKE, *args) in (kb.KB_ERR_INVALID_ARG, kb.KB_ERR_UNSUPPORTED)
    # chunk must fit in the cache
    assert kb.kb_attn_chunk(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 10, 100, 109) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 0, 0, 10) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 4, -1, 10) == kb.KB_ERR_INVALID_ARG
    # decode context within the cache
    assert kb.kb_attn_decode(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 11, 10) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 0, 10) == kb.KB_ERR_INVALID_ARG
    for shape in (1, 2, 6, -1):          # the tile kernel (3, 4, 5) and the packed kernel (0) only
        assert kb.kb_attn_chunk_cta_shape(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 4, 0, 10, shape) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_debug_wait_timeout(0) == kb.KB_ERR_INVALID_ARG


def test_paged_decode_arguments_rejected(kb):
    ok = (FAKE, FAKE, FAKE, FAKE, 2, 32, 8)
    assert kb.kb_attn_decode_paged(*ok, None, 4, 128, 10, FAKE) == kb.KB_ERR_INVALID_ARG      # no block table
    assert kb.kb_attn_decode_paged(*ok, FAKE, 4, 128, 10, None) == kb.KB_ERR_INVALID_ARG      # no ctx_lens
    assert kb.kb_attn_decode_paged(*ok, FAKE + 2, 4, 128, 10, FAKE) == kb.KB_ERR_INVALID_ARG  # misaligned table
    assert kb.kb_attn_decode_paged(*ok, FAKE, 4, 64, 10, FAKE) == kb.KB_ERR_INVALID_ARG       # page < 128 keys
    assert kb.kb_attn_decode_paged(*ok, FAKE, 4, 192, 10, FAKE) == kb.KB_ERR_UNSUPPORTED      # not a multiple of 128
    assert kb.kb_attn_decode_paged(*ok, FAKE, 0, 128, 10, FAKE) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode_paged(*ok, FAKE, 4, 128, 0, FAKE) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode_paged(FAKE, FAKE, FAKE, FAKE, 2, 32, 4, FAKE, 4, 128, 10, FAKE) == kb.KB_ERR_UNSUPPORTED


def test_training_entry_points_reject_bad_arguments(kb):
    args = (FAKE, FAKE, FAKE, FAKE)
    assert kb.kb_attn_prefill_lse(*args, None, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG       # no lse
    assert kb.kb_attn_prefill_lse(*args, FAKE + 2, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG   # misaligned lse
    assert kb.kb_attn_prefill_lse(*args, FAKE, 1, 32, 8, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_prefill_lse(*args, FAKE, 1, 32, 4, 64) == kb.KB_ERR_UNSUPPORTED       # Hq != 4 Hkv
    ok = (FAKE, FAKE, FAKE, FAKE, FAKE)                                                     # q k v o dout
    outs = (FAKE, FAKE, FAKE)                                                               # dq dk dv
    assert kb.kb_attn_backward(*ok, None, FAKE, *outs, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG   # no lse
    assert kb.kb_attn_backward(*ok, FAKE, None, *outs, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG   # no delta
    assert kb.kb_attn_backward(*ok, FAKE, FAKE, FAKE + 8, FAKE, FAKE, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_backward(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, *outs, 1, 32, 8, 64) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_backward(*ok, FAKE, FAKE, *outs, 1, 32, 8, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_backward(*ok, FAKE, FAKE, *outs, 1, 32, 2, 64) == kb.KB_ERR_UNSUPPORTED


def test_segmented_mode_rejects_bad_arguments(kb):
    args = (FAKE, FAKE, FAKE, FAKE, 1, 32, 8)
    assert kb.kb_attn_prefill_seg(*args, 64, 0) == kb.KB_ERR_INVALID_ARG                     # seg_tiles 0
    assert kb.kb_attn_prefill_seg(*args, 0, 2) == kb.KB_ERR_INVALID_ARG                      # S 0
    assert kb.kb_attn_decode_seg(*args, 100, 200, 0, FAKE, 1 << 20) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode_seg(*args, 300, 200, 2, FAKE, 1 << 20) == kb.KB_ERR_INVALID_ARG  # ctx > cap
    assert kb.kb_attn_decode_seg(*args, 100, 200, 2, None, 1 << 20) == kb.KB_ERR_INVALID_ARG  # no workspace
    need = kb.kb_attn_seg_workspace_bytes(1, 32, 1, 99, 2)
    assert need == 32 * 1 * 1 * 132 * 4
    assert kb.kb_attn_decode_seg(*args, 100, 200, 2, FAKE, need - 1) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode_seg(*args, 100, 200, 2, FAKE + 8, need) == kb.KB_ERR_INVALID_ARG  # misaligned
    assert kb.kb_attn_seg_workspace_bytes(1, 32, 33, 0, 2) == 0                              # L > 32: none needed
    assert kb.kb_attn_seg_workspace_bytes(1, 32, 1, 8191, 8) == 32 * 8 * 132 * 4
    # the static-scratch variant: 4 MiB of partials at most, checked before any CUDA call
    assert kb.kb_attn_decode_seg_static(*args, 100, 200, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_decode_seg_static(FAKE, FAKE, FAKE, FAKE, 64, 32, 8, 1 << 16, 1 << 16, 1) == \
        kb.KB_ERR_UNSUPPORTED


def test_packed_shape_limits(kb):
    assert kb.kb_attn_chunk_cta_shape(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 33, 0, 64, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_cta_shape(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 4, 0, 64, -1) == kb.KB_ERR_INVALID_ARG


def test_paged_chunk_arguments_rejected(kb):
    args = (FAKE, FAKE, FAKE, FAKE, 1, 32, 8)
    assert kb.kb_attn_chunk_paged(*args, 16, 0, None, 4, 128, 8) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_paged(*args, 16, 500, FAKE, 4, 128, 8) == kb.KB_ERR_INVALID_ARG   # past 4 pages
    assert kb.kb_attn_chunk_paged(*args, 16, 0, FAKE, 4, 100, 8) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_paged(*args, 16, 0, FAKE, 4, 192, 8) == kb.KB_ERR_UNSUPPORTED


def test_packed_path_host_checks_do_not_trap(kb):
    """Small chunks take the packed path; its host checks run without a GPU
    and end in a CUDA error here (no device), never in a host fault."""
    st = kb.kb_attn_chunk_paged(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 16, 0, FAKE, 4, 640, 8)
    assert st in (kb.KB_ERR_CUDA, kb.KB_ERR_INVALID_ARG)
    st = kb.kb_attn_chunk(FAKE, FAKE, FAKE, FAKE, 1, 32, 8, 16, 0, 64)
    assert st in (kb.KB_ERR_CUDA, kb.KB_ERR_INVALID_ARG)


def test_varlen_arguments_rejected(kb):
    args = (FAKE, FAKE, FAKE, FAKE, 2, 32, 8)
    assert kb.kb_attn_chunk_varlen(*args, 16, None, FAKE, 64, None, 0, 0, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_varlen(*args, 16, FAKE, FAKE + 2, 64, None, 0, 0, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_varlen(*args, 0, FAKE, FAKE, 64, None, 0, 0, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_varlen(*args, 65, FAKE, FAKE, 64, None, 0, 0, 0) == kb.KB_ERR_INVALID_ARG
    assert kb.kb_attn_chunk_varlen(*args, 16, FAKE, FAKE, 0, FAKE, 2, 192, 4) == kb.KB_ERR_UNSUPPORTED
