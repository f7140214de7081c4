"""ctypes binding of libkb_attn.so (C ABI in include/kb_attn.h).

Argument marshalling only: every step of the attention runs in the library's
CUDA kernels.  The functions named like the C entry points take raw device
pointers; ``prefill`` / ``chunk`` / ``decode`` accept torch CUDA tensors
(PyTorch is used here only for device memory and streams).

Importing this module loads the library and raises ``ImportError`` when it
has not been built: there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

from . import shapes

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkb_attn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with bitwise_aligned_causal_gb300.build.build()")
_lib = ctypes.CDLL(LIB_PATH)

KB_OK = 0
KB_ERR_INVALID_ARG = 1
KB_ERR_UNSUPPORTED = 2
KB_ERR_CUDA = 3
KB_ERR_TIMEOUT = 4

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "kb_attn_prefill": [_P, _P, _P, _P, _I, _I, _I, _I, _P],
    "kb_attn_chunk": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
    "kb_attn_decode": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P],
    "kb_attn_decode_paged": [_P, _P, _P, _P, _I, _I, _I, _P, _I, _I, _I, _P, _P],
    "kb_attn_chunk_paged": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I, _I, _I, _P],
    "kb_attn_chunk_varlen": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _I, _P, _I, _I, _I, _P],
    "kb_attn_check_device_status": [_P],
    "kb_attn_debug_wait_timeout": [_I, _P],
    "kb_attn_chunk_cta_shape": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P],
    "kb_attn_prefill_lse": [_P, _P, _P, _P, _P, _I, _I, _I, _I, _P],
    "kb_attn_prefill_seg": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _P],
    "kb_attn_chunk_seg": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P],
    "kb_attn_decode_seg": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P],
    "kb_attn_seg_workspace_bytes": [_I, _I, _I, _I, _I],
    "kb_attn_decode_seg_static": [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P],
    "kb_attn_backward": [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P],
    "kb_status_string": [_I],
    "kb_contract_version": [],
    "kb_attn_last_cuda_error": [],
    "kb_attn_last_cuda_error_string": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = (ctypes.c_char_p if _name.endswith("string")
                  else ctypes.c_size_t if _name.endswith("_bytes") else ctypes.c_int)

EXPORTED = tuple(_SIGS)


class KBError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {kb_status_string(status)} (status {status})"
        if status == KB_ERR_CUDA:
            msg += f": {kb_attn_last_cuda_error_string()} (cudaError {kb_attn_last_cuda_error()})"
        super().__init__(msg)


def kb_status_string(status: int) -> str:
    return _lib.kb_status_string(int(status)).decode()


def kb_contract_version() -> int:
    return int(_lib.kb_contract_version())


def kb_attn_last_cuda_error() -> int:
    return int(_lib.kb_attn_last_cuda_error())


def kb_attn_last_cuda_error_string() -> str:
    return _lib.kb_attn_last_cuda_error_string().decode()


# ---------------------------------------------------------------- raw C entry points

def kb_attn_prefill(q, k, v, o, B, Hq, Hkv, S, stream=None) -> int:
    return _lib.kb_attn_prefill(q, k, v, o, B, Hq, Hkv, S, stream)


def kb_attn_chunk(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, stream=None) -> int:
    return _lib.kb_attn_chunk(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, stream)


def kb_attn_decode(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, stream=None) -> int:
    return _lib.kb_attn_decode(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, stream)


def kb_attn_decode_paged(q, k_pages, v_pages, o, B, Hq, Hkv, block_table, pages_per_seq, page_size, num_pages,
                         ctx_lens, stream=None) -> int:
    return _lib.kb_attn_decode_paged(q, k_pages, v_pages, o, B, Hq, Hkv, block_table, pages_per_seq, page_size,
                                     num_pages, ctx_lens, stream)


def kb_attn_chunk_paged(q, k_pages, v_pages, o, B, Hq, Hkv, L, start, block_table, pages_per_seq, page_size,
                        num_pages, stream=None) -> int:
    return _lib.kb_attn_chunk_paged(q, k_pages, v_pages, o, B, Hq, Hkv, L, start, block_table, pages_per_seq,
                                    page_size, num_pages, stream)


def kb_attn_chunk_varlen(q, k, v, o, B, Hq, Hkv, L_max, starts, lens, kv_cap, block_table, pages_per_seq,
                         page_size, num_pages, stream=None) -> int:
    return _lib.kb_attn_chunk_varlen(q, k, v, o, B, Hq, Hkv, L_max, starts, lens, kv_cap, block_table, pages_per_seq,
                                     page_size, num_pages, stream)


def kb_attn_chunk_cta_shape(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, q_tiles_per_cta, stream=None) -> int:
    return _lib.kb_attn_chunk_cta_shape(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, q_tiles_per_cta, stream)


def kb_attn_prefill_lse(q, k, v, o, lse, B, Hq, Hkv, S, stream=None) -> int:
    return _lib.kb_attn_prefill_lse(q, k, v, o, lse, B, Hq, Hkv, S, stream)


def kb_attn_backward(q, k, v, o, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, stream=None) -> int:
    return _lib.kb_attn_backward(q, k, v, o, dout, lse, delta, dq, dk, dv, B, Hq, Hkv, S, stream)


def kb_attn_prefill_seg(q, k, v, o, B, Hq, Hkv, S, seg_tiles, stream=None) -> int:
    return _lib.kb_attn_prefill_seg(q, k, v, o, B, Hq, Hkv, S, seg_tiles, stream)


def kb_attn_chunk_seg(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, seg_tiles, workspace, workspace_bytes,
                      stream=None) -> int:
    return _lib.kb_attn_chunk_seg(q, k, v, o, B, Hq, Hkv, L, start, kv_cap, seg_tiles, workspace, workspace_bytes,
                                  stream)


def kb_attn_decode_seg(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, seg_tiles, workspace, workspace_bytes,
                       stream=None) -> int:
    return _lib.kb_attn_decode_seg(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, seg_tiles, workspace, workspace_bytes,
                                   stream)


def kb_attn_decode_seg_static(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, seg_tiles, stream=None) -> int:
    return _lib.kb_attn_decode_seg_static(q, k, v, o, B, Hq, Hkv, ctx_len, kv_cap, seg_tiles, stream)


def kb_attn_seg_workspace_bytes(B, Hq, L, start, seg_tiles) -> int:
    return int(_lib.kb_attn_seg_workspace_bytes(B, Hq, L, start, seg_tiles))


def kb_attn_check_device_status(stream=None) -> int:
    return _lib.kb_attn_check_device_status(stream)


def kb_attn_debug_wait_timeout(limit_us, stream=None) -> int:
    return _lib.kb_attn_debug_wait_timeout(limit_us, stream)


# ------------------------------------------------------------------ torch marshalling
#
# Every wrapper below checks each tensor's dtype, layout, device and full
# shape against the others (shapes.py) before the C call, so a caller's
# mistake raises here instead of becoming an out-of-bounds device access.
#
# Outputs are complete once the stream has run the kernels.  A bounded
# device-side wait that gave up, or a device-resident argument found out of
# range (a page index, a per-sequence length), leaves the affected rows
# unwritten and is reported only by check_device_status(), which also clears
# the library's error word; until that word is cleared, later calls on the
# device skip their work.  Pass check=True to call it after the launch.

def _torch():
    import torch

    return torch


def _stream(stream):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _on_current_device(t, name):
    torch = _torch()
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, not on the current device cuda:{torch.cuda.current_device()}")


def _check(t, name, ndim=4):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions [batch, heads, seq, head_dim]")
    _on_current_device(t, name)


def _check_i32(t, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    _on_current_device(t, name)


def _check_f32(t, name):
    torch = _torch()
    if not isinstance(t, torch.Tensor) or not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous float32 CUDA tensor")
    _on_current_device(t, name)


def _raise(status, where):
    if status != KB_OK:
        raise KBError(status, where)


def _out(q, out):
    o = _torch().empty_like(q) if out is None else out
    _check(o, "out")
    return o


def _finish(status, where, check, stream):
    _raise(status, where)
    if check:
        check_device_status(stream)


def prefill(q, k, v, out=None, stream=None, check=False):
    """Causal prefill: q [B,Hq,S,128], k/v [B,Hkv,S,128] -> o shaped like q."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, S = shapes.prefill(q.shape, k.shape, v.shape, None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, S, _stream(stream)),
            "kb_attn_prefill", check, stream)
    return o


def chunk(q, k, v, start, out=None, stream=None, q_tiles_per_cta=None, check=False):
    """Chunked forward: q [B,Hq,L,128] at positions start.., k/v caches [B,Hkv,cap,128]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, L, cap = shapes.chunk(q.shape, k.shape, v.shape, int(start), None if out is None else out.shape)
    o = _out(q, out)
    if q_tiles_per_cta is None:
        st = kb_attn_chunk(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, L, int(start), cap,
                           _stream(stream))
    else:
        st = kb_attn_chunk_cta_shape(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, L,
                                     int(start), cap, int(q_tiles_per_cta), _stream(stream))
    _finish(st, "kb_attn_chunk", check, stream)
    return o


def decode(q, k, v, ctx_len, out=None, stream=None, check=False):
    """One-token decode: q [B,Hq,1,128] at position ctx_len-1, k/v caches [B,Hkv,cap,128]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, cap = shapes.decode(q.shape, k.shape, v.shape, int(ctx_len), None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_decode(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, int(ctx_len), cap,
                           _stream(stream)), "kb_attn_decode", check, stream)
    return o


def decode_paged(q, k_pages, v_pages, block_table, ctx_lens, out=None, stream=None, check=False):
    """Paged decode: q [B,Hq,1,128]; pools [num_pages,Hkv,page_size,128]; block_table int32 [B,pages_per_seq];
    ctx_lens int32 [B] (all on the device)."""
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _check(t, n)
    for t, n in ((block_table, "block_table"), (ctx_lens, "ctx_lens")):
        _check_i32(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, num_pages, page_size, pps = shapes.decode_paged(
        q.shape, k_pages.shape, v_pages.shape, block_table.shape, ctx_lens.shape, None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), o.data_ptr(), B, Hq, Hkv,
                                 block_table.data_ptr(), pps, page_size, num_pages, ctx_lens.data_ptr(),
                                 _stream(stream)), "kb_attn_decode_paged", check, stream)
    return o


def chunk_paged(q, k_pages, v_pages, block_table, start, out=None, stream=None, check=False):
    """Chunked forward over a paged cache: q [B,Hq,L,128] at positions start..; pools
    [num_pages,Hkv,page_size,128]; block_table int32 [B,pages_per_seq] on the device."""
    for t, n in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _check(t, n)
    _check_i32(block_table, "block_table")
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, L, num_pages, page_size, pps = shapes.chunk_paged(
        q.shape, k_pages.shape, v_pages.shape, block_table.shape, int(start), None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_chunk_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(), o.data_ptr(), B, Hq, Hkv, L,
                                int(start), block_table.data_ptr(), pps, page_size, num_pages, _stream(stream)),
            "kb_attn_chunk_paged", check, stream)
    return o


def chunk_varlen(q, k, v, starts, lens, out=None, block_table=None, stream=None, check=False):
    """Ragged batch: q [B,Hq,L_max,128]; per-sequence starts/lens int32 [B] on the device; k/v either
    contiguous caches [B,Hkv,cap,128] or, with block_table [B,pages_per_seq], pools [num_pages,Hkv,page,128]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    for t, n in ((starts, "starts"), (lens, "lens")) + (((block_table, "block_table"),) if block_table is not None
                                                         else ()):
        _check_i32(t, n)
    if out is not None:
        _check(out, "out")
    sz = shapes.varlen(q.shape, k.shape, v.shape, starts.shape, lens.shape,
                       None if block_table is None else block_table.shape, None if out is None else out.shape)
    o = _out(q, out)
    if block_table is None:
        B, Hq, Hkv, L_max, cap = sz
        st = kb_attn_chunk_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, L_max,
                                  starts.data_ptr(), lens.data_ptr(), cap, None, 0, 0, 0, _stream(stream))
    else:
        B, Hq, Hkv, L_max, num_pages, page_size, pps = sz
        st = kb_attn_chunk_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, L_max,
                                  starts.data_ptr(), lens.data_ptr(), 0, block_table.data_ptr(), pps, page_size,
                                  num_pages, _stream(stream))
    _finish(st, "kb_attn_chunk_varlen", check, stream)
    return o


def check_device_status(stream=None):
    """Wait for `stream`, then raise KBError if a kernel since the last check gave up on a wait
    (KB_ERR_TIMEOUT) or found a device-resident argument out of range (KB_ERR_INVALID_ARG)."""
    _raise(kb_attn_check_device_status(_stream(stream)), "kb_attn_check_device_status")


def prefill_lse(q, k, v, out=None, lse=None, stream=None, check=False):
    """Training forward: (o, lse) with o bit-identical to prefill and lse [B,Hq,S] float32 the
    natural-log log-sum-exp of each row's scaled scores."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, S = shapes.prefill(q.shape, k.shape, v.shape, None if out is None else out.shape)
    o = _out(q, out)
    lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_f32(lse, "lse")
    shapes.vector_f32("lse", lse.shape, B, Hq, S)
    _finish(kb_attn_prefill_lse(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, Hq, Hkv,
                                S, _stream(stream)), "kb_attn_prefill_lse", check, stream)
    return o, lse


def backward(q, k, v, o, dout, lse, delta=None, dq=None, dk=None, dv=None, stream=None, check=False):
    """Gradients (dq, dk, dv) of the whole-sequence causal prefill for output gradient dout; o and
    lse from prefill_lse.  Also returns delta [B,Hq,S] float32 = rowsum(dout * o)."""
    torch = _torch()
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check(t, n)
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        if t is not None:
            _check(t, n)
    B, Hq, Hkv, S = shapes.backward(q.shape, k.shape, v.shape, o.shape, dout.shape,
                                    None if dq is None else dq.shape, None if dk is None else dk.shape,
                                    None if dv is None else dv.shape)
    _check_f32(lse, "lse")
    shapes.vector_f32("lse", lse.shape, B, Hq, S)
    delta = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device) if delta is None else delta
    _check_f32(delta, "delta")
    shapes.vector_f32("delta", delta.shape, B, Hq, S)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _finish(kb_attn_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(), lse.data_ptr(),
                             delta.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, S,
                             _stream(stream)), "kb_attn_backward", check, stream)
    return dq, dk, dv, delta


def _workspace(nbytes, device, workspace):
    torch = _torch()
    if workspace is None:
        return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)
    if not isinstance(workspace, torch.Tensor) or not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    _on_current_device(workspace, "workspace")
    return workspace


def prefill_seg(q, k, v, seg_tiles, out=None, stream=None, check=False):
    """Segmented-mode prefill (segments of seg_tiles 128-key tiles, folded left to right)."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, S = shapes.prefill(q.shape, k.shape, v.shape, None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_prefill_seg(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, S,
                                int(seg_tiles), _stream(stream)), "kb_attn_prefill_seg", check, stream)
    return o


def chunk_seg(q, k, v, start, seg_tiles, out=None, workspace=None, stream=None, check=False):
    """Segmented-mode chunk: q [B,Hq,L,128] at positions start.., caches [B,Hkv,cap,128]."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, L, cap = shapes.chunk(q.shape, k.shape, v.shape, int(start), None if out is None else out.shape)
    o = _out(q, out)
    ws = _workspace(kb_attn_seg_workspace_bytes(B, Hq, L, int(start), int(seg_tiles)), q.device, workspace)
    _finish(kb_attn_chunk_seg(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, L, int(start), cap,
                              int(seg_tiles), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
            "kb_attn_chunk_seg", check, stream)
    return o


def decode_seg(q, k, v, ctx_len, seg_tiles, out=None, workspace=None, stream=None, check=False):
    """Segmented-mode decode: q [B,Hq,1,128] at position ctx_len-1."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, cap = shapes.decode(q.shape, k.shape, v.shape, int(ctx_len), None if out is None else out.shape)
    o = _out(q, out)
    ws = _workspace(kb_attn_seg_workspace_bytes(B, Hq, 1, int(ctx_len) - 1, int(seg_tiles)), q.device, workspace)
    _finish(kb_attn_decode_seg(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv, int(ctx_len), cap,
                               int(seg_tiles), ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
            "kb_attn_decode_seg", check, stream)
    return o


def decode_seg_static(q, k, v, ctx_len, seg_tiles, out=None, stream=None, check=False):
    """Segmented-mode decode with the library's own scratch (no workspace argument, no allocation).
    Calls that overlap on the GPU share that scratch and must not run at the same time."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n)
    if out is not None:
        _check(out, "out")
    B, Hq, Hkv, cap = shapes.decode(q.shape, k.shape, v.shape, int(ctx_len), None if out is None else out.shape)
    o = _out(q, out)
    _finish(kb_attn_decode_seg_static(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, Hq, Hkv,
                                      int(ctx_len), cap, int(seg_tiles), _stream(stream)),
            "kb_attn_decode_seg_static", check, stream)
    return o
