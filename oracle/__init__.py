"""fp64 CPU oracle for causal grouped-query attention.

TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library never
imports, links or runs anything here, and this package never touches it.

The arithmetic lives in ``kb_oracle.c`` (plain definition of causal GQA
attention in double precision, and of its gradient with respect to q, k
and v; see the comments in that file).  This module
only builds it with gcc, loads it with ctypes and marshals numpy arrays.

Parity status: pinned.  ``tests/test_oracle_pins.py`` checks the forward
against closed forms, invariants of the definition and an independent brute
force; ``tests/test_oracle_backward_pins.py`` checks the gradient against
central finite differences of the forward oracle, float64 autograd of an
independent PyTorch expression, closed forms and invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kb_oracle.c")
_LIB = os.path.join(_HERE, "libkb_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile kb_oracle.c into libkb_oracle.so next to it (gcc, -O2)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-pthread", _SRC, "-lm", "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _bind(path: str):
    lib = ctypes.CDLL(path)
    lib.kb_oracle_rows.restype = ctypes.c_int
    lib.kb_oracle_rows.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.kb_oracle_backward.restype = ctypes.c_int
    lib.kb_oracle_backward.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    lib.kb_oracle_dq_rows.restype = ctypes.c_int
    lib.kb_oracle_dq_rows.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
        ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
    ]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            _lib = _bind(_LIB)
    return _lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def attention_rows(q_bits, k_bits, v_bits, rows, *, start: int = 0, n_threads: int | None = None,
                   _lib_override=None):
    """Oracle output (float64, [n_rows, D]) for the listed query rows.

    q_bits: uint16 bf16 bit patterns [B, Hq, Lq, D]; query row i sits at
        absolute position ``start + i`` and sees keys 0..start+i.
    k_bits, v_bits: uint16 [B, Hkv, cap, D].
    rows: int array [n, 3] of (b, h, i).
    """
    lib = _load() if _lib_override is None else _lib_override
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape:
        raise ValueError("q must be [B,Hq,Lq,D] and k, v [B,Hkv,cap,D]")
    B, Hq, Lq, D = q.shape
    Bk, Hkv, cap, Dk = k.shape
    if Bk != B or Dk != D:
        raise ValueError("batch / head_dim mismatch between q and k")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    out = np.empty((r.shape[0], D), dtype=np.float64)
    if r.shape[0] == 0:
        return out
    nt = default_threads() if n_threads is None else int(n_threads)
    rc = lib.kb_oracle_rows(
        q.ctypes.data, k.ctypes.data, v.ctypes.data,
        B, Hq, Hkv, Lq, D, int(start), cap,
        r.ctypes.data, r.shape[0], out.ctypes.data, nt,
    )
    if rc != 0:
        raise ValueError(f"kb_oracle_rows failed with code {rc}")
    return out


def attention_full(q_bits, k_bits, v_bits, *, start: int = 0, n_threads: int | None = None,
                   _lib_override=None):
    """Oracle output for every query row, shaped [B, Hq, Lq, D] (float64)."""
    B, Hq, Lq, D = np.shape(q_bits)
    bb, hh, ii = np.meshgrid(np.arange(B), np.arange(Hq), np.arange(Lq), indexing="ij")
    rows = np.stack([bb.ravel(), hh.ravel(), ii.ravel()], axis=1)
    out = attention_rows(q_bits, k_bits, v_bits, rows, start=start, n_threads=n_threads,
                         _lib_override=_lib_override)
    return out.reshape(B, Hq, Lq, D)


def _bwd_inputs(q_bits, k_bits, v_bits, dout_bits):
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    do = np.ascontiguousarray(dout_bits, dtype=np.uint16)
    if q.ndim != 4 or k.ndim != 4 or v.shape != k.shape or do.shape != q.shape:
        raise ValueError("q, dout must be [B,Hq,S,D] and k, v [B,Hkv,S,D]")
    B, Hq, S, D = q.shape
    if k.shape[0] != B or k.shape[2] != S or k.shape[3] != D:
        raise ValueError("k, v must cover the same batch, sequence and head_dim as q")
    return q, k, v, do


def backward(q_bits, k_bits, v_bits, dout_bits, *, n_threads: int | None = None, _lib_override=None):
    """Gradients (dq, dk, dv), float64, of causal GQA attention over a whole
    sequence (query row i at position i) for output gradient ``dout``.

    q_bits, dout_bits: uint16 bf16 bits [B, Hq, S, D]; k_bits, v_bits [B, Hkv, S, D].
    """
    lib = _load() if _lib_override is None else _lib_override
    q, k, v, do = _bwd_inputs(q_bits, k_bits, v_bits, dout_bits)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    dq = np.empty(q.shape, dtype=np.float64)
    dk = np.empty(k.shape, dtype=np.float64)
    dv = np.empty(k.shape, dtype=np.float64)
    nt = default_threads() if n_threads is None else int(n_threads)
    rc = lib.kb_oracle_backward(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data,
                                B, Hq, Hkv, S, D, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data, nt)
    if rc != 0:
        raise ValueError(f"kb_oracle_backward failed with code {rc}")
    return dq, dk, dv


def dq_rows(q_bits, k_bits, v_bits, dout_bits, rows, *, n_threads: int | None = None, _lib_override=None):
    """For listed rows (b, h, i) of a whole-sequence prefill: dq [n, D], the
    natural-log log-sum-exp of the row's scaled scores [n] and
    delta = sum_j P_ij dP_ij [n] (float64)."""
    lib = _load() if _lib_override is None else _lib_override
    q, k, v, do = _bwd_inputs(q_bits, k_bits, v_bits, dout_bits)
    B, Hq, S, D = q.shape
    Hkv = k.shape[1]
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32).reshape(-1, 3))
    n = r.shape[0]
    dq = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    delta = np.empty(n, dtype=np.float64)
    if n == 0:
        return dq, lse, delta
    nt = default_threads() if n_threads is None else int(n_threads)
    rc = lib.kb_oracle_dq_rows(q.ctypes.data, k.ctypes.data, v.ctypes.data, do.ctypes.data,
                               B, Hq, Hkv, S, D, r.ctypes.data, n, dq.ctypes.data, lse.ctypes.data,
                               delta.ctypes.data, nt)
    if rc != 0:
        raise ValueError(f"kb_oracle_dq_rows failed with code {rc}")
    return dq, lse, delta
