"""Shape rules of the entry points, as pure functions over shape tuples.

The C ABI receives plain pointers and sizes, so it cannot see how large the
caller's buffers are: a key cache shorter than the sequence, or an output
smaller than the query, would turn into reads or writes past an allocation.
The torch binding therefore checks every tensor's full shape against the
others with these functions before it makes any call into the library.
They hold no attention arithmetic and need neither a GPU nor the library, so
the CPU tests cover every mismatch.

Layouts (KernelBraid README, "Features": contiguous [batch, heads, seq,
head_dim], head_dim 128; "Usage": the output has the query's shape):
  q, o      [B, Hq, L, 128]
  k, v      [B, Hkv, cap, 128]                (contiguous cache)
  pools     [num_pages, Hkv, page_size, 128]  (paged cache)
Each function raises ValueError naming the first mismatch and returns the
sizes the C call takes.
"""

from __future__ import annotations

HEAD_DIM = 128


def _shape(t) -> tuple:
    return tuple(int(d) for d in t)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _rows(name: str, s: tuple) -> None:
    _need(len(s) == 4, f"{name} must have 4 dimensions [batch, heads, seq, head_dim], got {s}")
    _need(s[3] == HEAD_DIM, f"{name} must have head_dim {HEAD_DIM}, got {s}")
    _need(min(s) >= 1, f"{name} has an empty dimension: {s}")


def _same(name: str, s: tuple, ref_name: str, ref: tuple) -> None:
    _need(s == ref, f"{name} must have the shape of {ref_name} {ref}, got {s}")


def query_and_cache(q, k, v, out=None) -> tuple[int, int, int, int, int]:
    """q [B,Hq,L,128]; k = v [B,Hkv,cap,128]; out = q.  Returns (B, Hq, Hkv, L, cap)."""
    q, k, v = _shape(q), _shape(k), _shape(v)
    _rows("q", q)
    _rows("k", k)
    _same("v", v, "k", k)
    _need(k[0] == q[0], f"k must have q's batch {q[0]}, got {k[0]}")
    if out is not None:
        _same("out", _shape(out), "q", q)
    return q[0], q[1], k[1], q[2], k[2]


def prefill(q, k, v, out=None) -> tuple[int, int, int, int]:
    """Whole sequence: the cache holds exactly the query's S positions.  Returns (B, Hq, Hkv, S)."""
    B, Hq, Hkv, S, cap = query_and_cache(q, k, v, out)
    _need(cap == S, f"prefill needs k and v of q's sequence length {S}, got {cap}")
    return B, Hq, Hkv, S


def chunk(q, k, v, start: int, out=None) -> tuple[int, int, int, int, int]:
    """Rows start..start+L-1 against a cache of capacity cap >= start + L.  Returns (B, Hq, Hkv, L, cap)."""
    B, Hq, Hkv, L, cap = query_and_cache(q, k, v, out)
    _need(int(start) >= 0, f"start must be >= 0, got {start}")
    _need(int(start) + L <= cap, f"start + L = {int(start) + L} exceeds the cache capacity {cap}")
    return B, Hq, Hkv, L, cap


def decode(q, k, v, ctx_len: int, out=None) -> tuple[int, int, int, int]:
    """One query row at position ctx_len - 1.  Returns (B, Hq, Hkv, cap)."""
    B, Hq, Hkv, L, cap = query_and_cache(q, k, v, out)
    _need(L == 1, f"decode takes one query row per (batch, head), got {L}")
    _need(1 <= int(ctx_len) <= cap, f"ctx_len must lie in 1..{cap} (the cache capacity), got {ctx_len}")
    return B, Hq, Hkv, cap


def pools(q, k_pages, v_pages, block_table, out=None) -> tuple[int, int, int, int, int, int, int]:
    """Paged cache: pools [num_pages,Hkv,page,128], block_table [B, pages_per_seq].
    Returns (B, Hq, Hkv, L, num_pages, page_size, pages_per_seq)."""
    q, kp, vp, bt = _shape(q), _shape(k_pages), _shape(v_pages), _shape(block_table)
    _rows("q", q)
    _rows("k_pages", kp)
    _same("v_pages", vp, "k_pages", kp)
    _need(len(bt) == 2 and bt[0] == q[0] and bt[1] >= 1,
          f"block_table must be [batch {q[0]}, pages_per_seq >= 1], got {bt}")
    if out is not None:
        _same("out", _shape(out), "q", q)
    return q[0], q[1], kp[1], q[2], kp[0], kp[2], bt[1]


def chunk_paged(q, k_pages, v_pages, block_table, start: int, out=None):
    B, Hq, Hkv, L, num_pages, page, pps = pools(q, k_pages, v_pages, block_table, out)
    _need(int(start) >= 0, f"start must be >= 0, got {start}")
    _need(int(start) + L <= pps * page, f"start + L = {int(start) + L} exceeds the page table's {pps * page} rows")
    return B, Hq, Hkv, L, num_pages, page, pps


def decode_paged(q, k_pages, v_pages, block_table, ctx_lens, out=None):
    B, Hq, Hkv, L, num_pages, page, pps = pools(q, k_pages, v_pages, block_table, out)
    _need(L == 1, f"decode takes one query row per (batch, head), got {L}")
    _need(_shape(ctx_lens) == (B,), f"ctx_lens must have shape ({B},), got {_shape(ctx_lens)}")
    return B, Hq, Hkv, num_pages, page, pps


def varlen(q, k, v, starts, lens, block_table=None, out=None):
    """Ragged batch: starts, lens [B]; k/v a contiguous cache or (with block_table) pools.
    Returns (B, Hq, Hkv, L_max) plus (cap,) or (num_pages, page_size, pages_per_seq)."""
    qs = _shape(q)
    _rows("q", qs)
    B = qs[0]
    for name, t in (("starts", starts), ("lens", lens)):
        _need(_shape(t) == (B,), f"{name} must have shape ({B},), got {_shape(t)}")
    if block_table is None:
        B, Hq, Hkv, L_max, cap = query_and_cache(q, k, v, out)
        _need(L_max <= cap, f"L_max {L_max} exceeds the cache capacity {cap}")
        return B, Hq, Hkv, L_max, cap
    B, Hq, Hkv, L_max, num_pages, page, pps = pools(q, k, v, block_table, out)
    _need(L_max <= pps * page, f"L_max {L_max} exceeds the page table's {pps * page} rows")
    return B, Hq, Hkv, L_max, num_pages, page, pps


def vector_f32(name: str, t, B: int, Hq: int, S: int) -> None:
    """Per-row float32 outputs (log-sum-exp, delta): [B, Hq, S]."""
    _need(_shape(t) == (B, Hq, S), f"{name} must have shape {(B, Hq, S)}, got {_shape(t)}")


def backward(q, k, v, o, dout, dq=None, dk=None, dv=None) -> tuple[int, int, int, int]:
    """Gradients of the whole-sequence prefill: o, dout, dq like q; dk, dv like k.  Returns (B, Hq, Hkv, S)."""
    B, Hq, Hkv, S = prefill(q, k, v, o)
    qs, ks = _shape(q), _shape(k)
    _same("dout", _shape(dout), "q", qs)
    for name, t, ref_name, ref in (("dq", dq, "q", qs), ("dk", dk, "k", ks), ("dv", dv, "v", ks)):
        if t is not None:
            _same(name, _shape(t), ref_name, ref)
    return B, Hq, Hkv, S
