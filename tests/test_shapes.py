"""The binding's shape rules (bitwise_aligned_causal_gb300/shapes.py), on the CPU.

The C ABI takes plain pointers, so it cannot see a buffer's size: every
tensor shape is checked against the others before a call.  Each mismatch
below would otherwise let a kernel read or write past an allocation.
"""

import pytest

from bitwise_aligned_causal_gb300 import shapes

B, HQ, HKV, S, D = 2, 32, 8, 300, 128
Q = (B, HQ, S, D)
KV = (B, HKV, S, D)


def test_consistent_shapes_pass_and_return_the_call_sizes():
    assert shapes.prefill(Q, KV, KV, Q) == (B, HQ, HKV, S)
    assert shapes.chunk((B, HQ, 20, D), (B, HKV, 512, D), (B, HKV, 512, D), 100) == (B, HQ, HKV, 20, 512)
    assert shapes.decode((B, HQ, 1, D), (B, HKV, 512, D), (B, HKV, 512, D), 512) == (B, HQ, HKV, 512)
    assert shapes.backward(Q, KV, KV, Q, Q, Q, KV, KV) == (B, HQ, HKV, S)
    pool = (10, HKV, 256, D)
    assert shapes.chunk_paged((B, HQ, 5, D), pool, pool, (B, 3), 700) == (B, HQ, HKV, 5, 10, 256, 3)
    assert shapes.decode_paged((B, HQ, 1, D), pool, pool, (B, 3), (B,)) == (B, HQ, HKV, 10, 256, 3)
    assert shapes.varlen((B, HQ, 40, D), (B, HKV, 512, D), (B, HKV, 512, D), (B,), (B,)) == (B, HQ, HKV, 40, 512)
    assert shapes.varlen((B, HQ, 40, D), pool, pool, (B,), (B,), (B, 3)) == (B, HQ, HKV, 40, 10, 256, 3)


@pytest.mark.parametrize("q,k,v,out", [
    ((B, HQ, S, 64), KV, KV, None),                    # head_dim of q
    (Q, (B, HKV, S, 64), (B, HKV, S, 64), None),       # head_dim of k and v
    (Q, KV, (B, HKV, S - 1, D), None),                 # v shorter than k
    (Q, KV, (B, HKV + 1, S, D), None),                 # v with other heads
    (Q, (B, HKV, S - 1, D), (B, HKV, S - 1, D), None),  # cache shorter than the sequence
    (Q, (B, HKV, S + 1, D), (B, HKV, S + 1, D), None),  # cache longer than the sequence
    (Q, (B - 1, HKV, S, D), (B - 1, HKV, S, D), None),  # k batch smaller than q's
    (Q, (B + 1, HKV, S, D), (B + 1, HKV, S, D), None),  # k batch larger than q's
    (Q, KV, KV, (B, HQ, S - 1, D)),                    # out shorter than q
    (Q, KV, KV, (B, HQ - 1, S, D)),                    # out with fewer heads
    (Q, KV, KV, (B, HQ, S, D, 1)),                     # out of another rank
    ((B, HQ, S), KV, KV, None),                        # q of another rank
    ((B, HQ, 0, D), KV, KV, None),                     # empty q
])
def test_prefill_mismatches_are_refused(q, k, v, out):
    with pytest.raises(ValueError):
        shapes.prefill(q, k, v, out)


@pytest.mark.parametrize("q,k,v,start,out", [
    ((B, HQ, 20, D), (B, HKV, 119, D), (B, HKV, 119, D), 100, None),    # start + L past the cache
    ((B, HQ, 20, D), (B, HKV, 512, D), (B, HKV, 512, D), -1, None),     # negative start
    ((B, HQ, 20, D), (B, HKV, 512, D), (B, HKV, 511, D), 0, None),      # v capacity differs
    ((B, HQ, 20, D), (1, HKV, 512, D), (1, HKV, 512, D), 0, None),      # cache batch differs
    ((B, HQ, 20, D), (B, HKV, 512, D), (B, HKV, 512, D), 0, (B, HQ, 19, D)),   # out too small
])
def test_chunk_mismatches_are_refused(q, k, v, start, out):
    with pytest.raises(ValueError):
        shapes.chunk(q, k, v, start, out)


@pytest.mark.parametrize("q,k,ctx,out", [
    ((B, HQ, 2, D), (B, HKV, 512, D), 512, None),      # more than one query row
    ((B, HQ, 1, D), (B, HKV, 512, D), 513, None),      # context past the cache
    ((B, HQ, 1, D), (B, HKV, 512, D), 0, None),        # empty context
    ((B, HQ, 1, D), (B + 1, HKV, 512, D), 10, None),   # batch differs
    ((B, HQ, 1, D), (B, HKV, 512, D), 10, (B, HQ, 2, D)),  # out of another shape
])
def test_decode_mismatches_are_refused(q, k, ctx, out):
    with pytest.raises(ValueError):
        shapes.decode(q, k, k, ctx, out)


POOL = (10, HKV, 256, D)


@pytest.mark.parametrize("kp,vp,table,start", [
    (POOL, (9, HKV, 256, D), (B, 3), 0),           # pools differ
    (POOL, POOL, (B + 1, 3), 0),                   # table batch differs
    (POOL, POOL, (B,), 0),                         # table of another rank
    (POOL, POOL, (B, 3), 764),                     # chunk past the table's rows
    ((10, HKV, 256, 64), (10, HKV, 256, 64), (B, 3), 0),   # head_dim
])
def test_paged_chunk_mismatches_are_refused(kp, vp, table, start):
    with pytest.raises(ValueError):
        shapes.chunk_paged((B, HQ, 5, D), kp, vp, table, start)


def test_paged_decode_mismatches_are_refused():
    with pytest.raises(ValueError):
        shapes.decode_paged((B, HQ, 1, D), POOL, POOL, (B, 3), (B + 1,))     # ctx_lens length
    with pytest.raises(ValueError):
        shapes.decode_paged((B, HQ, 2, D), POOL, POOL, (B, 3), (B,))         # two query rows
    with pytest.raises(ValueError):
        shapes.decode_paged((B, HQ, 1, D), POOL, POOL, (B, 3), (B,), (B, HQ, 1, 64))   # out


def test_varlen_mismatches_are_refused():
    kv = (B, HKV, 512, D)
    with pytest.raises(ValueError):
        shapes.varlen((B, HQ, 40, D), kv, kv, (B + 1,), (B,))                # starts length
    with pytest.raises(ValueError):
        shapes.varlen((B, HQ, 40, D), kv, kv, (B,), (B, 1))                  # lens rank
    with pytest.raises(ValueError):
        shapes.varlen((B, HQ, 600, D), kv, kv, (B,), (B,))                   # L_max past the cache
    with pytest.raises(ValueError):
        shapes.varlen((B, HQ, 40, D), kv, (B, HKV, 511, D), (B,), (B,))      # v differs
    with pytest.raises(ValueError):
        shapes.varlen((B, HQ, 800, D), POOL, POOL, (B,), (B,), (B, 3))       # L_max past the pages


@pytest.mark.parametrize("which", ["o", "dout", "dq", "dk", "dv"])
def test_backward_mismatches_are_refused(which):
    t = {"o": Q, "dout": Q, "dq": Q, "dk": KV, "dv": KV}
    t[which] = (B, HQ if which in ("o", "dout", "dq") else HKV, S - 1, D)
    with pytest.raises(ValueError):
        shapes.backward(Q, KV, KV, t["o"], t["dout"], t["dq"], t["dk"], t["dv"])


def test_per_row_vectors():
    shapes.vector_f32("lse", (B, HQ, S), B, HQ, S)
    for bad in [(B, HQ, S - 1), (B, HQ), (B, HQ, S, 1)]:
        with pytest.raises(ValueError):
            shapes.vector_f32("lse", bad, B, HQ, S)
