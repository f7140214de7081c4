"""Bitwise-aligned causal GQA attention for GB300 (sm_103a).

One numerical contract makes full-sequence prefill, chunked forward against a
KV cache and one-token decode produce identical output bits for the same
query position and context (KernelBraid README, sections "Method" and
"Advantages").  The kernels live in ``libkb_attn.so`` (hand-written CUDA for
sm_103a, C ABI declared in ``include/kb_attn.h``); ``kb_attn`` is the thin
ctypes binding over it.  Importing this package does not load the library;
``from bitwise_aligned_causal_gb300 import kb_attn`` does, and raises if the
library has not been built.
"""

__all__ = ["kb_attn", "inputs", "build"]
