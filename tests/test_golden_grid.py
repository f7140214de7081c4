"""The workload grid printed by the pages (tests/golden/workload_grid.txt) matches ours."""

import os

from bitwise_aligned_causal_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "workload_grid.txt")


def load():
    out = {}
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, *vals = line.split()
        out[key] = [int(v) for v in vals]
    return out


def test_head_shape_constants():
    g = load()
    assert g["n_q_heads"] == [inputs.N_Q_HEADS]
    assert g["n_kv_heads"] == [inputs.N_KV_HEADS]
    assert g["head_dim"] == [inputs.HEAD_DIM]


def test_grid_size():
    g = load()
    n_prefill = 1 * len(g["prefill_lengths"])            # batch 1 only in the prefill bars
    n_decode = len(g["batch_sizes"]) * len(g["decode_contexts"])
    assert n_prefill + n_decode == g["configs_per_gpu"][0]
