"""Which inputs make the contract's rescale branch fire (host only, no GPU).

The row function moves a row's reference max only when a later key tile's
max exceeds it by more than 64 raw score units; only then is O rescaled.
With iid N(0, 1) inputs that is an 8-sigma event, so bitwise tests on such
inputs never exercise the branch; the stress recipe (q, k ~ N(0, 8^2), 1% of
keys x32) takes it on most rows.  These checks pin the host-side replay of
the decision that the GPU stress tests rely on.
"""

import numpy as np

from bitwise_aligned_causal_gb300 import inputs
from tests.gpu_util import rescale_after_first_tile, rescale_fraction


def _bits(a):
    return inputs.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_constructed_scores_decide_as_the_threshold_says():
    # q = e0 so the score of key j is k_j[0]; tile 0 holds max 10
    D, S = 128, 300
    q = np.zeros((3, D), np.float32)
    q[:, 0] = 1.0
    k = np.zeros((S, D), np.float32)
    k[5, 0] = 10.0
    k[200, 0] = 10.0 + 100.0       # tile 1: 100 above the max -> moves
    k[260, 0] = 10.0 + 30.0        # tile 2: below the 64 threshold
    pos = np.array([150, 210, 299])
    got = rescale_after_first_tile(_bits(q), _bits(k), pos)
    assert got.tolist() == [False, True, True]
    k[200, 0] = 10.0 + 50.0        # 50 above: no move anywhere
    got = rescale_after_first_tile(_bits(q), _bits(k), pos)
    assert got.tolist() == [False, False, False]
    k[260, 0] = 10.0 + 64.0        # exactly 64 above: the contract needs more than 64
    assert not rescale_after_first_tile(_bits(q), _bits(k), pos).any()
    k[260, 0] = 10.0 + 66.0
    assert rescale_after_first_tile(_bits(q), _bits(k), pos).tolist() == [False, False, True]


def test_masked_future_keys_do_not_count():
    D, S = 128, 300
    q = np.zeros((1, D), np.float32)
    q[0, 0] = 1.0
    k = np.zeros((S, D), np.float32)
    k[150, 0] = 500.0              # tile 1, but after the row's position
    assert not rescale_after_first_tile(_bits(q), _bits(k), np.array([140]))[0]
    assert rescale_after_first_tile(_bits(q), _bits(k), np.array([150]))[0]


def test_stress_inputs_rescale_and_iid_inputs_do_not():
    S = 1200
    rows = inputs.sample_rows(1, 32, S, 24, seed=5)
    rows = rows[rows[:, 2] >= 128]                 # rows that visit more than one tile
    stress = inputs.make_stress_qkv(1, S, seed=6)
    iid = inputs.make_qkv(1, S, seed=6)
    assert rescale_fraction(stress, rows) > 0.5
    assert rescale_fraction(iid, rows) == 0.0
