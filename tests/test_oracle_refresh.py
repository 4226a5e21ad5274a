"""Pins of the oracle's query-similarity refresh trigger ("RefreshKV: Updating
Small KV Cache During Long-form Generation", dynamic scheduling): closed-form
cosines on bf16-exact inputs, the zero-reference rule and the reference update."""
import math

import numpy as np
import torch


def _bits(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_identical_and_orthogonal(ref):
    d, Hq = 8, 4
    q = np.zeros((2, Hq, d), np.float32)
    q[0, :, 0] = 2.0                       # mean = 2 e0
    q[1, :, 1] = 3.0                       # mean = 3 e1
    q_ref = np.zeros((2, d))
    q_ref[0, 0] = 5.0                      # same direction as row 0
    q_ref[1, 0] = 1.0                      # orthogonal to row 1
    flag, sim, new = ref.refresh_decision(_bits(q), q_ref, 0.5)
    assert sim[0] == 1.0 and sim[1] == 0.0
    assert flag.tolist() == [0, 1]
    assert new[0, 0] == 5.0                # kept: no refresh
    assert new[1].tolist() == [0, 3, 0, 0, 0, 0, 0, 0]  # replaced by the current mean


def test_mean_over_heads_closed_form(ref):
    d, Hq = 4, 6
    q = np.zeros((1, Hq, d), np.float32)
    q[0, :3, 0] = 1.0
    q[0, 3:, 1] = 1.0                      # mean = (e0 + e1) / 2
    _, sim, _ = ref.refresh_decision(_bits(q), np.array([[1.0, 0, 0, 0]]), 0.0)
    assert abs(sim[0] - 1 / math.sqrt(2)) < 1e-15


def test_zero_reference_and_zero_query_refresh(ref):
    d, Hq = 4, 2
    q = np.ones((2, Hq, d), np.float32)
    q[1] = 0.0
    flag, sim, new = ref.refresh_decision(_bits(q), np.array([[0.0] * 4, [1.0] * 4]), -1.0)
    assert flag.tolist() == [1, 1] and sim.tolist() == [-2.0, -2.0]
    assert new[0].tolist() == [1.0] * 4 and new[1].tolist() == [0.0] * 4


def test_scale_invariance_and_strict_threshold(ref):
    d, Hq = 4, 1
    q = np.array([[[1.0, 1.0, 0.0, 0.0]]], np.float32)   # cos with e0 = 1/sqrt(2)
    for scale in (1e-3, 1.0, 7.5):
        _, sim, _ = ref.refresh_decision(_bits(q), np.array([[scale, 0, 0, 0]]), 0.0)
        assert abs(sim[0] - 1 / math.sqrt(2)) < 1e-15
    # equal to the threshold: no refresh (strictly below refreshes)
    q2 = np.array([[[1.0, 0.0, 0.0, 0.0]]], np.float32)
    flag, sim, _ = ref.refresh_decision(_bits(q2), np.array([[4.0, 0, 0, 0]]), 1.0)
    assert sim[0] == 1.0 and flag[0] == 0
