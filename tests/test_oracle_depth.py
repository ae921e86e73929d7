"""Pins for the oracle's draft-depth choice (CPU only).

"Speculative decoding and MTP on Apple silicon", Facts: mlx-dspark picks the
draft cap from measured verify and drafter cost curves; MTPLX keeps a depth
only if it beats plain decoding; OptiQ reports K=1..4 speedups of 1.36x,
1.34x, 0.94x and 0.74x on Qwen3.6-27B and ships depth 1.  Expected values
come from those reported outcomes, the geometric-series closed form and
invariants.
"""
import math

import numpy as np
import pytest

import oracle


def test_optiq_reported_speedups_pick_depth_one():
    """Costs built so that rate(K)/rate(0) are the reported 1.36, 1.34, 0.94,
    0.74: depth 1 wins, as OptiQ concluded."""
    accept = np.array([0.8, 0.6, 0.3, 0.1])
    tokens = 1 + np.concatenate([[0.0], np.cumsum(accept)])
    speedup = np.array([1.0, 1.36, 1.34, 0.94, 0.74])
    verify = tokens / speedup * 10.0  # plain decode step = 10 us
    k, rates = oracle.pick_depth(verify, accept)
    assert k == 1
    np.testing.assert_allclose(rates / rates[0], speedup, rtol=1e-12)


def test_only_losing_depths_keep_plain_decode():
    accept = np.array([0.5, 0.2])
    verify = np.array([10.0, 16.0, 25.0])  # 1.5/16 and 1.7/25 per us, both below 1/10
    k, _ = oracle.pick_depth(verify, accept)
    assert k == 0


def test_geometric_acceptance_closed_form():
    """i.i.d. acceptance a per draft: at least i accepted with probability
    a^i, so a round yields (1 - a^(K+1)) / (1 - a) tokens; with a flat verify
    cost the deepest depth wins."""
    a, Kmax = 0.7, 6
    accept = a ** np.arange(1, Kmax + 1)
    k, rates = oracle.pick_depth(np.full(Kmax + 1, 5.0), accept)
    assert k == Kmax
    for K in range(Kmax + 1):
        assert math.isclose(rates[K] * 5.0, (1 - a ** (K + 1)) / (1 - a), rel_tol=1e-12)


def test_linear_cost_optimum_by_enumeration_of_closed_forms():
    """Cost t0 (1 + c K) with geometric acceptance: the chosen depth maximises
    the closed-form yield over cost."""
    a, c, Kmax = 0.8, 0.15, 10
    accept = a ** np.arange(1, Kmax + 1)
    verify = 20.0 * (1 + c * np.arange(Kmax + 1))
    k, _ = oracle.pick_depth(verify, accept)
    closed = [(1 - a ** (K + 1)) / (1 - a) / (1 + c * K) for K in range(Kmax + 1)]
    assert k == int(np.argmax(closed)) and 0 < k < Kmax


def test_draft_cost_counts():
    """The same verify curve with an expensive drafter picks a shallower depth."""
    accept = np.array([0.9, 0.8, 0.7, 0.6])
    verify = np.array([10.0, 10.5, 11.0, 11.5, 12.0])
    k0, _ = oracle.pick_depth(verify, accept)
    k1, _ = oracle.pick_depth(verify, accept, draft_us=np.array([0.0, 4.0, 8.0, 12.0, 16.0]))
    assert k0 == 4 and k1 < k0


def test_ties_go_to_the_shallower_depth():
    accept = np.array([0.5])
    verify = np.array([10.0, 15.0])  # 1.5 / 15 == 1 / 10
    k, rates = oracle.pick_depth(verify, accept)
    assert rates[0] == rates[1] and k == 0


@pytest.mark.parametrize("bad", [
    dict(verify=[10.0, 0.0], accept=[0.5]),
    dict(verify=[10.0, 12.0], accept=[1.5]),
    dict(verify=[10.0, 12.0, 13.0], accept=[0.4, 0.6]),   # increasing
    dict(verify=[10.0, float("inf")], accept=[0.5]),
])
def test_invalid_inputs_rejected(bad):
    with pytest.raises(ValueError):
        oracle.pick_depth(np.array(bad["verify"]), np.array(bad["accept"]))


@pytest.mark.parametrize("mut", [oracle.MUT_DEPTH_NO_BONUS, oracle.MUT_DEPTH_CONDITIONAL,
                                 oracle.MUT_DEPTH_TIES_DEEPER])
def test_planted_mistakes_are_caught(mut):
    checks = [test_optiq_reported_speedups_pick_depth_one, test_geometric_acceptance_closed_form,
              test_ties_go_to_the_shallower_depth, test_only_losing_depths_keep_plain_decode]
    caught = 0
    with oracle.mutant(mut):
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
    assert caught >= 1, f"mutant {mut} slipped past every depth pin"
