"""spec_pick_depth (host code of the library) against the oracle, on the CPU.

The depth with the most tokens per microsecond from measured cost curves
("Speculative decoding and MTP on Apple silicon", Facts: mlx-dspark and MTPLX
depth tuning).  The choice is an integer: it must match exactly; the rates
within fp64 rounding.
"""
import numpy as np
import pytest

import oracle
import speculative_decoding_verify_08_gb300 as sv


def cases():
    rng = np.random.default_rng(0)
    for _ in range(300):
        kmax = int(rng.integers(0, 16))
        accept = np.sort(rng.random(kmax))[::-1]
        if rng.random() < 0.3:
            accept = accept * rng.random()
        verify = 10.0 + np.cumsum(rng.random(kmax + 1) * rng.choice([0.2, 2.0, 8.0]))
        draft = None if rng.random() < 0.5 else np.concatenate([[0.0], np.cumsum(rng.random(kmax))])
        yield verify, accept, draft


def test_random_curves_match_the_oracle():
    n_deep = 0
    for verify, accept, draft in cases():
        k, rates = sv.spec_pick_depth(verify, accept, draft)
        rk, rrates = oracle.pick_depth(verify, accept, draft)
        assert k == rk
        np.testing.assert_allclose(rates, rrates, rtol=1e-15, atol=0)
        n_deep += k > 0
    assert n_deep > 50  # the cases exercise both outcomes


def test_ties_and_edges_match_the_oracle():
    for verify, accept in [([10.0, 15.0], [0.5]), ([7.0], []), ([10.0, 10.0, 10.0], [1.0, 1.0]),
                           ([10.0, 10.0], [0.0])]:
        v, a = np.array(verify), np.array(accept)
        assert sv.spec_pick_depth(v, a)[0] == oracle.pick_depth(v, a)[0]


@pytest.mark.parametrize("verify,accept", [([10.0, -1.0], [0.5]), ([10.0, 12.0], [1.2]),
                                           ([10.0, 12.0, 13.0], [0.3, 0.4]),
                                           ([10.0, float("nan")], [0.5])])
def test_invalid_inputs_rejected(verify, accept):
    with pytest.raises(sv.SvError):
        sv.spec_pick_depth(np.array(verify), np.array(accept))
