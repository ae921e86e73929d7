"""Pins for the oracle's GatedDeltaNet verify step (CPU only).

Hybrid targets keep most layers as GatedDeltaNet layers with a fixed-size
recurrent state that cannot be trimmed after a rejected draft; MTPLX rolls it
back by replaying an "innovation tape" in its GDN kernel ("Speculative
decoding and MTP on Apple silicon", Facts).  The recurrence is the published
gated delta rule S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T,
o_t = S_t q_t.  Expected values here come from the rule's matrix form written
with numpy matmuls (the oracle updates row by row), closed forms and the
delta rule's recall property.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_08_gb300 import synth


def bf(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def make(M, Hk, Hv, dk, dv, seed):
    t = synth.gdn_inputs(M, Hk, Hv, dk, dv, seed=seed)
    return (t["state"].numpy().astype(np.float64), synth.bf16_bits(t["q"]), synth.bf16_bits(t["k"]),
            synth.bf16_bits(t["v"]), t["g"].numpy(), t["beta"].numpy())


def matrix_form(S0, q, k, v, g, beta):
    """Token by token with dense matrices: S <- a S (I - b k k^T) + b v k^T."""
    S = S0.copy()
    M, Hk, dk = q.shape
    Hv = S.shape[0]
    o = np.zeros((M, Hv, S.shape[1]))
    for t in range(M):
        for h in range(Hv):
            kk = bf(k[t, h // (Hv // Hk)])
            a, b = np.exp(np.float64(g[t, h])), np.float64(beta[t, h])
            S[h] = a * S[h] @ (np.eye(dk) - b * np.outer(kk, kk)) + b * np.outer(bf(v[t, h]), kk)
            o[t, h] = S[h] @ bf(q[t, h // (Hv // Hk)])
    return o, S


@pytest.mark.parametrize("dk,dv", [(16, 12), (8, 8)])
def test_matches_the_matrix_form(dk, dv):
    S0, q, k, v, g, b = make(4, 2, 6, dk, dv, seed=1)
    o, S = oracle.gdn(S0, q, k, v, g, b)
    o2, _ = matrix_form(S0, q, k, v, g, b)
    np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(S, S0)  # without a tape the state is untouched


def test_commit_replays_the_tape_then_verifies():
    """A call that commits n tokens of the previous round, then runs this
    round, equals the matrix form over those n tokens followed by this round."""
    S0, q0, k0, v0, g0, b0 = make(4, 2, 4, 16, 8, seed=2)
    _, q1, k1, v1, g1, b1 = make(3, 2, 4, 16, 8, seed=3)
    for n in (1, 2, 4):
        o, S = oracle.gdn(S0, q1, k1, v1, g1, b1, tape=(k0, v0, g0, b0), n_replay=n)
        _, Sn = matrix_form(S0, q0[:n], k0[:n], v0[:n], g0[:n], b0[:n])
        np.testing.assert_allclose(S, Sn, rtol=1e-11, atol=1e-12)
        o2, _ = matrix_form(Sn, q1, k1, v1, g1, b1)
        np.testing.assert_allclose(o, o2, rtol=1e-11, atol=1e-12)


def test_zero_write_strength_only_decays():
    """b = 0: S_t = (a_1 ... a_t) S_0, so o_t = prod(a) S_0 q_t."""
    S0, q, k, v, g, b = make(3, 1, 2, 8, 8, seed=4)
    b[:] = 0.0
    o, _ = oracle.gdn(S0, q, k, v, g, b)
    for t in range(3):
        for h in range(2):
            decay = np.exp(np.sum(g[: t + 1, h].astype(np.float64)))
            np.testing.assert_allclose(o[t, h], decay * S0[h] @ bf(q[t, 0]), rtol=1e-12, atol=1e-14)


def test_delta_rule_recalls_the_written_value():
    """a = 1, b = 1 and a unit-norm key: after the write S_t k_t = v_t, so
    reading with q_t = k_t returns v_t (within the key's bf16 norm error)."""
    M, Hk, Hv, dk, dv = 3, 1, 2, 16, 8
    S0, _, k, v, g, b = make(M, Hk, Hv, dk, dv, seed=5)
    g[:] = 0.0
    b[:] = 1.0
    o, _ = oracle.gdn(S0, k, k, v, g, b)
    for t in range(M):
        n2 = np.sum(bf(k[t, 0]) ** 2)  # |k|^2, 1 up to the bf16 rounding of the key
        assert abs(n2 - 1) < 1e-2
        for h in range(Hv):
            # S_t k = (1 - n2) S_{t-1} k + n2 v: within |1 - n2| (|v| + |S_{t-1} k|) of v,
            # and |v|, |S_{t-1} k| < 5 for these inputs
            np.testing.assert_allclose(o[t, h], bf(v[t, h]), atol=10 * abs(n2 - 1) + 1e-12)


def test_recall_is_exact_for_an_exactly_unit_key():
    """A key with one entry 1.0 (exact in bf16): the recall is exact."""
    M, Hk, Hv, dk, dv = 2, 1, 1, 8, 4
    S0, _, _, v, g, b = make(M, Hk, Hv, dk, dv, seed=6)
    k = np.zeros((M, Hk, dk), dtype=np.uint16)
    k[0, 0, 3] = 0x3F80
    k[1, 0, 5] = 0x3F80
    g[:] = 0.0
    b[:] = 1.0
    o, _ = oracle.gdn(S0, k, k, v, g, b)
    np.testing.assert_array_equal(o[:, 0], bf(v[:, 0]))


def test_value_heads_share_their_key_head():
    """Hv = 4 value heads over Hk = 2 key heads: heads 0,1 read key head 0 and
    2,3 read key head 1 (contiguous groups)."""
    S0, q, k, v, g, b = make(2, 2, 4, 8, 8, seed=7)
    S0[:] = S0[0]  # every head starts from the same state
    v[:] = v[:, :1]  # and writes the same values
    g[:] = g[:, :1]
    b[:] = b[:, :1]
    o, _ = oracle.gdn(S0, q, k, v, g, b)
    np.testing.assert_array_equal(o[:, 0], o[:, 1])
    np.testing.assert_array_equal(o[:, 2], o[:, 3])
    assert not np.allclose(o[:, 1], o[:, 2])


@pytest.mark.parametrize("mut", [oracle.MUT_GDN_NO_DECAY_IN_DELTA, oracle.MUT_GDN_OUTPUT_BEFORE,
                                 oracle.MUT_GDN_TRANSPOSED, oracle.MUT_GDN_HEAD_MODULO])
def test_planted_mistakes_are_caught(mut):
    checks = [lambda: test_matches_the_matrix_form(8, 8), test_commit_replays_the_tape_then_verifies,
              test_recall_is_exact_for_an_exactly_unit_key, test_value_heads_share_their_key_head]
    caught = 0
    with oracle.mutant(mut):
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
            except ValueError:
                pass  # the transposed mutant needs a square state; only the square check counts
    assert caught >= 1, f"mutant {mut} slipped past every GDN pin"
