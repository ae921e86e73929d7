"""Pins for the oracle's truncation and Leviathan-Chen acceptance (CPU only).

The rule: accept a draft x with probability min(1, p(x)/q(x)); on rejection
resample from (p - q)+; the emitted tokens then follow the target distribution
at any temperature ("The fastest way to run local LLMs on a Mac", section "Why
exact acceptance matters").  Draft and target are truncated identically
("Speculative decoding and MTP on Apple silicon", Facts).  Pins:

* hand-worked examples (tests/golden/accept_examples.json);
* the emission law integrated over stratified uniforms equals p (1e-4);
* chi-square of emitted tokens against p over many seeded rounds, at several
  temperatures and truncations, and a binomial test of the acceptance rate
  against sum_j min(p_j, q_j);
* negative controls: the greedy shortcut, the naive "sample both and compare"
  rule, a wrong residual, a reused uniform and one-sided truncation must each
  fail one of these pins (planted in the oracle through its mutant switch).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_examples.json")
with open(GOLDEN) as f:
    EX = json.load(f)


def logw(w):
    """Logits whose softmax is w / sum(w) (zero weight -> -inf)."""
    w = np.asarray(w, dtype=np.float64)
    with np.errstate(divide="ignore"):
        return np.log(w).astype(np.float32)


# ---------------------------------------------------------------- golden ---

@pytest.mark.parametrize("case", EX["dist"], ids=lambda c: c["name"])
def test_dist_worked_examples(case):
    p = oracle.dist(logw(case["w"]), case["T"], case["top_k"], case["top_p"])
    np.testing.assert_allclose(p, case["p"], rtol=2e-6, atol=1e-9)


@pytest.mark.parametrize("case", EX["dist_logits"], ids=lambda c: c["name"])
def test_dist_worked_examples_on_logits(case):
    p = oracle.dist(np.asarray(case["z"], np.float32), case["T"], case["top_k"], case["top_p"])
    expect = np.asarray(case.get("p", case.get("p_weights")), dtype=np.float64)
    expect = expect / expect.sum()
    np.testing.assert_allclose(p, expect, rtol=1e-12, atol=1e-15)


def _run_chain(case, logits_given):
    if logits_given:
        zt = np.asarray(case["target_z"], np.float32)
        zd = np.asarray(case["draft_z"], np.float32)
    else:
        zt = np.stack([logw(w) for w in case["target_w"]])
        zd = np.stack([logw(w) for w in case["draft_w"]])
    tok, n = oracle.accept(zt[None], zd[None], np.asarray([case["drafts"]], np.int32),
                           np.asarray([case["u"]], np.float32), case["T"],
                           case["top_k"], case["top_p"])
    return tok[0].tolist(), int(n[0])


@pytest.mark.parametrize("case", EX["chains"], ids=lambda c: c["name"])
def test_chain_worked_examples(case):
    assert _run_chain(case, False) == (case["tokens"], case["n"])


@pytest.mark.parametrize("case", EX["chains_logits"], ids=lambda c: c["name"])
def test_chain_worked_examples_on_logits(case):
    assert _run_chain(case, True) == (case["tokens"], case["n"])


def test_topp_boundary_is_strict():
    """A token whose mass above equals top_p exactly is dropped.

    z = [0, 0, -3, -3]: the two heads carry mass 2/(2 + 2e^-3); top_p is set
    to that very double (same libm exp, same summation order), so the tails sit
    exactly on the boundary and must go.
    """
    z = np.array([0, 0, -3, -3], np.float32)
    e3 = math.exp(-3.0)
    Z = ((1.0 + 1.0) + e3) + e3
    p0 = 1.0 / Z
    top_p = p0 + p0
    p = oracle.dist(z, 1.0, 0, top_p)
    np.testing.assert_allclose(p, [0.5, 0.5, 0, 0], rtol=1e-15)


# ---------------------------------------------------- stratified law -------

SETTINGS = [(1.0, 0, 1.0), (0.6, 0, 1.0), (0.6, 3, 1.0), (1.5, 0, 0.8), (0.3, 4, 0.9)]


def _pair(V, seed, draft_sigma=0.8):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, size=V).astype(np.float32)
    zd = (zt + rng.normal(0, draft_sigma, size=V)).astype(np.float32)
    return zt, zd


@pytest.mark.parametrize("T,k,tp", SETTINGS)
def test_emission_law_by_stratified_integration(T, k, tp):
    """P(emit j) = sum_t q(t) [A(t) 1{j=t} + (1 - A(t)) R_t(j)] equals p(j).

    A(t): share of a midpoint grid of u_0 that accepts draft t.  R_t: law of the
    resampled token over a midpoint grid of u_K, with u_0 pushed to the top of
    [0,1) so the draft is rejected.  Both come from running the oracle.
    """
    V, n = 6, 20000
    zt, zd = _pair(V, seed=11)
    p = oracle.dist(zt, T, k, tp)
    q = oracle.dist(zd, T, k, tp)
    grid = ((np.arange(n) + 0.5) / n).astype(np.float32)
    law = np.zeros(V)
    ztr = np.broadcast_to(np.stack([zt, zt])[None], (n, 2, V))
    zdr = np.broadcast_to(zd[None, None], (n, 1, V))
    for t in range(V):
        if q[t] == 0:
            continue
        dt = np.full((n, 1), t, np.int32)
        u = np.stack([grid, np.full(n, 0.5, np.float32)], axis=1)
        _, nacc = oracle.accept(ztr, zdr, dt, u, T, k, tp)
        A = nacc.mean()
        law[t] += q[t] * A
        if A < 1.0:
            u = np.stack([np.full(n, np.nextafter(np.float32(1), np.float32(0))), grid], axis=1)
            tok, nacc = oracle.accept(ztr, zdr, dt, u, T, k, tp)
            assert nacc.max() == 0
            R = np.bincount(tok[:, 0], minlength=V) / n
            law += q[t] * (1.0 - A) * R
    np.testing.assert_allclose(law, p, atol=1e-4)
    # the acceptance probability itself is min(1, p/q)
    # (checked through the integrated law above; spot-check one token)
    t = int(np.argmax(q))
    dt = np.full((n, 1), t, np.int32)
    u = np.stack([grid, np.full(n, 0.5, np.float32)], axis=1)
    _, nacc = oracle.accept(ztr, zdr, dt, u, T, k, tp)
    assert abs(nacc.mean() - min(1.0, p[t] / q[t])) <= 1.0 / n + 1e-12


# ------------------------------------------------------------ chi-square ---

def _rounds(V, K, T, k, tp, R, seed, sigma=0.7, draft_side=None):
    """R rounds sharing fixed logits; drafts sampled from q (or draft_side)."""
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    zd = (zt[:K] + rng.normal(0, sigma, size=(K, V))).astype(np.float32)
    dk, dp = (k, tp) if draft_side is None else draft_side
    qs = [oracle.dist(zd[i], T, dk, dp) for i in range(K)]
    drafts = np.stack([rng.choice(V, size=R, p=qs[i] / qs[i].sum()) for i in range(K)], axis=1)
    u = rng.random((R, K + 1), dtype=np.float32)
    zt_r = np.broadcast_to(zt[None], (R, K + 1, V))
    zd_r = np.broadcast_to(zd[None], (R, K, V))
    tok, n = oracle.accept(zt_r, zd_r, drafts.astype(np.int32), u, T, k, tp)
    ps = [oracle.dist(zt[i], T, k, tp) for i in range(K + 1)]
    qs_same = [oracle.dist(zd[i], T, k, tp) for i in range(K)]
    return tok, n, ps, qs_same


def _chi2_pvalue(samples, p):
    V = len(p)
    obs = np.bincount(samples, minlength=V).astype(np.float64)
    support = p > 0
    if obs[~support].sum() > 0:
        return 0.0
    exp = p[support] / p[support].sum() * obs.sum()
    if support.sum() == 1:
        return 1.0
    return stats.chisquare(obs[support], exp).pvalue


GRID = [(T, k, tp) for T in (0.3, 0.6, 1.0, 1.5)
        for (k, tp) in ((0, 1.0), (5, 1.0), (0, 0.9), (5, 0.9))]


@pytest.mark.parametrize("T,k,tp", GRID)
def test_emitted_tokens_follow_target(T, k, tp):
    V, K, R = 16, 3, 100_000
    tok, n, ps, qs = _rounds(V, K, T, k, tp, R, seed=int(T * 100) + 7 * k + int(tp * 10))
    # first emitted token ~ p_0
    assert _chi2_pvalue(tok[:, 0], ps[0]) > 1e-6
    # second token, given the first draft was accepted, ~ p_1
    sel = n >= 1
    assert _chi2_pvalue(tok[sel, 1], ps[1]) > 1e-6
    # bonus token after all K accepted ~ p_K
    sel = n == K
    if sel.sum() > 200:
        assert _chi2_pvalue(tok[sel, K], ps[K]) > 1e-6
    # acceptance rate at depth 0 ~ Binomial(R, sum min(p0, q0))
    alpha = float(np.minimum(ps[0], qs[0]).sum())
    acc0 = int((n >= 1).sum())
    assert stats.binomtest(acc0, R, alpha).pvalue > 1e-6
    # structural: tokens after the last emitted one are -1
    for r in range(0, R, 997):
        assert (tok[r, n[r] + 1:] == -1).all() and (tok[r, : n[r] + 1] >= 0).all()


def test_temperature_zero_is_greedy_with_correction():
    V, K, R = 16, 3, 2000
    tok, n, ps, qs = _rounds(V, K, 0.0, 0, 1.0, R, seed=5)
    am = [int(np.argmax(p)) for p in ps]
    assert (tok[:, 0] == am[0]).all()
    # depth-0 acceptance is all-or-nothing: the draft is q's argmax
    assert len(set((n >= 1).tolist())) == 1


def test_expected_accepted_length_closed_form():
    """E[n] = sum_{i=1..K} prod_{j<i} alpha_j with alpha_j = sum min(p_j, q_j)."""
    V, K, R = 16, 3, 100_000
    tok, n, ps, qs = _rounds(V, K, 1.0, 0, 1.0, R, seed=21)
    alpha = [float(np.minimum(ps[i], qs[i]).sum()) for i in range(K)]
    expect = sum(np.prod(alpha[:i + 1]) for i in range(K))
    se = n.std() / math.sqrt(R)
    assert abs(n.mean() - expect) < 6 * se


# ------------------------------------------------------ negative controls ---

def _law_ok(T=1.0, k=0, tp=1.0, seed=3, R=100_000, draft_side=None):
    V, K = 16, 3
    tok, n, ps, qs = _rounds(V, K, T, k, tp, R, seed=seed, draft_side=draft_side)
    law = _chi2_pvalue(tok[:, 0], ps[0]) > 1e-6
    alpha = float(np.minimum(ps[0], qs[0]).sum())
    rate = stats.binomtest(int((n >= 1).sum()), R, alpha).pvalue > 1e-6
    return law, rate, float((n >= 1).mean()), alpha


def test_reference_passes_both():
    law, rate, _, _ = _law_ok()
    assert law and rate


def test_greedy_shortcut_changes_the_law():
    with oracle.mutant(oracle.MUT_ACC_GREEDY):
        law, rate, _, _ = _law_ok()
    assert not law


def test_naive_sample_and_compare_collapses_acceptance():
    with oracle.mutant(oracle.MUT_ACC_NAIVE):
        law, rate, measured, alpha = _law_ok()
    assert law            # its emitted token is a target sample ...
    assert not rate       # ... but acceptance falls to sum p*q < sum min(p, q)
    assert measured < alpha


def test_wrong_residual_sign_fails():
    with oracle.mutant(oracle.MUT_ACC_RESIDUAL_SIGN):
        law, _, _, _ = _law_ok()
    assert not law


def test_reused_uniform_fails():
    with oracle.mutant(oracle.MUT_ACC_REUSE_UNIFORM):
        law, _, _, _ = _law_ok()
    assert not law


def test_one_sided_truncation_fails():
    with oracle.mutant(oracle.MUT_ACC_NO_DRAFT_TRUNC):
        law, rate, _, _ = _law_ok(T=1.0, k=5, tp=0.9)
    assert not (law and rate)


def test_mismatched_truncation_lowers_acceptance():
    """Drafts drawn without truncation, verified against truncated p: lower rate."""
    same = _law_ok(T=1.0, k=4, tp=1.0, seed=9)[2]
    with oracle.mutant(oracle.MUT_ACC_NO_DRAFT_TRUNC):
        mixed = _law_ok(T=1.0, k=4, tp=1.0, seed=9, draft_side=(0, 1.0))[2]
    assert mixed < same - 0.02


def test_topp_inclusive_mutant_caught():
    with oracle.mutant(oracle.MUT_ACC_TOPP_INCLUSIVE):
        with pytest.raises(AssertionError):
            test_topp_boundary_is_strict()


def test_rejects_bad_parameters():
    z = np.zeros((1, 2, 4), np.float32)
    d = np.zeros((1, 1, 4), np.float32)
    for T, k, tp in ((-1.0, 0, 1.0), (1.0, -1, 1.0), (1.0, 0, 0.0), (1.0, 0, 1.5)):
        with pytest.raises(ValueError):
            oracle.accept(z, d, np.zeros((1, 1), np.int32), np.zeros((1, 2), np.float32), T, k, tp)
