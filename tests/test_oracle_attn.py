"""Pins for the oracle's multi-row verify attention (CPU only).

Row i of the M verify rows is the token in cache slot L-M+i and attends to
slots 0..L-M+i; query head h reads KV head h // (Hq/Hkv)
("Speculative decoding and MTP on Apple silicon", Facts: multi-row attention
verify over the KV cache, 2-8 query rows; "The fastest way to run local LLMs
on a Mac", "Why token 1,000 is faster than token 100,000").  Expected values
come from closed forms, scipy's softmax, or invariants -- never from the
oracle's own loops.
"""
import math

import numpy as np
import pytest
from scipy.special import softmax

import oracle
from speculative_decoding_verify_08_gb300 import synth


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def to_bf16(a):
    """bf16 bits by truncation (the tests use the resulting values exactly)."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def make(M, Hq, Hkv, D, L, cap=None, seed=0):
    t = synth.attn_inputs(M, Hq, Hkv, D, L, cap=cap, seed=seed)
    return synth.bf16_bits(t["q"]), synth.bf16_bits(t["k"]), synth.bf16_bits(t["v"])


def test_single_slot_returns_v0():
    q, k, v = make(1, 4, 2, 16, 1, seed=1)
    o = oracle.attn(q, k, v, 1, 0.25)
    V = bf16_to_f64(v)
    for h in range(4):
        assert np.array_equal(o[0, h], V[h // 2, 0])


def test_zero_keys_average_visible_values():
    """K = 0 gives uniform weights: row i is the mean of V over slots 0..L-M+i."""
    M, Hq, Hkv, D, L = 4, 4, 1, 32, 11
    q, k, v = make(M, Hq, Hkv, D, L, seed=2)
    k[:] = 0
    o = oracle.attn(q, k, v, L, 1.0 / math.sqrt(D))
    V = bf16_to_f64(v)
    for i in range(M):
        expect = V[0, : L - M + i + 1].mean(axis=0)
        for h in range(Hq):
            np.testing.assert_allclose(o[i, h], expect, rtol=1e-13, atol=1e-14)


def test_two_slot_closed_form():
    """Scores 0 and a: weight of slot 1 is 1 / (1 + exp(-a))."""
    D = 8
    qf = np.zeros((1, 1, D), np.float32)
    qf[0, 0, 0] = 1.0
    kf = np.zeros((1, 2, D), np.float32)
    kf[0, 1, 0] = 1.5
    vf = np.zeros((1, 2, D), np.float32)
    vf[0, 0, :] = 2.0
    vf[0, 1, :] = -1.0
    scale = 0.5
    o = oracle.attn(to_bf16(qf), to_bf16(kf), to_bf16(vf), 2, scale)
    w1 = 1.0 / (1.0 + math.exp(-1.5 * scale))
    np.testing.assert_allclose(o[0, 0], (1 - w1) * 2.0 + w1 * (-1.0), rtol=1e-14)


def test_single_row_is_textbook_attention():
    """M = 1 (no draft mask): softmax(scale * q K^T) V with scipy's softmax."""
    Hq, Hkv, D, L = 6, 2, 64, 37
    q, k, v = make(1, Hq, Hkv, D, L, seed=3)
    scale = 1.0 / math.sqrt(D)
    o = oracle.attn(q, k, v, L, scale)
    Q, K, V = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        w = softmax(scale * (K[g] @ Q[0, h]))
        np.testing.assert_allclose(o[0, h], w @ V[g], rtol=1e-12, atol=1e-13)


def test_draft_rows_match_shorter_single_row_calls():
    """Row i of an M-row call equals a 1-row call over the first L-M+i+1 slots."""
    M, Hq, Hkv, D, L = 4, 4, 2, 32, 20
    q, k, v = make(M, Hq, Hkv, D, L, seed=4)
    o = oracle.attn(q, k, v, L, 0.2)
    Q, K, V = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    for i in range(M):
        n = L - M + i + 1
        for h in range(Hq):
            g = h // (Hq // Hkv)
            w = softmax(0.2 * (K[g, :n] @ Q[i, h]))
            np.testing.assert_allclose(o[i, h], w @ V[g, :n], rtol=1e-12, atol=1e-13)


def test_mask_locality():
    """Changing slots after L-M+i leaves row i alone and moves the last row."""
    M, Hq, Hkv, D, L = 4, 2, 1, 16, 12
    q, k, v = make(M, Hq, Hkv, D, L, seed=5)
    o = oracle.attn(q, k, v, L, 0.25)
    k2, v2 = k.copy(), v.copy()
    j = L - 2  # visible only to rows M-2 and M-1
    k2[:, j] = to_bf16(np.full(D, 3.0))
    v2[:, j] = to_bf16(np.full(D, 7.0))
    o2 = oracle.attn(q, k2, v2, L, 0.25)
    assert np.array_equal(o[: M - 2], o2[: M - 2])
    assert not np.allclose(o[M - 1], o2[M - 1])


def test_gqa_head_mapping():
    """KV head g holds V = g+1 everywhere, so head h must return h//group + 1."""
    M, Hq, Hkv, D, L = 2, 12, 4, 16, 9
    q, k, v = make(M, Hq, Hkv, D, L, seed=6)
    for g in range(Hkv):
        v[g] = to_bf16(np.full((L, D), g + 1.0))
    o = oracle.attn(q, k, v, L, 0.25)
    for h in range(Hq):
        np.testing.assert_allclose(o[:, h], h // (Hq // Hkv) + 1.0, rtol=1e-14)


def test_cache_stride_beyond_length():
    """Slots beyond kv_len in a larger cache are never read."""
    M, Hq, Hkv, D, L = 3, 4, 2, 16, 10
    q, k, v = make(M, Hq, Hkv, D, L, cap=16, seed=7)
    k[:, L:] = to_bf16(np.full(D, 50.0))
    v[:, L:] = to_bf16(np.full(D, 1e4))
    o = oracle.attn(q, k, v, L, 0.25)
    o_tight = oracle.attn(q, k[:, :L], v[:, :L], L, 0.25)
    assert np.array_equal(o, o_tight)


def test_rows_are_convex_combinations():
    M, Hq, Hkv, D, L = 4, 4, 1, 8, 30
    q, k, v = make(M, Hq, Hkv, D, L, seed=8)
    v[:] = to_bf16(np.ones((Hkv, L, D)))
    o = oracle.attn(q, k, v, L, 1.0)
    np.testing.assert_allclose(o, 1.0, rtol=1e-14)


@pytest.mark.parametrize("mut", [oracle.MUT_ATTN_NO_CAUSAL,
                                 oracle.MUT_ATTN_MASK_OFF_BY_ONE,
                                 oracle.MUT_ATTN_GQA_MODULO])
def test_planted_mistakes_are_caught(mut):
    checks = [test_zero_keys_average_visible_values,
              test_draft_rows_match_shorter_single_row_calls,
              test_mask_locality, test_gqa_head_mapping]
    caught = 0
    with oracle.mutant(mut):
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
    assert caught >= 1, f"mutant {mut} slipped past every attention pin"


# ---- draft trees ("Speculative decoding and MTP on Apple silicon", Facts:
# ddtree-mlx verifies a draft tree with tree-attention masks; ReDrafter's
# dynamic tree attention).  Row i sees every slot before L-M and draft slot
# L-M+j iff bit j of mask[i] is set.

def random_tree_masks(M, rng):
    """Each draft node sees its ancestors and itself; node 0 is the root."""
    mask = np.zeros(M, dtype=np.uint32)
    mask[0] = 1
    for i in range(1, M):
        parent = int(rng.integers(0, i))
        mask[i] = mask[parent] | np.uint32(1 << i)
    return mask


def brute_tree_attention(q, k, v, L, scale, mask):
    """Textbook softmax attention over an explicit visibility matrix (numpy
    and scipy only)."""
    M, Hq, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    qf, kf, vf = bf16_to_f64(q), bf16_to_f64(k), bf16_to_f64(v)
    out = np.zeros((M, Hq, D))
    for i in range(M):
        vis = np.ones(L, dtype=bool)
        for j in range(M):
            vis[L - M + j] = bool((int(mask[i]) >> j) & 1)
        idx = np.nonzero(vis)[0]
        for h in range(Hq):
            g = h // G
            s = scale * (kf[g, idx] @ qf[i, h])
            out[i, h] = softmax(s) @ vf[g, idx]
    return out


@pytest.mark.parametrize("M", [2, 4, 6, 8])
def test_tree_masks_match_brute_force(M):
    rng = np.random.default_rng(40 + M)
    Hq, Hkv, D, L = 6, 2, 16, 40
    q, k, v = make(M, Hq, Hkv, D, L, seed=50 + M)
    mask = random_tree_masks(M, rng)
    if M > 2:
        assert not np.array_equal(mask, (2 ** np.arange(1, M + 1) - 1).astype(np.uint32))
    o = oracle.attn(q, k, v, L, 0.3, mask=mask)
    np.testing.assert_allclose(o, brute_tree_attention(q, k, v, L, 0.3, mask), rtol=1e-10, atol=1e-12)


def test_chain_mask_is_the_causal_case():
    M, Hq, Hkv, D, L = 5, 4, 1, 8, 21
    q, k, v = make(M, Hq, Hkv, D, L, seed=61)
    chain = (2 ** np.arange(1, M + 1) - 1).astype(np.uint32)
    np.testing.assert_allclose(oracle.attn(q, k, v, L, 0.5, mask=chain), oracle.attn(q, k, v, L, 0.5),
                               rtol=0, atol=0)


def test_planted_mask_bit_order_is_caught():
    """Reading the draft bits in reverse order breaks the brute-force pin."""
    with oracle.mutant(oracle.MUT_ATTN_MASK_BIT_ORDER):
        with pytest.raises(AssertionError):
            test_tree_masks_match_brute_force(6)
