"""Pins for the oracle's 8-bit quantised matmul (CPU only).

y = x @ W^T with W[n, k] = s[n, k//64]*q[n, k] + b[n, k//64], q in 0..255
packed four per uint32 word, lowest k in the lowest byte: the 8-bit affine
pack ("Speculative decoding and MTP on Apple silicon", Facts: skinny_qmm covers
4-bit and 8-bit weights; 8-bit is the sweet spot for the speedup ratio).  The
expected values here come from unpacking by hexadecimal digit pairs (not
shifts), numpy's float64 matmul, closed forms, and the independently pinned
4-bit oracle; the last tests plant mistakes in the oracle and show that a pin
catches each one.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_08_gb300 import synth

from test_oracle_qmm import bf16_to_f64, f32_to_bf16_exact


def unpack_hex8(codes):
    """Codes [N, K] from words [N, K/4] via pairs of hexadecimal digits."""
    N, W = codes.shape
    out = np.zeros((N, W * 4), dtype=np.int64)
    for n in range(N):
        for j in range(W):
            digits = format(int(codes[n, j]), "08x")  # most significant first
            for i in range(4):
                out[n, 4 * j + i] = int(digits[6 - 2 * i: 8 - 2 * i], 16)
    return out


def make8(M, N, K, seed=0):
    t = synth.qmm_inputs(M, N, K, seed=seed, bits=8)
    return (synth.bf16_bits(t["x"]), synth.u32_bits(t["codes"]),
            synth.bf16_bits(t["scales"]), synth.bf16_bits(t["biases"]))


def reference(x, codes, s, b, group=64):
    q = unpack_hex8(codes).astype(np.float64)
    S = np.repeat(bf16_to_f64(s), group, axis=1)
    B = np.repeat(bf16_to_f64(b), group, axis=1)
    return bf16_to_f64(x) @ (S * q + B).T


def test_unpacker_reads_little_endian_bytes():
    w = np.array([[0x04030201, 0xFFEE0080]], dtype=np.uint32)
    assert unpack_hex8(w).tolist() == [[1, 2, 3, 4, 0x80, 0, 0xEE, 0xFF]]
    assert np.array_equal(unpack_hex8(w), w.view(np.uint8).reshape(1, -1))


def test_matches_float64_matmul():
    x, c, s, b = make8(3, 10, 192, seed=1)
    np.testing.assert_allclose(oracle.qmm8(x, c, s, b), reference(x, c, s, b), rtol=1e-12, atol=1e-12)


def test_codes_span_the_full_byte():
    _, c, _, _ = make8(1, 64, 512, seed=2)
    q = unpack_hex8(c)
    assert q.min() == 0 and q.max() == 255 and (q >= 128).mean() > 0.4


def test_constant_code_closed_form():
    """All codes = 200, scale 1/8, bias -3 (exact in bf16): every weight is 22,
    so y[m][n] = 22 * sum_k x[m][k]."""
    M, N, K = 2, 5, 128
    x, _, _, _ = make8(M, N, K, seed=3)
    codes = np.full((N, K // 4), 0xC8C8C8C8, dtype=np.uint32)
    s = f32_to_bf16_exact(np.full((N, K // 64), 0.125))
    b = f32_to_bf16_exact(np.full((N, K // 64), -3.0))
    y = oracle.qmm8(x, codes, s, b)
    expect = 22.0 * bf16_to_f64(x).sum(axis=1)
    np.testing.assert_allclose(y, np.repeat(expect[:, None], N, axis=1), rtol=1e-13)


def test_one_hot_row_picks_one_weight():
    """x = e_k picks W[n, k] = s*q + b exactly."""
    N, K = 4, 256
    _, c, s, b = make8(1, N, K, seed=4)
    q = unpack_hex8(c)
    for k in (0, 3, 64, 129, 255):
        x = np.zeros((1, K), dtype=np.uint16)
        x[0, k] = 0x3F80  # 1.0
        y = oracle.qmm8(x, c, s, b)[0]
        g = k // 64
        np.testing.assert_array_equal(y, bf16_to_f64(s[:, g]) * q[:, k] + bf16_to_f64(b[:, g]))


def test_small_codes_equal_the_4bit_oracle():
    """Codes below 16 mean the same weights in either pack, so the 8-bit
    oracle must agree with the separately pinned 4-bit one."""
    M, N, K = 2, 6, 128
    x, _, s, b = make8(M, N, K, seed=5)
    rng = np.random.default_rng(5)
    q = rng.integers(0, 16, size=(N, K))
    w8 = np.zeros((N, K // 4), dtype=np.uint32)
    w4 = np.zeros((N, K // 8), dtype=np.uint32)
    for k in range(K):
        w8[:, k // 4] |= (q[:, k] << (8 * (k % 4))).astype(np.uint32)
        w4[:, k // 8] |= (q[:, k] << (4 * (k % 8))).astype(np.uint32)
    np.testing.assert_array_equal(oracle.qmm8(x, w8, s, b), oracle.qmm(x, w4, s, b))


def test_byte_split_identity():
    """q = lo + 16*hi: the 8-bit product equals a 4-bit product over the low
    nibbles plus one over the high nibbles with 16*s and no bias."""
    M, N, K = 3, 4, 192
    x, c, s, b = make8(M, N, K, seed=6)
    q = unpack_hex8(c)
    lo, hi = q % 16, q // 16
    w_lo = np.zeros((N, K // 8), dtype=np.uint32)
    w_hi = np.zeros((N, K // 8), dtype=np.uint32)
    for k in range(K):
        w_lo[:, k // 8] |= (lo[:, k] << (4 * (k % 8))).astype(np.uint32)
        w_hi[:, k // 8] |= (hi[:, k] << (4 * (k % 8))).astype(np.uint32)
    s16 = f32_to_bf16_exact(bf16_to_f64(s) * 16.0)
    zero = np.zeros_like(b)
    y = oracle.qmm(x, w_lo, s, b) + oracle.qmm(x, w_hi, s16, zero)
    np.testing.assert_allclose(oracle.qmm8(x, c, s, b), y, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("mut", [oracle.MUT_QMM8_BYTE_HIGH_FIRST, oracle.MUT_QMM8_SIGNED,
                                 oracle.MUT_QMM_GROUP_OFF_BY_ONE, oracle.MUT_QMM_DROP_BIAS])
def test_planted_mistakes_are_caught(mut):
    checks = [test_matches_float64_matmul, test_one_hot_row_picks_one_weight,
              test_constant_code_closed_form]
    caught = 0
    with oracle.mutant(mut):
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
    assert caught >= 1, f"mutant {mut} slipped past every 8-bit pin"
