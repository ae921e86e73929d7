"""Pins for the oracle's quantised matmul (CPU only).

The oracle computes y = x @ W^T with W[n, k] = s[n, k//64]*q[n, k] + b[n, k//64]
and 4-bit codes packed eight per uint32 word, lowest k in the lowest nibble
("Speculative decoding and MTP on Apple silicon", Facts: small-M 4-bit
quantized matmul; "The fastest way to run local LLMs on a Mac", "Decode is a
memory-bandwidth problem").  Each pin below is checked against something other
than the oracle's own formula: codes are unpacked here by reading hexadecimal
digits or little-endian bytes (not shifts), and the expected values are closed
forms or a library matmul.  The last test plants mistakes in the oracle and
shows that some pin catches each one.
"""
import numpy as np
import pytest

import oracle
from speculative_decoding_verify_08_gb300 import synth

BF16_ONE = 0x3F80


def bf16_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_exact(a):
    """bf16 bits of values that are exactly representable (asserted)."""
    f = np.asarray(a, dtype=np.float32)
    bits = (f.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(bf16_to_f64(bits), f.astype(np.float64))
    return bits


def unpack_hex(codes):
    """Codes [N, K] from words [N, K/8] via hexadecimal digits (tiny shapes)."""
    N, W = codes.shape
    out = np.zeros((N, W * 8), dtype=np.int64)
    for n in range(N):
        for j in range(W):
            digits = format(int(codes[n, j]), "08x")  # most significant first
            for i in range(8):
                out[n, 8 * j + i] = int(digits[7 - i], 16)
    return out


def unpack_bytes(codes):
    """Codes [N, K] via the little-endian byte view: byte i = nibbles 2i, 2i+1."""
    b = np.ascontiguousarray(codes, dtype="<u4").view(np.uint8)
    lo = (b & 0x0F).astype(np.int64)
    hi = (b >> 4).astype(np.int64)
    return np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)


def make(M, N, K, seed=0):
    t = synth.qmm_inputs(M, N, K, seed=seed)
    return (synth.bf16_bits(t["x"]), synth.u32_bits(t["codes"]),
            synth.bf16_bits(t["scales"]), synth.bf16_bits(t["biases"]))


def test_unpackers_agree():
    _, codes, _, _ = make(1, 8, 128, seed=3)
    assert np.array_equal(unpack_hex(codes), unpack_bytes(codes))
    # a hand-written word: 0x76543210 holds codes 0,1,...,7 in k order
    assert unpack_hex(np.array([[0x76543210]], dtype=np.uint32)).tolist() == [list(range(8))]


def test_integer_matmul_when_scale_one_bias_zero():
    """s = 1, b = 0: y is the exact integer product x @ Q^T."""
    rng = np.random.default_rng(1)
    M, N, K = 3, 16, 256
    xi = rng.integers(-4, 5, size=(M, K))
    x = f32_to_bf16_exact(xi)
    codes = rng.integers(0, 2 ** 32, size=(N, K // 8), dtype=np.uint64).astype(np.uint32)
    s = np.full((N, K // 64), BF16_ONE, dtype=np.uint16)
    b = np.zeros((N, K // 64), dtype=np.uint16)
    y = oracle.qmm(x, codes, s, b)
    expect = xi @ unpack_hex(codes).T
    assert np.array_equal(y, expect.astype(np.float64))


def test_one_hot_rows_return_dequantised_weights():
    """x = e_r returns column r of W: pins nibble order and group indexing."""
    M, N, K = 4, 8, 256
    _, codes, s, b = make(M, N, K, seed=2)
    Q = unpack_hex(codes)
    S, B = bf16_to_f64(s), bf16_to_f64(b)
    for r in (0, 1, 7, 8, 63, 64, 65, 130, 255):
        xr = np.zeros((1, K), dtype=np.float32)
        xr[0, r] = 1.0
        y = oracle.qmm(f32_to_bf16_exact(xr), codes, s, b)
        expect = S[:, r // 64] * Q[:, r] + B[:, r // 64]
        assert np.array_equal(y[0], expect), r


def test_constant_code_closed_form():
    """Every code = c: y[m, n] = sum_g (s[n,g]*c + b[n,g]) * sum_{k in g} x[m, k]."""
    M, N, K = 2, 4, 192
    x, _, s, b = make(M, N, K, seed=4)
    X, S, B = bf16_to_f64(x), bf16_to_f64(s), bf16_to_f64(b)
    for c in (0, 5, 15):
        codes = np.full((N, K // 8), c * 0x11111111, dtype=np.uint32)
        y = oracle.qmm(x, codes, s, b)
        xg = X.reshape(M, K // 64, 64).sum(axis=2)  # [M, G]
        expect = xg @ (S * c + B).T
        np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_matches_library_matmul_on_dequantised_weights():
    """Dequantise independently (byte view), then numpy's fp64 matmul."""
    M, N, K = 5, 48, 320
    x, codes, s, b = make(M, N, K, seed=5)
    Q = unpack_bytes(codes).astype(np.float64)
    S = np.repeat(bf16_to_f64(s), 64, axis=1)
    B = np.repeat(bf16_to_f64(b), 64, axis=1)
    W = S * Q + B
    expect = bf16_to_f64(x).reshape(M, K) @ W.T
    y = oracle.qmm(x, codes, s, b)
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-12)


def test_permutation_within_group():
    M, N, K = 2, 8, 128
    x, codes, s, b = make(M, N, K, seed=6)
    y = oracle.qmm(x, codes, s, b)
    # permuting k inside one group of both x and the codes leaves y unchanged
    Q = unpack_bytes(codes)
    perm = np.arange(K)
    perm[64:128] = perm[64:128][::-1]
    Qp = Q[:, perm]
    packed = np.zeros((N, K // 8), dtype=np.uint64)
    for i in range(8):
        packed |= Qp[:, i::8].astype(np.uint64) << np.uint64(4 * i)
    yp = oracle.qmm(x[:, perm], packed.astype(np.uint32), s, b)
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-12)


def test_ragged_and_empty_shapes():
    x, codes, s, b = make(3, 5, 64, seed=7)
    y = oracle.qmm(x, codes, s, b)
    assert y.shape == (3, 5)
    y0 = oracle.qmm(x[:0], codes, s, b)
    assert y0.shape == (0, 5)


@pytest.mark.parametrize("mut", [oracle.MUT_QMM_NIBBLE_HIGH_FIRST,
                                 oracle.MUT_QMM_GROUP_OFF_BY_ONE,
                                 oracle.MUT_QMM_DROP_BIAS])
def test_planted_mistakes_are_caught(mut):
    checks = [test_one_hot_rows_return_dequantised_weights,
              test_constant_code_closed_form,
              test_matches_library_matmul_on_dequantised_weights,
              test_integer_matmul_when_scale_one_bias_zero]
    caught = 0
    with oracle.mutant(mut):
        for chk in checks:
            try:
                chk()
            except AssertionError:
                caught += 1
    assert caught >= 1, f"mutant {mut} slipped past every qmm pin"
