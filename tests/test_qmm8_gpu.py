"""qmm8_small_m against the oracle (GPU).

y = x @ W^T over 8-bit affine group-quantised weights, the 8-bit pack
("Speculative decoding and MTP on Apple silicon", Facts: skinny_qmm covers
4-bit and 8-bit weights; 8-bit is the sweet spot for the speedup ratio).  Bar:
max abs error <= 2e-2 * RMS of the oracle's output (fp32 accumulation).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import SCALE_EXPS, assert_close, assert_close_per_column, qmm_gpu, qmm_ref, scaled_rows
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def check(sv, M, N, K, seed, device="cpu", rows=None, out_dtype=torch.float32):
    t = synth.qmm_inputs(M, N, K, seed=seed, device=device, bits=8)
    y = qmm_gpu(sv, t, M, N, K, out_dtype=out_dtype, bits=8)
    if rows is None:
        assert_close(y, qmm_ref(t, bits=8), what=f"qmm8 {M}x{N}x{K}")
    else:
        assert_close(y[:, rows], qmm_ref(t, rows, bits=8), what=f"qmm8 {M}x{N}x{K} sampled")
    return t, y


@pytest.mark.parametrize("M,N,K", [
    (4, 1024, 512),
    (3, 1000, 512),     # ragged N (partial last tile)
    (1, 17, 64),        # one group, two tiles
    (5, 40, 192),
    (2, 4096, 2560),    # 40 groups, 8 batches
])
def test_small_shapes(cuda_lib, M, N, K):
    check(cuda_lib, M, N, K, seed=M * 37 + N)


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 15, 16])
def test_row_counts(cuda_lib, M):
    check(cuda_lib, M, 2048, 1024, seed=200 + M)


def test_bf16_output(cuda_lib):
    check(cuda_lib, 4, 1024, 512, seed=8, out_dtype=torch.bfloat16)


def test_extreme_codes(cuda_lib):
    """Every code 0 or 255 (the high nibble's full range): the split into
    128 + lo and 2048 + 16*hi must stay exact at both ends."""
    M, N, K = 4, 256, 512
    t = synth.qmm_inputs(M, N, K, seed=9, bits=8)
    rng = np.random.default_rng(9)
    words = np.where(rng.random((N, K // 4)) < 0.5, 0xFFFFFFFF, 0x00000000).astype(np.uint32)
    words[::3] = 0xFF00FF00
    t["codes"] = torch.from_numpy(words.view(np.int32))
    assert_close(qmm_gpu(cuda_lib, t, M, N, K, bits=8), qmm_ref(t, bits=8), what="qmm8 extreme codes")


@pytest.mark.parametrize("name,N,K,M", [
    ("qkv", 6144, 5120, 16),
    ("o", 5120, 5120, 8),
    ("down", 5120, 17408, 4),
])
def test_projection_shapes_full(cuda_lib, name, N, K, M):
    check(cuda_lib, M, N, K, seed=21, device="cuda")


@pytest.mark.parametrize("name,N,K,M", [("gate_up", 34816, 5120, M) for M in (1, 2, 4, 8, 16)] +
                         [("lm_head", 152064, 5120, 4)])
def test_large_shapes_sampled(cuda_lib, name, N, K, M):
    """Full-size launches with whole batches per CTA at every row count the
    benchmark times; the oracle computes 512 sampled columns, the last one
    included."""
    rows = np.sort(np.random.default_rng(2).choice(N, size=512, replace=False))
    rows[-1] = N - 1
    check(cuda_lib, M, N, K, seed=23 + M, device="cuda", rows=rows)


@pytest.mark.parametrize("M", [1, 4, 8, 16])
def test_whole_batches_per_cta_full(cuda_lib, M):
    """N = 20000 (157 batches, more than the SMs, last tile ragged): whole
    batches per CTA; every output column against the oracle."""
    check(cuda_lib, M, 20000, 1024, seed=210 + M, device="cuda")


def test_long_k_several_windows(cuda_lib):
    """Rows longer than one activation window (window reloads, wrap-around)."""
    N, K = 1500, 64 * 4200
    rows = np.sort(np.random.default_rng(3).choice(N, size=64, replace=False))
    rows[-1] = N - 1
    check(cuda_lib, 4, N, K, seed=29, device="cuda", rows=rows)


def test_determinism_and_row_class_invariance(cuda_lib):
    N, K = 3072, 5120
    t = synth.qmm_inputs(8, N, K, seed=31, device="cuda", bits=8)
    packed = cuda_lib.prepack(t["codes"], t["scales"], t["biases"], bits=8)
    ws = cuda_lib.workspace(cuda_lib.qmm8_workspace_bytes(8, N, K))

    def run(M):
        tm = dict(t)
        tm["x"] = t["x"][:M].contiguous()
        return qmm_gpu(cuda_lib, tm, M, N, K, packed=packed, ws=ws, bits=8)

    y8 = run(8)
    assert np.array_equal(y8, run(8))
    for M in (1, 4):
        assert np.array_equal(run(M), y8[:M]), M


def test_small_codes_match_the_4bit_path(cuda_lib):
    """Codes below 16 packed both ways: the 8-bit and 4-bit kernels compute
    the same weights and agree within the tolerance."""
    M, N, K = 4, 2048, 1024
    t8 = synth.qmm_inputs(M, N, K, seed=33, bits=8)
    rng = np.random.default_rng(33)
    q = rng.integers(0, 16, size=(N, K)).astype(np.uint32)
    w8 = np.zeros((N, K // 4), dtype=np.uint32)
    w4 = np.zeros((N, K // 8), dtype=np.uint32)
    for j in range(4):
        w8 |= q[:, j::4] << (8 * j)
    for j in range(8):
        w4 |= q[:, j::8] << (4 * j)
    t8["codes"] = torch.from_numpy(w8.view(np.int32))
    t4 = dict(t8)
    t4["codes"] = torch.from_numpy(w4.view(np.int32))
    y8 = qmm_gpu(cuda_lib, t8, M, N, K, bits=8)
    y4 = qmm_gpu(cuda_lib, t4, M, N, K, bits=4)
    assert_close(y8, qmm_ref(t4), what="qmm8 small codes")
    assert_close(y4, qmm_ref(t4), what="qmm4 small codes")


def test_scale_magnitudes_across_bf16_range(cuda_lib):
    """The 8-bit prepack stores every scale times 64 (exact over bf16's range,
    subnormal scales included): every output column meets the tolerance
    against the oracle at its own magnitude."""
    M, N, K = 4, 1000, 512
    t = scaled_rows(synth.qmm_inputs(M, N, K, seed=31, bits=8), SCALE_EXPS, seed=31)
    assert_close_per_column(qmm_gpu(cuda_lib, t, M, N, K, bits=8), qmm_ref(t, bits=8), "qmm8 scale magnitudes")
