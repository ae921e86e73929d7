"""qmm_small_m against the oracle (GPU).

y = x @ W^T over 4-bit affine group-quantised weights ("Speculative decoding
and MTP on Apple silicon", Facts: small-M quantized matmul).  Bar: max abs
error <= 2e-2 * RMS of the oracle's output (fp32 accumulation).
"""
import numpy as np
import pytest
import torch

from gpu_helpers import SCALE_EXPS, assert_close, assert_close_per_column, qmm_gpu, qmm_ref, scaled_rows
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [
    (4, 1024, 512),     # tiny workload
    (3, 1000, 512),     # ragged N (partial last tile)
    (1, 17, 64),        # one group, two tiles
    (5, 40, 192),
    (2, 4096, 2560),    # 40 groups, 8 batches
])
def test_small_shapes(cuda_lib, M, N, K):
    t = synth.qmm_inputs(M, N, K, seed=M * 31 + N)
    assert_close(qmm_gpu(cuda_lib, t, M, N, K), qmm_ref(t), what=f"qmm {M}x{N}x{K}")


@pytest.mark.parametrize("M", [1, 2, 4, 7, 8, 9, 15, 16])
def test_row_counts(cuda_lib, M):
    N, K = 2048, 1024
    t = synth.qmm_inputs(M, N, K, seed=100 + M)
    assert_close(qmm_gpu(cuda_lib, t, M, N, K), qmm_ref(t), what=f"qmm M={M}")


def test_bf16_output(cuda_lib):
    M, N, K = 4, 1024, 512
    t = synth.qmm_inputs(M, N, K, seed=7)
    y = qmm_gpu(cuda_lib, t, M, N, K, out_dtype=torch.bfloat16)
    assert_close(y, qmm_ref(t), what="qmm bf16 out")


@pytest.mark.parametrize("name,N,K,M", [
    ("qkv", 6144, 5120, 16),
    ("o", 5120, 5120, 8),
    ("down", 5120, 17408, 8),
])
def test_projection_shapes_full(cuda_lib, name, N, K, M):
    t = synth.qmm_inputs(M, N, K, seed=11, device="cuda")
    assert_close(qmm_gpu(cuda_lib, t, M, N, K), qmm_ref(t), what=name)


@pytest.mark.parametrize("name,N,K,M", [("gate_up", 34816, 5120, M) for M in (1, 2, 3, 4, 8, 16)] +
                         [("lm_head", 152064, 5120, M) for M in (1, 4, 8, 16)])
def test_large_shapes_sampled(cuda_lib, name, N, K, M):
    """Full-size launches with at least one 128-row batch per CTA (whole
    batches per CTA, no cross-CTA merge) at every row count the benchmark
    times: the plan's stage size, activation window and the second n8 half
    (M > 8) change with M.  The oracle computes 512 sampled output columns,
    the last one included."""
    t = synth.qmm_inputs(M, N, K, seed=13 + M, device="cuda")
    y = qmm_gpu(cuda_lib, t, M, N, K)
    rows = np.sort(np.random.default_rng(0).choice(N, size=512, replace=False))
    rows[-1] = N - 1
    assert_close(y[:, rows], qmm_ref(t, rows), what=name)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 8, 9, 16])
def test_whole_batches_per_cta_full(cuda_lib, M):
    """N = 20000 (157 batches of 128 rows, more than the SMs; the last tile
    ragged): the plan gives each CTA whole batches.  Every output column is
    compared with the oracle."""
    N, K = 20000, 1024
    t = synth.qmm_inputs(M, N, K, seed=200 + M, device="cuda")
    assert_close(qmm_gpu(cuda_lib, t, M, N, K), qmm_ref(t), what=f"qmm whole batches M={M}")


@pytest.mark.parametrize("M,G", [(4, 4200), (16, 1800)])
def test_long_k_several_windows(cuda_lib, M, G):
    """Three batches of very long rows: each CTA's share of the group-blocks
    is larger than the activation window it keeps in shared memory (80
    groups at M = 4, 56 at M = 16), so it reloads the rows in two windows,
    and the windows of CTAs that cross a batch boundary wrap around the end
    of the row.  The oracle computes 64 sampled output columns."""
    N, K = 1500, 64 * G
    t = synth.qmm_inputs(M, N, K, seed=19 + M, device="cuda")
    y = qmm_gpu(cuda_lib, t, M, N, K)
    rows = np.sort(np.random.default_rng(1).choice(N, size=64, replace=False))
    rows[-1] = N - 1
    assert_close(y[:, rows], qmm_ref(t, rows), what=f"qmm long K M={M}")


def test_batch_invariance_and_determinism(cuda_lib):
    """Row r of an M-row call equals row r of any other call in the same row
    class (M <= 8, or 9 <= M <= 16) bit for bit: the split plan depends only
    on N, K and the row class.  Repeated calls agree."""
    N, K = 3072, 5120
    t = synth.qmm_inputs(16, N, K, seed=17, device="cuda")
    packed = cuda_lib.prepack(t["codes"], t["scales"], t["biases"])
    ws = cuda_lib.workspace(max(cuda_lib.qmm_workspace_bytes(16, N, K),
                                cuda_lib.qmm_workspace_bytes(8, N, K)))

    def run(M):
        tm = dict(t)
        tm["x"] = t["x"][:M].contiguous()
        return qmm_gpu(cuda_lib, tm, M, N, K, packed=packed, ws=ws)

    y8, y8b = run(8), run(8)
    assert np.array_equal(y8, y8b)
    for M in (1, 3, 4):
        assert np.array_equal(run(M), y8[:M]), M
    y16, y16b = run(16), run(16)
    assert np.array_equal(y16, y16b)
    for M in (9, 12):
        assert np.array_equal(run(M), y16[:M]), M


@pytest.mark.parametrize("cuda_cores", [False, True])
def test_scale_magnitudes_across_bf16_range(cuda_lib, cuda_cores):
    """The prepack stores each scale times a power of two (64, or 4 for the
    rows whose codes enter the MMA sixteen times larger); the scaling is exact
    over bf16's range, subnormal scales included, so every output column meets
    the tolerance against the oracle at its own magnitude.  The CUDA-core
    comparison path divides the factors back out."""
    M, N, K = 4, 1000, 512
    t = scaled_rows(synth.qmm_inputs(M, N, K, seed=29), SCALE_EXPS, seed=29)
    old = cuda_lib.sv_get_launch_flags()
    if cuda_cores:
        cuda_lib.sv_set_launch_flags(old | cuda_lib.SV_LAUNCH_QMM_CUDA_CORES)
    try:
        y = qmm_gpu(cuda_lib, t, M, N, K)
    finally:
        cuda_lib.sv_set_launch_flags(old)
    assert_close_per_column(y, qmm_ref(t), "qmm scale magnitudes")


def test_prepack_rows_beyond_n_are_zero(cuda_lib):
    """N = 20: one batch of eight 16-row tiles; rows 20..127 carry zero
    codes, scales and biases.  Group-block g holds tile j's 576 bytes at j*576."""
    N, K = 20, 128
    t = synth.qmm_inputs(1, N, K, seed=3, device="cuda")
    packed = cuda_lib.prepack(t["codes"], t["scales"], t["biases"]).cpu().numpy()
    assert packed.size == 1 * (K // 64) * 8 * 576
    blocks = packed.reshape(K // 64, 8, 576)
    assert (blocks[:, 2:, :] == 0).all()          # tiles 2..7: rows 32..127
    sb = blocks[:, 1, 512:].copy().view(np.uint16).reshape(K // 64, 8, 4)  # tile 1: rows 16..31
    assert (sb[:, 4:, :] == 0).all()  # rows 20..23 (s, b) and 28..31 (s, b)
    assert (sb[:, :4, 1] == 0).all() and (sb[:, :4, 3] == 0).all()  # rows 24..27
    assert (sb[:, :4, 0] != 0).any()  # rows 16..19 are real


@pytest.mark.parametrize("M", [1, 4])
@pytest.mark.parametrize("N,K", [(1000, 512), (6144, 5120)])
def test_cuda_core_comparison_path(cuda_lib, M, N, K):
    """The FFMA (CUDA-core) variant selected by SV_LAUNCH_QMM_CUDA_CORES, kept
    to time tensor cores against CUDA cores, meets the same tolerance."""
    t = synth.qmm_inputs(M, N, K, seed=23 + M)
    old = cuda_lib.sv_get_launch_flags()
    cuda_lib.sv_set_launch_flags(old | cuda_lib.SV_LAUNCH_QMM_CUDA_CORES)
    try:
        y = qmm_gpu(cuda_lib, t, M, N, K)
    finally:
        cuda_lib.sv_set_launch_flags(old)
    assert_close(y, qmm_ref(t), what=f"qmm cuda-core M={M} {N}x{K}")
