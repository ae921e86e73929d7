"""verify_attn against the oracle (GPU).

Multi-row verify attention, causal among the M draft rows, GQA head groups
("Speculative decoding and MTP on Apple silicon", Facts: multi-row attention
verify).  Bar: max abs error <= 2e-2 * RMS of the oracle's output.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, attn_gpu, attn_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["mma_sync", "tcgen05"], autouse=True)
def attn_kernel(request, cuda_lib):
    """Every case runs on both attention kernels."""
    old = cuda_lib.sv_get_launch_flags()
    bit = {"mma_sync": cuda_lib.SV_LAUNCH_ATTN_MMA_SYNC,
           "tcgen05": cuda_lib.SV_LAUNCH_ATTN_TCGEN05}[request.param]
    cuda_lib.sv_set_launch_flags(old | bit)
    yield request.param
    cuda_lib.sv_set_launch_flags(old)


def case(sv, M, Hq, Hkv, D, L, cap=None, seed=0, device="cpu"):
    cap = L if cap is None else cap
    t = synth.attn_inputs(M, Hq, Hkv, D, L, cap=cap, seed=seed, device=device)
    scale = 1.0 / math.sqrt(D)
    got = attn_gpu(sv, t, M, Hq, Hkv, D, L, cap, scale)
    ref = attn_ref(t, L, scale)
    assert_close(got, ref, what=f"attn M={M} Hq={Hq} Hkv={Hkv} D={D} L={L}")
    return t, got


def test_tiny(cuda_lib):
    case(cuda_lib, 4, 4, 1, 128, 256)


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("D", [128, 256])
def test_rows_and_head_dims(cuda_lib, M, D):
    case(cuda_lib, M, 24, 4, D, 1000, seed=M + D)


@pytest.mark.parametrize("L", [4, 63, 64, 65, 66, 127, 129, 500])
def test_ragged_lengths(cuda_lib, L):
    """Partial last blocks, blocks fully masked for early draft rows, L = M."""
    case(cuda_lib, 4, 12, 2, 256, L, cap=L + 37, seed=L)


def test_group_sizes(cuda_lib):
    case(cuda_lib, 8, 8, 8, 128, 300, seed=1)     # MHA, G = 1
    case(cuda_lib, 3, 16, 1, 128, 700, seed=2)    # MQA, R = 48
    case(cuda_lib, 6, 32, 4, 128, 333, seed=3)    # G = 8, R = 48


@pytest.mark.parametrize("L", [8192, 32768])
@pytest.mark.parametrize("M", [1, 4, 8])
def test_long_context(cuda_lib, M, L):
    case(cuda_lib, M, 24, 4, 256, L, seed=L + M, device="cuda")


def test_128k_context(cuda_lib):
    case(cuda_lib, 8, 24, 4, 256, 131072, seed=5, device="cuda")


def test_mask_locality(cuda_lib):
    """Changing the slots only the last draft row may see leaves rows 0..M-2."""
    M, Hq, Hkv, D, L = 4, 24, 4, 256, 2000
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=9)
    scale = 1.0 / 16
    o1 = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, scale)
    t2 = dict(t)
    k2, v2 = t["k"].clone(), t["v"].clone()
    k2[:, L - 1] = 3.0
    v2[:, L - 1] = 7.0
    t2["k"], t2["v"] = k2, v2
    o2 = attn_gpu(cuda_lib, t2, M, Hq, Hkv, D, L, L, scale)
    assert np.array_equal(o1[: M - 1], o2[: M - 1])
    assert not np.array_equal(o1[M - 1], o2[M - 1])


def test_deterministic(cuda_lib):
    M, Hq, Hkv, D, L = 8, 24, 4, 256, 5000
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=4)
    a = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 0.0625)
    b = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 0.0625)
    assert np.array_equal(a, b)


# ---- draft trees: verify_attn_masked ("Speculative decoding and MTP on Apple
# silicon", Facts: tree-attention masks in ddtree-mlx, ReDrafter's dynamic
# tree attention)

@pytest.mark.parametrize("M", [2, 4, 6, 8])
@pytest.mark.parametrize("L", [300, 2049])
def test_tree_masks(cuda_lib, M, L):
    Hq, Hkv, D = 24, 4, 256
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=70 + M + L)
    mask = synth.draft_tree_masks(M, seed=M * 1000 + L)
    scale = 1.0 / 16
    got = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, scale, mask=mask)
    assert_close(got, attn_ref(t, L, scale, mask=mask), what=f"tree attn M={M} L={L}")


def test_tree_mask_32k(cuda_lib):
    M, Hq, Hkv, D, L = 8, 24, 4, 256, 32768
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=77, device="cuda")
    mask = synth.draft_tree_masks(M, seed=5)
    got = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 1.0 / 16, mask=mask)
    assert_close(got, attn_ref(t, L, 1.0 / 16, mask=mask), what="tree attn 32K")


def test_chain_mask_equals_verify_attn(cuda_lib):
    """The chain written as a mask gives verify_attn's output bit for bit."""
    M, Hq, Hkv, D, L = 5, 24, 4, 128, 700
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=78)
    chain = (2 ** np.arange(1, M + 1) - 1).astype(np.uint32)
    a = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 0.08)
    b = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 0.08, mask=chain)
    assert np.array_equal(a, b)


# ---- wider drafts: up to 16 verify rows ("Speculative decoding and MTP on
# Apple silicon", Facts: ddtree-mlx verifies trees of up to 16 drafts), i.e.
# up to 96 query rows per KV head at 6 query heads per KV head (six m16 tiles)

@pytest.mark.parametrize("M", [9, 12, 16])
@pytest.mark.parametrize("D", [128, 256])
def test_wide_drafts_chain(cuda_lib, M, D):
    case(cuda_lib, M, 24, 4, D, 1500, seed=90 + M + D)


@pytest.mark.parametrize("M,Hq,Hkv", [(16, 16, 1), (12, 32, 4), (11, 8, 1), (16, 96, 16)])
def test_wide_drafts_group_shapes(cuda_lib, M, Hq, Hkv):
    """R = M*Hq/Hkv from 88 to 256 rows: at most 96 run, more are refused."""
    R = M * (Hq // Hkv)
    if R > 96:
        t = synth.attn_inputs(M, Hq, Hkv, 128, 300, seed=1)
        dev = torch.device("cuda")
        o = torch.empty((M, Hq, 128), dtype=torch.bfloat16, device=dev)
        ws = cuda_lib.workspace(cuda_lib.verify_attn_workspace_bytes(M, Hq, Hkv, 128, 300))
        with pytest.raises(cuda_lib.SvError) as err:
            cuda_lib.verify_attn(t["q"].to(dev), t["k"].to(dev), t["v"].to(dev), o, M, Hq, Hkv,
                                 128, 300, 300, 0.1, ws)
        assert err.value.status == cuda_lib.SV_ERR_UNSUPPORTED
        return
    case(cuda_lib, M, Hq, Hkv, 128, 777, cap=800, seed=R)


@pytest.mark.parametrize("L", [16, 17, 64, 80, 4099])
def test_wide_drafts_ragged(cuda_lib, L):
    """Draft rows spanning two KV blocks, L = M, partial last blocks."""
    case(cuda_lib, 16, 24, 4, 256, L, cap=L + 5, seed=L + 16)


@pytest.mark.parametrize("M", [12, 16])
def test_wide_tree_masks(cuda_lib, M):
    Hq, Hkv, D, L = 24, 4, 256, 3000
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=95 + M)
    mask = synth.draft_tree_masks(M, seed=M)
    got = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, 1.0 / 16, mask=mask)
    assert_close(got, attn_ref(t, L, 1.0 / 16, mask=mask), what=f"tree attn M={M}")


def test_wide_drafts_32k(cuda_lib):
    M, Hq, Hkv, D, L = 16, 24, 4, 256, 32768
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=99, device="cuda")
    scale = 1.0 / 16
    got = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, scale)
    assert_close(got, attn_ref(t, L, scale), what="attn M=16 32K")
    mask = synth.draft_tree_masks(M, seed=6)
    got = attn_gpu(cuda_lib, t, M, Hq, Hkv, D, L, L, scale, mask=mask)
    assert_close(got, attn_ref(t, L, scale, mask=mask), what="tree attn M=16 32K")
