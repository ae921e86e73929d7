"""verify_attn_noalloc: the allocation-free variant of verify_attn.

Some callers cannot allocate device memory when they run the attention (a
plugin inside another engine's enqueue, code inside a stream capture, a
service with a fixed device-memory budget).  For them the library keeps the
split-KV partials in a fixed 16 MiB device array.  This test calls that entry
point through the C ABI and checks that, on two calls in a row with
different inputs, it returns what verify_attn returns (within the attention
parity tolerance).  It sits in a file of its own that pytest collects last.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, assert_close
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def _both(sv, M, Hq, Hkv, D, L, cap, seed):
    dev = torch.device("cuda")
    t = synth.attn_inputs(M, Hq, Hkv, D, L, cap=cap, seed=seed, device=dev)
    scale = 1.0 / math.sqrt(D)
    o_ws = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = sv.workspace(sv.verify_attn_workspace_bytes(M, Hq, Hkv, D, L))
    sv.verify_attn(t["q"], t["k"], t["v"], o_ws, M, Hq, Hkv, D, L, cap, scale, ws)
    o_na = torch.full((M, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    sv.verify_attn_noalloc(t["q"], t["k"], t["v"], o_na, M, Hq, Hkv, D, L, cap, scale)
    assert sv.sv_last_device_error() == sv.SV_OK
    return o_na.float().cpu().numpy(), o_ws.float().cpu().numpy()


def test_noalloc_matches_workspace_variant_twice(cuda_lib):
    # two calls in a row, different inputs and shapes, sharing the fixed array
    got, ref = _both(cuda_lib, 4, 24, 4, 256, 32768, 32768, seed=21)
    assert_close(got, ref, tol=TOL, what="noalloc call 1")
    got, ref = _both(cuda_lib, 8, 24, 4, 256, 5000, 5100, seed=22)
    assert_close(got, ref, tol=TOL, what="noalloc call 2")


def test_noalloc_rejects_oversized_scratch(cuda_lib):
    """Short context over very many KV heads needs more partials than the
    fixed array holds: rejected with SV_ERR_WORKSPACE, nothing launched."""
    dev = torch.device("cuda")
    M, Hkv, G, D, L = 3, 1024, 16, 256, 64
    Hq = Hkv * G
    assert cuda_lib.verify_attn_workspace_bytes(M, Hq, Hkv, D, L) > (16 << 20)
    q = torch.zeros((M, Hq, D), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((Hkv, L, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    o = torch.zeros_like(q)
    with pytest.raises(cuda_lib.SvError) as ei:
        cuda_lib.verify_attn_noalloc(q, k, v, o, M, Hq, Hkv, D, L, L, 0.0625)
    assert ei.value.status == cuda_lib.SV_ERR_WORKSPACE
