"""verify_attn_noalloc: the allocation-free variant of verify_attn.

Some callers cannot allocate device memory when they run the attention (a
plugin inside another engine's enqueue, code inside a stream capture, a
service with a fixed device-memory budget).  For them the library keeps the
split-KV partials in a fixed 16 MiB device array.  This test calls that entry
point through the C ABI on two calls in a row with different inputs and
shapes, and checks each output against the CPU oracle and against
verify_attn with a caller's workspace (within the attention parity
tolerance; the two share one implementation, so they agree bit for bit).  It
sits in a file of its own that pytest collects last.
"""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, assert_close, attn_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def _run(sv, M, Hq, Hkv, D, L, cap, seed):
    dev = torch.device("cuda")
    t = synth.attn_inputs(M, Hq, Hkv, D, L, cap=cap, seed=seed, device=dev)
    scale = 1.0 / math.sqrt(D)
    o_ws = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = sv.workspace(sv.verify_attn_workspace_bytes(M, Hq, Hkv, D, L))
    sv.verify_attn(t["q"], t["k"], t["v"], o_ws, M, Hq, Hkv, D, L, cap, scale, ws)
    o_na = torch.full((M, Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    sv.verify_attn_noalloc(t["q"], t["k"], t["v"], o_na, M, Hq, Hkv, D, L, cap, scale)
    assert sv.sv_last_device_error() == sv.SV_OK
    return t, scale, o_na.float().cpu().numpy(), o_ws.float().cpu().numpy()


def test_noalloc_matches_oracle_and_workspace_variant_twice(cuda_lib):
    # two calls in a row, different inputs and shapes, sharing the fixed array:
    # M = 4 (two 16-row tiles per KV head) and M = 8 (three tiles, the largest
    # that fits the array at 24/4 heads, D = 256) on a ragged, strided cache
    for (M, L, cap, seed) in ((4, 32768, 32768, 21), (8, 5000, 5100, 22)):
        t, scale, got, ws_out = _run(cuda_lib, M, 24, 4, 256, L, cap, seed)
        assert_close(got, attn_ref(t, L, scale), tol=TOL, what=f"noalloc M={M} vs oracle")
        assert_close(got, ws_out, tol=TOL, what=f"noalloc M={M} vs verify_attn")
        assert np.array_equal(got, ws_out)


def test_noalloc_rejects_oversized_scratch(cuda_lib):
    """Nine drafts at 24/4 heads and D = 256 need four 16-row tiles of
    partials per KV head, more than the fixed array holds: rejected with
    SV_ERR_WORKSPACE, nothing launched (the output keeps its contents)."""
    dev = torch.device("cuda")
    M, Hq, Hkv, D, L = 9, 24, 4, 256, 8192
    assert cuda_lib.verify_attn_workspace_bytes(M, Hq, Hkv, D, L) > (16 << 20)
    assert cuda_lib.verify_attn_workspace_bytes(8, Hq, Hkv, D, L) <= (16 << 20)
    q = torch.zeros((M, Hq, D), dtype=torch.bfloat16, device=dev)
    k = torch.zeros((Hkv, L, D), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    o = torch.full_like(q, 3.0)
    with pytest.raises(cuda_lib.SvError) as ei:
        cuda_lib.verify_attn_noalloc(q, k, v, o, M, Hq, Hkv, D, L, L, 0.0625)
    assert ei.value.status == cuda_lib.SV_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((o == 3.0).all())
