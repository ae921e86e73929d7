"""Bounded device waits (GPU): a wait that runs out is reported, not hung.

Every device wait of the library gives up after about 1.5 s of SM clocks,
records SV_ERR_TIMEOUT in the device error word and lets the kernel finish.
Here the test aid SV_LAUNCH_TEST_STALL_COPY makes the mma.sync attention
kernel arm its first KV copy without issuing it, so its consumers' and
producer's waits run out; nothing faults, traps or spins unbounded.  The call
must report the timeout, and the next call on the same context must be correct.
"""
import math
import time

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, attn_gpu, attn_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def test_stalled_copy_times_out_and_context_stays_usable(cuda_lib):
    sv = cuda_lib
    M, Hq, Hkv, D, L = 1, 24, 4, 256, 1024
    t = synth.attn_inputs(M, Hq, Hkv, D, L, seed=3)
    dev = torch.device("cuda")
    q, k, v = t["q"].to(dev), t["k"].to(dev), t["v"].to(dev)
    o = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = sv.workspace(sv.verify_attn_workspace_bytes(M, Hq, Hkv, D, L))
    old = sv.sv_get_launch_flags()
    assert sv.sv_last_device_error() == sv.SV_OK
    try:
        sv.sv_set_launch_flags(sv.SV_LAUNCH_ATTN_MMA_SYNC | sv.SV_LAUNCH_TEST_STALL_COPY)
        t0 = time.monotonic()
        sv.verify_attn(q, k, v, o, M, Hq, Hkv, D, L, L, 1.0 / math.sqrt(D), ws)
        status = sv.sv_last_device_error()
        elapsed = time.monotonic() - t0
    finally:
        sv.sv_set_launch_flags(old)
    assert status == sv.SV_ERR_TIMEOUT
    assert elapsed < 60.0
    # the error word was cleared by the read, and the context is usable
    assert sv.sv_last_device_error() == sv.SV_OK
    scale = 1.0 / math.sqrt(D)
    got = attn_gpu(sv, t, M, Hq, Hkv, D, L, L, scale)
    assert_close(got, attn_ref(t, L, scale), what="attention after a timed-out call")
