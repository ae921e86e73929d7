"""Bounded device waits of the quantised matmul (GPU): a wait that runs out is
reported, not hung, and leaves the workspace usable.

With the test aid SV_LAUNCH_TEST_STALL_COPY the matmul's producer arms the
barrier of its first weight stage for the stage's bytes but issues no copy,
so the consumers' wait on it and the producer's wait for the consumers run
out (about 1.5 s of SM clocks each); nothing faults, traps or spins
unbounded.  The call must report SV_ERR_TIMEOUT, and the next call on the
same context and the same workspace must match the oracle: under the plans
that merge a batch's partial sums through global memory (each batch split
over a few CTAs; the even stream-K split) every CTA still makes its arrival,
so the per-batch arrival counters are left ready.  (The aid is not honoured
under the thread-block cluster plan.)
"""
import time

import pytest
import torch

from gpu_helpers import assert_close, qmm_gpu, qmm_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,M,N,K", [
    ("whole batches per CTA", 4, 20000, 1024),
    ("batches split over 3 CTAs", 4, 6144, 5120),
    ("stream-K split", 4, 5120, 17408),
])
def test_stalled_copy_times_out_and_workspace_stays_usable(cuda_lib, name, M, N, K):
    sv = cuda_lib
    dev = torch.device("cuda")
    t = synth.qmm_inputs(M, N, K, seed=41, device=dev)
    packed = sv.prepack(t["codes"], t["scales"], t["biases"])
    ws = sv.workspace(sv.qmm_workspace_bytes(M, N, K))
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    old = sv.sv_get_launch_flags()
    assert sv.sv_last_device_error() == sv.SV_OK
    try:
        sv.sv_set_launch_flags(old | sv.SV_LAUNCH_TEST_STALL_COPY)
        t0 = time.monotonic()
        sv.qmm_small_m(t["x"], packed, y, M, N, K, ws)
        status = sv.sv_last_device_error()
        elapsed = time.monotonic() - t0
    finally:
        sv.sv_set_launch_flags(old)
    assert status == sv.SV_ERR_TIMEOUT, name
    assert elapsed < 60.0
    assert sv.sv_last_device_error() == sv.SV_OK
    # the same workspace, twice: the arrival counters were left at zero
    for _ in range(2):
        got = qmm_gpu(sv, t, M, N, K, packed=packed, ws=ws)
        assert_close(got, qmm_ref(t), what=f"qmm after a timed-out call ({name})")
