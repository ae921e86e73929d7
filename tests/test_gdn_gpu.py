"""gdn_verify against the oracle (GPU).

The GatedDeltaNet verify step of a hybrid target with deferred commit: the
previous round's accepted prefix is replayed from its tape into the state,
then this round's rows run from the committed state ("Speculative decoding
and MTP on Apple silicon", Facts: GDN state cannot be trimmed; MTPLX's GDN
kernel replays an innovation tape).  Bar: outputs and committed state within
max-abs 2e-2 of their RMS (fp32 arithmetic against the oracle's fp64).
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def bits(t):
    return synth.bf16_bits(t)


def run_case(sv, M, Hk, Hv, dk, dv, n_replay, seed, out_dtype=torch.float32, M_prev=4):
    prev = synth.gdn_inputs(M_prev, Hk, Hv, dk, dv, seed=seed)
    cur = synth.gdn_inputs(M, Hk, Hv, dk, dv, seed=seed + 1)
    dev = torch.device("cuda")
    state = prev["state"].to(dev).contiguous()
    o = torch.empty((M, Hv, dv), dtype=out_dtype, device=dev)
    tape = tuple(prev[n].to(dev) for n in ("k", "v", "g", "beta")) if n_replay else None
    sv.gdn_verify(state, cur["q"].to(dev), cur["k"].to(dev), cur["v"].to(dev), cur["g"].to(dev),
                  cur["beta"].to(dev), o, tape=tape, n_replay=n_replay)
    assert sv.sv_last_device_error() == sv.SV_OK
    ro, rs = oracle.gdn(prev["state"].numpy(), bits(cur["q"]), bits(cur["k"]), bits(cur["v"]),
                        cur["g"].numpy(), cur["beta"].numpy(),
                        tape=(bits(prev["k"]), bits(prev["v"]), prev["g"].numpy(), prev["beta"].numpy()),
                        n_replay=n_replay)
    assert_close(o.float().cpu().numpy(), ro, what=f"gdn o M={M} n={n_replay}")
    assert_close(state.cpu().numpy(), rs, what=f"gdn state n={n_replay}")
    if n_replay == 0:
        assert torch.equal(state.cpu(), prev["state"])  # nothing committed: untouched


@pytest.mark.parametrize("n_replay", [0, 1, 2, 4])
@pytest.mark.parametrize("dk", [64, 128, 256])
def test_replay_then_verify(cuda_lib, dk, n_replay):
    run_case(cuda_lib, 4, 2, 6, dk, 40, n_replay, seed=dk + n_replay)


@pytest.mark.parametrize("M", [1, 2, 8, 16, 64])
def test_row_counts(cuda_lib, M):
    run_case(cuda_lib, M, 4, 8, 128, 128, 2, seed=100 + M)


@pytest.mark.parametrize("M,n_replay", [(8, 16), (4, 8), (20, 5), (3, 17), (0, 20), (13, 35)])
def test_tape_and_row_mixes(cuda_lib, M, n_replay):
    """Longer tapes than one round of drafts, more rows than the tape and the
    reverse, and a commit-only call of 20 tokens."""
    if M == 0:
        prev = synth.gdn_inputs(n_replay, 2, 4, 128, 48, seed=300 + n_replay)
        dev = torch.device("cuda")
        state = prev["state"].to(dev).contiguous()
        tape = tuple(prev[x].to(dev) for x in ("k", "v", "g", "beta"))
        cuda_lib.gdn_verify(state, None, None, None, None, None, None, tape=tape, n_replay=n_replay)
        assert cuda_lib.sv_last_device_error() == cuda_lib.SV_OK
        _, rs = oracle.gdn(prev["state"].numpy(), np.zeros((0, 2, 128), np.uint16),
                           np.zeros((0, 2, 128), np.uint16), np.zeros((0, 4, 48), np.uint16),
                           np.zeros((0, 4), np.float32), np.zeros((0, 4), np.float32),
                           tape=(bits(prev["k"]), bits(prev["v"]), prev["g"].numpy(), prev["beta"].numpy()),
                           n_replay=n_replay)
        assert_close(state.cpu().numpy(), rs, what=f"gdn commit only n={n_replay}")
        return
    run_case(cuda_lib, M, 2, 4, 128, 48, n_replay, seed=300 + M, M_prev=n_replay)


def test_longest_tape_and_ragged_rows(cuda_lib):
    """64 replayed tokens and 64 verify rows (the per-call limits) at dk 256,
    with dv = 76 (a CTA takes 8 rows of a head: the last one holds 4)."""
    run_case(cuda_lib, 64, 2, 4, 256, 76, 64, seed=201, M_prev=64)


def test_27b_class_layer(cuda_lib):
    """16 key heads, 48 value heads, 128 x 128 state per head, M = 4, two
    tokens of the previous round committed; bf16 outputs."""
    run_case(cuda_lib, 4, 16, 48, 128, 128, 2, seed=7, out_dtype=torch.bfloat16)


def test_commit_only(cuda_lib):
    """M = 0: the call only commits the tape."""
    prev = synth.gdn_inputs(4, 2, 4, 128, 64, seed=9)
    dev = torch.device("cuda")
    state = prev["state"].to(dev).contiguous()
    tape = tuple(prev[n].to(dev) for n in ("k", "v", "g", "beta"))
    cuda_lib.gdn_verify(state, None, None, None, None, None, None, tape=tape, n_replay=3)
    _, rs = oracle.gdn(prev["state"].numpy(), np.zeros((0, 2, 128), np.uint16),
                       np.zeros((0, 2, 128), np.uint16), np.zeros((0, 4, 64), np.uint16),
                       np.zeros((0, 4), np.float32), np.zeros((0, 4), np.float32),
                       tape=(bits(prev["k"]), bits(prev["v"]), prev["g"].numpy(), prev["beta"].numpy()),
                       n_replay=3)
    assert_close(state.cpu().numpy(), rs, what="gdn commit only")


def test_two_rounds_equal_one_sequential_pass(cuda_lib):
    """A first verify round (4 rows) accepts 2 drafts; the next round commits
    that round's rows 0..2 and verifies 4 new rows: the committed state equals
    running the first round's 3 tokens one call at a time."""
    Hk, Hv, dk, dv = 2, 4, 128, 64
    r1 = synth.gdn_inputs(4, Hk, Hv, dk, dv, seed=11)
    r2 = synth.gdn_inputs(4, Hk, Hv, dk, dv, seed=12)
    dev = torch.device("cuda")
    s_a = r1["state"].to(dev).contiguous()
    o = torch.empty((4, Hv, dv), dtype=torch.float32, device=dev)
    d1 = {n: r1[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    d2 = {n: r2[n].to(dev) for n in ("q", "k", "v", "g", "beta")}
    cuda_lib.gdn_verify(s_a, d1["q"], d1["k"], d1["v"], d1["g"], d1["beta"], o)
    cuda_lib.gdn_verify(s_a, d2["q"], d2["k"], d2["v"], d2["g"], d2["beta"], o,
                        tape=(d1["k"], d1["v"], d1["g"], d1["beta"]), n_replay=3)
    # the same three tokens committed one at a time
    s_b = r1["state"].to(dev).contiguous()
    for t in range(3):
        sl = lambda x: x[t:t + 1].contiguous()
        cuda_lib.gdn_verify(s_b, None, None, None, None, None, None,
                            tape=(sl(d1["k"]), sl(d1["v"]), sl(d1["g"]), sl(d1["beta"])), n_replay=1)
    torch.testing.assert_close(s_a, s_b, rtol=1e-5, atol=1e-6)
    _, rs = oracle.gdn(r1["state"].numpy(), bits(r2["q"]), bits(r2["k"]), bits(r2["v"]),
                       r2["g"].numpy(), r2["beta"].numpy(),
                       tape=(bits(r1["k"]), bits(r1["v"]), r1["g"].numpy(), r1["beta"].numpy()),
                       n_replay=3)
    assert_close(s_a.cpu().numpy(), rs, what="gdn two rounds")
