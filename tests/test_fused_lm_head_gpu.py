"""The lm_head fused with the acceptance's top-k selection (GPU).

qmm_small_m_topk writes the logits and, per CTA and row, the top-k of its
vocabulary columns; spec_accept_draft_select selects the draft rows' sets and
spec_accept_lists merges the lists for the target rows
("The fastest way to run local LLMs on a Mac", "Why native MTP doubles
decode" and "Why exact acceptance matters").  The pair must give exactly what
the unfused pair (qmm_small_m, then spec_accept on the logits) gives: the same
logits bit for bit, and the same accepted counts and tokens -- which in turn
equal the oracle's acceptance on those logits.  The logits themselves meet
the matmul tolerance against the oracle's matmul on sampled columns.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, qmm_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def lm_head(sv, N, K, M, seed, x_scale=0.25, period=None):
    """Random 4-bit weights [N, K] (rows repeating with `period` when given,
    which ties their logits) and activations [M, K]."""
    dev = torch.device("cuda")
    t = synth.qmm_inputs(M, N, K, seed=seed, device=dev)
    if period:
        idx = torch.arange(N, device=dev) % period
        for key in ("codes", "scales", "biases"):
            t[key] = t[key][idx].contiguous()
    t["x"] = (t["x"].float() * x_scale).to(torch.bfloat16)
    packed = sv.prepack(t["codes"], t["scales"], t["biases"])
    return t, packed


def run_pair(sv, t, packed, R, Kd, N, K, T, k, p, seed, fused_k=None):
    """Unfused and fused pair on the same inputs; returns logits, tokens and
    counts of both, and the draft inputs."""
    dev = torch.device("cuda")
    M = R * (Kd + 1)
    ws_q = sv.workspace(sv.qmm_workspace_bytes(M, N, K))
    y = torch.empty((M, N), dtype=torch.float32, device=dev)
    sv.qmm_small_m(t["x"], packed, y, M, N, K, ws_q)
    # draft logits: the target rows plus noise, drafts sampled from them
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    tgt = y.view(R, Kd + 1, N)
    drf = (tgt[:, :Kd] + torch.randn((R, Kd, N), generator=g, device=dev) * 0.5).contiguous()
    dtok = synth.synthetic_drafter(drf, T, k, seed=seed)
    u = torch.rand((R, Kd + 1), generator=g, device=dev)
    ws_a = sv.workspace(sv.spec_accept_workspace_bytes(R, Kd, N))
    tok = torch.full((R, Kd + 1), -7, dtype=torch.int32, device=dev)
    n = torch.full((R,), -7, dtype=torch.int32, device=dev)
    sv.spec_accept(tgt, drf, dtok, u, T, k, p, R, Kd, N, tok, n, ws_a)
    assert sv.sv_last_device_error() == sv.SV_OK
    # fused
    y2 = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    lists = torch.zeros(sv.qmm_topk_lists_bytes(M, N, K), dtype=torch.uint8, device=dev)
    ws_q2 = sv.workspace(sv.qmm_workspace_bytes(M, N, K))
    fk = k if fused_k is None else fused_k
    sv.qmm_small_m_topk(t["x"], packed, y2, M, N, K, T, fk, p, lists, ws_q2)
    ws_a2 = sv.workspace(sv.spec_accept_workspace_bytes(R, Kd, N))
    tok2 = torch.full((R, Kd + 1), -7, dtype=torch.int32, device=dev)
    n2 = torch.full((R,), -7, dtype=torch.int32, device=dev)
    sv.spec_accept_draft_select(drf, T, k, p, R, Kd, N, ws_a2)
    sv.spec_accept_lists(lists, dtok, u, T, k, p, R, Kd, N, tok2, n2, ws_a2)
    status = sv.sv_last_device_error()
    return dict(y=y.cpu().numpy(), y2=y2.cpu().numpy(), tok=tok.cpu().numpy(), n=n.cpu().numpy(),
                tok2=tok2.cpu().numpy(), n2=n2.cpu().numpy(), status=status, drf=drf, dtok=dtok, u=u)


def check(sv, N, K, R, Kd, T, k, p, seed, period=None):
    t, packed = lm_head(sv, N, K, R * (Kd + 1), seed, period=period)
    o = run_pair(sv, t, packed, R, Kd, N, K, T, k, p, seed)
    assert o["status"] == sv.SV_OK
    assert np.array_equal(o["y"], o["y2"]), "fused logits differ from qmm_small_m"
    assert np.array_equal(o["tok2"], o["tok"]) and np.array_equal(o["n2"], o["n"])
    # the oracle's acceptance on the same logits
    rtok, rn = oracle.accept(o["y"].reshape(R, Kd + 1, N), o["drf"].cpu().numpy(),
                             o["dtok"].cpu().numpy(), o["u"].cpu().numpy(),
                             float(np.float32(T)), k, float(np.float32(p)))
    assert np.array_equal(o["tok2"], rtok) and np.array_equal(o["n2"], rn)
    # the logits against the oracle's matmul on sampled columns
    cols = np.sort(np.random.default_rng(seed).choice(N, size=256, replace=False))
    cols[-1] = N - 1
    assert_close(o["y2"][:, cols], qmm_ref(t, cols), what="fused lm_head logits")
    return o


@pytest.mark.parametrize("R,Kd,T,k,p", [(1, 3, 0.6, 20, 0.95), (2, 3, 0.0, 0, 1.0),
                                        (4, 3, 0.8, 50, 0.9), (1, 7, 1.0, 5, 1.0)])
def test_vocab_152064(cuda_lib, R, Kd, T, k, p):
    """The 27B-class lm_head (5120 -> 152064): one round at top-k 20 as in
    the verify step, greedy, four rounds (16 rows), and seven drafts."""
    check(cuda_lib, 152064, 5120, R, Kd, T, k, p, seed=300 + R + Kd)


def test_top_k_beyond_cta_ranges(cuda_lib):
    """top-k 1024 is at least every CTA's column range, so the lists hold the
    whole ranges and the merge compacts them in batches."""
    check(cuda_lib, 152064, 5120, 1, 3, 1.0, 1024, 0.9, seed=310)


def test_tied_logits(cuda_lib):
    """Weight rows repeating every 37 rows: every logit value is shared by
    about 540 columns spread over all CTAs; the top-k sets keep all ties."""
    o = check(cuda_lib, 20000, 512, 2, 3, 1.0, 20, 1.0, seed=311, period=37)
    y = o["y"][0]
    assert int((y == y.max()).sum()) > 20


def test_smaller_aligned_vocab(cuda_lib):
    """N = 20000 (157 batches of 128 columns: at least one per CTA)."""
    check(cuda_lib, 20000, 1024, 2, 3, 0.7, 40, 0.8, seed=312)


def test_lists_for_a_smaller_top_k_are_refused(cuda_lib):
    """Lists made with top-k 5 cannot give top-k 20 sets: the device reports
    SV_ERR_INVALID_ARG and marks the round."""
    N, K = 152064, 5120
    t, packed = lm_head(cuda_lib, N, K, 4, seed=313)
    o = run_pair(cuda_lib, t, packed, 1, 3, N, K, 0.6, 20, 0.95, seed=313, fused_k=5)
    assert o["status"] == cuda_lib.SV_ERR_INVALID_ARG
    assert (o["n2"] == -1).all()


def test_draft_lists_from_the_drafters_lm_head(cuda_lib):
    """The MTP head's own lm_head (same weights, the drafter's hidden states)
    makes the draft rows' lists too: spec_accept_lists then merges every row
    and reads no logits at all.  Equal to spec_accept on both sets of logits
    and to the oracle."""
    sv = cuda_lib
    dev = torch.device("cuda")
    N, K, R, Kd, T, k, p = 152064, 5120, 2, 3, 0.8, 30, 0.9
    t, packed = lm_head(sv, N, K, R * (Kd + 1), seed=320)
    Mt, Md = R * (Kd + 1), R * Kd
    ws_q = sv.workspace(max(sv.qmm_workspace_bytes(Mt, N, K), sv.qmm_workspace_bytes(Md, N, K)))
    y = torch.empty((Mt, N), dtype=torch.float32, device=dev)
    tl = torch.zeros(sv.qmm_topk_lists_bytes(Mt, N, K), dtype=torch.uint8, device=dev)
    sv.qmm_small_m_topk(t["x"], packed, y, Mt, N, K, T, k, p, tl, ws_q)
    g = torch.Generator(device=dev)
    g.manual_seed(320)
    xd = (t["x"][:Md].float() + 0.1 * torch.randn((Md, K), generator=g, device=dev)).to(torch.bfloat16)
    yd = torch.empty((Md, N), dtype=torch.float32, device=dev)
    dl = torch.zeros(sv.qmm_topk_lists_bytes(Md, N, K), dtype=torch.uint8, device=dev)
    sv.qmm_small_m_topk(xd, packed, yd, Md, N, K, T, k, p, dl, ws_q)
    drf = yd.view(R, Kd, N)
    dtok = synth.synthetic_drafter(drf, T, k, seed=320)
    u = torch.rand((R, Kd + 1), generator=g, device=dev)
    ws = sv.workspace(sv.spec_accept_workspace_bytes(R, Kd, N))
    tok = torch.full((R, Kd + 1), -7, dtype=torch.int32, device=dev)
    n = torch.full((R,), -7, dtype=torch.int32, device=dev)
    sv.spec_accept_lists(tl, dtok, u, T, k, p, R, Kd, N, tok, n, ws, draft_lists=dl)
    assert sv.sv_last_device_error() == sv.SV_OK
    ws2 = sv.workspace(sv.spec_accept_workspace_bytes(R, Kd, N))
    tok2 = torch.full((R, Kd + 1), -7, dtype=torch.int32, device=dev)
    n2 = torch.full((R,), -7, dtype=torch.int32, device=dev)
    sv.spec_accept(y.view(R, Kd + 1, N), drf, dtok, u, T, k, p, R, Kd, N, tok2, n2, ws2)
    assert sv.sv_last_device_error() == sv.SV_OK
    assert np.array_equal(tok.cpu().numpy(), tok2.cpu().numpy())
    assert np.array_equal(n.cpu().numpy(), n2.cpu().numpy())
    rtok, rn = oracle.accept(y.view(R, Kd + 1, N).cpu().numpy(), drf.cpu().numpy(), dtok.cpu().numpy(),
                             u.cpu().numpy(), float(np.float32(T)), k, float(np.float32(p)))
    assert np.array_equal(tok.cpu().numpy(), rtok) and np.array_equal(n.cpu().numpy(), rn)
    assert (n.cpu().numpy() >= 1).any()
