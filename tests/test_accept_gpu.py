"""spec_accept against the oracle (GPU): accepted counts and emitted tokens
must match bit for bit on the same logits and uniforms ("The fastest way to
run local LLMs on a Mac", "Why exact acceptance matters"; "Speculative
decoding and MTP on Apple silicon", Facts: identical truncation)."""
import numpy as np
import pytest
import torch

from gpu_helpers import accept_gpu, accept_ref
from speculative_decoding_verify_08_gb300 import synth

pytestmark = pytest.mark.gpu


def accept_margins(a, T, k, p, rounds, dtype=torch.float32):
    """Smallest relative margins of the oracle's decisions in `rounds`: the
    ratio tests |u_i q(x) - p(x)| / p(x) up to the round's first rejection.
    A parity failure whose margin is within rounding (below ~1e-12) is a
    near-tie of the kind the pages warn about, not a logic error."""
    import oracle
    zt = a["target"].to(dtype).float().cpu().numpy()
    zd = a["draft"].to(dtype).float().cpu().numpy()
    u = a["uniforms"].cpu().numpy()
    d = a["draft_tokens"].cpu().numpy()
    Tf, pf = float(np.float32(T)), float(np.float32(p))
    out = []
    for r in rounds:
        m = np.inf
        for i in range(d.shape[1]):
            pp = oracle.dist(zt[r, i], Tf, k, pf)
            qq = oracle.dist(zd[r, i], Tf, k, pf)
            x = int(d[r, i])
            px = pp[x] if 0 <= x < pp.size else 0.0
            qx = qq[x] if 0 <= x < qq.size else 0.0
            if px > 0:
                m = min(m, abs(float(u[r, i]) * qx - px) / px)
            if not float(u[r, i]) * qx < px:
                break
        out.append(m)
    return out


def check(sv, a, T, k, p, dtype=torch.float32, ws=None):
    tok, n, status = accept_gpu(sv, a, T, k, p, dtype, ws=ws)
    assert status == sv.SV_OK
    rtok, rn = accept_ref(a, T, k, p, dtype)
    bad = np.nonzero((tok != rtok).any(axis=1) | (n != rn))[0]
    if bad.size:
        margins = accept_margins(a, T, k, p, bad[:5], dtype)
        raise AssertionError(
            f"{bad.size} rounds differ, first {bad[:5]} (ratio-test margins {margins}): "
            f"gpu {tok[bad[:3]]} {n[bad[:3]]} ref {rtok[bad[:3]]} {rn[bad[:3]]}")
    return tok, n


def test_tiny_vocab_whole_row(cuda_lib):
    """Vocabulary 1000, 3 drafts, temperature 1, no truncation, seed 0."""
    a = synth.accept_inputs(64, 3, 1000, (1.0, 1.0, 1.0), 1.0, seed=0)
    tok, n = check(cuda_lib, a, 1.0, 0, 1.0)
    assert 0 < n.mean() < 3


def test_acceptance_batch(cuda_lib):
    """256 rounds, vocabulary 152064, T=0.6, top-k 20, top-p 0.95, calibrated
    per-depth draft noise."""
    a = synth.accept_inputs(256, 3, 152064, synth.ACCEPT_BATCH_SIGMA, 0.6, top_k=20,
                            seed=1, device="cuda")
    tok, n = check(cuda_lib, a, 0.6, 20, 0.95)
    assert n.mean() > 1.5


@pytest.mark.parametrize("T,k,p", [(1.0, 0, 0.9), (0.7, 50, 1.0), (1.3, 5, 0.8), (0.0, 0, 1.0),
                                   (0.3, 1, 1.0), (2.0, 999, 0.5)])
def test_settings_small_vocab(cuda_lib, T, k, p):
    a = synth.accept_inputs(128, 4, 1000, (0.5, 1.0, 1.5, 2.0), T, top_k=k, seed=3)
    check(cuda_lib, a, T, k, p)


def test_long_candidate_lists(cuda_lib):
    """top-k 700 over a 20000-token vocabulary: the lists are longer than the
    shared-memory capacity of the distribution kernel (256), so it works in
    the lists' global scratch space."""
    a = synth.accept_inputs(32, 3, 20000, (0.5, 0.8, 1.1), 1.0, top_k=700, seed=8, device="cuda")
    check(cuda_lib, a, 1.0, 700, 0.97)


@pytest.mark.parametrize("R", [1, 2])
def test_large_top_k_few_rounds(cuda_lib, R):
    """top-k 700 over the full vocabulary with one or two rounds: the rows are
    split over several CTAs, and the chunks' top-k lists must still fit the
    merging CTA (no overflow)."""
    a = synth.accept_inputs(R, 3, 152064, (0.5, 0.8, 1.1), 1.0, top_k=700, seed=9, device="cuda")
    check(cuda_lib, a, 1.0, 700, 0.95)


def test_greedy_large_vocab(cuda_lib):
    a = synth.accept_inputs(32, 3, 152064, (0.3, 0.3, 0.3), 0.0, seed=4, device="cuda")
    check(cuda_lib, a, 0.0, 0, 1.0)


def test_bf16_logits(cuda_lib):
    a = synth.accept_inputs(64, 3, 32000, (0.2, 0.4, 0.6), 0.8, top_k=40, seed=5, device="cuda")
    check(cuda_lib, a, 0.8, 40, 0.9, dtype=torch.bfloat16)


def test_ties_at_the_top_k_boundary(cuda_lib):
    """Logits rounded to a coarse grid create ties at the k-th value; every
    tied token must be kept on both sides."""
    a = synth.accept_inputs(64, 3, 5000, (0.5, 0.5, 0.5), 1.0, top_k=10, seed=6)
    for key in ("target", "draft"):
        a[key] = torch.round(a[key] * 2) / 2
    a["draft_tokens"] = synth.synthetic_drafter(a["draft"], 1.0, 10, seed=6)
    check(cuda_lib, a, 1.0, 10, 1.0)
    check(cuda_lib, a, 1.0, 10, 0.7)


def test_tied_top_k_lists_over_a_thousand_long(cuda_lib):
    """top-k 1000 over integer logits (std 3): ties at the k-th value make
    every list 1266-1349 entries long (the top-k set with every token tied
    at its boundary), far beyond the 256 entries evaluated in shared memory."""
    a = synth.accept_inputs(8, 3, 3000, (0.5, 0.5, 0.5), 1.0, top_k=1000, seed=11)
    for key in ("target", "draft"):
        a[key] = torch.round(a[key])
    z = a["target"][0, 0]
    assert int((z >= torch.topk(z, 1000).values[-1]).sum()) > 1024
    a["draft_tokens"] = synth.synthetic_drafter(a["draft"], 1.0, 1000, seed=11)
    check(cuda_lib, a, 1.0, 1000, 1.0)
    check(cuda_lib, a, 1.0, 1000, 0.9)


@pytest.mark.parametrize("V,dtype", [(5001, torch.float32), (30001, torch.bfloat16)])
def test_rows_not_16_byte_aligned(cuda_lib, V, dtype):
    """Odd vocabulary sizes: rows start off 16-byte boundaries, so the select
    pass reads the logits one by one instead of 16 bytes at a time."""
    a = synth.accept_inputs(8, 3, V, (0.4, 0.6, 0.8), 0.9, top_k=30, seed=V)
    check(cuda_lib, a, 0.9, 30, 0.9, dtype=dtype)
    check(cuda_lib, a, 0.0, 0, 1.0, dtype=dtype)


def test_out_of_range_draft_is_rejected(cuda_lib):
    a = synth.accept_inputs(8, 2, 500, (0.5, 0.5), 1.0, seed=7)
    a["draft_tokens"][:, 0] = torch.tensor([-1, 500, 10 ** 6, 0, 1, 2, 3, 499], dtype=torch.int32)
    check(cuda_lib, a, 1.0, 0, 1.0)


@pytest.mark.parametrize("R", [1, 2, 5])
def test_few_rounds_full_vocab(cuda_lib, R):
    """Few rounds: each logits row is split over many CTAs and merged."""
    a = synth.accept_inputs(R, 3, 152064, synth.ACCEPT_BATCH_SIGMA, 0.6, top_k=20,
                            seed=40 + R, device="cuda")
    check(cuda_lib, a, 0.6, 20, 0.95)
    check(cuda_lib, a, 0.0, 0, 1.0)


@pytest.mark.parametrize("T,k,tp", [(1.0, 0, 1.0), (0.6, 5, 0.9), (1.5, 5, 1.0)])
def test_gpu_emission_law_chi_square(cuda_lib, T, k, tp):
    """60000 rounds sharing fixed logits (V = 16, K = 3) with drafts drawn from
    q: the GPU's first emitted token follows p_0, the second (given the first
    draft was accepted) follows p_1, and the depth-0 acceptance count is
    Binomial(R, sum min(p_0, q_0)) -- the exactness property ("The fastest way to
    run local LLMs on a Mac", "Why exact acceptance matters") checked at scale
    against the distributions themselves, not against the oracle's tokens."""
    from scipy import stats
    import oracle
    V, K, R = 16, 3, 60_000
    rng = np.random.default_rng(int(T * 100) + k)
    zt = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    zd = (zt[:K] + rng.normal(0, 0.7, size=(K, V))).astype(np.float32)
    Tf, tpf = float(np.float32(T)), float(np.float32(tp))
    ps = [oracle.dist(zt[i], Tf, k, tpf) for i in range(K + 1)]
    qs = [oracle.dist(zd[i], Tf, k, tpf) for i in range(K)]
    drafts = np.stack([rng.choice(V, size=R, p=qs[i] / qs[i].sum()) for i in range(K)], axis=1)
    a = {"target": torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zt[None], (R, K + 1, V)))),
         "draft": torch.from_numpy(np.ascontiguousarray(np.broadcast_to(zd[None], (R, K, V)))),
         "draft_tokens": torch.from_numpy(drafts.astype(np.int32)),
         "uniforms": torch.from_numpy(rng.random((R, K + 1), dtype=np.float32))}
    tok, n, status = accept_gpu(cuda_lib, a, T, k, tp)
    assert status == cuda_lib.SV_OK

    def pvalue(samples, p):
        obs = np.bincount(samples, minlength=V).astype(np.float64)
        sup = p > 0
        assert obs[~sup].sum() == 0, "a token outside the target's support was emitted"
        if sup.sum() == 1:
            return 1.0
        return stats.chisquare(obs[sup], p[sup] / p[sup].sum() * obs.sum()).pvalue

    assert pvalue(tok[:, 0], ps[0]) > 1e-6
    assert pvalue(tok[n >= 1, 1], ps[1]) > 1e-6
    alpha = float(np.minimum(ps[0], qs[0]).sum())
    assert stats.binomtest(int((n >= 1).sum()), R, alpha).pvalue > 1e-6


# ------------------------------------------------ whole-vocabulary path ---
# Every setting with temperature > 0 whose top-k is off, at least V, or above
# the candidate lists' 1024: exact integer sums of exp(z/T - zmax/T) over the
# whole row (accept_whole.cu).

@pytest.mark.parametrize("R", [1, 256])
@pytest.mark.parametrize("T,k,p", [(1.0, 0, 1.0), (0.6, 0, 0.95), (0.8, 5000, 0.9)])
def test_whole_vocab(cuda_lib, R, T, k, p):
    """The full 152064-token vocabulary with no top-k (no truncation at all,
    or top-p 0.95 only) and with top-k 5000 beyond the candidate lists."""
    a = synth.accept_inputs(R, 3, 152064, synth.ACCEPT_BATCH_SIGMA, T, top_k=k,
                            seed=60 + R + int(10 * T), device="cuda")
    tok, n = check(cuda_lib, a, T, k, p)
    assert (n >= 0).all()


def test_whole_vocab_tied_logits(cuda_lib):
    """Integer logits: thousands of tokens share each value, so the bucket of
    the k-th largest and the top-p band hold more tokens than one CTA sorts;
    the select kernel narrows them over key ranges down to a single tie
    group."""
    a = synth.accept_inputs(4, 3, 152064, (0.5, 0.5, 0.5), 1.0, seed=61, device="cuda")
    for key in ("target", "draft"):
        a[key] = torch.round(a[key])
    a["draft_tokens"] = synth.synthetic_drafter(a["draft"], 1.0, 0, seed=61)
    check(cuda_lib, a, 1.0, 0, 0.9)
    a["draft_tokens"] = synth.synthetic_drafter(a["draft"], 1.0, 5000, seed=61)
    check(cuda_lib, a, 1.0, 5000, 0.9)
    check(cuda_lib, a, 1.0, 5000, 1.0)


def test_whole_vocab_high_temperature(cuda_lib):
    """T = 500: every weight is within 5% of the largest, so the mass bounds
    put some ten thousand distinct logits in the top-p band and the select
    kernel narrows the band by exact masses before sorting."""
    a = synth.accept_inputs(2, 3, 152064, (0.5, 0.5, 0.5), 500.0, seed=62, device="cuda")
    check(cuda_lib, a, 500.0, 0, 0.5)
    check(cuda_lib, a, 500.0, 3000, 0.3)


@pytest.mark.parametrize("V", [4096, 4097, 9000])
@pytest.mark.parametrize("T,k,p", [(1.0, 0, 0.9), (0.7, 2000, 0.95), (1.2, 0, 1.0), (0.9, 1500, 1.0)])
def test_whole_vocab_around_the_list_capacity(cuda_lib, V, T, k, p):
    """Rows of up to 4096 tokens are handled by one CTA per row; longer rows
    by the multi-CTA passes."""
    a = synth.accept_inputs(16, 3, V, (0.4, 0.8, 1.2), T, top_k=k, seed=V + k, device="cuda")
    check(cuda_lib, a, T, k, p)


def test_whole_vocab_bf16(cuda_lib):
    """bf16 logits (8-bit mantissas: many ties) over the full vocabulary."""
    a = synth.accept_inputs(8, 3, 152064, (0.3, 0.5, 0.7), 0.9, seed=63, device="cuda")
    check(cuda_lib, a, 0.9, 0, 0.92, dtype=torch.bfloat16)
    check(cuda_lib, a, 0.9, 4000, 1.0, dtype=torch.bfloat16)


def test_whole_vocab_top_k_at_least_vocab_is_off(cuda_lib):
    a = synth.accept_inputs(8, 3, 3000, (0.5, 0.5, 0.5), 1.0, seed=64)
    t0, n0 = check(cuda_lib, a, 1.0, 0, 0.8)
    t1, n1 = check(cuda_lib, a, 1.0, 3000, 0.8)
    t2, n2 = check(cuda_lib, a, 1.0, 10 ** 6, 0.8)
    assert np.array_equal(t0, t1) and np.array_equal(t0, t2)


def test_whole_vocab_32_drafts(cuda_lib):
    """K = 32 (a full warp of ratio tests) with small draft noise, so that
    some rounds accept every draft and sample the bonus row."""
    a = synth.accept_inputs(16, 32, 5000, [0.01] * 32, 1.0, seed=65, device="cuda")
    tok, n = check(cuda_lib, a, 1.0, 0, 0.97)
    assert (n == 32).any()


def test_workspace_reused_across_settings(cuda_lib):
    """One workspace through calls on both paths and every pass of the
    whole-vocabulary path: each call leaves it ready for the next."""
    R, K, V = 4, 3, 152064
    ws = cuda_lib.workspace(cuda_lib.spec_accept_workspace_bytes(R, K, V))
    a = synth.accept_inputs(R, K, V, (0.3, 0.6, 0.9), 0.8, seed=66, device="cuda")
    for (T, k, p) in [(0.8, 0, 0.9), (0.8, 20, 0.95), (0.8, 5000, 0.9), (0.8, 0, 1.0),
                      (0.0, 0, 1.0), (0.8, 5000, 1.0), (0.8, 0, 0.9)]:
        check(cuda_lib, a, T, k, p, ws=ws)
