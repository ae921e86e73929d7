"""The seeded input generators: determinism, shapes, and the stored sigmas."""
import json
import os

import numpy as np
import torch

from speculative_decoding_verify_08_gb300 import synth

HERE = os.path.dirname(__file__)


def test_sigma_constants_match_calibration():
    with open(os.path.join(HERE, "golden", "accept_sigma.json")) as f:
        d = json.load(f)
    assert tuple(d["sigma"]) == synth.ACCEPT_BATCH_SIGMA
    assert d["vocab"] == 152064 and d["top_k"] == 20 and d["top_p"] == 0.95


def test_generators_are_deterministic_and_shaped():
    a = synth.qmm_inputs(4, 32, 128, seed=3)
    b = synth.qmm_inputs(4, 32, 128, seed=3)
    c = synth.qmm_inputs(4, 32, 128, seed=4)
    for k in a:
        assert torch.equal(a[k], b[k])
    assert not torch.equal(a["codes"], c["codes"])
    assert a["x"].dtype == torch.bfloat16 and a["codes"].shape == (32, 16)
    assert (a["scales"].float() >= 0).all()
    t = synth.attn_inputs(2, 4, 2, 16, 10, cap=12, seed=1)
    assert t["k"].shape == (2, 12, 16) and (t["k"][:, 10:] == 0).all()
    acc = synth.accept_inputs(3, 2, 50, (0.1, 0.2), 1.0, top_k=5, seed=0)
    assert acc["target"].shape == (3, 3, 50) and acc["draft_tokens"].dtype == torch.int32
    u = acc["uniforms"]
    assert (u >= 0).all() and (u < 1).all()
    # drafts come from the draft row's top-k
    top = torch.topk(acc["draft"], 5, dim=-1).indices
    assert (top == acc["draft_tokens"].long()[..., None]).any(-1).all()


def test_code_words_cover_all_nibbles():
    a = synth.qmm_inputs(1, 64, 512, seed=0)
    w = synth.u32_bits(a["codes"]).ravel()
    nib = np.concatenate([(w >> (4 * i)) & 15 for i in range(8)])
    counts = np.bincount(nib, minlength=16)
    assert counts.min() > 0.8 * counts.mean()


def test_draft_tree_masks_are_trees():
    """Node 0 is the root; each node sees itself and exactly its parent's set."""
    for M in (1, 2, 5, 8, 16):
        m = synth.draft_tree_masks(M, seed=M)
        assert m.dtype == np.uint32 and m.shape == (M,)
        assert m[0] == 1
        for i in range(1, M):
            assert (m[i] >> i) & 1 and m[i] < (1 << (i + 1))
            parent = m[i] & ~np.uint32(1 << i)
            assert any(m[j] == parent for j in range(i)), (M, i)
