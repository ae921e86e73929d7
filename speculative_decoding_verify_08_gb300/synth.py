"""Seeded synthetic inputs for the verify-step kernels.

This module is shared by the CUDA path's tests/benchmark and by the CPU
oracle's tests, so it holds none of the method's arithmetic: no dequantising,
no attention, no truncation or acceptance.  It only draws tensors.

Every tensor is drawn from its own ``torch.Generator`` seeded with
``(seed, tensor id)``, on the device asked for.  CPU and CUDA generators give
different streams, so a comparison always hands both sides the *same bytes*
(generate once, copy to the other side); nothing relies on two devices
reproducing one another's random numbers.

Distributions (standard deviations, ``torch.randn() * sigma`` convention):

* quantised weights: 4-bit codes uniform in 0..15 (random 32-bit words, eight
  codes per word), scales ``|N(0, 0.02)|`` and biases ``N(0, 0.01)`` as bf16;
  activations ``N(0, 1)`` bf16;
* attention: Q, K, V ``N(0, 1)`` bf16;
* acceptance: target logits ``N(0, 3)`` fp32, draft logits = target +
  ``N(0, sigma_i)`` per draft depth, uniforms in [0, 1) (fp32, 24-bit grid),
  draft tokens from a synthetic drafter (Gumbel-max over the draft row's
  top-k logits at the sampling temperature; the drafter model itself is not
  part of the verify step).
"""
from __future__ import annotations

import math

import numpy as np
import torch

# tensor ids: keep stable, they seed the streams
_T_X, _T_CODES, _T_SCALES, _T_BIASES = 1, 2, 3, 4
_T_Q, _T_K, _T_V = 11, 12, 13
_T_ZT, _T_NOISE, _T_U, _T_GUMBEL = 21, 22, 23, 24

# Draft-logit noise per depth for the 256-round acceptance batch (vocab
# 152064, T=0.6, top-k 20, top-p 0.95), chosen so that the mean per-row
# acceptance sum_j min(p_j, q_j) is about 0.95 / 0.88 / 0.80.  Written by
# tests/golden/calibrate_sigma.py (which calls only the oracle) into
# tests/golden/accept_sigma.json; a CPU test checks the two agree.
ACCEPT_BATCH_SIGMA = (0.0732, 0.1845, 0.3128)


def _gen(seed: int, tid: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((int(seed) * 1_000_003 + tid * 7919) & 0x7FFF_FFFF_FFFF_FFFF)
    return g


def qmm_inputs(M: int, N: int, K: int, group: int = 64, seed: int = 0,
               device="cpu", bits: int = 4):
    """Activations and canonical 4-bit (or 8-bit) weights for ``y = x @ W^T``.

    Returns x bf16 [M, K], codes int32 [N, K*bits/32] (bit pattern of the
    uint32 code words; lowest k in the lowest nibble or byte, every code
    uniform over its range), scales bf16 [N, K/group], biases bf16
    [N, K/group].  8-bit scales are 1/17 of the 4-bit ones, so that both
    weight sets span about the same range.
    """
    assert bits in (4, 8) and K % 8 == 0 and K % group == 0
    dev = torch.device(device)
    x = torch.randn((M, K), generator=_gen(seed, _T_X, dev), device=dev)
    codes = torch.randint(-(2 ** 31), 2 ** 31, (N, K * bits // 32), dtype=torch.int64,
                          generator=_gen(seed, _T_CODES, dev), device=dev)
    codes = codes.to(torch.int32)
    s = torch.randn((N, K // group), generator=_gen(seed, _T_SCALES, dev), device=dev)
    b = torch.randn((N, K // group), generator=_gen(seed, _T_BIASES, dev), device=dev)
    return {
        "x": x.to(torch.bfloat16),
        "codes": codes,
        "scales": (s.abs() * (0.02 if bits == 4 else 0.02 / 17)).to(torch.bfloat16),
        "biases": (b * 0.01).to(torch.bfloat16),
    }


def gdn_inputs(M: int, Hk: int, Hv: int, dk: int, dv: int, seed: int = 0, device="cpu"):
    """One round of GatedDeltaNet inputs: q, k bf16 [M, Hk, dk] with unit-norm
    rows (the layer normalises them before the recurrence), v bf16 [M, Hv, dv]
    N(0,1), log-decays g fp32 [M, Hv] uniform in (-0.2, -0.01), write
    strengths beta fp32 [M, Hv] uniform in (0.05, 0.95), and a prior state fp32
    [Hv, dv, dk] N(0, 0.1)."""
    dev = torch.device(device)
    gq, gk, gv = (_gen(seed, t, dev) for t in (_T_Q, _T_K, _T_V))
    q = torch.randn((M, Hk, dk), generator=gq, device=dev)
    k = torch.randn((M, Hk, dk), generator=gk, device=dev)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    v = torch.randn((M, Hv, dv), generator=gv, device=dev)
    gs = _gen(seed, _T_SCALES, dev)
    g = -(0.01 + 0.19 * torch.rand((M, Hv), generator=gs, device=dev))
    beta = 0.05 + 0.9 * torch.rand((M, Hv), generator=gs, device=dev)
    state = 0.1 * torch.randn((Hv, dv, dk), generator=_gen(seed, _T_BIASES, dev), device=dev)
    return {"q": q.to(torch.bfloat16), "k": k.to(torch.bfloat16), "v": v.to(torch.bfloat16),
            "g": g.float(), "beta": beta.float(), "state": state.float()}


def attn_inputs(M: int, Hq: int, Hkv: int, D: int, kv_len: int, cap: int | None = None,
                seed: int = 0, device="cpu"):
    """Q bf16 [M, Hq, D]; K, V bf16 [Hkv, cap, D] with slots >= kv_len zero."""
    cap = kv_len if cap is None else cap
    assert cap >= kv_len
    dev = torch.device(device)
    q = torch.randn((M, Hq, D), generator=_gen(seed, _T_Q, dev), device=dev)
    k = torch.zeros((Hkv, cap, D), device=dev, dtype=torch.bfloat16)
    v = torch.zeros((Hkv, cap, D), device=dev, dtype=torch.bfloat16)
    if kv_len > 0:
        gk = _gen(seed, _T_K, dev)
        gv = _gen(seed, _T_V, dev)
        for h in range(Hkv):  # per head keeps the fp32 temporary small
            k[h, :kv_len] = torch.randn((kv_len, D), generator=gk, device=dev).to(torch.bfloat16)
            v[h, :kv_len] = torch.randn((kv_len, D), generator=gv, device=dev).to(torch.bfloat16)
    return {"q": q.to(torch.bfloat16), "k": k, "v": v}


def draft_tree_masks(M: int, seed: int = 0) -> np.ndarray:
    """uint32 [M] masks of a random draft tree: node 0 is the root, node i
    (i >= 1) hangs under a uniformly drawn earlier node, and bit j of mask[i]
    is set iff node j is node i or one of its ancestors."""
    rng = np.random.default_rng(seed)
    mask = np.zeros(M, dtype=np.uint32)
    mask[0] = 1
    for i in range(1, M):
        parent = int(rng.integers(0, i))
        mask[i] = mask[parent] | np.uint32(1 << i)
    return mask


def accept_inputs(R: int, K: int, V: int, sigmas, temperature: float,
                  top_k: int = 0, seed: int = 0, device="cpu",
                  target_std: float = 3.0):
    """Logits, draft tokens and uniforms for R independent speculative rounds.

    target fp32 [R, K+1, V] ~ N(0, target_std); draft fp32 [R, K, V] = target
    rows 0..K-1 + N(0, sigmas[i]); uniforms fp32 [R, K+1] in [0, 1);
    draft_tokens int32 [R, K] from the synthetic drafter (Gumbel-max over the
    draft row's top-k logits divided by the temperature; argmax at T = 0).
    """
    dev = torch.device(device)
    sig = list(sigmas) if hasattr(sigmas, "__len__") else [float(sigmas)] * K
    assert len(sig) == K
    zt = torch.randn((R, K + 1, V), generator=_gen(seed, _T_ZT, dev), device=dev)
    zt.mul_(target_std)
    gn = _gen(seed, _T_NOISE, dev)
    zd = torch.empty((R, K, V), device=dev, dtype=torch.float32)
    for i in range(K):
        zd[:, i] = zt[:, i] + torch.randn((R, V), generator=gn, device=dev) * sig[i]
    u = torch.rand((R, K + 1), generator=_gen(seed, _T_U, dev), device=dev)
    tokens = synthetic_drafter(zd, temperature, top_k, seed=seed)
    return {"target": zt, "draft": zd, "uniforms": u, "draft_tokens": tokens}


def synthetic_drafter(draft_logits: torch.Tensor, temperature: float, top_k: int,
                      seed: int = 0) -> torch.Tensor:
    """Draft tokens int32 [R, K] standing in for the MTP head's own samples."""
    R, K, V = draft_logits.shape
    dev = draft_logits.device
    kk = V if (top_k <= 0 or top_k >= V) else top_k
    vals, idx = torch.topk(draft_logits, kk, dim=-1)
    if temperature == 0.0:
        pick = torch.zeros((R, K, 1), dtype=torch.int64, device=dev)
    else:
        g = torch.rand(vals.shape, generator=_gen(seed, _T_GUMBEL, dev), device=dev)
        g = -torch.log(-torch.log(g.clamp_min(1e-12)))
        pick = torch.argmax(vals / temperature + g, dim=-1, keepdim=True)
    return torch.gather(idx, -1, pick).squeeze(-1).to(torch.int32)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (on the CPU)."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u32_bits(t: torch.Tensor):
    """uint32 numpy view of an int32 tensor's bit patterns (on the CPU)."""
    import numpy as np
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def attn_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
