"""Shared helpers of the GPU parity tests: run a kernel through the C ABI,
run the oracle on the same bytes, compare."""
import numpy as np
import torch

import oracle
from speculative_decoding_verify_08_gb300 import synth

TOL = 2e-2  # max |gpu - oracle| <= TOL * RMS(oracle), fp32 accumulation


def assert_close(got, ref, tol=TOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    err = float(np.max(np.abs(got - ref))) if got.size else 0.0
    assert err <= tol * rms, f"{what}: max abs err {err:.3e} > {tol} * rms {rms:.3e}"
    return err / rms if rms > 0 else 0.0


def scaled_rows(t, exps, seed):
    """Scales of row n near 2^exps[n % len(exps)] (bf16, subnormal at 2^-133),
    biases about -8 times the scale: the same codes and activations."""
    rng = np.random.default_rng(seed)
    N, G = t["scales"].shape
    e = np.asarray(exps, dtype=np.float64)[np.arange(N) % len(exps)][:, None]
    s = np.exp2(e) * rng.uniform(1.0, 2.0, size=(N, G))
    b = -8.0 * s * rng.uniform(0.5, 1.5, size=(N, G))
    out = dict(t)
    out["scales"] = torch.from_numpy(s).to(torch.bfloat16).to(t["scales"].device)
    out["biases"] = torch.from_numpy(b).to(torch.bfloat16).to(t["biases"].device)
    return out


def assert_close_per_column(got, ref, what, tol=2e-2):
    """Each output column against its own scale: max |gpu - oracle| over the
    rows <= tol * RMS of the oracle's column."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    rms = np.sqrt(np.mean(ref ** 2, axis=0))
    err = np.max(np.abs(got - ref), axis=0)
    bad = np.nonzero(err > tol * rms)[0]
    assert bad.size == 0, f"{what}: columns {bad[:8]} err {err[bad[:8]]} rms {rms[bad[:8]]}"


# row magnitudes from a subnormal bf16 scale (2^-133) to 2^100: the outputs
# stay finite at 4 and 8 bits
SCALE_EXPS = [-133, -126, -100, -40, -7, 0, 40, 100]


def qmm_gpu(sv, t, M, N, K, out_dtype=torch.float32, packed=None, ws=None, bits=4):
    dev = torch.device("cuda")
    if packed is None:
        packed = sv.prepack(t["codes"].to(dev), t["scales"].to(dev), t["biases"].to(dev), bits=bits)
    if ws is None:
        ws = sv.workspace((sv.qmm_workspace_bytes if bits == 4 else sv.qmm8_workspace_bytes)(M, N, K))
    x = t["x"].to(dev)
    y = torch.empty((M, N), dtype=out_dtype, device=dev)
    (sv.qmm_small_m if bits == 4 else sv.qmm8_small_m)(x, packed, y, M, N, K, ws)
    assert sv.sv_last_device_error() == sv.SV_OK
    return y.float().cpu().numpy()


def qmm_ref(t, rows=None, bits=4):
    x = synth.bf16_bits(t["x"])
    codes = synth.u32_bits(t["codes"])
    s = synth.bf16_bits(t["scales"])
    b = synth.bf16_bits(t["biases"])
    if rows is not None:
        codes, s, b = codes[rows], s[rows], b[rows]
    return (oracle.qmm if bits == 4 else oracle.qmm8)(x, codes, s, b)


def attn_gpu(sv, t, M, Hq, Hkv, D, L, cap, scale, mask=None):
    dev = torch.device("cuda")
    q, k, v = t["q"].to(dev), t["k"].to(dev), t["v"].to(dev)
    o = torch.empty((M, Hq, D), dtype=torch.bfloat16, device=dev)
    ws = sv.workspace(sv.verify_attn_workspace_bytes(M, Hq, Hkv, D, L))
    if mask is None:
        sv.verify_attn(q, k, v, o, M, Hq, Hkv, D, L, cap, scale, ws)
    else:
        mk = torch.from_numpy(mask.astype(np.int64).astype(np.int32)).to(dev)
        sv.verify_attn_masked(q, k, v, o, M, Hq, Hkv, D, L, cap, scale, mk, ws)
    assert sv.sv_last_device_error() == sv.SV_OK
    return o.float().cpu().numpy()


def attn_ref(t, L, scale, mask=None):
    return oracle.attn(synth.bf16_bits(t["q"]), synth.bf16_bits(t["k"]), synth.bf16_bits(t["v"]),
                       L, scale, mask=mask)


def accept_gpu(sv, a, T, top_k, top_p, logit_dtype=torch.float32, ws=None):
    dev = torch.device("cuda")
    zt = a["target"].to(dev).to(logit_dtype)
    zd = a["draft"].to(dev).to(logit_dtype)
    R, K1, V = zt.shape
    K = K1 - 1
    tok = torch.full((R, K + 1), -7, dtype=torch.int32, device=dev)
    n = torch.full((R,), -7, dtype=torch.int32, device=dev)
    if ws is None:
        ws = sv.workspace(sv.spec_accept_workspace_bytes(R, K, V))
    sv.spec_accept(zt, zd, a["draft_tokens"].to(dev), a["uniforms"].to(dev), T, top_k, top_p,
                   R, K, V, tok, n, ws)
    status = sv.sv_last_device_error()
    return tok.cpu().numpy(), n.cpu().numpy(), status


def accept_ref(a, T, top_k, top_p, logit_dtype=torch.float32):
    zt = a["target"].to(logit_dtype).float().cpu().numpy()
    zd = a["draft"].to(logit_dtype).float().cpu().numpy()
    # the library receives fp32 settings: hand the oracle the same values
    return oracle.accept(zt, zd, a["draft_tokens"].cpu().numpy(), a["uniforms"].cpu().numpy(),
                         float(np.float32(T)), top_k, float(np.float32(top_p)))
