"""GB300-native K-draft verify step for MTP speculative decoding.

Thin ctypes binding over ``libspecverify.so`` (see ``include/specverify.h``).
Every compute function has the same name and argument order as its C entry
point; this module only marshals torch tensors (device memory) and the
current CUDA stream into pointers and sizes.  All arithmetic happens in the
library's CUDA kernels; there is no Python or CPU fallback, and a missing
library raises immediately.

    import speculative_decoding_verify_08_gb300 as sv
    packed = sv.prepack(codes, scales, biases)          # once per matrix
    ws = sv.workspace(sv.qmm_workspace_bytes(M, N, K))  # zeroed scratch
    sv.qmm_small_m(x, packed, y, M, N, K, ws)           # y = x @ W^T
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "load", "SvError", "SV_OK", "SV_ERR_INVALID_ARG", "SV_ERR_UNSUPPORTED", "SV_ERR_CUDA",
    "SV_ERR_TIMEOUT", "SV_ERR_WORKSPACE", "SV_ERR_OVERFLOW", "SV_BF16", "SV_F32", "SV_LAUNCH_PDL",
    "SV_LAUNCH_QMM_CUDA_CORES", "SV_LAUNCH_ATTN_MMA_SYNC", "SV_LAUNCH_ATTN_TCGEN05",
    "SV_LAUNCH_TEST_STALL_COPY",
    "qmm_packed_bytes", "qmm_prepack", "qmm_workspace_bytes", "qmm_small_m",
    "qmm8_packed_bytes", "qmm8_prepack", "qmm8_workspace_bytes", "qmm8_small_m",
    "verify_attn_workspace_bytes", "verify_attn", "verify_attn_masked", "verify_attn_noalloc", "spec_accept_workspace_bytes", "spec_accept",
    "qmm_topk_lists_bytes", "qmm_small_m_topk", "spec_accept_draft_select", "spec_accept_lists",
    "sv_status_string", "sv_last_device_error", "sv_set_launch_flags", "sv_get_launch_flags",
    "sv_kernel_launch_count", "prepack", "workspace", "library_path", "spec_pick_depth",
    "gdn_verify",
]

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED, SV_ERR_CUDA = 0, 1, 2, 3
SV_ERR_TIMEOUT, SV_ERR_WORKSPACE, SV_ERR_OVERFLOW = 4, 5, 6
SV_BF16, SV_F32 = 0, 1
SV_LAUNCH_PDL = 1
SV_LAUNCH_QMM_CUDA_CORES = 2  # measurement aid: qmm on CUDA-core FFMA at M = 1 and 4
SV_LAUNCH_ATTN_MMA_SYNC = 4  # verify_attn on the mma.sync kernel
SV_LAUNCH_ATTN_TCGEN05 = 8   # verify_attn on the tcgen05 kernel
SV_LAUNCH_TEST_STALL_COPY = 0x10000  # test aid: the attention (mma.sync) and matmul waits run out

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libspecverify.so")
_lock = threading.Lock()
_lib = None


class SvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {sv_status_string(status)} (status {status})")


class _Sampling(ctypes.Structure):
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_int32),
                ("top_p", ctypes.c_float)]


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libspecverify.so (built by ``__graft_entry__.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        lib = ctypes.CDLL(_LIB_PATH)
        P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        L = ctypes.c_int64
        sig = {
            "qmm_packed_bytes": (Z, [I, I, I]),
            "qmm_prepack": (I, [P, P, P, I, I, I, P, Z, P]),
            "qmm_workspace_bytes": (Z, [I, I, I]),
            "qmm_small_m": (I, [P, P, P, I, I, I, I, I, P, Z, P]),
            "qmm8_packed_bytes": (Z, [I, I, I]),
            "qmm8_prepack": (I, [P, P, P, I, I, I, P, Z, P]),
            "qmm8_workspace_bytes": (Z, [I, I, I]),
            "qmm8_small_m": (I, [P, P, P, I, I, I, I, I, P, Z, P]),
            "verify_attn_workspace_bytes": (Z, [I, I, I, I, L]),
            "verify_attn": (I, [P, P, P, P, I, I, I, I, L, L, ctypes.c_float, P, Z, P]),
            "verify_attn_noalloc": (I, [P, P, P, P, I, I, I, I, L, L, ctypes.c_float, P]),
            "verify_attn_masked": (I, [P, P, P, P, I, I, I, I, L, L, ctypes.c_float, P, P, Z, P]),
            "spec_accept_workspace_bytes": (Z, [I, I, I]),
            "spec_accept": (I, [P, P, I, P, P, _Sampling, I, I, I, P, P, P, Z, P]),
            "qmm_topk_lists_bytes": (Z, [I, I, I]),
            "qmm_small_m_topk": (I, [P, P, P, I, I, I, I, _Sampling, P, Z, P, Z, P]),
            "spec_accept_draft_select": (I, [P, I, _Sampling, I, I, I, P, Z, P]),
            "spec_accept_lists": (I, [P, P, P, P, _Sampling, I, I, I, P, P, P, Z, P]),
            "sv_status_string": (ctypes.c_char_p, [I]),
            "sv_last_device_error": (I, [P]),
            "sv_set_launch_flags": (None, [ctypes.c_uint]),
            "sv_get_launch_flags": (ctypes.c_uint, []),
            "sv_kernel_launch_count": (ctypes.c_uint64, []),
            "spec_pick_depth": (I, [P, P, P, I, P]),
            "gdn_verify": (I, [P, P, P, P, P, I, P, P, P, P, P, P, I, I, I, I, I, I, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str):
    if status != SV_OK:
        raise SvError(status, where)


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


# ------------------------------------------------------------- queries ----
def sv_status_string(status: int) -> str:
    return load().sv_status_string(int(status)).decode()


def qmm_packed_bytes(N: int, K: int, group: int = 64) -> int:
    return load().qmm_packed_bytes(N, K, group)


def qmm_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().qmm_workspace_bytes(M, N, K)


def qmm8_packed_bytes(N: int, K: int, group: int = 64) -> int:
    return load().qmm8_packed_bytes(N, K, group)


def qmm8_workspace_bytes(M: int, N: int, K: int) -> int:
    return load().qmm8_workspace_bytes(M, N, K)


def verify_attn_workspace_bytes(M: int, Hq: int, Hkv: int, D: int, kv_len: int) -> int:
    return load().verify_attn_workspace_bytes(M, Hq, Hkv, D, kv_len)


def spec_accept_workspace_bytes(R: int, K: int, V: int) -> int:
    return load().spec_accept_workspace_bytes(R, K, V)


def sv_set_launch_flags(flags: int) -> None:
    load().sv_set_launch_flags(int(flags))


def sv_get_launch_flags() -> int:
    return load().sv_get_launch_flags()


def sv_kernel_launch_count() -> int:
    return load().sv_kernel_launch_count()


def sv_last_device_error(stream=None) -> int:
    return load().sv_last_device_error(_stream(stream))


# ------------------------------------------------------------- compute ----
def qmm_prepack(codes, scales, biases, N: int, K: int, group: int, packed_out, stream=None):
    _check(load().qmm_prepack(_ptr(codes), _ptr(scales), _ptr(biases), N, K, group,
                              _ptr(packed_out), _nbytes(packed_out), _stream(stream)),
           "qmm_prepack")


def qmm_small_m(x, packed_w, y, M: int, N: int, K: int, workspace=None, group: int = 64,
                stream=None):
    ydt = SV_F32 if y.dtype == torch.float32 else SV_BF16
    _check(load().qmm_small_m(_ptr(x), _ptr(packed_w), _ptr(y), ydt, M, N, K, group,
                              _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "qmm_small_m")


def qmm8_prepack(codes, scales, biases, N: int, K: int, group: int, packed_out, stream=None):
    _check(load().qmm8_prepack(_ptr(codes), _ptr(scales), _ptr(biases), N, K, group,
                               _ptr(packed_out), _nbytes(packed_out), _stream(stream)),
           "qmm8_prepack")


def qmm8_small_m(x, packed_w, y, M: int, N: int, K: int, workspace=None, group: int = 64,
                 stream=None):
    ydt = SV_F32 if y.dtype == torch.float32 else SV_BF16
    _check(load().qmm8_small_m(_ptr(x), _ptr(packed_w), _ptr(y), ydt, M, N, K, group,
                               _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "qmm8_small_m")


def verify_attn(q, k_cache, v_cache, o, M: int, Hq: int, Hkv: int, D: int, kv_len: int,
                kv_stride_tokens: int, scale: float, workspace=None, stream=None):
    _check(load().verify_attn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, Hq, Hkv, D,
                              kv_len, kv_stride_tokens, float(scale), _ptr(workspace),
                              _nbytes(workspace), _stream(stream)),
           "verify_attn")


def verify_attn_masked(q, k_cache, v_cache, o, M: int, Hq: int, Hkv: int, D: int, kv_len: int,
                       kv_stride_tokens: int, scale: float, draft_mask, workspace=None, stream=None):
    """verify_attn over a draft tree: draft_mask is a device int32/uint32
    tensor [M]; bit j of draft_mask[i] lets row i see draft slot kv_len-M+j."""
    _check(load().verify_attn_masked(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, Hq, Hkv,
                                     D, kv_len, kv_stride_tokens, float(scale), _ptr(draft_mask),
                                     _ptr(workspace), _nbytes(workspace), _stream(stream)),
           "verify_attn_masked")


def verify_attn_noalloc(q, k_cache, v_cache, o, M: int, Hq: int, Hkv: int, D: int,
                        kv_len: int, kv_stride_tokens: int, scale: float, stream=None):
    """verify_attn without a workspace argument, for callers that cannot
    allocate device memory; its scratch is a fixed 16 MiB array inside the
    library (see include/specverify.h for the rules of use)."""
    _check(load().verify_attn_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(o), M, Hq,
                                      Hkv, D, kv_len, kv_stride_tokens, float(scale),
                                      _stream(stream)),
           "verify_attn_noalloc")


def spec_accept(target_logits, draft_logits, draft_tokens, uniforms, temperature: float,
                top_k: int, top_p: float, R: int, K: int, V: int, out_tokens,
                out_num_accepted, workspace=None, stream=None):
    dt = SV_BF16 if target_logits.dtype == torch.bfloat16 else SV_F32
    sp = _Sampling(float(temperature), int(top_k), float(top_p))
    _check(load().spec_accept(_ptr(target_logits), _ptr(draft_logits), dt, _ptr(draft_tokens),
                              _ptr(uniforms), sp, R, K, V, _ptr(out_tokens),
                              _ptr(out_num_accepted), _ptr(workspace), _nbytes(workspace),
                              _stream(stream)),
           "spec_accept")


def qmm_topk_lists_bytes(M: int, N: int, K: int) -> int:
    return load().qmm_topk_lists_bytes(M, N, K)


def qmm_small_m_topk(x, packed_w, y, M: int, N: int, K: int, temperature: float, top_k: int,
                     top_p: float, lists, workspace=None, group: int = 64, stream=None):
    sp = _Sampling(float(temperature), int(top_k), float(top_p))
    _check(load().qmm_small_m_topk(_ptr(x), _ptr(packed_w), _ptr(y), M, N, K, group, sp, _ptr(lists),
                                   _nbytes(lists), _ptr(workspace), _nbytes(workspace),
                                   _stream(stream)),
           "qmm_small_m_topk")


def spec_accept_draft_select(draft_logits, temperature: float, top_k: int, top_p: float, R: int,
                             K: int, V: int, workspace, stream=None):
    dt = SV_BF16 if draft_logits.dtype == torch.bfloat16 else SV_F32
    sp = _Sampling(float(temperature), int(top_k), float(top_p))
    _check(load().spec_accept_draft_select(_ptr(draft_logits), dt, sp, R, K, V, _ptr(workspace),
                                           _nbytes(workspace), _stream(stream)),
           "spec_accept_draft_select")


def spec_accept_lists(target_lists, draft_tokens, uniforms, temperature: float, top_k: int,
                      top_p: float, R: int, K: int, V: int, out_tokens, out_num_accepted,
                      workspace, draft_lists=None, stream=None):
    sp = _Sampling(float(temperature), int(top_k), float(top_p))
    _check(load().spec_accept_lists(_ptr(target_lists), _ptr(draft_lists), _ptr(draft_tokens),
                                    _ptr(uniforms), sp, R, K, V, _ptr(out_tokens),
                                    _ptr(out_num_accepted), _ptr(workspace), _nbytes(workspace),
                                    _stream(stream)),
           "spec_accept_lists")


# ------------------------------------------------------------- helpers ----
def workspace(nbytes: int, device=None):
    """Zero-filled device scratch of at least ``nbytes`` bytes (None if 0)."""
    if nbytes <= 0:
        return None
    dev = device if device is not None else torch.device("cuda")
    return torch.zeros(((nbytes + 255) // 256) * 256, dtype=torch.uint8, device=dev)


def prepack(codes, scales, biases, group: int = 64, stream=None, bits: int = 4):
    """Allocate and fill the prepacked weight buffer of an [N, K] matrix
    (4-bit codes [N, K/8], or 8-bit codes [N, K/4] with bits=8)."""
    if bits not in (4, 8):
        raise SvError(SV_ERR_UNSUPPORTED, "prepack")
    N, KW = codes.shape
    K = KW * (32 // bits)
    nb = (qmm_packed_bytes if bits == 4 else qmm8_packed_bytes)(N, K, group)
    if nb == 0:
        raise SvError(SV_ERR_UNSUPPORTED, "qmm_packed_bytes")
    out = torch.empty(nb, dtype=torch.uint8, device=codes.device)
    (qmm_prepack if bits == 4 else qmm8_prepack)(codes, scales, biases, N, K, group, out, stream=stream)
    return out


def spec_pick_depth(verify_us, accept, draft_us=None):
    """Draft depth with the most tokens per microsecond (0 unless it beats
    plain decoding) and every depth's rate.  verify_us[K]: cost of a verify
    pass with K+1 rows; accept[i-1]: P(at least i drafts accepted)."""
    import numpy as np
    v = np.ascontiguousarray(verify_us, dtype=np.float64).ravel()
    a = np.ascontiguousarray(accept, dtype=np.float64).ravel()
    kmax = v.shape[0] - 1
    if a.shape[0] != kmax:
        raise SvError(SV_ERR_INVALID_ARG, "spec_pick_depth")
    d = None if draft_us is None else np.ascontiguousarray(draft_us, dtype=np.float64).ravel()
    rates = np.zeros(kmax + 1, dtype=np.float64)
    k = load().spec_pick_depth(v.ctypes.data, None if d is None else d.ctypes.data,
                               a.ctypes.data if kmax > 0 else None, kmax, rates.ctypes.data)
    if k < 0:
        raise SvError(SV_ERR_INVALID_ARG, "spec_pick_depth")
    return k, rates


def gdn_verify(state, q, k, v, g, beta, o, tape=None, n_replay=0, stream=None):
    """GatedDeltaNet verify step: commits the first n_replay tokens of the
    previous round's tape (k, v, g, beta) into `state` (fp32 [Hv, dv, dk]),
    then runs this round's rows into `o`.  q, k bf16 [M, Hk, dk]; v bf16
    [M, Hv, dv]; g, beta fp32 [M, Hv]."""
    Hv, dv, dk = state.shape
    M, Hk = (k.shape[0], k.shape[1]) if k is not None else (0, tape[0].shape[1])
    tk, tv, tg, tb = tape if tape is not None else (None, None, None, None)
    odt = SV_F32 if (o is not None and o.dtype == torch.float32) else SV_BF16
    _check(load().gdn_verify(_ptr(state), _ptr(tk), _ptr(tv), _ptr(tg), _ptr(tb), int(n_replay),
                             _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(o), odt, M, Hk, Hv,
                             dk, dv, _stream(stream)),
           "gdn_verify")
