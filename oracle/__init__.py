"""CPU oracle for the K-draft verify step (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64); this module compiles it
with gcc on first use and marshals numpy arrays through ctypes.  Functions:

* :func:`qmm`    -- y = x @ dequant(codes, scales, biases)^T, affine 4-bit
  group quantisation ("Speculative decoding and MTP on Apple silicon", Facts:
  the small-M 4-bit quantized matmul; "The fastest way to run local LLMs on a
  Mac", "Decode is a memory-bandwidth problem").
* :func:`qmm8`   -- the same with 8-bit codes (four per uint32), the 8-bit
  affine pack ("Speculative decoding and MTP on Apple silicon", Facts:
  skinny_qmm covers 4-bit and 8-bit weights; 8-bit is the ratio sweet spot).
* :func:`attn`   -- multi-row verify attention, causal among the M draft rows
  ("Speculative decoding and MTP on Apple silicon", Facts: multi-row verify
  attention reads each KV tile once for 2-8 query rows).
* :func:`gdn` -- GatedDeltaNet verify step that first commits the previous
  round from its tape ("Speculative decoding and MTP on Apple silicon", Facts:
  GDN state cannot be trimmed; MTPLX's GDN kernel replays an innovation tape).
* :func:`pick_depth` -- the draft depth with the most tokens per microsecond
  from measured verify / draft cost curves ("Speculative decoding and MTP on
  Apple silicon", Facts: mlx-dspark and MTPLX depth tuning).
* :func:`dist`, :func:`accept` -- truncated sampling distribution and the
  Leviathan-Chen acceptance chain ("The fastest way ...", "Why exact
  acceptance matters"; "Speculative decoding and MTP on Apple silicon", Facts:
  rejection sampling and identical truncation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_handle = None

# planted-mistake codes (see oracle.c); tests use them to show pins bite
MUT_NONE = 0
MUT_QMM_NIBBLE_HIGH_FIRST = 1
MUT_QMM_GROUP_OFF_BY_ONE = 2
MUT_QMM_DROP_BIAS = 3
MUT_ATTN_NO_CAUSAL = 4
MUT_ATTN_MASK_OFF_BY_ONE = 5
MUT_ATTN_GQA_MODULO = 6
MUT_ACC_RESIDUAL_SIGN = 7
MUT_ACC_REUSE_UNIFORM = 8
MUT_ACC_NO_DRAFT_TRUNC = 9
MUT_ACC_GREEDY = 10
MUT_ACC_TOPP_INCLUSIVE = 11
MUT_ACC_NAIVE = 12
MUT_ATTN_MASK_BIT_ORDER = 13
MUT_QMM8_BYTE_HIGH_FIRST = 14
MUT_QMM8_SIGNED = 15
MUT_DEPTH_NO_BONUS = 16
MUT_DEPTH_CONDITIONAL = 17
MUT_DEPTH_TIES_DEEPER = 18
MUT_GDN_NO_DECAY_IN_DELTA = 19
MUT_GDN_OUTPUT_BEFORE = 20
MUT_GDN_TRANSPOSED = 21
MUT_GDN_HEAD_MODULO = 22


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``oracle/lib/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _lib():
    global _handle
    with _lock:
        if _handle is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            L = ctypes.c_int64
            lib.oracle_qmm.argtypes = [P, P, P, P, I, I, I, I, P, I]
            lib.oracle_qmm8.argtypes = [P, P, P, P, I, I, I, I, P, I]
            lib.oracle_attn.argtypes = [P, P, P, I, I, I, I, L, L, D, P, I]
            lib.oracle_attn_masked.argtypes = [P, P, P, I, I, I, I, L, L, D, P, P, I]
            lib.oracle_dist.argtypes = [P, I, D, I, D, P]
            lib.oracle_accept.argtypes = [P, P, P, P, I, I, I, D, I, D, P, P, I]
            lib.oracle_pick_depth.argtypes = [P, P, P, I, P]
            lib.oracle_pick_depth.restype = I
            lib.oracle_gdn.argtypes = [P, P, P, P, P, I, P, P, P, P, P, I, I, I, I, I, P, I]
            lib.oracle_gdn.restype = I
            lib.oracle_set_mutant.argtypes = [I]
            for f in (lib.oracle_qmm, lib.oracle_qmm8, lib.oracle_attn, lib.oracle_attn_masked, lib.oracle_dist,
                      lib.oracle_accept):
                f.restype = I
            lib.oracle_set_mutant.restype = None
            _handle = lib
    return _handle


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def set_mutant(code: int) -> None:
    """Plant a named mistake in the oracle (tests only); 0 restores it."""
    _lib().oracle_set_mutant(int(code))


class mutant:
    """Context manager planting one mistake for the duration of a block."""

    def __init__(self, code: int):
        self.code = code

    def __enter__(self):
        set_mutant(self.code)
        return self

    def __exit__(self, *exc):
        set_mutant(MUT_NONE)
        return False


def qmm(x_bf16: np.ndarray, codes: np.ndarray, scales_bf16: np.ndarray,
        biases_bf16: np.ndarray, group: int = 64, threads: int = 0) -> np.ndarray:
    """fp64 [M, N] = x @ W^T with W[n, k] = s[n, k//group]*q[n, k] + b[n, k//group].

    x_bf16: uint16 bf16 bits [M, K]; codes: uint32 [N, K/8] (low nibble = lowest
    k); scales_bf16, biases_bf16: uint16 bf16 bits [N, K/group].
    """
    x = _c(x_bf16, np.uint16)
    wq = _c(codes, np.uint32)
    s = _c(scales_bf16, np.uint16)
    b = _c(biases_bf16, np.uint16)
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K // 8) and s.shape == (N, K // group) == b.shape
    y = np.zeros((M, N), dtype=np.float64)
    rc = _lib().oracle_qmm(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), M, N, K, group,
                           _ptr(y), threads)
    if rc != 0:
        raise ValueError("oracle_qmm rejected its arguments")
    return y


def qmm8(x_bf16: np.ndarray, codes: np.ndarray, scales_bf16: np.ndarray,
         biases_bf16: np.ndarray, group: int = 64, threads: int = 0) -> np.ndarray:
    """fp64 [M, N] = x @ W^T with 8-bit codes: W[n, k] = s[n, k//group]*q[n, k] +
    b[n, k//group], q in 0..255.

    codes: uint32 [N, K/4] (lowest byte = lowest k); other arguments as qmm.
    """
    x = _c(x_bf16, np.uint16)
    wq = _c(codes, np.uint32)
    s = _c(scales_bf16, np.uint16)
    b = _c(biases_bf16, np.uint16)
    M, K = x.shape
    N = wq.shape[0]
    assert wq.shape == (N, K // 4) and s.shape == (N, K // group) == b.shape
    y = np.zeros((M, N), dtype=np.float64)
    rc = _lib().oracle_qmm8(_ptr(x), _ptr(wq), _ptr(s), _ptr(b), M, N, K, group,
                            _ptr(y), threads)
    if rc != 0:
        raise ValueError("oracle_qmm8 rejected its arguments")
    return y


def attn(q_bf16: np.ndarray, k_bf16: np.ndarray, v_bf16: np.ndarray,
         kv_len: int, scale: float, threads: int = 0, mask=None) -> np.ndarray:
    """fp64 [M, Hq, D] verify attention; row i sees slots 0..kv_len-M+i, or,
    with a draft mask (uint32 [M]), every slot before kv_len-M and draft slot
    kv_len-M+j iff bit j of mask[i] is set.

    q_bf16: uint16 [M, Hq, D]; k_bf16, v_bf16: uint16 [Hkv, cap, D], cap >= kv_len.
    """
    q = _c(q_bf16, np.uint16)
    k = _c(k_bf16, np.uint16)
    v = _c(v_bf16, np.uint16)
    M, Hq, D = q.shape
    Hkv, cap, Dk = k.shape
    assert Dk == D and v.shape == k.shape
    o = np.zeros((M, Hq, D), dtype=np.float64)
    if mask is None:
        rc = _lib().oracle_attn(_ptr(q), _ptr(k), _ptr(v), M, Hq, Hkv, D,
                                int(kv_len), int(cap), float(scale), _ptr(o), threads)
    else:
        mk = _c(np.asarray(mask, dtype=np.uint32), np.uint32)
        assert mk.shape == (M,)
        rc = _lib().oracle_attn_masked(_ptr(q), _ptr(k), _ptr(v), M, Hq, Hkv, D, int(kv_len),
                                       int(cap), float(scale), _ptr(mk), _ptr(o), threads)
    if rc != 0:
        raise ValueError("oracle_attn rejected its arguments")
    return o


def dist(z: np.ndarray, temperature: float, top_k: int = 0,
         top_p: float = 1.0) -> np.ndarray:
    """Truncated sampling distribution (fp64, length V) of one fp32 logits row."""
    zz = _c(z, np.float32).ravel()
    p = np.zeros(zz.shape[0], dtype=np.float64)
    rc = _lib().oracle_dist(_ptr(zz), zz.shape[0], float(temperature),
                            int(top_k), float(top_p), _ptr(p))
    if rc != 0:
        raise ValueError("oracle_dist rejected its arguments")
    return p


def accept(target_logits: np.ndarray, draft_logits: np.ndarray,
           draft_tokens: np.ndarray, uniforms: np.ndarray, temperature: float,
           top_k: int = 0, top_p: float = 1.0, threads: int = 0):
    """Run R independent speculative rounds.

    target_logits fp32 [R, K+1, V]; draft_logits fp32 [R, K, V]; draft_tokens
    int32 [R, K]; uniforms fp32 [R, K+1].  Returns (tokens int32 [R, K+1] with
    -1 padding, n_accepted int32 [R]).
    """
    zt = _c(target_logits, np.float32)
    zd = _c(draft_logits, np.float32)
    dt = _c(draft_tokens, np.int32)
    u = _c(uniforms, np.float32)
    R, K1, V = zt.shape
    K = K1 - 1
    assert zd.shape == (R, K, V) and dt.shape == (R, K) and u.shape == (R, K + 1)
    tok = np.full((R, K + 1), -1, dtype=np.int32)
    n = np.zeros((R,), dtype=np.int32)
    rc = _lib().oracle_accept(_ptr(zt), _ptr(zd), _ptr(dt), _ptr(u), R, K, V,
                              float(temperature), int(top_k), float(top_p),
                              _ptr(tok), _ptr(n), threads)
    if rc != 0:
        raise ValueError("oracle_accept rejected its arguments")
    return tok, n


def pick_depth(verify_us, accept, draft_us=None):
    """Depth K in 0..Kmax with the most tokens per microsecond, 0 unless it
    beats plain decoding; returns (K, rates[0..Kmax]).  verify_us[K]: cost of a
    verify pass with K+1 rows; accept[i-1]: P(at least i drafts accepted)."""
    v = _c(verify_us, np.float64).ravel()
    Kmax = v.shape[0] - 1
    a = _c(accept, np.float64).ravel()
    assert a.shape[0] == Kmax
    d = None if draft_us is None else _c(draft_us, np.float64).ravel()
    rates = np.zeros(Kmax + 1, dtype=np.float64)
    k = _lib().oracle_pick_depth(_ptr(v), None if d is None else _ptr(d),
                                 _ptr(a) if Kmax > 0 else None, Kmax, _ptr(rates))
    if k < 0:
        raise ValueError("oracle_pick_depth rejected its arguments")
    return k, rates


def gdn(state, q, k, v, g, beta, tape=None, n_replay=0, threads=0):
    """GatedDeltaNet verify with deferred commit.  state fp32/fp64 [Hv, dv, dk]
    (not modified); q, k bf16 bits [M, Hk, dk]; v bf16 bits [M, Hv, dv]; g, beta
    fp32 [M, Hv]; tape = (k, v, g, beta) of the previous round, of which the
    first n_replay tokens are committed first.  Returns (o fp64 [M, Hv, dv],
    committed state fp64 [Hv, dv, dk])."""
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    Hv, dv, dk = S.shape
    qq, kk, vv = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    gg, bb = _c(g, np.float32), _c(beta, np.float32)
    M, Hk, _ = kk.shape
    if tape is None:
        tk = np.zeros((0, Hk, dk), np.uint16); tv = np.zeros((0, Hv, dv), np.uint16)
        tg = np.zeros((0, Hv), np.float32); tb = np.zeros((0, Hv), np.float32)
    else:
        tk, tv = _c(tape[0], np.uint16), _c(tape[1], np.uint16)
        tg, tb = _c(tape[2], np.float32), _c(tape[3], np.float32)
    assert n_replay <= tk.shape[0]
    o = np.zeros((M, Hv, dv), dtype=np.float64)
    P = lambda a: _ptr(a) if a.size else None
    rc = _lib().oracle_gdn(_ptr(S), P(tk), P(tv), P(tg), P(tb), int(n_replay), P(qq), P(kk), P(vv),
                           P(gg), P(bb), M, Hk, Hv, dk, dv, P(o), threads)
    if rc != 0:
        raise ValueError("oracle_gdn rejected its arguments")
    return o, S
