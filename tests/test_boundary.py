"""The C-ABI library: it builds, loads without a GPU, exports every symbol the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import os
import re

import pytest

from speculative_decoding_verify_08_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def lib():
    path = build_lib.build()
    import speculative_decoding_verify_08_gb300 as sv
    return sv.load()


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"SV_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for n in ("qmm_small_m", "qmm_prepack", "qmm_packed_bytes", "qmm_workspace_bytes",
              "qmm8_small_m", "qmm8_prepack", "qmm8_packed_bytes", "qmm8_workspace_bytes",
              "gdn_verify", "spec_pick_depth",
              "verify_attn", "verify_attn_workspace_bytes", "spec_accept",
              "spec_accept_workspace_bytes", "sv_status_string", "sv_last_device_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(build_lib.LIB)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_status_strings(lib):
    import speculative_decoding_verify_08_gb300 as sv
    for code in range(7):
        assert sv.sv_status_string(code) and sv.sv_status_string(code) != "unknown status"
    assert sv.sv_status_string(99) == "unknown status"


def test_packed_bytes(lib):
    assert lib.qmm_packed_bytes(1024, 512, 64) == 64 * 8 * 576
    assert lib.qmm_packed_bytes(17, 128, 64) == 1 * 2 * 8 * 576  # rows padded to 128
    assert lib.qmm_packed_bytes(16, 100, 64) == 0            # K not a multiple of 64
    assert lib.qmm_packed_bytes(16, 128, 32) == 0            # group 32 unsupported
    assert lib.qmm_packed_bytes(0, 128, 64) == 0
    # 8-bit: 1024 code bytes + 64 scale/bias bytes per 16-row tile and group
    assert lib.qmm8_packed_bytes(1024, 512, 64) == 64 * 8 * 1088  # tiles x groups x 1088
    assert lib.qmm8_packed_bytes(17, 128, 64) == 1 * 2 * 8 * 1088
    assert lib.qmm8_packed_bytes(16, 100, 64) == 0
    assert lib.qmm8_packed_bytes(16, 128, 32) == 0


A = 256  # a 16-byte aligned stand-in pointer value; never dereferenced


def test_qmm_rejects_on_host(lib):
    f = lib.qmm_small_m
    assert f(None, A, A, 0, 4, 64, 64, 64, None, 0, None) == 1
    assert f(A, A, A, 0, 0, 64, 64, 64, None, 0, None) == 1     # M = 0
    assert f(A, A, A, 7, 4, 64, 64, 64, None, 0, None) == 1     # bad dtype
    assert f(A, A, A, 0, 17, 64, 64, 64, None, 0, None) == 2    # M > 16
    assert f(A, A, A, 0, 4, 64, 96, 64, None, 0, None) == 2     # K % 64
    assert f(A, A, A, 0, 4, 64, 64, 32, None, 0, None) == 2     # group
    assert f(A + 2, A, A, 0, 4, 64, 64, 64, None, 0, None) == 1  # misaligned x
    p = lib.qmm_prepack
    assert p(None, A, A, 16, 64, 64, A, 576, None) == 1
    assert p(A, A, A, 16, 64, 64, A, 100, None) == 1            # buffer too small
    assert p(A, A, A, 16, 64, 32, A, 576, None) == 2
    f8 = lib.qmm8_small_m
    assert f8(None, A, A, 0, 4, 64, 64, 64, None, 0, None) == 1
    assert f8(A, A, A, 0, 17, 64, 64, 64, None, 0, None) == 2   # M > 16
    assert f8(A, A, A, 0, 4, 64, 96, 64, None, 0, None) == 2    # K % 64
    assert f8(A + 2, A, A, 0, 4, 64, 64, 64, None, 0, None) == 1  # misaligned x
    p8 = lib.qmm8_prepack
    assert p8(A, A, A, 16, 64, 64, A, 8 * 576, None) == 1       # a 4-bit-sized buffer is too small
    assert p8(A, A, A, 16, 64, 32, A, 8 * 1088, None) == 2


def test_attn_rejects_on_host(lib):
    f = lib.verify_attn
    assert f(None, A, A, A, 4, 4, 1, 128, 256, 256, 0.1, A, 1 << 20, None) == 1
    assert f(A, A, A, A, 4, 6, 4, 128, 256, 256, 0.1, A, 1 << 20, None) == 1   # Hq % Hkv
    assert f(A, A, A, A, 4, 4, 1, 128, 3, 256, 0.1, A, 1 << 20, None) == 1     # L < M
    assert f(A, A, A, A, 4, 4, 1, 128, 300, 256, 0.1, A, 1 << 20, None) == 1   # stride < L
    assert f(A, A, A, A, 4, 4, 1, 128, 256, 256, -1.0, A, 1 << 20, None) == 1  # scale
    assert f(A, A, A, A, 4, 4, 1, 64, 256, 256, 0.1, A, 1 << 20, None) == 2    # D
    assert f(A, A, A, A, 17, 24, 4, 256, 256, 256, 0.1, A, 1 << 20, None) == 2  # 102 rows


def test_masked_attn_rejects_on_host(lib):
    f = lib.verify_attn_masked
    assert f(A, A, A, A, 4, 4, 1, 128, 256, 256, 0.1, None, A, 1 << 20, None) == 1    # no mask
    assert f(A, A, A, A, 4, 4, 1, 128, 256, 256, 0.1, A + 2, A, 1 << 20, None) == 1   # misaligned
    assert f(A, A, A, A, 33, 1, 1, 128, 256, 256, 0.1, A, A, 1 << 20, None) == 2      # M > 32
    assert f(A, A, A, A, 4, 6, 4, 128, 256, 256, 0.1, A, A, 1 << 20, None) == 1       # Hq % Hkv


def test_gdn_rejects_on_host(lib):
    f = lib.gdn_verify
    args = lambda **kw: [kw.get("state", A), kw.get("tk", None), kw.get("tv", None), kw.get("tg", None),
                         kw.get("tb", None), kw.get("n", 0), A, A, A, A, A, A, kw.get("odt", 0),
                         kw.get("M", 4), kw.get("Hk", 2), kw.get("Hv", 4), kw.get("dk", 128),
                         kw.get("dv", 128), None]
    assert f(*args(state=None)) == 1
    assert f(*args(M=0)) == 1                      # nothing to do
    assert f(*args(Hv=6, Hk=4)) == 1               # Hv % Hk
    assert f(*args(dk=96)) == 2                    # unsupported key dim
    assert f(*args(n=2)) == 1                      # replay without a tape
    assert f(*args(odt=7)) == 1
    assert f(*args(state=A + 4)) == 1              # misaligned state
    assert f(*args(M=65)) == 2                     # more than 64 verify rows


def test_accept_rejects_on_host(lib):
    import speculative_decoding_verify_08_gb300 as sv

    def call(T=1.0, k=0, p=1.0, R=2, K=3, V=100, ws=None, wsb=0, dt=1):
        sp = sv._Sampling(T, k, p)
        return lib.spec_accept(A, A, dt, A, A, sp, R, K, V, A, A, ws, wsb, None)

    assert call(T=-1.0) == 1
    assert call(T=float("nan")) == 1
    assert call(p=0.0) == 1
    assert call(p=1.5) == 1
    assert call(k=-1) == 1
    assert call(R=0) == 1
    assert call(dt=5) == 1
    assert call(K=33) == 2
    assert call(k=0, V=5000) == 5                                # whole vocabulary, no workspace
    assert call(k=2000, V=100000) == 5                           # large top-k, no workspace
    assert call(k=20, V=152064) == 5                             # no workspace
    assert call(T=0.0, V=152064, ws=A, wsb=10) == 5              # workspace too small
    assert call(T=1e-35, V=100, ws=A, wsb=1 << 40) == 2          # log2(e)/T beyond 2^100
    # Without a device the library plans one chunk per row (with one, the
    # chunk counts follow its SM count).  Candidate-list path: counters +
    # lists; whole-vocabulary path: row headers, round jobs, counters and
    # chunk sums, and (V > 4096) bucket counts and band lists per row
    import torch
    if not torch.cuda.is_available():
        rows = 256 * 7
        lists = 7168 + rows * (16 + 21 * 2048)
        whole = rows * 128 + 256 * 16 + 1024 + 256 * 16 + rows * (8192 * 4 + 4096 * 8)
        assert lib.spec_accept_workspace_bytes(256, 3, 152064) == lists + whole
    small = 2 * 7 * 128 + 256 + 256 + 256
    lists2 = (256 + 2 * 7 * (16 + 21 * 2048) + 255) // 256 * 256
    assert lib.spec_accept_workspace_bytes(2, 3, 1000) == lists2 + small


def test_fused_lm_head_rejects_on_host(lib):
    import speculative_decoding_verify_08_gb300 as sv

    def topk(T=0.6, k=20, p=0.95, M=4, N=152064, K=5120, lists=A, y=A):
        return lib.qmm_small_m_topk(A, A, y, M, N, K, 64, sv._Sampling(T, k, p), lists, 1 << 30,
                                    A, 1 << 30, None)

    assert topk(y=None) == 1
    assert topk(M=0) == 1
    assert topk(T=-1.0) == 1
    assert topk(M=17) == 2
    assert topk(k=0) == 2                    # top-k off: the logits path
    assert topk(k=2000) == 2                 # beyond the candidate lists
    assert topk(T=0.0, k=0, lists=A + 4) == 1  # greedy is supported; misaligned lists

    def acc(T=0.6, k=20, p=0.95, ws=A, wsb=1 << 40, lists=A):
        return lib.spec_accept_lists(lists, None, A, A, sv._Sampling(T, k, p), 1, 3, 152064, A, A,
                                     ws, wsb, None)

    assert acc(lists=None) == 1
    assert acc(k=0) == 2
    assert acc(k=2000) == 2
    assert acc(ws=None, wsb=0) == 5
    assert acc(lists=A + 8) == 1
    assert lib.spec_accept_lists(A, A + 4, A, A, sv._Sampling(0.6, 20, 0.95), 1, 3, 152064, A, A,
                                 A, 1 << 40, None) == 1   # misaligned draft lists

    def drafts(T=0.6, k=20, p=0.95, ws=A, wsb=1 << 40, logits=A, dt=1):
        return lib.spec_accept_draft_select(logits, dt, sv._Sampling(T, k, p), 1, 3, 152064, ws, wsb,
                                            None)

    assert drafts(logits=None) == 1
    assert drafts(dt=4) == 1
    assert drafts(k=0) == 2
    assert drafts(ws=None, wsb=0) == 5


def test_launch_flags(lib):
    import speculative_decoding_verify_08_gb300 as sv
    old = sv.sv_get_launch_flags()
    sv.sv_set_launch_flags(sv.SV_LAUNCH_PDL)
    assert sv.sv_get_launch_flags() == sv.SV_LAUNCH_PDL
    sv.sv_set_launch_flags(0xFF | sv.SV_LAUNCH_TEST_STALL_COPY)
    assert sv.sv_get_launch_flags() & sv.SV_LAUNCH_TEST_STALL_COPY
    sv.sv_set_launch_flags(0xFF)
    assert sv.sv_get_launch_flags() == (sv.SV_LAUNCH_PDL | sv.SV_LAUNCH_QMM_CUDA_CORES |
                                        sv.SV_LAUNCH_ATTN_MMA_SYNC | sv.SV_LAUNCH_ATTN_TCGEN05)  # unknown bits dropped
    sv.sv_set_launch_flags(old)
