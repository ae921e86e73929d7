"""Benchmark of the K=3 verify step on GB300.

One step = the data-parallel verify pass of a 27B-class model with M = 4
rows (last token + 3 drafts): 64 layers of 4-bit projections (qkv 5120->6144,
o 5120->5120, gate+up 5120->34816, down 17408->5120), 16 verify-attention
layers over a 32K-slot bf16 KV cache (24 query heads, 4 KV heads, head dim
256), the 4-bit lm_head (5120->152064, fp32 logits) and the exact acceptance
of 3 drafts at T=0.6, top-k 20, top-p 0.95.  Weights, caches and activations
are synthetic and random (seeded); 14.3 GB of weights and KV are read per
step, far more than L2, so no L2 flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same step and extrapolates to one step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("µs per K=3 verify step + achieved HBM GB/s (% of GB300 peak), "
          "M=4/8 vs M=1")

# workload: 27B-class verify step, M = K + 1 = 4 rows
HIDDEN, FFN, QKV, VOCAB = 5120, 17408, 6144, 152064
LAYERS, ATTN_LAYERS = 64, 16
HQ, HKV, HD, CTX = 24, 4, 256, 32768
KD, T_SAMPLE, TOP_K, TOP_P = 3, 0.6, 20, 0.95
M = KD + 1
PROJ = [("qkv", HIDDEN, QKV), ("o", HIDDEN, HIDDEN), ("gate_up", HIDDEN, 2 * FFN),
        ("down", FFN, HIDDEN)]  # (name, K, N)
FALLBACK_PEAK_GBS = 6800.0


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_PEAK_GBS, "fallback"


def qmm_bytes(M_, N, K, out_bytes):
    return N * K // 2 + N * (K // 64) * 4 + M_ * K * 2 + M_ * N * out_bytes


def qmm8_bytes(M_, N, K, out_bytes):
    return N * K + N * (K // 64) * 4 + M_ * K * 2 + M_ * N * out_bytes


# GatedDeltaNet layers of the hybrid 27B-class target (48 recurrent layers):
# 16 key heads, 48 value heads, 128 x 128 fp32 state per value head
GDN_LAYERS, GDN_HK, GDN_HV, GDN_DK, GDN_DV = 48, 16, 48, 128, 128
GDN_REPLAY = 3  # tokens committed per round (the round's first row + 2 accepted drafts)


def gdn_bytes(M_, n_replay):
    state = GDN_HV * GDN_DV * GDN_DK * 4
    per_tok = (2 * GDN_HK * GDN_DK + GDN_HV * GDN_DV) * 2 + 2 * GDN_HV * 4
    return 2 * state + n_replay * (GDN_HK * GDN_DK + GDN_HV * GDN_DV) * 2 + n_replay * 2 * GDN_HV * 4 + \
        M_ * per_tok + M_ * GDN_HV * GDN_DV * 2


def attn_bytes(M_, L):
    return 4 * L * HKV * HD + 4 * M_ * HQ * HD


def accept_bytes(R, K, V):
    return 4 * R * (2 * K + 1) * V + 16 * R * (K + 1)


# the timed workload, named the same by both arms
WORKLOAD = ("27B-class K=3 verify step: 64x{qkv 5120->6144, o 5120->5120, gate+up 5120->34816, "
            "down 17408->5120} 4-bit g64 qmm at M=4, 16x verify_attn (24q/4kv heads, d256, 32K ctx, "
            "M=4), 4-bit lm_head 5120->152064 fp32 logits, spec_accept (V=152064, T=0.6, top-k 20, "
            "top-p 0.95)")


def step_bytes():
    b = 0
    for _, K, N in PROJ:
        b += LAYERS * qmm_bytes(M, N, K, 2)
    b += ATTN_LAYERS * attn_bytes(M, CTX)
    b += qmm_bytes(M, VOCAB, HIDDEN, 4)
    b += accept_bytes(1, KD, VOCAB)
    return b


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        sm = []
        for p in rows:
            try:
                sm.append(float(p[1]))
            except ValueError:
                pass
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        try:
            smax = float(rows[-1][2])
        except ValueError:
            smax = None
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------- the model --
class VerifyStep:
    """All device buffers of one verify step and the launch sequence."""

    def __init__(self, sv, seed=0, keep_layer0_host=False, fused=False):
        from speculative_decoding_verify_08_gb300 import synth
        self.sv = sv
        # the lm_head selects the target rows' top-k in its epilogue and the
        # acceptance merges those lists (qmm_small_m_topk + spec_accept_lists)
        self.fused = fused
        dev = torch.device("cuda")
        self.dev = dev
        self.layer0_host = {}
        self.weights = []  # [layer][proj] packed
        for layer in range(LAYERS):
            per = []
            for pi, (name, K, N) in enumerate(PROJ):
                t = synth.qmm_inputs(1, N, K, seed=seed * 1000 + layer * 4 + pi, device=dev)
                per.append(sv.prepack(t["codes"], t["scales"], t["biases"]))
                if keep_layer0_host and layer == 0:
                    self.layer0_host[name] = {k: v.cpu() for k, v in t.items() if k != "x"}
                del t
            self.weights.append(per)
        t = synth.qmm_inputs(1, VOCAB, HIDDEN, seed=seed * 1000 + 999, device=dev)
        self.lm_head = sv.prepack(t["codes"], t["scales"], t["biases"])
        if keep_layer0_host:
            self.layer0_host["lm_head"] = {k: v.cpu() for k, v in t.items() if k != "x"}
        del t
        torch.cuda.synchronize()
        self.kv = []
        for a in range(ATTN_LAYERS):
            kvt = synth.attn_inputs(M, HQ, HKV, HD, CTX, seed=seed * 100 + a, device=dev)
            self.kv.append((kvt["k"], kvt["v"]))
            if a == 0:
                self.q_host = kvt["q"].cpu()
                if keep_layer0_host:
                    self.layer0_host["attn"] = {"k": kvt["k"].cpu(), "v": kvt["v"].cpu()}
        g = torch.Generator(device=dev)
        g.manual_seed(seed + 7)
        self.x_hidden = (torch.randn((M, HIDDEN), generator=g, device=dev)).to(torch.bfloat16)
        self.x_ffn = (torch.randn((M, FFN), generator=g, device=dev)).to(torch.bfloat16)
        self.q = self.q_host.to(dev)
        self.y = {name: torch.empty((M, N), dtype=torch.bfloat16, device=dev) for name, _, N in PROJ}
        self.attn_out = torch.empty((M, HQ, HD), dtype=torch.bfloat16, device=dev)
        self.logits = torch.empty((M, VOCAB), dtype=torch.float32, device=dev)
        acc = synth.accept_inputs(1, KD, VOCAB, synth.ACCEPT_BATCH_SIGMA, T_SAMPLE, top_k=TOP_K,
                                  seed=seed + 11, device=dev)
        self.uniforms = acc["uniforms"]
        # the drafter: the MTP head's own lm_head over its hidden states (the
        # target's input rows plus noise), run before the verify pass; its
        # epilogue makes the draft rows' top-k lists beside the draft logits
        gd = torch.Generator(device=dev)
        gd.manual_seed(seed + 13)
        self.x_draft = (self.x_hidden[:KD].float() +
                        0.3 * torch.randn((KD, HIDDEN), generator=gd, device=dev)).to(torch.bfloat16)
        self.draft_lists = torch.zeros(sv.qmm_topk_lists_bytes(KD, VOCAB, HIDDEN), dtype=torch.uint8,
                                       device=dev)
        yd = torch.empty((KD, VOCAB), dtype=torch.float32, device=dev)
        ws_d = sv.workspace(sv.qmm_workspace_bytes(KD, VOCAB, HIDDEN))
        sv.qmm_small_m_topk(self.x_draft, self.lm_head, yd, KD, VOCAB, HIDDEN, T_SAMPLE, TOP_K, TOP_P,
                            self.draft_lists, ws_d)
        self.draft_logits = yd.view(1, KD, VOCAB)
        self.draft_tokens = synth.synthetic_drafter(self.draft_logits, T_SAMPLE, TOP_K, seed=seed + 13)
        # tokens and count side by side, so the host reads the result in one copy
        self.out = torch.empty((KD + 2,), dtype=torch.int32, device=dev)
        self.out_tokens = self.out[:KD + 1].view(1, KD + 1)
        self.out_n = self.out[KD + 1:]
        # workspaces (one per projection shape, one per attention, one for acceptance)
        self.ws = {name: sv.workspace(sv.qmm_workspace_bytes(M, N, K)) for name, K, N in PROJ}
        self.ws["lm_head"] = sv.workspace(sv.qmm_workspace_bytes(M, VOCAB, HIDDEN))
        self.ws_attn = sv.workspace(sv.verify_attn_workspace_bytes(M, HQ, HKV, HD, CTX))
        self.ws_acc = sv.workspace(sv.spec_accept_workspace_bytes(1, KD, VOCAB))
        self.lists = torch.zeros(sv.qmm_topk_lists_bytes(M, VOCAB, HIDDEN), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def qmm(self, layer, pi):
        name, K, N = PROJ[pi]
        x = self.x_ffn if name == "down" else self.x_hidden
        self.sv.qmm_small_m(x, self.weights[layer][pi], self.y[name], M, N, K, self.ws[name])

    def attn(self, a, M_=M, L=CTX, q=None, o=None, ws=None):
        k, v = self.kv[a]
        self.sv.verify_attn(self.q if q is None else q, k, v, self.attn_out if o is None else o,
                            M_, HQ, HKV, HD, L, CTX, 1.0 / math.sqrt(HD),
                            self.ws_attn if ws is None else ws)

    def lm_head_call(self, fused=None):
        if self.fused if fused is None else fused:
            self.sv.qmm_small_m_topk(self.x_hidden, self.lm_head, self.logits, M, VOCAB, HIDDEN,
                                     T_SAMPLE, TOP_K, TOP_P, self.lists, self.ws["lm_head"])
        else:
            self.sv.qmm_small_m(self.x_hidden, self.lm_head, self.logits, M, VOCAB, HIDDEN,
                                self.ws["lm_head"])

    def draft_select(self):
        self.sv.spec_accept_draft_select(self.draft_logits, T_SAMPLE, TOP_K, TOP_P, 1, KD, VOCAB,
                                         self.ws_acc)

    def accept(self, fused=None):
        if self.fused if fused is None else fused:
            self.sv.spec_accept_lists(self.lists, self.draft_tokens, self.uniforms, T_SAMPLE, TOP_K,
                                      TOP_P, 1, KD, VOCAB, self.out_tokens, self.out_n, self.ws_acc,
                                      draft_lists=self.draft_lists)
        else:
            self.sv.spec_accept(self.logits.view(1, M, VOCAB), self.draft_logits, self.draft_tokens,
                                self.uniforms, T_SAMPLE, TOP_K, TOP_P, 1, KD, VOCAB, self.out_tokens,
                                self.out_n, self.ws_acc)

    def run_layers(self):
        a = 0
        for layer in range(LAYERS):
            self.qmm(layer, 0)
            if layer % (LAYERS // ATTN_LAYERS) == LAYERS // ATTN_LAYERS - 1:
                self.attn(a)
                a += 1
            for pi in (1, 2, 3):
                self.qmm(layer, pi)

    def run_tail(self):
        self.lm_head_call()
        self.accept()

    def run(self):
        self.run_layers()
        self.run_tail()


def capture(fn, pdl=True, extra_flags=0):
    """CUDA graph of fn(); PDL launch attributes when possible (extra_flags
    are OR-ed into the library's launch flags during the capture)."""
    import speculative_decoding_verify_08_gb300 as sv
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    old = sv.sv_get_launch_flags()
    sv.sv_set_launch_flags(old | extra_flags)
    with torch.cuda.stream(s):
        fn()  # warm (sets smem attributes, tensor-map entry point)
    torch.cuda.synchronize()
    for use_pdl in ([True, False] if pdl else [False]):
        sv.sv_set_launch_flags((sv.SV_LAUNCH_PDL if use_pdl else 0) | extra_flags)
        g = torch.cuda.CUDAGraph()
        try:
            c0 = sv.sv_kernel_launch_count()
            with torch.cuda.graph(g, stream=s):
                fn()
            launches = sv.sv_kernel_launch_count() - c0
            sv.sv_set_launch_flags(old)
            return g, launches, use_pdl
        except RuntimeError:
            torch.cuda.synchronize()
            continue
    sv.sv_set_launch_flags(old)
    raise RuntimeError("graph capture failed")


def time_graph(g, reps, warmup):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(reps):
        g.replay()
    e1.record(s)
    e1.synchronize()
    return e0.elapsed_time(e1) / reps  # ms per replay


# dram__bytes_read.sum + dram__bytes_write.sum of one gate+up launch at M=4
# (whole batches per CTA), from an ncu capture of
#   python bench.py --only qmm_gate_up --m 4 --steps 3
# (100,391,936 B read + 2,862,592 B written).  Set back to None whenever the
# qmm kernel or its launch plan changes.
GATE_UP_DRAM_BYTES = 103254528


# launches per timed graph in the kernel table (at least 100, each weight or
# cache copy reused only after all the others, so nothing is served from L2)
QMM_PASSES = 2        # x 64 distinct matrices = 128 launches
ATTN_PASSES = 7       # x 16 distinct caches = 112 launches
SINGLE_LAUNCHES = 100  # lm_head (438 MB, larger than L2) and acceptance


def kernel_table(step, sweep=True):
    """Per-kernel launch time (events around graphs of at least 100 launches
    over distinct weights / caches) and M ratios."""
    sv = step.sv
    res = {}
    # projections at M=4: one launch per layer (64 distinct matrices)
    for pi, (name, K, N) in enumerate(PROJ):
        g, n, _ = capture(lambda: [step.qmm(l, pi) for _ in range(QMM_PASSES) for l in range(LAYERS)])
        ms = time_graph(g, 3, 2)
        t_us = ms * 1e3 / (QMM_PASSES * LAYERS)
        b = qmm_bytes(M, N, K, 2)
        res[f"qmm_{name}_M4"] = {"us": t_us, "gbs": b / t_us / 1e3, "bytes": b}
        del g
    g, n, _ = capture(lambda: [step.attn(a) for _ in range(ATTN_PASSES) for a in range(ATTN_LAYERS)])
    ms = time_graph(g, 3, 2)
    t_us = ms * 1e3 / (ATTN_PASSES * ATTN_LAYERS)
    b = attn_bytes(M, CTX)
    res["verify_attn_M4_32K"] = {"us": t_us, "gbs": b / t_us / 1e3, "bytes": b}
    del g
    # GatedDeltaNet verify with the previous round's commit, one launch per
    # recurrent layer (48 distinct states, 151 MB), three passes
    from speculative_decoding_verify_08_gb300 import synth
    dev = step.dev
    gi = synth.gdn_inputs(M, GDN_HK, GDN_HV, GDN_DK, GDN_DV, seed=5, device=dev)
    states = [torch.randn((GDN_HV, GDN_DV, GDN_DK), device=dev) * 0.1 for _ in range(GDN_LAYERS)]
    go = torch.empty((M, GDN_HV, GDN_DV), dtype=torch.bfloat16, device=dev)
    tape = (gi["k"], gi["v"], gi["g"], gi["beta"])
    g, n, _ = capture(lambda: [sv.gdn_verify(st, gi["q"], gi["k"], gi["v"], gi["g"], gi["beta"], go,
                                             tape=tape, n_replay=GDN_REPLAY)
                               for _ in range(3) for st in states])
    ms = time_graph(g, 3, 1) / (3 * GDN_LAYERS)
    b = gdn_bytes(M, GDN_REPLAY)
    res["gdn_verify_M4"] = {"us": ms * 1e3, "gbs": b / (ms * 1e3) / 1e3, "bytes": b}
    del g, states
    b = qmm_bytes(M, VOCAB, HIDDEN, 4)
    for label, fused in (("qmm_lm_head_M4", False), ("qmm_lm_head_topk_M4", True)):
        g, n, _ = capture(lambda: [step.lm_head_call(fused) for _ in range(SINGLE_LAUNCHES)])
        ms = time_graph(g, 2, 1) / SINGLE_LAUNCHES
        res[label] = {"us": ms * 1e3, "gbs": b / (ms * 1e3) / 1e3, "bytes": b}
        del g
    b = accept_bytes(1, KD, VOCAB)
    # (spec_accept_lists_R1: every row's set merged from the target's and the
    # drafter's lists, the distributions and the chain)
    for label, fused in (("spec_accept_R1", False), ("spec_accept_lists_R1", True)):
        g, n, _ = capture(lambda: [step.accept(fused) for _ in range(SINGLE_LAUNCHES)])
        ms = time_graph(g, 2, 1) / SINGLE_LAUNCHES
        res[label] = {"us": ms * 1e3, "gbs": b / (ms * 1e3) / 1e3, "bytes": b}
        del g
    res.update(accept_table(step))
    if not sweep:
        return res, {}
    ratios = {}
    dev = step.dev
    for pi, (name, K, N) in enumerate(PROJ):
        times = {}
        for Mx in (1, 2, 3, 4, 8, 16):
            x = torch.randn((Mx, K), device=dev).to(torch.bfloat16)
            y = torch.empty((Mx, N), dtype=torch.bfloat16, device=dev)
            ws = step.ws[name]
            g, _, _ = capture(lambda: [sv.qmm_small_m(x, step.weights[l][pi], y, Mx, N, K, ws)
                                       for _ in range(QMM_PASSES) for l in range(LAYERS)])
            times[Mx] = time_graph(g, 3, 1) * 1e3 / (QMM_PASSES * LAYERS)
            del g
        ratios[f"qmm_{name}"] = {"us": {str(k): round(v, 3) for k, v in times.items()},
                                 "ratio_vs_M1": {str(k): round(v / times[1], 3) for k, v in times.items()},
                                 "gbs_M8": round(qmm_bytes(8, N, K, 2) / times[8] / 1e3, 1)}
    # tensor cores against CUDA-core FFMA on the same kernel (gate+up, M = 1, 4)
    name, K, N = PROJ[2]
    cmp = {}
    for Mx in (1, 4):
        x = torch.randn((Mx, K), device=dev).to(torch.bfloat16)
        y = torch.empty((Mx, N), dtype=torch.bfloat16, device=dev)
        ws = step.ws[name]
        for label, fl in (("tensor_core_mma", 0), ("cuda_core_ffma", sv.SV_LAUNCH_QMM_CUDA_CORES)):
            g, _, _ = capture(lambda: [sv.qmm_small_m(x, step.weights[l][2], y, Mx, N, K, ws)
                                       for _ in range(QMM_PASSES) for l in range(LAYERS)],
                              extra_flags=fl)
            us = time_graph(g, 3, 1) * 1e3 / (QMM_PASSES * LAYERS)
            cmp[f"{label}_M{Mx}"] = {"us": round(us, 3), "gbs": round(qmm_bytes(Mx, N, K, 2) / us / 1e3, 1)}
            del g
    ratios["qmm_gate_up_tensor_vs_cuda_cores"] = cmp
    # the 8-bit pack: gate+up and down, four distinct matrices each (more
    # than L2 together), rotated over 128 launches
    from speculative_decoding_verify_08_gb300 import synth
    for name, K, N in (PROJ[2], PROJ[3]):
        mats = []
        for c in range(4):
            t = synth.qmm_inputs(1, N, K, seed=900 + c, device=dev, bits=8)
            mats.append(sv.prepack(t["codes"], t["scales"], t["biases"], bits=8))
            del t
        ws8 = sv.workspace(max(sv.qmm8_workspace_bytes(Mx, N, K) for Mx in (1, 16)))
        times = {}
        for Mx in (1, 2, 4, 8, 16):
            x = torch.randn((Mx, K), device=dev).to(torch.bfloat16)
            y = torch.empty((Mx, N), dtype=torch.bfloat16, device=dev)
            g, _, _ = capture(lambda: [sv.qmm8_small_m(x, mats[i % 4], y, Mx, N, K, ws8) for i in range(128)])
            times[Mx] = time_graph(g, 3, 1) * 1e3 / 128
            del g
        ratios[f"qmm8_{name}"] = {"us": {str(k): round(v, 3) for k, v in times.items()},
                                  "ratio_vs_M1": {str(k): round(v / times[1], 3) for k, v in times.items()},
                                  "gbs_M8": round(qmm8_bytes(8, N, K, 2) / times[8] / 1e3, 1)}
        del mats, ws8
    for L in (8192, 32768, 131072):
        times = {}
        for Mx in (1, 2, 3, 4, 8, 16):
            q = torch.randn((Mx, HQ, HD), device=dev).to(torch.bfloat16)
            o = torch.empty((Mx, HQ, HD), dtype=torch.bfloat16, device=dev)
            ws = sv.workspace(sv.verify_attn_workspace_bytes(Mx, HQ, HKV, HD, min(L, CTX)))
            if L <= CTX:
                g, _, _ = capture(lambda: [step.attn(a, Mx, L, q, o, ws) for _ in range(ATTN_PASSES)
                                           for a in range(ATTN_LAYERS)])
                times[Mx] = time_graph(g, 3, 1) * 1e3 / (ATTN_PASSES * ATTN_LAYERS)
            else:
                times[Mx] = long_ctx_attn(step, Mx, L, q, o)
            del ws
        ratios[f"verify_attn_{L // 1024}K"] = {
            "us": {str(k): round(v, 3) for k, v in times.items()},
            "ratio_vs_M1": {str(k): round(v / times[1], 3) for k, v in times.items()},
            "gbs_M8": round(attn_bytes(8, L) / times[8] / 1e3, 1)}
    # Draft depth per context from these cost curves (spec_pick_depth): a
    # verify pass with M = K+1 rows costs the 64 layers' projections and the
    # 16 attention layers at M rows plus the lm_head and the acceptance; a
    # drafted token costs one pass of the model's own MTP head (one decoder
    # layer and the lm_head at one row); acceptance is the pages' reported
    # MTPLX per-position profile (at least 1, 2, 3 drafts accepted).
    accept = [0.73, 0.48, 0.32]
    qsum = {Mx: sum(ratios[f"qmm_{n}"]["us"][str(Mx)] for n, _, _ in PROJ) for Mx in (1, 2, 3, 4)}
    head = res["qmm_lm_head_M4"]["us"]
    table = {}
    for L in (8192, 32768, 131072):
        a = ratios[f"verify_attn_{L // 1024}K"]["us"]
        verify = [LAYERS * qsum[K + 1] + ATTN_LAYERS * a[str(K + 1)] + head + res["spec_accept_R1"]["us"]
                  for K in range(len(accept) + 1)]
        draft = [K * (qsum[1] + a["1"] + head) for K in range(len(accept) + 1)]
        k, rates = sv.spec_pick_depth(verify, accept, draft)
        table[f"{L // 1024}K"] = {"verify_us": [round(v, 1) for v in verify],
                                  "draft_us": [round(d, 1) for d in draft],
                                  "tokens_per_ms": [round(r * 1e3, 3) for r in rates],
                                  "depth": int(k), "speedup_vs_plain": round(rates[k] / rates[0], 3)}
    ratios["depth_table"] = {"accept_at_least": accept, "contexts": table}
    return res, ratios


# acceptance settings timed on their own: the 256-round batch (top-k 20,
# candidate lists) and the whole-vocabulary path (top-k off, or top-k 5000)
ACCEPT_SETTINGS = [("k20_p095_T06", 0.6, 20, 0.95), ("whole_T1", 1.0, 0, 1.0),
                   ("whole_p095_T06", 0.6, 0, 0.95), ("whole_k5000_p09_T08", 0.8, 5000, 0.9)]
ACCEPT_R1_COPIES = 120  # x 4.26 MB of logits: four times L2, read in turn


def accept_table(step):
    """spec_accept per call: R = 256 rounds (1.09 GB of logits per call, more
    than L2) and R = 1 round rotated over 120 distinct input sets."""
    sv = step.sv
    from speculative_decoding_verify_08_gb300 import synth
    dev = step.dev
    res = {}
    for R, copies in ((256, 1), (1, ACCEPT_R1_COPIES)):
        for label, T, k, p in ACCEPT_SETTINGS:
            sets = [synth.accept_inputs(R, KD, VOCAB, synth.ACCEPT_BATCH_SIGMA, T, top_k=k,
                                        seed=700 + c, device=dev) for c in range(copies)]
            tok = torch.empty((R, KD + 1), dtype=torch.int32, device=dev)
            n = torch.empty((R,), dtype=torch.int32, device=dev)
            ws = sv.workspace(sv.spec_accept_workspace_bytes(R, KD, VOCAB))
            calls = 10 if R > 1 else copies
            g, _, _ = capture(lambda: [sv.spec_accept(a["target"], a["draft"], a["draft_tokens"],
                                                      a["uniforms"], T, k, p, R, KD, VOCAB, tok, n, ws)
                                       for a in (sets * calls)[:calls]])
            ms = time_graph(g, 2, 1) / calls
            b = accept_bytes(R, KD, VOCAB)
            res[f"spec_accept_R{R}_{label}"] = {"us": ms * 1e3, "gbs": b / (ms * 1e3) / 1e3, "bytes": b}
            del g, sets, ws
    # the small-vocabulary case (V = 1000, 3 drafts, temperature 1, no
    # truncation, 16 rounds per call), rotated over 120 input sets
    R, V = 16, 1000
    sets = [synth.accept_inputs(R, KD, V, (1.0, 1.0, 1.0), 1.0, seed=800 + c, device=dev)
            for c in range(ACCEPT_R1_COPIES)]
    tok = torch.empty((R, KD + 1), dtype=torch.int32, device=dev)
    n = torch.empty((R,), dtype=torch.int32, device=dev)
    ws = sv.workspace(sv.spec_accept_workspace_bytes(R, KD, V))
    g, _, _ = capture(lambda: [sv.spec_accept(a["target"], a["draft"], a["draft_tokens"], a["uniforms"],
                                              1.0, 0, 1.0, R, KD, V, tok, n, ws) for a in sets])
    ms = time_graph(g, 2, 1) / len(sets)
    b = accept_bytes(R, KD, V)
    res["spec_accept_R16_V1000_T1"] = {"us": ms * 1e3, "gbs": b / (ms * 1e3) / 1e3, "bytes": b}
    del g, sets, ws
    assert sv.sv_last_device_error() == sv.SV_OK
    return res


_LONG = {}


def long_ctx_attn(step, Mx, L, q, o):
    """128K-slot caches: four distinct 537 MB caches (more than L2) in turn."""
    sv = step.sv
    from speculative_decoding_verify_08_gb300 import synth
    if L not in _LONG:
        caches = []
        for c in range(4):
            t = synth.attn_inputs(1, HQ, HKV, HD, L, seed=500 + c, device=step.dev)
            caches.append((t["k"], t["v"]))
        _LONG[L] = caches
    caches = _LONG[L]
    ws = sv.workspace(sv.verify_attn_workspace_bytes(Mx, HQ, HKV, HD, L))
    g, _, _ = capture(lambda: [sv.verify_attn(q, k, v, o, Mx, HQ, HKV, HD, L, L,
                                              1.0 / math.sqrt(HD), ws) for (k, v) in caches * 25])
    t = time_graph(g, 2, 1) * 1e3 / 100
    del g
    return t


# ---------------------------------------------------------- CPU oracle ---
def cpu_oracle_sample(step_host, budget_s=25.0):
    """Time the oracle on the host cores on a bounded sample of one step and
    extrapolate to a whole step."""
    import oracle
    from speculative_decoding_verify_08_gb300 import synth
    oracle.build()
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    parts = {}
    t_total = 0.0
    # projections of one layer, on a slice of output columns each
    frac_cols = 1.0 / 16
    for name, K, N in PROJ:
        h = step_host[name]
        cols = max(16, int(N * frac_cols))
        x = (torch.randn((M, K)) ).to(torch.bfloat16)
        t0 = time.perf_counter()
        oracle.qmm(synth.bf16_bits(x), synth.u32_bits(h["codes"][:cols]),
                   synth.bf16_bits(h["scales"][:cols]), synth.bf16_bits(h["biases"][:cols]),
                   threads=threads)
        dt = (time.perf_counter() - t0) * N / cols
        parts[f"qmm_{name}"] = dt
        t_total += LAYERS * dt
    h = step_host["lm_head"]
    cols = VOCAB // 64
    x = torch.randn((M, HIDDEN)).to(torch.bfloat16)
    t0 = time.perf_counter()
    oracle.qmm(synth.bf16_bits(x), synth.u32_bits(h["codes"][:cols]),
               synth.bf16_bits(h["scales"][:cols]), synth.bf16_bits(h["biases"][:cols]), threads=threads)
    dt = (time.perf_counter() - t0) * VOCAB / cols
    parts["qmm_lm_head"] = dt
    t_total += dt
    # one attention layer on one KV head's query group (rows of 1 of 4 heads)
    a = step_host["attn"]
    q = torch.randn((M, HQ // HKV, HD)).to(torch.bfloat16)
    t0 = time.perf_counter()
    oracle.attn(synth.bf16_bits(q), synth.bf16_bits(a["k"][:1]), synth.bf16_bits(a["v"][:1]), CTX,
                1.0 / math.sqrt(HD), threads=threads)
    dt = (time.perf_counter() - t0) * HKV
    parts["verify_attn"] = dt
    t_total += ATTN_LAYERS * dt
    acc = synth.accept_inputs(1, KD, VOCAB, synth.ACCEPT_BATCH_SIGMA, T_SAMPLE, top_k=TOP_K, seed=3)
    t0 = time.perf_counter()
    oracle.accept(acc["target"].numpy(), acc["draft"].numpy(), acc["draft_tokens"].numpy(),
                  acc["uniforms"].numpy(), float(np.float32(T_SAMPLE)), TOP_K,
                  float(np.float32(TOP_P)), threads=threads)
    dt = time.perf_counter() - t0
    parts["spec_accept"] = dt
    t_total += dt
    sample = ("one layer's 4 projections on 1/16 of their output columns, the lm_head on 1/64, "
              "one 32K attention layer on 1 of 4 KV heads, one acceptance round; "
              "scaled to 64 + 1 + 16 + 1 calls of one step")
    return t_total * 1e6, threads, sample, {k: round(v * 1e6, 1) for k, v in parts.items()}


def host_step_inputs():
    """Host copy of a synthetic verify step for the reference arm (no GPU)."""
    from speculative_decoding_verify_08_gb300 import synth
    out = {}
    for pi, (name, K, N) in enumerate(PROJ):
        cols = max(16, N // 16)
        t = synth.qmm_inputs(1, cols, K, seed=pi)
        out[name] = {k: v for k, v in t.items() if k != "x"}
    t = synth.qmm_inputs(1, VOCAB // 64, HIDDEN, seed=9)
    out["lm_head"] = {k: v for k, v in t.items() if k != "x"}
    a = synth.attn_inputs(1, HQ // HKV, 1, HD, CTX, seed=5)
    out["attn"] = {"k": a["k"], "v": a["v"]}
    return out


def max_over_ranks(x, dist, device):
    """Largest x over all ranks (the slowest replica sets the job's time);
    x itself when not distributed."""
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_step(ms_max, world):
    """Whole-job microseconds per verify step: each of the `world` replicas
    completes one step every ms_max milliseconds."""
    return ms_max * 1e3 / world


def run_reference(args, rank, world):
    """The CPU oracle as the reference arm; under torchrun rank 0 alone runs
    and prints, the other ranks exit at once."""
    if rank != 0:
        return
    host = host_step_inputs()
    for _ in range(args.warmup):
        cpu_oracle_sample(host)  # untimed
    vals = []
    info = None
    for _ in range(max(1, args.steps)):
        us, cores, sample, parts = cpu_oracle_sample(host)
        vals.append(us)
        info = (cores, sample, parts)
    v = statistics.median(vals)
    cores, sample, parts = info
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us/step",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "bytes_per_step": step_bytes(),
                   "l2": "n/a (CPU)", "parallelism": "host cores"},
        "cpu_baseline": {"value": round(v, 1), "unit": "us/step", "cores": cores,
                         "kind": "oracle", "sample": sample, "parts_us": parts},
        "e2e": {"value": round(v, 1), "unit": "us/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ----------------------------------------------------- one-kernel runs ---
def run_only(args):
    """A few launches of one kernel at its full-size workload shape (for
    profiler captures of a small, single-kernel program)."""
    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_08_gb300 as sv
    from speculative_decoding_verify_08_gb300 import synth
    dev = torch.device("cuda")
    reps = max(1, args.steps)
    if args.cuda_cores:
        sv.sv_set_launch_flags(sv.sv_get_launch_flags() | sv.SV_LAUNCH_QMM_CUDA_CORES)
    if args.attn_kernel != "auto":
        bit = sv.SV_LAUNCH_ATTN_MMA_SYNC if args.attn_kernel == "mma_sync" else sv.SV_LAUNCH_ATTN_TCGEN05
        sv.sv_set_launch_flags(sv.sv_get_launch_flags() | bit)
    name = args.only
    if name == "qmm_lm_head_topk":
        # the lm_head with the acceptance's top-k lists in its epilogue
        Mx = args.m
        mats = []
        for c in range(3):
            t = synth.qmm_inputs(Mx, VOCAB, HIDDEN, seed=c, device=dev)
            mats.append(sv.prepack(t["codes"], t["scales"], t["biases"]))
            x = t["x"]
        ws = sv.workspace(sv.qmm_workspace_bytes(Mx, VOCAB, HIDDEN))
        y = torch.empty((Mx, VOCAB), dtype=torch.float32, device=dev)
        lists = torch.zeros(sv.qmm_topk_lists_bytes(Mx, VOCAB, HIDDEN), dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()
        for i in range(reps):
            sv.qmm_small_m_topk(x, mats[i % 3], y, Mx, VOCAB, HIDDEN, T_SAMPLE, TOP_K, TOP_P, lists, ws)
    elif name.startswith("qmm_") or name.startswith("qmm8_"):
        bits = 8 if name.startswith("qmm8_") else 4
        proj = {p[0]: p for p in PROJ}
        proj["lm_head"] = ("lm_head", HIDDEN, VOCAB)
        _, K, N = proj[name.split("_", 1)[1]]
        Mx = args.m
        mats = []
        for c in range(3):
            t = synth.qmm_inputs(Mx, N, K, seed=c, device=dev, bits=bits)
            mats.append(sv.prepack(t["codes"], t["scales"], t["biases"], bits=bits))
            x = t["x"]
        ws = sv.workspace((sv.qmm_workspace_bytes if bits == 4 else sv.qmm8_workspace_bytes)(Mx, N, K))
        y = torch.empty((Mx, N), dtype=torch.bfloat16, device=dev)
        run = sv.qmm_small_m if bits == 4 else sv.qmm8_small_m
        torch.cuda.synchronize()
        for i in range(reps):
            run(x, mats[i % 3], y, Mx, N, K, ws)
    elif name == "verify_attn":
        Mx, L = args.m, args.ctx
        caches = [synth.attn_inputs(Mx, HQ, HKV, HD, L, seed=c, device=dev) for c in range(2)]
        o = torch.empty((Mx, HQ, HD), dtype=torch.bfloat16, device=dev)
        ws = sv.workspace(sv.verify_attn_workspace_bytes(Mx, HQ, HKV, HD, L))
        torch.cuda.synchronize()
        for i in range(reps):
            c = caches[i % 2]
            sv.verify_attn(c["q"], c["k"], c["v"], o, Mx, HQ, HKV, HD, L, L, 1.0 / math.sqrt(HD), ws)
    elif name == "gdn_verify":
        gi = synth.gdn_inputs(args.m, GDN_HK, GDN_HV, GDN_DK, GDN_DV, seed=5, device=dev)
        states = [torch.randn((GDN_HV, GDN_DV, GDN_DK), device=dev) * 0.1 for _ in range(4)]
        o = torch.empty((args.m, GDN_HV, GDN_DV), dtype=torch.bfloat16, device=dev)
        tape = (gi["k"], gi["v"], gi["g"], gi["beta"])
        torch.cuda.synchronize()
        for i in range(reps):
            sv.gdn_verify(states[i % 4], gi["q"], gi["k"], gi["v"], gi["g"], gi["beta"], o, tape=tape,
                          n_replay=min(GDN_REPLAY, args.m))
    elif name == "spec_accept":
        R = args.rounds
        _, T, k, p = {lab: (lab, T, k, p) for lab, T, k, p in ACCEPT_SETTINGS}[args.accept]
        a = synth.accept_inputs(R, KD, VOCAB, synth.ACCEPT_BATCH_SIGMA, T, top_k=k,
                                seed=1, device=dev)
        tok = torch.empty((R, KD + 1), dtype=torch.int32, device=dev)
        n = torch.empty((R,), dtype=torch.int32, device=dev)
        ws = sv.workspace(sv.spec_accept_workspace_bytes(R, KD, VOCAB))
        torch.cuda.synchronize()
        for i in range(reps):
            sv.spec_accept(a["target"], a["draft"], a["draft_tokens"], a["uniforms"], T, k, p,
                           R, KD, VOCAB, tok, n, ws)
    else:
        raise SystemExit(f"unknown --only {name}")
    torch.cuda.synchronize()
    assert sv.sv_last_device_error() == sv.SV_OK
    print(json.dumps({"only": name, "launches": reps}), flush=True)


# ------------------------------------------------------------------ main --
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-table", action="store_true", help="skip the per-kernel table")
    ap.add_argument("--only", default=None,
                    help="run one kernel only: qmm_{qkv,o,gate_up,down,lm_head}, qmm8_{...}, qmm_lm_head_topk, "
                         "verify_attn, gdn_verify, "
                         "spec_accept (for profiler captures)")
    ap.add_argument("--m", type=int, default=M, help="rows for --only")
    ap.add_argument("--ctx", type=int, default=CTX, help="KV slots for --only verify_attn")
    ap.add_argument("--attn-kernel", default="auto", choices=["auto", "mma_sync", "tcgen05"],
                    help="--only verify_attn: force one of the two attention kernels")
    ap.add_argument("--cuda-cores", action="store_true",
                    help="--only qmm_*: the CUDA-core FFMA comparison path (M = 1 or 4)")
    ap.add_argument("--rounds", type=int, default=256, help="rounds for --only spec_accept")
    ap.add_argument("--accept", default=ACCEPT_SETTINGS[0][0], choices=[a[0] for a in ACCEPT_SETTINGS],
                    help="sampling setting for --only spec_accept")
    args = ap.parse_args()
    if args.only:
        run_only(args)
        return
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import __graft_entry__
    __graft_entry__.build()
    import speculative_decoding_verify_08_gb300 as sv
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    peak, peak_kind = measured_peaks()

    step = VerifyStep(sv, seed=rank, keep_layer0_host=(rank == 0 and not args.no_cpu))
    graph, launches_per_step, pdl = capture(step.run)
    for _ in range(max(3, args.warmup)):
        graph.replay()
    torch.cuda.synchronize()
    assert sv.sv_last_device_error() == sv.SV_OK

    # ---- timed region: K replays of the whole step ----
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(s)
        for _ in range(args.steps):
            graph.replay()
        e1.record(s)
        e1.synchronize()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dist, "cuda")
    if dist:
        dist.barrier()
    clocks = clk.summary()
    # the same step with the lm_head fused with the acceptance's top-k
    # selection (qmm_small_m_topk, spec_accept_lists on the target's and the
    # drafter's lists); the timed step above keeps them unfused, which
    # measures as fast or faster at one round
    step.fused = True
    graph_f, _, _ = capture(step.run)
    step.fused = False
    ms_fused = time_graph(graph_f, args.steps, 3)
    del graph_f

    # ---- end to end: pinned host inputs in, tokens out, every step ----
    # The step replays as two graphs here: the layers, then the lm_head and
    # the acceptance.  The activation rows are copied first; the drafter's
    # logits, tokens and the uniforms, which only the acceptance reads, are
    # copied on a second stream while the layers run.
    tok_graph, n_graph = step.out_tokens.cpu(), step.out_n.cpu()
    graph_layers, _, _ = capture(step.run_layers)
    graph_tail, _, _ = capture(step.run_tail)
    side = torch.cuda.Stream()
    h_x = step.x_hidden.cpu().pin_memory()
    h_draft = step.draft_logits.cpu().pin_memory()
    h_dtok = step.draft_tokens.cpu().pin_memory()
    h_u = step.uniforms.cpu().pin_memory()
    h_out = torch.empty_like(step.out, device="cpu").pin_memory()
    h_tok, h_n = h_out[:KD + 1].view(1, KD + 1), h_out[KD + 1:]
    bi = sum(t.numel() * t.element_size() for t in (h_x, h_draft, h_dtok, h_u))
    bo = h_tok.numel() * 4 + h_n.numel() * 4
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    cur = torch.cuda.current_stream()

    def e2e_step():
        # (the previous step ended with a synchronize, so the side stream's
        # copies cannot overwrite inputs that its acceptance still reads)
        step.x_hidden.copy_(h_x, non_blocking=True)
        graph_layers.replay()
        with torch.cuda.stream(side):
            step.draft_logits.copy_(h_draft, non_blocking=True)
            step.draft_tokens.copy_(h_dtok, non_blocking=True)
            step.uniforms.copy_(h_u, non_blocking=True)
        cur.wait_stream(side)
        graph_tail.replay()
        h_out.copy_(step.out, non_blocking=True)
        cur.synchronize()

    for _ in range(max(3, args.warmup)):
        e2e_step()
    e2.record(s)
    for _ in range(args.steps):
        e2e_step()
    e3.record(s)
    e3.synchronize()
    e2e_ms = max_over_ranks(e2.elapsed_time(e3) / args.steps, dist, "cuda")
    assert sv.sv_last_device_error() == sv.SV_OK
    assert torch.equal(h_tok, tok_graph) and torch.equal(h_n, n_graph), "e2e tokens differ"

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return

    kernels, ratios, roofline = {}, {}, None
    if not args.no_table:
        kernels, ratios = kernel_table(step, sweep=not args.no_sweep)
        dom = "qmm_gate_up_M4"
        kd = kernels[dom]
        roofline = {"kernel": "qmm_small_m gate+up (5120->34816) M=4", "bound": "hbm",
                    "achieved": round(kd["gbs"], 1), "peak": peak, "unit": "GB/s",
                    "frac": round(kd["gbs"] / peak, 4), "traffic": GATE_UP_DRAM_BYTES,
                    "peak_kind": peak_kind, "bytes_per_launch": kd["bytes"],
                    "us_per_launch": round(kd["us"], 3)}
    sb = step_bytes()
    us = ms * 1e3
    value = job_us_per_step(ms, world)
    cpu = None
    if not args.no_cpu:
        cus, cores, sample, parts = cpu_oracle_sample(step.layer0_host)
        cpu = {"value": round(cus, 1), "unit": "us/step", "cores": cores, "kind": "oracle",
               "sample": sample, "parts_us": parts}
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "us/step", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD,
                   "bytes_per_step": sb, "graph_launches_per_step": launches_per_step,
                   "pdl": pdl, "l2": "inputs larger than L2 (14.3 GB read per step)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "hbm_gbs": round(sb / us / 1e3, 1), "hbm_frac_of_peak": round(sb / us / 1e3 / peak, 4),
        "roofline_step_us": round(sb / (peak * 1e3), 1),
        "step_us_lm_head_fused": round(ms_fused * 1e3, 2),
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": round(job_us_per_step(e2e_ms, world), 2), "unit": "us/step",
                "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
        "kernels": {k: {"us": round(v["us"], 3), "gbs": round(v["gbs"], 1)} for k, v in kernels.items()},
        "m_sweep": ratios,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
