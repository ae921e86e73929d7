"""Calibrate the draft-logit noise of the 256-round acceptance batch.

Target logits ~ N(0, 3) over a 152064-token vocabulary; draft logits = target +
N(0, sigma).  With temperature 0.6, top-k 20 and top-p 0.95 applied to both
sides, find per draft depth the sigma whose mean per-row acceptance
sum_j min(p_j, q_j) is 0.95, 0.88 and 0.80 -- the per-depth acceptance quoted
for the 27B pack in "The fastest way to run local LLMs on a Mac", section "Why
native MTP doubles decode".

Calls only the CPU oracle (oracle.dist).  Writes accept_sigma.json beside this
file; the synthetic-input module carries the same numbers as constants and a
CPU test checks that the two agree.

    python tests/golden/calibrate_sigma.py [--rounds 48]
"""
import argparse
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402

V, T, TOP_K, TOP_P = 152064, 0.6, 20, 0.95
TARGETS = (0.95, 0.88, 0.80)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--rounds", type=int, default=48)
    ap.add_argument("--seed", type=int, default=2024)
    args = ap.parse_args()
    rng = np.random.default_rng(args.seed)
    zt = (rng.standard_normal((args.rounds, V)) * 3.0).astype(np.float32)
    eps = rng.standard_normal((args.rounds, V)).astype(np.float32)
    ps = [oracle.dist(zt[r], T, TOP_K, TOP_P) for r in range(args.rounds)]

    def alpha(sigma):
        acc = 0.0
        for r in range(args.rounds):
            q = oracle.dist((zt[r] + np.float32(sigma) * eps[r]).astype(np.float32), T, TOP_K, TOP_P)
            acc += float(np.minimum(ps[r], q).sum())
        return acc / args.rounds

    sigmas, measured = [], []
    for target in TARGETS:
        lo, hi = 0.0, 4.0
        for _ in range(22):
            mid = 0.5 * (lo + hi)
            if alpha(mid) > target:
                lo = mid
            else:
                hi = mid
        s = round(0.5 * (lo + hi), 4)
        sigmas.append(s)
        measured.append(round(alpha(s), 4))
        print(f"target {target:.2f}: sigma {s:.4f} -> mean acceptance {measured[-1]:.4f}")
    out = {
        "what": "draft-logit noise sigma per depth for the acceptance batch",
        "vocab": V, "temperature": T, "top_k": TOP_K, "top_p": TOP_P,
        "target_std": 3.0, "rounds": args.rounds, "seed": args.seed,
        "target_acceptance": list(TARGETS), "sigma": sigmas,
        "measured_acceptance": measured,
    }
    with open(os.path.join(HERE, "accept_sigma.json"), "w") as f:
        json.dump(out, f, indent=1)


if __name__ == "__main__":
    main()
