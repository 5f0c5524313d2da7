"""Find the W_lm scale at which the b32k8 generator gives a mean acceptance
of 4 to 5 draft tokens per cycle (test infrastructure; uses the oracle).

With the literal generator (W_lm ~ N(0, 0.02)) the drafter's logits have a
standard deviation of about 0.9 over 151936 tokens, the target's softmax is
nearly flat, and almost no draft is accepted.  Scaling the standard
deviation of W_lm by s sharpens both distributions; this script bisects s
on the oracle's full cycle (same seeds as b32k8, the first `--seqs`
sequences) and prints the result, which synth records as the workload
"b32k8cal" (scale 4*sqrt(2) = 5.657: mean 4.5 accepted over the 32
sequences).  Run: python tests/calibrate_b32k8.py --seqs 32 --lo 4 --hi 8
"""
import argparse
import math
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import oracle  # noqa: E402
import synth  # noqa: E402
from parity import draft_logits_oracle, f64  # noqa: E402


def mean_accepted(s, seqs):
    base = synth.get("b32k8")
    w = base.with_(w_lm_sd=base.w_lm_sd * s)
    x = synth.make_inputs(w)
    L = synth.target_logits(w, draft_logits_oracle(x, w))
    sub = slice(0, seqs)
    r = oracle.draft_verify_cycle(
        f64(x["h"][sub, :w.K]), f64(x["w_conv"]), f64(x["w_lm"]),
        f64(x["w_gate"]), f64(x["e_in"]), f64(x["e_out"]),
        np.asarray(x["anchor"][sub]), np.asarray(L[sub]), w.T, w.seed, 0,
        w.dtype)
    return float(np.mean(r["n"]))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--seqs", type=int, default=8)
    ap.add_argument("--lo", type=float, default=1.0)
    ap.add_argument("--hi", type=float, default=64.0)
    ap.add_argument("--iters", type=int, default=8)
    a = ap.parse_args()
    lo, hi = math.log(a.lo), math.log(a.hi)
    for _ in range(a.iters):
        mid = 0.5 * (lo + hi)
        n = mean_accepted(math.exp(mid), a.seqs)
        print(f"s = {math.exp(mid):8.3f}  mean accepted {n:.3f}", flush=True)
        if 4.0 <= n <= 5.0:
            break
        if n < 4.0:
            lo = mid
        else:
            hi = mid
    print(f"scale {math.exp(mid):.4f}")


if __name__ == "__main__":
    main()
