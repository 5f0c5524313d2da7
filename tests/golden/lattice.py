"""Loader for the hand-built lattice fixture (no method arithmetic here).

Turns ``lattice_figure.json`` into the input arrays of one draft-verify
cycle (fp32 storage, B = 1) and the expected results written in it.
"""
import json
import math
import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
C = 16


def load():
    with open(os.path.join(HERE, "lattice_figure.json")) as f:
        fx = json.load(f)
    vocab = fx["vocab"]
    tok = {w: i for i, w in enumerate(vocab)}
    V, K, H, r = len(vocab), fx["K"], fx["H"], fx["r"]
    h = np.zeros((1, K, H), np.float32)
    for t in range(K):
        h[0, t, t] = 1.0
    w_lm = np.full((V, H), fx["other_logits"], np.float32)
    for t, row in fx["drafter_logits"].items():
        for w, v in row.items():
            w_lm[tok[w], int(t)] = v
    e_in = np.zeros((V, r), np.float32)
    e_out = np.zeros((V, r), np.float32)
    for w, v in fx["e_in"].items():
        e_in[tok[w]] = v
    for w, v in fx["e_out"].items():
        e_out[tok[w]] = v
    L = np.zeros((1, K + 1, V), np.float32)
    for t, w in enumerate(fx["target_argmax"]):
        L[0, t, tok[w]] = 5.0
    ex = fx["expected"]
    e2 = math.e ** 2
    lse = np.array([math.log(e2 + math.e ** 1.8 + math.e + 8),
                    math.log(e2 + math.e ** 1.2 + math.e + 8),
                    math.log(e2 + math.e ** 1.5 + 9)])
    ids = lambda ws: [tok[w] if w is not None else -1 for w in ws]
    return {
        "V": V, "K": K, "H": H, "r": r, "vocab": vocab, "tok": tok,
        "h": h, "w_lm": w_lm, "w_gate": np.zeros((r, H), np.float32),
        "e_in": e_in, "e_out": e_out,
        "anchor": np.array([fx["anchor"]], np.int32), "L": L,
        "lse": lse,
        "topi0_first3": ids(ex["topi_0_first3"]),
        "independent": ids(ex["independent_top1_tokens"]),
        "path_tokens": ids(ex["selector_path_tokens"]),
        "path_slots": ex["selector_path_slots"],
        "path_scores": ex["selector_path_scores"],
        "verify_selector": (ex["greedy_verify_selector"]["n"],
                            ids(ex["greedy_verify_selector"]["out"])),
        "verify_independent": (ex["greedy_verify_independent"]["n"],
                               ids(ex["greedy_verify_independent"]["out"])),
    }
