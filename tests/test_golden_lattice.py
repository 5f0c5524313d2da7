"""The lattice figure of "DFlash 2: Keep Drafting Parallel" as a worked case.

Independent top-1 picks repeat a word; the pair selector walks the coherent
path; greedy verify accepts it.  Expected values are derived by hand in
tests/golden/lattice_figure.json.
"""
import numpy as np

import oracle
from golden import lattice


def test_oracle_reproduces_hand_derived_lattice():
    fx = lattice.load()
    K, H = fx["K"], fx["H"]
    topv, topi, lse = oracle.lmhead_topk(fx["h"][0].astype(np.float64),
                                         fx["w_lm"])
    assert list(topi[0, :3]) == fx["topi0_first3"]
    assert list(topi[0, fx["V"]:]) == [-1] * (16 - fx["V"])
    # 1.8 and 1.2 are stored in fp32: agree to that resolution
    np.testing.assert_allclose(lse, fx["lse"], rtol=1e-7)
    topv = topv.reshape(1, K, 16)
    topi = topi.reshape(1, K, 16)
    g = oracle.gate(fx["h"], fx["w_gate"])
    S = oracle.pair_score(topv, topi, fx["anchor"], g, fx["e_in"],
                          fx["e_out"]).astype(np.float32)
    slot, draft, q, _ = oracle.path_walk(S, topi, 0.0, None)
    assert list(slot[0]) == fx["path_slots"]
    assert list(draft[0]) == fx["path_tokens"]
    prev = 0
    for t in range(K):
        np.testing.assert_allclose(S[0, t, prev, slot[0, t]],
                                   fx["path_scores"][t], rtol=1e-6)
        prev = slot[0, t]
    # zeroed selector: independent top-1 (the same word twice)
    E0 = np.zeros_like(fx["e_in"])
    S0 = oracle.pair_score(topv, topi, fx["anchor"], g, E0, E0)
    _, d0, q0, _ = oracle.path_walk(S0.astype(np.float32), topi, 0.0, None)
    assert list(d0[0]) == fx["independent"]
    n, out, _ = oracle.verify(fx["L"], draft, topi, q, 0.0, None, None)
    assert (int(n[0]), list(out[0])) == fx["verify_selector"]
    n, out, _ = oracle.verify(fx["L"], d0, topi, q0, 0.0, None, None)
    assert (int(n[0]), list(out[0])) == fx["verify_independent"]
