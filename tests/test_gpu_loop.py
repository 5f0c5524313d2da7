"""The draft-verify loop over many cycles: dflash_draft, dflash_verify and
dflash_commit with the anchor handed over from cycle to cycle, against the
oracle's loop (every cycle: new hidden states and target logits)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import draft_logits_oracle, f64, np_, to_dev

pytestmark = pytest.mark.gpu


def _weights(x):
    return {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out")}


def _cycle_inputs(w, base, c):
    """Hidden states of cycle c (their own seed) with the shared weights,
    and the target logits built from them."""
    wc = w.with_(seed=1000 + c)
    x = dict(base)
    x["h"] = synth.make_inputs(wc)["h"]
    L = synth.target_logits(wc, draft_logits_oracle(x, w))
    return x, L


@pytest.mark.parametrize("name,T", [("tiny", 0.0), ("tiny", 1.0),
                                    ("tiny_conv", 1.0)])
def test_loop_matches_oracle(lib, name, T):
    w = synth.get(name, T=T).with_(B=6)
    base = synth.make_inputs(w)
    B, K, cap, cycles, seed = w.B, w.K, 64, 10, 3
    dv = lib.DraftVerify(B, K, w.H, w.V, w.r, _weights(base))
    anchor_d = to_dev(base["anchor"]).clone()
    tokens_d = torch.full((B, cap), -1, dtype=torch.int32, device="cuda")
    length_d = torch.zeros(B, dtype=torch.int32, device="cuda")
    stats_d = torch.zeros(lib.COMMIT_STATS, dtype=torch.int64, device="cuda")
    anchor_o = np_(base["anchor"]).astype(np.int64)
    tokens_o = np.full((B, cap), -1, np.int64)
    length_o = np.zeros(B, np.int64)
    stats_o = np.zeros(lib.COMMIT_STATS, np.int64)
    for c in range(cycles):
        x, L = _cycle_inputs(w, base, c)
        dv.draft_all(to_dev(x["h"][:, :K]), anchor_d, T, seed, c)
        dv.verify(to_dev(L), T, seed, c)
        dv.commit(anchor_d, tokens_d, length_d, stats_d)
        r = oracle.draft_verify_cycle(
            f64(x["h"][:, :K]), f64(x["w_conv"]), f64(x["w_lm"]),
            f64(x["w_gate"]), f64(x["e_in"]), f64(x["e_out"]),
            anchor_o.copy(), np_(L), T, seed, c, w.dtype)
        oracle.commit(r["n"], r["out"], anchor_o, tokens_o, length_o, stats_o)
    torch.cuda.synchronize()
    lib.dflash_check()
    assert np.array_equal(np_(length_d), length_o)
    assert np.array_equal(np_(anchor_d), anchor_o)
    assert np.array_equal(np_(tokens_d), tokens_o)
    assert np.array_equal(np_(stats_d), stats_o)
    assert stats_o[1] == B * cycles


def test_commit_flags_a_full_buffer_and_a_bad_count(lib):
    B, K, cap = 2, 3, 4
    n = torch.tensor([3, 2], dtype=torch.int32, device="cuda")
    out = torch.tensor([[1, 2, 3, 4], [5, 6, 7, -1]], dtype=torch.int32,
                       device="cuda")
    anchor = torch.zeros(B, dtype=torch.int32, device="cuda")
    tokens = torch.full((B, cap), -1, dtype=torch.int32, device="cuda")
    length = torch.tensor([2, 0], dtype=torch.int32, device="cuda")
    stats = torch.zeros(lib.COMMIT_STATS, dtype=torch.int64, device="cuda")
    lib.dflash_commit(n, out, anchor, tokens, length, stats)
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_check()
    assert e.value.status == 6                  # DFLASH_ERR_BAD_INDEX
    assert np_(tokens).tolist() == [[-1, -1, 1, 2], [5, 6, 7, -1]]
    assert np_(length).tolist() == [6, 3] and np_(anchor).tolist() == [4, 7]
    bad = torch.tensor([5, 0], dtype=torch.int32, device="cuda")
    lib.dflash_commit(bad, out, anchor, tokens, length, stats)
    with pytest.raises(lib.DFlashError):
        lib.dflash_check()
    assert np_(length).tolist() == [6, 4]       # sequence 0 left unchanged
    s = np_(stats)
    assert s[:3].tolist() == [5, 3, 8]
