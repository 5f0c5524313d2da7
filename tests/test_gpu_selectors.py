"""Selector variants and diagnostics: the Viterbi walk (global max-sum path
through the K x 16 lattice) and recall@16 by position, against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import np_, to_dev

pytestmark = pytest.mark.gpu

C = 16


def _lattice(B, K, seed, n_pad=3):
    """Normal(0, 1) pair scores with a few padded candidates (-inf columns,
    as a row with fewer than 16 finite candidates has) and distinct topi."""
    g = np.random.default_rng(seed)
    S = g.normal(size=(B, K, C, C)).astype(np.float32)
    S[:, 0] = S[:, 0, :1]                     # position 0: the anchor's row
    for b in range(0, B, 5):
        S[b, :, :, C - n_pad:] = -np.inf
    topi = g.integers(0, 151936, size=(B, K, C)).astype(np.int32)
    return S, topi


def _run_viterbi(lib, S, topi):
    B, K = S.shape[:2]
    Sd = torch.from_numpy(S).cuda()
    Td = torch.from_numpy(topi).cuda()
    slot = torch.empty(B, K, dtype=torch.int32, device="cuda")
    draft = torch.empty_like(slot)
    q = torch.empty(B, K, C, dtype=torch.float32, device="cuda")
    lib.dflash_path_viterbi(Sd, Td, slot, draft, q)
    torch.cuda.synchronize()
    lib.dflash_check()
    return np_(slot), np_(draft), np_(q)


def _check_viterbi(S, topi, slot, draft, q):
    """The CUDA path must be a maximal path: its float64 total equal to the
    oracle's maximum within the fp32 accumulation error of K sums; where
    the paths differ the two totals are within that band (a near-tie)."""
    o_slot, o_draft, o_q, o_total = oracle.path_viterbi(S.astype(np.float64),
                                                        topi)
    tot = oracle.path_total(S.astype(np.float64), slot)
    K = S.shape[1]
    mag = np.abs(np.where(np.isfinite(S), S, 0)).max(axis=(1, 2, 3))
    band = 4 * K * np.finfo(np.float32).eps * (K * mag + 1)
    assert np.all(np.isfinite(tot))
    assert np.all(np.abs(tot - o_total) <= band)
    same = np.all(slot == o_slot, axis=1)
    assert same.mean() >= 0.99
    B = S.shape[0]
    assert np.array_equal(draft, topi[np.arange(B)[:, None],
                                      np.arange(K)[None, :], slot])
    assert np.array_equal(q, np.eye(C, dtype=np.float32)[slot])
    return same


@pytest.mark.parametrize("B,K", [(1, 1), (3, 2), (37, 8), (4096, 16)])
def test_viterbi_matches_oracle(lib, B, K):
    S, topi = _lattice(B, K, seed=B * 100 + K)
    _check_viterbi(S, topi, *_run_viterbi(lib, S, topi))


def test_viterbi_on_the_drafter_lattice_beats_greedy(lib):
    """On the pair scores the fused drafter wrote, the Viterbi path is
    maximal and its total is at least the greedy walk's."""
    w = synth.get("tiny", T=0.0).with_(B=9, K=6)
    x = synth.make_inputs(w)
    weights = {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                         "e_out")}
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, weights)
    dv.draft_all(to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), 0.0, 1, 0)
    torch.cuda.synchronize()
    S = np_(dv.scores)
    topi = np_(dv.topi).reshape(w.B, w.K, C)
    slot, draft, q = _run_viterbi(lib, S, topi)
    _check_viterbi(S, topi, slot, draft, q)
    greedy = oracle.path_total(S.astype(np.float64), np_(dv.slot))
    vit = oracle.path_total(S.astype(np.float64), slot)
    assert np.all(vit >= greedy - 1e-5 * (1 + np.abs(greedy)))


def test_viterbi_flags_a_sequence_without_a_finite_path(lib):
    S, topi = _lattice(4, 3, seed=7)
    S[2] = -np.inf
    Sd, Td = torch.from_numpy(S).cuda(), torch.from_numpy(topi).cuda()
    slot = torch.empty(4, 3, dtype=torch.int32, device="cuda")
    lib.dflash_path_viterbi(Sd, Td, slot, torch.empty_like(slot),
                            torch.empty(4, 3, C, device="cuda"))
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_check()
    assert e.value.status == 6                  # DFLASH_ERR_BAD_INDEX


def _recall_inputs(B, K, V, seed):
    """Target logits with planted ties at the maximum (the first index must
    win) and candidate lists holding the argmax at about half the rows."""
    g = np.random.default_rng(seed)
    L = g.normal(size=(B, K + 1, V)).astype(np.float32)
    topi = g.integers(0, V, size=(B, K, C)).astype(np.int32)
    for b in range(B):
        for t in range(K):
            if (b + t) % 3 == 0:               # a tie: two equal maxima
                i, j = sorted(g.choice(V, 2, replace=False))
                L[b, t, i] = L[b, t, j] = 9.0
                if t % 2:
                    topi[b, t, g.integers(C)] = j   # the later one: a miss
            if (b * 7 + t) % 2 == 0:
                a = int(np.argmax(L[b, t]))
                topi[b, t, g.integers(C)] = a
    return L, topi


@pytest.mark.parametrize("B,K,V", [(1, 1, 7), (5, 4, 1001), (4, 8, 151936),
                                   (32, 8, 4096)])
def test_top16_recall_matches_oracle(lib, B, K, V):
    L, topi = _recall_inputs(B, K, V, seed=V + B)
    Ld, Td = torch.from_numpy(L).cuda(), torch.from_numpy(topi).cuda()
    arg = torch.empty(B, K, dtype=torch.int32, device="cuda")
    hit = torch.empty_like(arg)
    lib.dflash_top16_recall(Ld, Td, arg, hit)
    torch.cuda.synchronize()
    lib.dflash_check()
    o_arg, o_hit = oracle.top16_recall(L, topi)
    assert np.array_equal(np_(arg), o_arg)
    assert np.array_equal(np_(hit), o_hit)
    from bench import recall_by_position
    recall, accept = recall_by_position(hit)
    assert np.allclose(recall.cpu().numpy(), o_hit.mean(axis=0))
    lead = np.array([np.argmin(np.append(h, 0)) for h in o_hit])
    assert np.isclose(float(accept), lead.mean())


def test_top16_recall_flags_a_nan_logit(lib):
    L, topi = _recall_inputs(2, 2, 64, seed=3)
    L[1, 0, 5] = np.nan
    arg = torch.empty(2, 2, dtype=torch.int32, device="cuda")
    lib.dflash_top16_recall(torch.from_numpy(L).cuda(),
                            torch.from_numpy(topi).cuda(), arg,
                            torch.empty_like(arg))
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_check()
    assert e.value.status != 0
