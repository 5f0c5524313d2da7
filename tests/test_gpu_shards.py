"""Vocabulary shards on one GPU: the vocabulary is split into S contiguous
ranges, each shard's calls run in turn on its own slices (as separate
devices would hold them), and the merged results are compared with the
oracle on the whole vocabulary (the sharded decomposition must not change
what the path computes) and with the library's own whole-vocabulary calls."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (ERR_C, check_topk, check_verify, draft_logits_oracle, f64,
                    np_, to_dev)

pytestmark = pytest.mark.gpu
C = 16


def _bounds(V, S, rng):
    """S contiguous ranges of uneven sizes covering [0, V), one of them
    shorter than 16 tokens when S > 2."""
    if S == 1:
        return [0, V]
    cuts = sorted(rng.choice(np.arange(20, V - 20), S - 1, replace=False))
    b = [0] + [int(c) for c in cuts] + [V]
    if S > 2:
        b[2] = b[1] + 7            # a shard of 7 tokens
    return b


def _weights(x):
    return {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out")}


@pytest.mark.parametrize("S,dtype", [(1, "bf16"), (2, "bf16"), (4, "bf16"),
                                     (3, "fp32")])
def test_lmhead_shards_merge_to_the_whole_vocabulary(lib, S, dtype):
    B, K, H, V = 5, 4, (192 if dtype == "bf16" else 64), 5003
    w = synth.Workload("shards", B=B, K=K, V=V, H=H, r=32, dtype=dtype,
                       T=1.0, seed=61 + S, w_lm_sd=0.1, conv_sd=0.05,
                       sel_sd=0.1, target=("affine", 0.9, 1.0))
    x = synth.make_inputs(w)
    h = to_dev(x["h"][:, :K])
    wc, wl = to_dev(x["w_conv"]), to_dev(x["w_lm"])
    M = B * K
    bnd = _bounds(V, S, np.random.default_rng(S))
    pv = torch.empty(S, M, C, device="cuda")
    pi = torch.empty(S, M, C, dtype=torch.int32, device="cuda")
    pm = torch.empty(S, M, device="cuda")
    ps = torch.empty(S, M, device="cuda")
    ys = []
    for s in range(S):
        v0, v1 = bnd[s], bnd[s + 1]
        ws = torch.empty(lib.dflash_workspace_bytes(0, B, K, H, v1 - v0),
                         dtype=torch.uint8, device="cuda")
        lib.dflash_lmhead_topk_shard(h, wc, wl[v0:v1].contiguous(), v0, pv[s],
                                     pi[s], pm[s], ps[s], ws)
        es = 2 if dtype == "bf16" else 4
        ys.append(ws[:M * H * es].view(h.dtype).clone())
    topv = torch.empty(M, C, device="cuda")
    topi = torch.empty(M, C, dtype=torch.int32, device="cuda")
    lse = torch.empty(M, device="cuda")
    lib.dflash_topk_merge_shards(pv, pi, pm, ps, topv, topi, lse)
    torch.cuda.synchronize()
    lib.dflash_check()
    for y in ys[1:]:                  # every shard computed the same y
        assert torch.equal(y, ys[0])
    y64 = f64(ys[0]).reshape(M, H)
    W64 = f64(x["w_lm"])
    ref = oracle.lmhead_topk(y64, W64, want_logits=True)
    A = np.abs(y64) @ np.abs(W64).T
    check_topk(topv, topi, lse, ref, A, ERR_C[dtype])
    # and the whole-vocabulary call: the same logits, so the same candidates
    dv = lib.DraftVerify(B, K, H, V, w.r, _weights(x))
    dv.lmhead(h)
    torch.cuda.synchronize()
    assert torch.equal(dv.topi, topi)
    assert torch.equal(dv.topv, topv)
    np.testing.assert_allclose(np_(lse), np_(dv.lse), rtol=2e-6, atol=0)


def _sharded_verify(lib, L, draft, topi, q, T, seed, cycle, bnd):
    B, K1, V = L.shape
    K = K1 - 1
    S = len(bnd) - 1
    stats = torch.empty(S, B * K1, lib.SHARD_STATS, device="cuda")
    parts, wss = [], []
    for s in range(S):
        v0, v1 = bnd[s], bnd[s + 1]
        Ls = L[:, :, v0:v1].contiguous()
        ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, v1 - v0),
                         dtype=torch.uint8, device="cuda")
        lib.dflash_verify_shard_stats(Ls, draft, topi, v0, V, T, stats[s], ws)
        parts.append(Ls)
        wss.append(ws)
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, K1), -7, dtype=torch.int32, device="cuda")
    plan = torch.empty(B, lib.SHARD_PLAN, device="cuda")
    lib.dflash_verify_shard_decide(stats, draft, topi, q, V, T, seed, cycle,
                                   n, out, plan)
    for s in range(S):
        lib.dflash_verify_shard_draw(parts[s], plan, topi, q, s, bnd[s], T,
                                     out, wss[s])
    torch.cuda.synchronize()
    lib.dflash_check()
    return n, out


@pytest.mark.parametrize("S,T,V", [(1, 1.0, 4099), (2, 1.0, 4099),
                                   (3, 0.7, 4099), (5, 1.0, 20011),
                                   (3, 0.0, 4099), (4, 1.0, 3001)])
def test_verify_shards_match_the_oracle(lib, S, T, V):
    """Drafts from the library's own draft step; target logits built so
    that some drafts are accepted and the draws fall in every shard."""
    w = synth.Workload("vshards", B=24, K=6, V=V, H=128, r=32, dtype="bf16",
                       T=T, seed=71 + S, w_lm_sd=0.3, conv_sd=0.05,
                       sel_sd=0.1, target=("affine", 1.0, 0.4))
    x = synth.make_inputs(w)
    L = to_dev(synth.target_logits(w, draft_logits_oracle(x, w)))
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x))
    seed, cycle = 13, 2
    dv.draft_all(to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), T, seed,
                 cycle)
    topi = dv.topi.view(w.B, w.K, C)
    bnd = _bounds(V, S, np.random.default_rng(100 + S))
    n, out = _sharded_verify(lib, L, dv.draft, topi, dv.q, T, seed, cycle,
                             bnd)
    ties, o_n, o_out = check_verify(n, out, np_(L), np_(dv.draft), np_(topi),
                                    np_(dv.q), T, seed, cycle)
    # the whole-vocabulary verify decides the same, but for near-ties of
    # either against the oracle
    dv.verify(L, T, seed, cycle)
    torch.cuda.synchronize()
    ties_whole, _, _ = check_verify(dv.n, dv.out, np_(L), np_(dv.draft),
                                    np_(topi), np_(dv.q), T, seed, cycle)
    same = (np_(dv.n) == np_(n)) & np.all(np_(dv.out) == np_(out), axis=1)
    assert same.sum() >= w.B - ties - ties_whole
    owners = set()
    for b in range(w.B):
        tok = int(np_(out)[b, int(np_(n)[b])])
        owners.add(int(np.searchsorted(bnd, tok, side="right") - 1))
    print(f"S={S} T={T} mean accepted {np_(n).mean():.2f} ties {ties} "
          f"shards drawn from {sorted(owners)}")
    assert np.all(np_(out) >= -1)


def test_verify_shards_full_size_b32k8cal(lib):
    """The calibrated b32k8 workload (about 4.5 accepted drafts per cycle)
    with V = 151936 split over 4 shards."""
    w = synth.get("b32k8cal")
    x = synth.make_inputs(w)
    L = to_dev(synth.target_logits(w, draft_logits_oracle(x, w)))
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x))
    seed, cycle = w.seed, 0
    dv.draft_all(to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), w.T, seed,
                 cycle)
    topi = dv.topi.view(w.B, w.K, C)
    bnd = [0, 37984, 75968, 113952, w.V]
    n, out = _sharded_verify(lib, L, dv.draft, topi, dv.q, w.T, seed, cycle,
                             bnd)
    ties, _, _ = check_verify(n, out, np_(L), np_(dv.draft), np_(topi),
                              np_(dv.q), w.T, seed, cycle)
    print("b32k8cal over 4 shards: mean accepted", np_(n).mean(), "ties",
          ties)
    assert np_(n).mean() > 2.0
