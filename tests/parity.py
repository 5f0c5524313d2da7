"""Comparison helpers for the GPU parity tests (tie-aware, stage-wise).

Each stage of the CUDA path is compared with the oracle run on the CUDA
path's own upstream outputs.  Integer results (indices, slots, lengths,
tokens) must be identical except where the oracle's own margin at that
decision is below the stated epsilon; such cases are counted as ties and the
CUDA choice must then be one of the near-equal alternatives.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from oracle import philox

C = 16
# Tie epsilons (absolute logit gap / relative CDF distance).
EPS_LOGIT_BF16 = 1e-4
EPS_LOGIT_FP32 = 1e-5
EPS_CDF = 1e-5
EPS_ACCEPT = 1e-5


def f64(t):
    if t is None:
        return None
    return t.detach().float().cpu().numpy().astype(np.float64)


def np_(t):
    return t.detach().cpu().numpy()


def check_y(y_gpu, y_ref64, y_abs64, dtype):
    """y: bf16 results equal the oracle's rounding except at rounding
    near-ties; fp32 within the accumulation bound.  ``y_abs64`` is the same
    conv of |h| with |W| (the sum of the magnitudes of every term), which
    bounds the fp32 accumulation error.  Returns the tie count."""
    g = np_(y_gpu.float()).astype(np.float64)
    band = 1e-5 * y_abs64 + 1e-30
    if dtype == "fp32":
        assert np.all(np.abs(g - y_ref64) <= band)
        return 0
    o = oracle.round_bf16(y_ref64).astype(np.float64)
    diff = g != o
    if not diff.any():
        return 0
    # a mismatch is allowed only when the exact value sits on the rounding
    # boundary between the two neighbouring bf16 values
    mid = 0.5 * (g[diff] + o[diff])
    near = np.abs(y_ref64[diff] - mid) <= band[diff]
    step = np.abs(g[diff] - o[diff]) <= np.abs(o[diff]) * 2.0 ** -7 + 1e-30
    assert np.all(near & step), (
        f"{int((~(near & step)).sum())} y values differ beyond rounding ties")
    return int(diff.sum())


def check_topk(topv, topi, lse, ref, eps, lse_rtol):
    """Compare the CUDA top-16 / lse with the oracle's ``ref`` = (topv, topi,
    lse, U) computed from the CUDA path's own y (U = float64 logits [M, V]).
    Returns the number of rows whose lists differ by near-ties."""
    topv, topi, lse = np_(topv), np_(topi), np_(lse)
    _, o_i, o_lse, U = ref
    M, V = U.shape
    np.testing.assert_allclose(lse, o_lse, rtol=lse_rtol, atol=0)
    n = min(C, V)
    ties = 0
    for m in range(M):
        gi, oi = topi[m, :n], o_i[m, :n]
        assert np.all((gi >= 0) & (gi < V)), f"row {m}: index out of range"
        assert len(set(gi.tolist())) == n, f"row {m}: repeated index"
        assert np.all(topi[m, n:] == -1) and np.all(np.isneginf(topv[m, n:]))
        # reported values belong to their indices
        np.testing.assert_allclose(topv[m, :n], U[m, gi], rtol=1e-5,
                                   atol=eps * 0.1)
        if not np.array_equal(gi, oi):
            ties += 1
            # rank by rank, the chosen tokens' exact logits agree within eps
            gap = np.abs(U[m, gi] - U[m, oi])
            assert np.all(gap <= eps), (
                f"row {m}: top-16 differs beyond ties: {gi} vs {oi}, gap "
                f"{gap.max()}")
    return ties


def check_scores(S_gpu, S_ref, rtol=1e-5, atol=1e-5):
    g = np_(S_gpu).astype(np.float64)
    inf_g, inf_o = np.isneginf(g), np.isneginf(S_ref)
    assert np.array_equal(inf_g, inf_o), "padding pattern differs"
    np.testing.assert_allclose(g[~inf_g], S_ref[~inf_o], rtol=rtol, atol=atol)


def check_walk(slot, draft, q, S32, topi, T, seed, cycle, eps):
    """Oracle walk on the CUDA scores; identical slots except near-ties
    (after which the rest of that sequence is not comparable)."""
    slot, draft, q = np_(slot), np_(draft), np_(q)
    B, K = slot.shape
    u = philox.walk_uniforms(seed, cycle, B, K) if T > 0 else None
    o_slot, o_draft, o_q, margin = oracle.path_walk(S32, topi, T, u)
    ties = 0
    for b in range(B):
        for t in range(K):
            if slot[b, t] != o_slot[b, t]:
                assert margin[b, t] < eps, (
                    f"walk b={b} t={t}: slot {slot[b, t]} vs {o_slot[b, t]}, "
                    f"margin {margin[b, t]}")
                ties += 1
                break
            assert draft[b, t] == topi[b, t, slot[b, t]]
            np.testing.assert_allclose(q[b, t], o_q[b, t], rtol=1e-5,
                                       atol=1e-6)
    return ties


def check_verify(n, out, L, draft, topi, q, T, seed, cycle):
    """Oracle verify on the CUDA drafts; identical n and tokens except at
    near-tie accept tests or draws."""
    n, out = np_(n), np_(out)
    B, K1, V = L.shape
    K = K1 - 1
    ua = philox.accept_uniforms(seed, cycle, B, K) if T > 0 else None
    ur = philox.resample_uniforms(seed, cycle, B, K) if T > 0 else None
    o_n, o_out, mg = oracle.verify(L, draft, topi, q, T, ua, ur)
    ties = 0
    for b in range(B):
        if n[b] == o_n[b] and np.array_equal(out[b], o_out[b]):
            continue
        assert T > 0, f"greedy verify differs at b={b}: {out[b]} vs {o_out[b]}"
        k = min(int(n[b]), int(o_n[b]))
        if n[b] != o_n[b]:
            assert mg["accept"][b, k] < EPS_ACCEPT, (
                f"verify b={b}: n {n[b]} vs {o_n[b]}, accept margin "
                f"{mg['accept'][b, k]}")
        else:
            assert mg["resample"][b] < EPS_CDF, (
                f"verify b={b}: token {out[b, n[b]]} vs {o_out[b, n[b]]}, "
                f"margin {mg['resample'][b]}")
        ties += 1
    return ties, o_n, o_out


def to_dev(t, dev="cuda"):
    return None if t is None else t.to(dev).contiguous()


def draft_logits_oracle(x, w):
    """The drafter's fp32 logits of all K+1 rows (oracle), used to build the
    target logits of a workload."""
    h = f64(x["h"])
    y = oracle.to_storage(oracle.conv2tap(h, f64(x["w_conv"])), w.dtype)
    _, _, _, U = oracle.lmhead_topk(y.reshape(-1, w.H).astype(np.float64),
                                    f64(x["w_lm"]), want_logits=True)
    return U.reshape(w.B, w.K + 1, w.V).astype(np.float32)


def tie_eps(dtype):
    return EPS_LOGIT_BF16 if dtype == "bf16" else EPS_LOGIT_FP32


__all__ = ["check_y", "check_topk", "check_scores", "check_walk",
           "check_verify", "to_dev", "draft_logits_oracle", "f64", "np_",
           "tie_eps", "torch"]
