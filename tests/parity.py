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
# Tie epsilons of the sampled decisions (relative CDF distance / relative
# accept-test margin).
EPS_CDF = 1e-5
EPS_ACCEPT = 1e-5


def f64(t):
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().float().cpu().numpy().astype(np.float64)


def np_(t):
    if isinstance(t, np.ndarray):
        return t
    return t.detach().cpu().numpy()


def _ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def check_y(y_gpu, y_ref64, y_abs64, dtype):
    """Conv output y.  The exact value y_ref is known to float64; the CUDA
    value may differ by its fp32 accumulation error, at most 1e-6 of the sum
    of term magnitudes y_abs (measured on GB300: 1.25e-7).  A bf16 result
    must therefore be the correct rounding of some value within that band:
    |y - y_ref| <= band + ulp(y)/2.  Where the two taps cancel, the band can
    span several bf16 steps.  Returns the count of results that differ from
    the round-to-nearest-even of y_ref (legitimate near-ties)."""
    g = np_(y_gpu.float()).astype(np.float64)
    band = 1e-6 * y_abs64 + 1e-30
    if dtype == "fp32":
        assert np.all(np.abs(g - y_ref64) <= band)
        return 0
    half = 0.5 * np.maximum(_ulp_bf16(g), _ulp_bf16(y_ref64))
    ok = np.abs(g - y_ref64) <= band + half
    if not np.all(ok):
        idx = np.nonzero(~ok.reshape(-1))[0][:5]
        gv, rv, bv = g.reshape(-1), y_ref64.reshape(-1), band.reshape(-1)
        det = "; ".join(f"#{i}: gpu {gv[i]!r} exact {rv[i]!r} band {bv[i]:.3g}"
                        for i in idx)
        raise AssertionError(f"{int((~ok).sum())} y values outside the "
                             f"accumulation band: {det}")
    return int((g != oracle.round_bf16(y_ref64)).sum())


# Error model of a logit computed with fp32 accumulation: |error| <= c *
# sum_k |y_k W_vk|.  Measured on GB300 for the tensor-core path: at most
# 6.6e-7 of that sum (b32k8); c = 2e-6 leaves a 3x margin.  Sequential fp32
# accumulation over H <= 64 terms is bounded by H * 2^-24 < 4e-6.
ERR_C = {"bf16": 2e-6, "fp32": 4e-6}


def check_topk(topv, topi, lse, ref, A, c):
    """Compare the CUDA top-16 / lse with the oracle's ``ref`` = (topv, topi,
    lse, U) computed from the CUDA path's own y.  ``A`` = |y| |W|^T (the
    sum of term magnitudes per logit) scales the accumulation bound c * A.
    Two tokens may trade ranks only if their exact logits are within the sum
    of their bounds.  Returns the number of rows whose lists differ."""
    topv, topi, lse = np_(topv), np_(topi), np_(lse)
    _, o_i, o_lse, U = ref
    M, V = U.shape
    lse_tol = c * A.max(axis=1) + 1e-6 * np.abs(o_lse)
    bad = ~(np.abs(lse - o_lse) <= lse_tol)   # NaN counts as bad
    assert not bad.any(), (f"lse rows {np.nonzero(bad)[0][:5]}: "
                           f"{lse[bad][:5]} vs {o_lse[bad][:5]}")
    n = min(C, V)
    ties = 0
    for m in range(M):
        gi, oi = topi[m, :n], o_i[m, :n]
        assert np.all((gi >= 0) & (gi < V)), f"row {m}: index out of range"
        assert len(set(gi.tolist())) == n, f"row {m}: repeated index"
        assert np.all(topi[m, n:] == -1) and np.all(np.isneginf(topv[m, n:]))
        eg = c * A[m, gi] + 1e-7
        assert np.all(np.abs(topv[m, :n] - U[m, gi]) <= eg), (
            f"row {m}: topv off by {np.abs(topv[m, :n] - U[m, gi]).max()}")
        if not np.array_equal(gi, oi):
            ties += 1
            gap = np.abs(U[m, gi] - U[m, oi])
            assert np.all(gap <= eg + c * A[m, oi] + 1e-7), (
                f"row {m}: top-16 differs beyond ties: {gi} vs {oi}, gap "
                f"{gap.max()}")
    return ties


def check_scores(S_gpu, S_ref, rtol=1e-5, atol=1e-5):
    g = np_(S_gpu).astype(np.float64)
    inf_g, inf_o = np.isneginf(g), np.isneginf(S_ref)
    assert np.array_equal(inf_g, inf_o), "padding pattern differs"
    np.testing.assert_allclose(g[~inf_g], S_ref[~inf_o], rtol=rtol, atol=atol)


def check_walk(slot, draft, q, S32, topi, T, seed, cycle, eps, bidx=None):
    """Oracle walk on the CUDA scores; identical slots except near-ties
    (after which the rest of that sequence is not comparable).  ``bidx``:
    the batch indices of the given sequences (their Philox streams), when
    they are a sample of a larger batch."""
    slot, draft, q = np_(slot), np_(draft), np_(q)
    B, K = slot.shape
    u = None
    if T > 0:
        bi = np.arange(B) if bidx is None else np.asarray(bidx)
        u = philox.uniforms(seed, cycle, bi[:, None], np.arange(K)[None, :],
                            philox.PURPOSE_WALK)
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


def check_verify(n, out, L, draft, topi, q, T, seed, cycle, bidx=None):
    """Oracle verify on the CUDA drafts; identical n and tokens except at
    near-tie accept tests or draws.  ``bidx`` as in check_walk."""
    n, out = np_(n), np_(out)
    B, K1, V = L.shape
    K = K1 - 1
    ua = ur = None
    if T > 0:
        bi = np.arange(B) if bidx is None else np.asarray(bidx)
        ua = philox.uniforms(seed, cycle, bi[:, None], np.arange(K)[None, :],
                             philox.PURPOSE_ACCEPT)
        ur = philox.uniforms(seed, cycle, bi, np.full(B, K),
                             philox.PURPOSE_RESAMPLE)
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




__all__ = ["ERR_C", "check_y", "check_topk", "check_scores", "check_walk",
           "check_verify", "to_dev", "draft_logits_oracle", "f64", "np_",
           "torch"]
