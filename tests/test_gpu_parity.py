"""Parity of the CUDA path with the CPU oracle, stage by stage, through the
C ABI (ctypes binding).  Needs a GB300 (sm_103a)."""
import math

import numpy as np
import pytest
import torch
from scipy import stats

import oracle
import synth
from golden import lattice
from oracle import philox
from parity import (ERR_C, check_scores, check_topk, check_verify,
                    check_walk, check_y, draft_logits_oracle, f64, np_, to_dev)

pytestmark = pytest.mark.gpu
C = 16


def _weights(x):
    return {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out")}


def run_stagewise(lib, w, x, L, seed=7, cycle=3):
    """Run the four calls and check each against the oracle fed with the
    previous CUDA stage's outputs.  Returns a dict of tie counts and the
    CUDA results."""
    B, K, H, V, r = w.B, w.K, w.H, w.V, w.r
    h = to_dev(x["h"][:, :K])
    anchor = to_dev(x["anchor"])
    Ld = to_dev(L)
    dv = lib.DraftVerify(B, K, H, V, r, _weights(x))
    ties = {}
    dv.lmhead(h)
    torch.cuda.synchronize()
    lib.dflash_check()
    h64 = f64(h)
    if x["w_conv"] is not None:
        y = dv.y()
        W = f64(x["w_conv"])
        ties["y"] = check_y(y, oracle.conv2tap(h64, W),
                            oracle.conv2tap(np.abs(h64), np.abs(W)), w.dtype)
        y64 = f64(y).reshape(-1, H)
    else:
        y64 = h64.reshape(-1, H)
    W_lm = f64(x["w_lm"])
    ref = oracle.lmhead_topk(y64, W_lm, want_logits=True)
    A = np.abs(y64) @ np.abs(W_lm).T
    ties["topk"] = check_topk(dv.topv, dv.topi, dv.lse, ref, A, ERR_C[w.dtype])
    dv.pair_score(h, anchor)
    torch.cuda.synchronize()
    topv = np_(dv.topv).reshape(B, K, C)
    topi = np_(dv.topi).reshape(B, K, C)
    g = oracle.gate(h64, f64(x["w_gate"]))
    S = oracle.pair_score(topv, topi, np_(anchor), g, f64(x["e_in"]),
                          f64(x["e_out"]))
    check_scores(dv.scores, S)
    dv.walk(w.T, seed, cycle)
    torch.cuda.synchronize()
    S32 = np_(dv.scores)
    ties["walk"] = check_walk(dv.slot, dv.draft, dv.q, S32, topi, w.T, seed,
                              cycle, 1e-5)
    dv.verify(Ld, w.T, seed, cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    ties["verify"], o_n, _ = check_verify(dv.n, dv.out, np_(Ld), np_(dv.draft),
                                          topi, np_(dv.q), w.T, seed, cycle)
    return {"ties": ties, "n": np_(dv.n), "out": np_(dv.out), "dv": dv}


def run_fused(lib, w, x, L, seed=7, cycle=3):
    """dflash_draft (steps a1-a4 in one call, the gate computed inside the
    conv launch for bf16) then dflash_verify; every output is checked
    against the oracle fed with the CUDA path's own upstream outputs."""
    B, K, H, V, r = w.B, w.K, w.H, w.V, w.r
    h = to_dev(x["h"][:, :K])
    anchor = to_dev(x["anchor"])
    Ld = to_dev(L)
    dv = lib.DraftVerify(B, K, H, V, r, _weights(x))
    ties = {}
    dv.draft_all(h, anchor, w.T, seed, cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    h64 = f64(h)
    if x["w_conv"] is not None:
        y = dv.y(fused=True)
        W = f64(x["w_conv"])
        ties["y"] = check_y(y, oracle.conv2tap(h64, W),
                            oracle.conv2tap(np.abs(h64), np.abs(W)), w.dtype)
        y64 = f64(y).reshape(-1, H)
    else:
        y64 = h64.reshape(-1, H)
    W_lm = f64(x["w_lm"])
    ref = oracle.lmhead_topk(y64, W_lm, want_logits=True)
    A = np.abs(y64) @ np.abs(W_lm).T
    ties["topk"] = check_topk(dv.topv, dv.topi, dv.lse, ref, A, ERR_C[w.dtype])
    topv = np_(dv.topv).reshape(B, K, C)
    topi = np_(dv.topi).reshape(B, K, C)
    g = oracle.gate(h64, f64(x["w_gate"]))
    S = oracle.pair_score(topv, topi, np_(anchor), g, f64(x["e_in"]),
                          f64(x["e_out"]))
    check_scores(dv.scores, S)
    S32 = np_(dv.scores)
    ties["walk"] = check_walk(dv.slot, dv.draft, dv.q, S32, topi, w.T, seed,
                              cycle, 1e-5)
    dv.verify(Ld, w.T, seed, cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    ties["verify"], _, _ = check_verify(dv.n, dv.out, np_(Ld), np_(dv.draft),
                                        topi, np_(dv.q), w.T, seed, cycle)
    return {"ties": ties, "n": np_(dv.n), "out": np_(dv.out), "dv": dv}


def _make(w):
    x = synth.make_inputs(w)
    L = synth.target_logits(w, draft_logits_oracle(x, w))
    return x, L


# --------------------------------------------------------------------------
def test_library_loads_and_device_is_sm103(lib):
    assert torch.cuda.get_device_capability() == (10, 3)
    lib.load()


def test_philox_bit_exact_with_oracle(lib):
    n = 1 << 20
    rng = np.random.default_rng(0)
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64)
    ctr[:4096, 0] = np.arange(4096)
    ctr[:4096, 1:] = 0
    seed = 0x0123456789ABCDEF
    dev_ctr = torch.from_numpy(ctr.astype(np.uint32).view(np.int32)).cuda()
    out = torch.empty_like(dev_ctr)
    lib.dflash_philox4x32(dev_ctr, seed, out)
    got = np_(out).view(np.uint32)
    ref = philox.philox4x32_10(ctr, philox.seed_key(seed))
    assert np.array_equal(got, ref)


def test_philox_published_known_answers_on_gpu(lib):
    """The kernels' generator against the published Philox4x32-10
    known-answer vectors (Random123): the key is passed as the 64-bit seed
    (k0 = low word, k1 = high word)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(__file__), "golden",
                           "philox_kat.json")) as f:
        vec = json.load(f)["vectors"]
    h = lambda ws: [int(w, 16) for w in ws]
    for v in vec:
        ctr = np.array([h(v["ctr"])], np.uint32)
        k0, k1 = h(v["key"])
        dev_ctr = torch.from_numpy(ctr.view(np.int32)).cuda()
        out = torch.empty_like(dev_ctr)
        lib.dflash_philox4x32(dev_ctr, k0 | (k1 << 32), out)
        assert [int(x) for x in np_(out).view(np.uint32)[0]] == h(v["out"])


@pytest.mark.parametrize("name,T", [("tiny", 0.0), ("tiny", 1.0),
                                    ("tiny_conv", 0.0), ("tiny_conv", 1.0)])
def test_tiny_fp32(lib, name, T):
    w = synth.get(name, T=T)
    x, L = _make(w)
    r = run_stagewise(lib, w, x, L)
    assert r["ties"]["topk"] == 0


@pytest.mark.parametrize("B,K,H,V,r,T", [
    (3, 5, 192, 5003, 64, 1.0),     # ragged V (not a multiple of 4 or 256)
    (2, 16, 256, 3000, 256, 0.0),   # K = 16, full rank
    (2, 16, 256, 3000, 256, 0.7),
    (4, 1, 64, 777, 16, 1.0),       # K = 1
    (9, 3, 128, 2051, 32, 1.5),     # M not a multiple of 8
    (5, 3, 200, 1999, 48, 1.0),     # H not a multiple of 64 (ragged K tail)
    (16, 16, 256, 3000, 256, 0.0),  # M = 256: two row tiles (CTA pair)
    (20, 15, 136, 4099, 64, 1.0),   # M = 300: pair with an empty odd tile
])
def test_small_bf16(lib, B, K, H, V, r, T):
    w = synth.Workload("small", B=B, K=K, V=V, H=H, r=r, dtype="bf16", T=T,
                       seed=11 + B, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 1.0))
    x, L = _make(w)
    run_stagewise(lib, w, x, L)


def test_vocab_smaller_than_candidates(lib):
    w = synth.Workload("v10", B=2, K=3, V=10, H=16, r=8, dtype="fp32", T=1.0,
                       seed=5, w_lm_sd=0.5, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 1.0, 0.3))
    x, L = _make(w)
    r = run_stagewise(lib, w, x, L)
    dv = r["dv"]
    assert np.all(np_(dv.topi)[:, 10:] == -1)
    assert np.all(np_(dv.q).reshape(-1, C)[:, 10:] == 0)


def test_golden_lattice_figure(lib):
    fx = lattice.load()
    K, H, V, r = fx["K"], fx["H"], fx["V"], fx["r"]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    weights = {"w_conv": None, "w_lm": dev(fx["w_lm"]),
               "w_gate": dev(fx["w_gate"]), "e_in": dev(fx["e_in"]),
               "e_out": dev(fx["e_out"])}
    dv = lib.DraftVerify(1, K, H, V, r, weights)
    n, out = dv.cycle(dev(fx["h"]), dev(fx["anchor"]), dev(fx["L"]), 0.0, 0, 0)
    torch.cuda.synchronize()
    lib.dflash_check()
    np.testing.assert_allclose(np_(dv.lse), fx["lse"], rtol=1e-6)
    assert list(np_(dv.topi)[0, :3]) == fx["topi0_first3"]
    assert list(np_(dv.slot)[0]) == fx["path_slots"]
    assert list(np_(dv.draft)[0]) == fx["path_tokens"]
    assert (int(np_(n)[0]), list(np_(out)[0])) == fx["verify_selector"]


def test_greedy_verify_is_target_argmax_prefix(lib):
    B, K, V = 64, 8, 4099
    rng = np.random.default_rng(3)
    L = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    am = L.argmax(-1)
    n_true = rng.integers(0, K + 1, B)
    draft = am[:, :K].copy()
    for b in range(B):
        if n_true[b] < K:
            draft[b, n_true[b]] = (am[b, n_true[b]] + 1) % V
    topi = np.full((B, K, C), -1, np.int32)
    topi[:, :, 0] = draft
    q = np.zeros((B, K, C), np.float32)
    q[:, :, 0] = 1
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(d(L), d(draft.astype(np.int32)), d(topi), d(q), 0.0, 0,
                      0, n, out, ws)
    lib.dflash_check()
    assert np.array_equal(np_(n), n_true)
    for b in range(B):
        k = n_true[b]
        assert list(np_(out)[b, :k + 1]) == list(am[b, :k + 1])
        assert np.all(np_(out)[b, k + 1:] == -1)


def _engineered_walk(lib, q0, B, seed):
    """Drafts from q0 (V = len(q0) <= 16) drawn by the CUDA walk."""
    V = len(q0)
    S = np.full((B, 1, C, C), -np.inf, np.float32)
    S[:, 0, :, :V] = np.log(q0)
    topi = np.full((B, 1, C), -1, np.int32)
    topi[:, :, :V] = np.arange(V)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    slot = torch.empty(B, 1, dtype=torch.int32, device="cuda")
    draft = torch.empty_like(slot)
    q = torch.empty(B, 1, C, dtype=torch.float32, device="cuda")
    lib.dflash_path_walk(d(S), d(topi), 1.0, seed, 0, slot, draft, q)
    return draft, q, d(topi)


def test_sampler_is_lossless_on_gpu(lib):
    """Emitted first token ~ p0 and accept rate = sum min(p, q) (V = 8)."""
    V, B = 8, 200000
    rng = np.random.default_rng(21)
    q0 = rng.dirichlet(np.ones(V) * 0.8)
    p0 = rng.dirichlet(np.ones(V) * 0.8)
    draft, q, topi = _engineered_walk(lib, q0, B, seed=31)
    L = np.zeros((B, 2, V), np.float32)
    L[:, 0] = np.log(p0)
    Ld = torch.from_numpy(L).cuda()
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, 2, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, 1, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(Ld, draft, topi, q, 1.0, 77, 0, n, out, ws)
    lib.dflash_check()
    # the walk's drafts follow q0
    cd = np.bincount(np_(draft)[:, 0], minlength=V)
    assert stats.chisquare(cd, q0 * B).pvalue > 1e-3
    pa = np.minimum(p0, q0).sum()
    assert abs(np_(n).mean() - pa) < 4 * math.sqrt(pa * (1 - pa) / B)
    c0 = np.bincount(np_(out)[:, 0], minlength=V)
    assert stats.chisquare(c0, p0 * B).pvalue > 1e-3


def test_bonus_draw_follows_target_row_K_on_gpu(lib):
    """Every draft accepted with certainty (position t drafts token t with
    q = 1 and the target puts all its mass there): the bonus token follows
    p_K = softmax(L[:, K] / T) (chi-square, V = 8, 200k sequences), not
    row K-1 (all mass on token K-1)."""
    V, B, K, T = 8, 200000, 2, 0.7
    rng = np.random.default_rng(41)
    pK = rng.dirichlet(np.ones(V) * 0.5)
    draft = np.tile(np.arange(K, dtype=np.int32), (B, 1))
    topi = np.full((B, K, C), -1, np.int32)
    topi[:, :, 0] = draft
    q = np.zeros((B, K, C), np.float32)
    q[:, :, 0] = 1.0
    L = np.full((B, K + 1, V), -np.inf, np.float32)
    L[:, np.arange(K), np.arange(K)] = 0.0
    L[:, K] = T * np.log(pK)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(d(L), d(draft), d(topi), d(q), T, 45, 0, n, out, ws)
    lib.dflash_check()
    assert np.all(np_(n) == K)
    assert np.array_equal(np_(out)[:, :K], draft)
    cK = np.bincount(np_(out)[:, K], minlength=V)
    assert stats.chisquare(cK, pK * B).pvalue > 1e-3



@pytest.mark.parametrize("T", [1.0, 0.0])
def test_verify_position_order_with_mixed_acceptance(lib, T):
    """Rows run in position order and a row after a known rejection stops
    reading.  B = 64, V = 40000 (3 blocks per row): positions 0-1 go in 3
    chunks per row, the later ones in 1, so both chunkings and the stops
    meet.  Sequence b accepts about m_b drafts (m_b spread over 0..K: the
    target puts nearly all its mass on drafts 0..m_b-1 and almost none on
    draft m_b); every sequence's n and tokens must match the oracle."""
    B, K, V = 64, 8, 40000
    rng = np.random.default_rng(71)
    L = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    m = rng.integers(0, K + 1, size=B)
    draft = rng.integers(0, V, size=(B, K)).astype(np.int32)
    for b in range(B):
        for t in range(K):
            if t < m[b]:
                L[b, t, draft[b, t]] = 20.0
            else:
                L[b, t, draft[b, t]] = -20.0
    topi = np.full((B, K, C), -1, np.int32)
    topi[:, :, 0] = draft
    q = np.zeros((B, K, C), np.float32)
    q[:, :, 0] = 1.0
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(d(L), d(draft), d(topi), d(q), T, 13, 2, n, out, ws)
    torch.cuda.synchronize()
    lib.dflash_check()
    _, o_n, _ = check_verify(n, out, L, draft, topi, q, T, 13, 2)
    assert np.array_equal(np_(n), o_n)
    # the construction spreads the accepted lengths over 0..K
    assert len(set(np_(n).tolist())) >= K - 1


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_verify_rows_after_the_first_rejection_do_not_matter(lib, T):
    """Rows after a sequence's first rejection are never emitted (the CUDA
    verify stops reading them once the rejection is known): replacing them
    with other finite values leaves n and every token identical, bit for
    bit, whichever of them the launch happened to read."""
    B, K, V = 64, 8, 40000
    rng = np.random.default_rng(73)
    L = rng.standard_normal((B, K + 1, V)).astype(np.float32)
    m = rng.integers(0, K + 1, size=B)
    draft = rng.integers(0, V, size=(B, K)).astype(np.int32)
    for b in range(B):
        for t in range(K):
            L[b, t, draft[b, t]] = 20.0 if t < m[b] else -20.0
    topi = np.full((B, K, C), -1, np.int32)
    topi[:, :, 0] = draft
    q = np.zeros((B, K, C), np.float32)
    q[:, :, 0] = 1.0
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")

    def run(Lx):
        n = torch.empty(B, dtype=torch.int32, device="cuda")
        out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
        lib.dflash_verify(d(Lx), d(draft), d(topi), d(q), T, 21, 4, n, out,
                          ws)
        torch.cuda.synchronize()
        lib.dflash_check()
        return np_(n).copy(), np_(out).copy()

    n1, o1 = run(L)
    L2 = L.copy()
    for b in range(B):
        L2[b, n1[b] + 1:] = rng.standard_normal((K - n1[b], V)) * 4
    n2, o2 = run(L2)
    assert len(set(n1.tolist())) >= K - 1
    assert np.array_equal(n1, n2)
    assert np.array_equal(o1, o2)

def test_p_equals_q_accepts_all(lib):
    V, K, B = 12, 4, 512
    rng = np.random.default_rng(5)
    qv = rng.dirichlet(np.ones(V), size=(B, K)).astype(np.float32)
    topi = np.full((B, K, C), -1, np.int32)
    topi[:, :, :V] = np.arange(V)
    q = np.zeros((B, K, C), np.float32)
    q[:, :, :V] = qv
    draft = np.array([[rng.choice(V, p=qv[b, t] / qv[b, t].sum())
                       for t in range(K)] for b in range(B)], np.int32)
    L = np.zeros((B, K + 1, V), np.float32)
    L[:, :K] = np.log(qv)
    d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(d(L), d(draft), d(topi), d(q), 1.0, 3, 1, n, out, ws)
    lib.dflash_check()
    assert np.all(np_(n) == K)
    assert np.array_equal(np_(out)[:, :K], draft)


def test_invalid_arguments_are_rejected(lib):
    B, K, V = 2, 17, 100
    L = torch.zeros(B, K + 1, V, device="cuda")
    draft = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    topi = torch.zeros(B, K, C, dtype=torch.int32, device="cuda")
    q = torch.zeros(B, K, C, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_verify(L, draft, topi, q, 1.0, 0, 0, n, out, ws)
    assert e.value.status == 1
    h = torch.zeros(1, 2, 12, dtype=torch.bfloat16, device="cuda")
    w_lm = torch.zeros(50, 12, dtype=torch.bfloat16, device="cuda")
    tv = torch.empty(2, C, device="cuda")
    ti = torch.empty(2, C, dtype=torch.int32, device="cuda")
    ls = torch.empty(2, device="cuda")
    with pytest.raises(lib.DFlashError) as e:          # H % 8 != 0
        lib.dflash_lmhead_topk(h, None, w_lm, tv, ti, ls, ws)
    assert e.value.status == 1


def test_nonfinite_target_logit_is_reported(lib):
    # in row 0, which is always read (rows after a sequence's first
    # rejection may stop being read once it is known)
    B, K, V = 1, 2, 64
    L = torch.zeros(B, K + 1, V, device="cuda")
    L[0, 0, 5] = float("nan")
    draft = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    topi = torch.zeros(B, K, C, dtype=torch.int32, device="cuda")
    topi[:, :, 1:] = -1
    q = torch.zeros(B, K, C, device="cuda")
    q[:, :, 0] = 1
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dflash_workspace_bytes(1, B, K, 0, V),
                     dtype=torch.uint8, device="cuda")
    lib.dflash_verify(L, draft, topi, q, 1.0, 0, 0, n, out, ws)
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_check()
    assert e.value.status == 4
    lib.dflash_check()  # cleared


def test_cycle_is_deterministic(lib):
    w = synth.Workload("det", B=4, K=6, V=9000, H=128, r=64, dtype="bf16",
                       T=1.0, seed=9, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 1.0))
    x, L = _make(w)
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x))
    h, a, Ld = to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), to_dev(L)
    res = []
    for _ in range(2):
        n, out = dv.cycle(h, a, Ld, w.T, 5, 6)
        res.append((np_(n).copy(), np_(out).copy(), np_(dv.scores).copy(),
                    np_(dv.lse).copy()))
    for a0, a1 in zip(res[0], res[1]):
        assert np.array_equal(a0, a1)


# --------------------------------------------------------------------------
# full-size workloads, in the launch configuration the benchmark times
# --------------------------------------------------------------------------
@pytest.mark.parametrize("name", ["b1k8", "b32k8"])
def test_full_size_workload(lib, name):
    w = synth.get(name)
    x, L = _make(w)
    r = run_stagewise(lib, w, x, L, seed=w.seed, cycle=0)
    print(name, "ties", r["ties"], "mean accepted", r["n"].mean())


# --------------------------------------------------------------------------
# dflash_draft: steps a1-a4 in one call
@pytest.mark.parametrize("B,K,H,V,r,T", [
    (3, 5, 192, 5003, 64, 1.0),     # ragged V, one row tile
    (9, 3, 128, 2051, 40, 1.5),     # r not a multiple of 64 (partial gate tile)
    (5, 3, 200, 1999, 48, 0.0),     # ragged K tail, greedy
    (20, 15, 136, 4099, 256, 1.0),  # M = 300: CTA pairs, full rank
    (65, 16, 200, 3001, 200, 1.0),  # M = 1040: 128-channel conv tiles,
                                    # ragged H and a partial gate tile
    (6, 5, 224, 3001, 32, 1.0),     # ragged K (224 = 3.5 k-blocks)
    (20, 15, 256, 4099, 128, 0.7),  # M = 300, one full 128-row gate tile
    (17, 9, 200, 3001, 200, 1.0),   # M = 153: conv K split over a cluster
                                    # with ragged H, a ragged second row
                                    # tile and a partial gate tile
    (9, 16, 128, 2051, 40, 0.0),    # M = 144: K split into single blocks,
                                    # one partial gate tile, greedy
])
def test_fused_draft_bf16(lib, B, K, H, V, r, T):
    w = synth.Workload("small", B=B, K=K, V=V, H=H, r=r, dtype="bf16", T=T,
                       seed=31 + B, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 1.0))
    x, L = _make(w)
    run_fused(lib, w, x, L)


@pytest.mark.parametrize("name,T", [("tiny", 1.0), ("tiny_conv", 0.0)])
def test_fused_draft_fp32(lib, name, T):
    """fp32 storage (and no conv) take the separate kernels inside the call."""
    w = synth.get(name, T=T)
    x, L = _make(w)
    r = run_fused(lib, w, x, L)
    assert r["ties"]["topk"] == 0


def test_fused_draft_matches_separate_calls(lib):
    """Same LM head kernels: identical candidates; lse and scores within
    fp32 rounding (the fused path folds the lse pairs and accumulates the
    gate in other orders)."""
    w = synth.Workload("small", B=6, K=8, V=3001, H=256, r=256, dtype="bf16",
                       T=1.0, seed=5, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 1.0))
    x = synth.make_inputs(w)
    h = to_dev(x["h"][:, :w.K])
    anchor = to_dev(x["anchor"])
    a = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x))
    b = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x))
    a.lmhead(h)
    a.pair_score(h, anchor)
    b.draft_all(h, anchor, w.T, 7, 3)
    torch.cuda.synchronize()
    lib.dflash_check()
    assert torch.equal(a.topi, b.topi) and torch.equal(a.topv, b.topv)
    np.testing.assert_allclose(np_(b.lse), np_(a.lse), rtol=2e-6, atol=0)
    np.testing.assert_allclose(np_(b.scores), np_(a.scores), rtol=1e-5,
                               atol=1e-5)


def test_fused_draft_full_size_b32k8(lib):
    w = synth.get("b32k8")
    x, L = _make(w)
    r = run_fused(lib, w, x, L, seed=w.seed, cycle=0)
    print("b32k8 fused ties", r["ties"], "mean accepted", r["n"].mean())


def test_fused_full_size_b32k8cal(lib):
    """The calibrated workload (mean 4.5 accepted drafts per cycle): the
    accept tests and residual draws of every position are exercised."""
    w = synth.get("b32k8cal")
    x, L = _make(w)
    r = run_fused(lib, w, x, L, seed=w.seed, cycle=0)
    print("b32k8cal ties", r["ties"], "mean accepted", r["n"].mean())
    assert r["n"].mean() > 2.0


@pytest.mark.parametrize("e4m3", [False, True])
def test_fused_draft_exact_ties_across_strips(lib, e4m3):
    """W_lm built from 40 distinct rows repeated over V = 5003 tokens: every
    logit value occurs about 125 times, spread over all vocab strips, so the
    top 16 of a row are 16 copies of its largest value and must be the 16
    lowest ids that carry it (ties to the lower id through the first-tile
    threshold, the shared row maxima and the merge of the strips)."""
    import synth as _s
    w = _s.Workload("ties", B=4, K=4, V=5003, H=128, r=32, dtype="bf16",
                    T=1.0, seed=77, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                    target=("affine", 0.9, 1.0))
    x = _s.make_inputs(w)
    base = x["w_lm"][:40].clone()
    x["w_lm"] = base.repeat((w.V + 39) // 40, 1)[: w.V].contiguous()
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights(x), lm_e4m3=e4m3)
    h = to_dev(x["h"][:, : w.K])
    dv.draft_all(h, to_dev(x["anchor"]), w.T, 5, 0)
    torch.cuda.synchronize()
    lib.dflash_check()
    if e4m3:
        yc, ys = dv.y_e4m3()
        wc, ws = oracle.quantize_e4m3_rows(x["w_lm"].float().numpy())
        y64 = oracle.dequantize_e4m3_rows(np_(yc), np_(ys))
        W64 = oracle.dequantize_e4m3_rows(wc, ws)
    else:
        y64 = f64(dv.y(fused=True)).reshape(-1, w.H)
        W64 = f64(x["w_lm"])
    _, o_i, _ = oracle.lmhead_topk(y64, W64)
    gi = np_(dv.topi)
    for m in range(w.M):
        # the GPU's 16 values are equal copies of one logit (same W rows,
        # same accumulation order), so the ids must be the lowest 16
        gv = np_(dv.topv)[m]
        assert np.all(gv == gv[0]), f"row {m}: values differ {gv}"
        assert np.array_equal(gi[m], o_i[m]), f"row {m}: {gi[m]} vs {o_i[m]}"


@pytest.mark.parametrize("B,K", [(3, 5), (20, 15)])
def test_bf16_without_conv(lib, B, K):
    """bf16 storage with no conv (y = h): the tensor-core LM head runs
    without the shared row maxima (nothing resets them), single CTAs at
    M = 15 and CTA pairs at M = 300, through the separate calls and
    through dflash_draft."""
    w = synth.Workload("noconv", B=B, K=K, V=4099, H=136, r=64,
                       dtype="bf16", T=1.0, seed=13 + B, w_lm_sd=0.1,
                       conv_sd=None, sel_sd=0.1, target=("affine", 0.9, 1.0))
    x, L = _make(w)
    run_stagewise(lib, w, x, L)
    run_fused(lib, w, x, L)


def test_vocab_smaller_than_candidates_tensor_cores(lib):
    """V = 10 < 16 on the bf16 tensor-core path (conv, LM head, draft
    tail): lists padded with (-inf, -1), scores of padded candidates -inf."""
    w = synth.Workload("v10bf", B=2, K=3, V=10, H=32, r=8, dtype="bf16",
                       T=1.0, seed=6, w_lm_sd=0.5, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 1.0, 0.3))
    x, L = _make(w)
    run_stagewise(lib, w, x, L)
    r = run_fused(lib, w, x, L)
    assert np.all(np_(r["dv"].topi)[:, 10:] == -1)
