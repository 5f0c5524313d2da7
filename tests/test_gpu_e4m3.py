"""The LM head on 8-bit operands (E4M3 codes with one fp32 scale per row):
the quantization kernel bit-exact against the oracle's codec, and
dflash_draft_e4m3 stage by stage against the oracle fed the CUDA path's own
upstream outputs (the same tie policy as the bf16 path)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (ERR_C, check_scores, check_topk, check_verify,
                    check_walk, check_y, draft_logits_oracle, f64, np_,
                    to_dev)

pytestmark = pytest.mark.gpu

C = 16


def _weights(x):
    return {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out")}


def _quantize(lib, X):
    R, H = X.shape
    codes = torch.empty(R, H, dtype=torch.uint8, device="cuda")
    scale = torch.empty(R, dtype=torch.float32, device="cuda")
    lib.dflash_quantize_e4m3_rows(X, codes, scale)
    torch.cuda.synchronize()
    lib.dflash_check()
    return np_(codes), np_(scale)


@pytest.mark.parametrize("R,H", [(1, 16), (37, 208), (300, 2048)])
def test_quantize_rows_bit_exact(lib, R, H):
    g = np.random.default_rng(R * 7 + H)
    X = (g.standard_normal((R, H)) *
         np.exp2(g.uniform(-20, 20, size=(R, 1)))).astype(np.float32)
    X[0, : H // 2] = 0.0
    if R > 3:
        X[1] = 0.0                              # all-zero row: scale 1
        X[2] = -0.0
        X[3, :] = np.float32(1e-3)
        X[3, 5] = np.float32(-7.0)              # wide range: subnormal codes
    Xb = torch.from_numpy(X).to(torch.bfloat16)
    codes, scale = _quantize(lib, Xb.cuda())
    o_codes, o_scale = oracle.quantize_e4m3_rows(Xb.float().numpy())
    assert np.array_equal(scale, o_scale)
    assert np.array_equal(codes, o_codes), (
        f"{int((codes != o_codes).sum())} codes differ")


def test_quantize_flags_a_nonfinite_input(lib):
    X = torch.ones(4, 32, dtype=torch.bfloat16, device="cuda")
    X[2, 3] = float("inf")
    codes = torch.empty(4, 32, dtype=torch.uint8, device="cuda")
    scale = torch.empty(4, dtype=torch.float32, device="cuda")
    lib.dflash_quantize_e4m3_rows(X, codes, scale)
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_check()
    assert e.value.status == 4                  # DFLASH_ERR_NONFINITE


def run_e4m3(lib, w, x, L, seed=7, cycle=3):
    B, K, H, V, r = w.B, w.K, w.H, w.V, w.r
    h = to_dev(x["h"][:, :K])
    anchor = to_dev(x["anchor"])
    dv = lib.DraftVerify(B, K, H, V, r, _weights(x), lm_e4m3=True)
    torch.cuda.synchronize()
    lib.dflash_check()
    wc, ws = oracle.quantize_e4m3_rows(x["w_lm"].float().numpy())
    assert np.array_equal(np_(dv.w_scale), ws)
    assert np.array_equal(np_(dv.w_codes), wc)
    ties = {}
    dv.draft_all(h, anchor, w.T, seed, cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    h64 = f64(h)
    y = dv.y(fused=True)
    W = f64(x["w_conv"])
    ties["y"] = check_y(y, oracle.conv2tap(h64, W),
                        oracle.conv2tap(np.abs(h64), np.abs(W)), "bf16")
    yc, ys = dv.y_e4m3()
    o_yc, o_ys = oracle.quantize_e4m3_rows(np_(y.float()).reshape(-1, H))
    assert np.array_equal(np_(ys), o_ys)
    assert np.array_equal(np_(yc), o_yc)
    yq = oracle.dequantize_e4m3_rows(o_yc, o_ys)
    Wq = oracle.dequantize_e4m3_rows(wc, ws)
    ref = oracle.lmhead_topk(yq, Wq, want_logits=True)
    A = np.abs(yq) @ np.abs(Wq).T
    ties["topk"] = check_topk(dv.topv, dv.topi, dv.lse, ref, A,
                              ERR_C["bf16"])
    topv = np_(dv.topv).reshape(B, K, C)
    topi = np_(dv.topi).reshape(B, K, C)
    g = oracle.gate(h64, f64(x["w_gate"]))
    S = oracle.pair_score(topv, topi, np_(anchor), g, f64(x["e_in"]),
                          f64(x["e_out"]))
    check_scores(dv.scores, S)
    ties["walk"] = check_walk(dv.slot, dv.draft, dv.q, np_(dv.scores), topi,
                              w.T, seed, cycle, 1e-5)
    Ld = to_dev(L)
    dv.verify(Ld, w.T, seed, cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    ties["verify"], _, _ = check_verify(dv.n, dv.out, np_(Ld), np_(dv.draft),
                                        topi, np_(dv.q), w.T, seed, cycle)
    return {"ties": ties, "n": np_(dv.n), "dv": dv}


def _make(w):
    x = synth.make_inputs(w)
    L = synth.target_logits(w, draft_logits_oracle(x, w))
    return x, L


@pytest.mark.parametrize("B,K,H,V,r,T", [
    (3, 5, 192, 5003, 64, 1.0),     # ragged V, one row tile
    (9, 3, 128, 2051, 40, 1.5),     # one k-block of 128 codes
    (5, 3, 208, 1999, 48, 0.0),     # ragged K tail (208 = 128 + 80), greedy
    (20, 15, 144, 4099, 256, 1.0),  # M = 300: CTA pairs, full rank
    (65, 16, 208, 3001, 200, 1.0),  # M = 1040: 128-channel conv tiles
])
def test_draft_e4m3_small(lib, B, K, H, V, r, T):
    w = synth.Workload("small", B=B, K=K, V=V, H=H, r=r, dtype="bf16", T=T,
                       seed=41 + B, w_lm_sd=0.1, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 1.0))
    x, L = _make(w)
    run_e4m3(lib, w, x, L)


def test_draft_e4m3_full_size_b32k8cal(lib):
    """B=32, K=8, V=151936, H=2048 with the calibrated W_lm: every output
    against the oracle; the target is built from the bf16 drafter, so the
    acceptance shows what the 8-bit head costs."""
    w = synth.get("b32k8cal")
    x, L = _make(w)
    r = run_e4m3(lib, w, x, L, seed=w.seed, cycle=0)
    print("b32k8cal e4m3 ties", r["ties"], "mean accepted", r["n"].mean())


def test_draft_e4m3_vocab_smaller_than_candidates(lib):
    """V = 10 < 16: every list ends in (-inf, -1) padding, one vocab tile
    whose columns beyond V take no part (and no unit publishes to most
    shared-maxima slots)."""
    w = synth.Workload("v10", B=2, K=3, V=10, H=32, r=8, dtype="bf16",
                       T=1.0, seed=5, w_lm_sd=0.5, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 1.0, 0.3))
    x, L = _make(w)
    r = run_e4m3(lib, w, x, L)
    topi = np_(r["dv"].topi)
    assert np.all(topi[:, 10:] == -1)
    assert np.all(np.isneginf(np_(r["dv"].topv)[:, 10:]))
