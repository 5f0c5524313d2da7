"""Full-size parity in the launch configuration the benchmark times
(dflash_draft + dflash_verify), on sequences sampled so that every 128-row
tile of the LM head and conv launches, and both CTAs of every LM-head CTA
pair, hold a checked sequence.

  * b128k16zipf (B=128, K=16, V=151936, H=2560, Zipf-skewed target): one
    sequence in each of the 16 row tiles (rows 0..2047).
  * the sweep's corners (V=262144, H=3072, r=256): K=16 B=256 (M=4096,
    32 row tiles, 16 CTA-pair row groups, every verify row of 128
    segments) and K=4 B=1 (one row tile, single-CTA LM head), each at T=0
    and T=1.

Each stage of the sampled sequences is compared with the oracle fed the
CUDA path's own upstream outputs (conv y, top-16 and logsumexp, pair
scores, walk, verify), as in test_gpu_parity.py.  The target logits are
drawn on the device with torch ops (input synthesis only; both sides read
the same tensor)."""
import functools

import numpy as np
import pytest
import torch

import oracle
import synth
from parity import (ERR_C, check_scores, check_topk, check_verify,
                    check_walk, check_y, f64, np_, to_dev)

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
C = 16
ROW_TILE = 128


def sampled_sequences(B, K, offset=3):
    """One sequence per 128-row tile (all of them when the batch fits one
    tile), at a position inside the tile that varies from tile to tile."""
    per_tile = max(1, ROW_TILE // K)
    tiles = (B * K + ROW_TILE - 1) // ROW_TILE
    if tiles == 1:
        return list(range(B))
    out = []
    for tile in range(tiles):
        b = tile * per_tile + (tile * offset) % per_tile
        if b < B:
            out.append(b)
    return out


def drafter_logits_device(w, x, dev="cuda"):
    """The drafter's fp32 logits of all K+1 rows [B, K+1, V], from torch
    ops on the device (conv in fp32, y rounded to bf16, fp32 matmul)."""
    torch.backends.cuda.matmul.allow_tf32 = False
    h = x["h"].to(dev).float()
    H = w.H
    wc = x["w_conv"].to(dev).float()
    prev = torch.zeros_like(h)
    prev[:, 1:] = h[:, :-1]
    y = ((h @ wc[:H].T) * h + (h @ wc[H:].T) * prev).to(
        torch.bfloat16).float().reshape(-1, H)
    del h, prev, wc
    wl = x["w_lm"].to(dev)
    U = torch.empty(y.shape[0], w.V, device=dev)
    for v0 in range(0, w.V, 16384):
        U[:, v0:v0 + 16384] = y @ wl[v0:v0 + 16384].float().T
    return U.reshape(w.B, w.K + 1, w.V)


def affine_target_device(w, x, seed):
    """target = a * drafter logits + N(0, sd), noise from a seeded torch
    generator on the device."""
    kind, a, sd = w.target
    assert kind == "affine"
    L = drafter_logits_device(w, x)
    g = torch.Generator(device="cuda").manual_seed(seed)
    flat = L.view(-1, w.V)
    for r0 in range(0, flat.shape[0], 1024):
        blk = flat[r0:r0 + 1024]
        blk.mul_(a).add_(torch.randn(blk.shape, generator=g,
                                     device="cuda") * sd)
    return L


def check_sampled(w, x, dv, L, seqs, seed, cycle, W64=None):
    """Every stage of the sequences ``seqs`` against the oracle.  Returns
    the tie counts per stage."""
    K, H = w.K, w.H
    bi = np.asarray(seqs)
    rows = (bi[:, None] * K + np.arange(K)[None, :]).reshape(-1)
    ties = {}
    h64 = f64(x["h"][torch.as_tensor(bi), :K])
    Wc = f64(x["w_conv"])
    y = dv.y(fused=True)[torch.as_tensor(bi, device="cuda")]
    ties["y"] = check_y(y, oracle.conv2tap(h64, Wc),
                        oracle.conv2tap(np.abs(h64), np.abs(Wc)), w.dtype)
    y64 = f64(y).reshape(-1, H)
    if W64 is None:
        W64 = f64(x["w_lm"])
    ref = oracle.lmhead_topk(y64, W64, want_logits=True)
    ay = np.abs(y64)
    A = np.empty((y64.shape[0], w.V))
    for v0 in range(0, w.V, 32768):                # |y| |W|^T by blocks
        A[:, v0:v0 + 32768] = ay @ np.abs(W64[v0:v0 + 32768]).T
    ri = torch.as_tensor(rows, device="cuda")
    ties["topk"] = check_topk(dv.topv[ri], dv.topi[ri], dv.lse[ri], ref, A,
                              ERR_C[w.dtype])
    topv = np_(dv.topv).reshape(w.B, K, C)[bi]
    topi = np_(dv.topi).reshape(w.B, K, C)[bi]
    g = oracle.gate(h64, f64(x["w_gate"]))
    S = oracle.pair_score(topv, topi, np_(x["anchor"])[bi], g,
                          f64(x["e_in"]), f64(x["e_out"]))
    check_scores(dv.scores[torch.as_tensor(bi, device="cuda")], S)
    S32 = np_(dv.scores)[bi]
    sel = lambda t: np_(t)[bi]
    ties["walk"] = check_walk(sel(dv.slot), sel(dv.draft), sel(dv.q), S32,
                              topi, w.T, seed, cycle, 1e-5, bidx=bi)
    Lh = L[torch.as_tensor(bi, device=L.device)].cpu().numpy()
    ties["verify"], _, _ = check_verify(sel(dv.n), sel(dv.out), Lh,
                                        sel(dv.draft), topi, sel(dv.q), w.T,
                                        seed, cycle, bidx=bi)
    return ties


def _weights_dev(x):
    return {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out")}


def test_sampled_sequences_cover_every_tile_and_pair_half():
    for B, K in ((128, 16), (256, 16), (1, 4), (32, 8)):
        seqs = sampled_sequences(B, K)
        tiles = sorted({(b * K) // ROW_TILE for b in seqs})
        assert tiles == list(range((B * K + ROW_TILE - 1) // ROW_TILE))
        if len(tiles) >= 2:
            assert {t % 2 for t in tiles} == {0, 1}


def test_full_size_b128k16zipf_every_row_tile(lib):
    """B=128, K=16, H=2560, Zipf target, T=1: the whole cycle at full size,
    one checked sequence in each of the 16 row tiles (both CTAs of all 8
    CTA pairs)."""
    w = synth.get("b128k16zipf")
    x = synth.make_inputs(w)
    U = drafter_logits_device(w, x).cpu().numpy()
    L = synth.target_logits(w, U).cuda()
    del U
    seed, cycle = w.seed, 0
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, _weights_dev(x))
    dv.cycle(to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), L, w.T, seed,
             cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    seqs = sampled_sequences(w.B, w.K)
    assert len(seqs) == 16
    ties = check_sampled(w, x, dv, L, seqs, seed, cycle)
    print("b128k16zipf sequences", seqs, "ties", ties,
          "mean accepted (all)", np_(dv.n).mean())


@functools.lru_cache(maxsize=1)
def _sweep_weights():
    """The sweep grid's weights (V=262144, H=3072, r=256; one draw shared
    by every point, as in the sweep) on the host, in float64 for the
    oracle's LM head, and on the device."""
    w = [p for p in synth.sweep_points() if p.K == 16 and p.B == 256][0]
    x = synth.make_inputs(w, tensors=("w_conv", "w_lm", "w_gate", "e_in",
                                      "e_out"))
    return x, f64(x["w_lm"]), _weights_dev(x)


@pytest.mark.parametrize("K,B,T", [(16, 256, 1.0), (16, 256, 0.0),
                                   (4, 1, 1.0), (4, 1, 0.0)])
def test_full_size_sweep_corner(lib, K, B, T):
    """A sweep corner at full size through dflash_draft + dflash_verify:
    V=262144 (1024 vocab tiles, verify rows of 128 segments), H=3072.
    K=16 B=256 has M=4096 rows (32 row tiles, 16 CTA-pair row groups,
    128-channel conv tiles); K=4 B=1 runs the single-CTA LM head."""
    w = [p for p in synth.sweep_points()
         if p.K == K and p.B == B and p.T == T][0]
    xw, W64, wdev = _sweep_weights()
    x = dict(xw)
    x.update({k: v for k, v in synth.make_inputs(
        w, tensors=("h", "anchor")).items() if v is not None})
    L = affine_target_device(w, x, seed=1000 + K * 1000 + B)
    seed, cycle = w.seed, 11
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, wdev)
    dv.cycle(to_dev(x["h"][:, :w.K]), to_dev(x["anchor"]), L, w.T, seed,
             cycle)
    torch.cuda.synchronize()
    lib.dflash_check()
    seqs = sampled_sequences(w.B, w.K)
    ties = check_sampled(w, x, dv, L, seqs, seed, cycle, W64=W64)
    print(w.name, "checked sequences", len(seqs), "ties", ties,
          "mean accepted (all)", np_(dv.n).mean())
    del dv, L
    torch.cuda.empty_cache()
