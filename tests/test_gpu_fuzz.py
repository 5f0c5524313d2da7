"""Seeded random shapes through the fused draft (bf16 and 8-bit LM heads)
and verify, each stage against the oracle: ragged V (including last tiles
whose second half lies beyond V), ragged H, single CTAs and CTA pairs,
several row groups, T = 0 and T > 0."""
import numpy as np
import pytest

import synth
from parity import draft_logits_oracle

pytestmark = pytest.mark.gpu


def _shapes(n=12, seed=2024):
    g = np.random.default_rng(seed)
    out = []
    for i in range(n):
        B = int(g.integers(1, 24))
        K = int(g.integers(1, 17))
        H = int(16 * g.integers(2, 17))          # 32..256, multiple of 16
        V = int(g.integers(17, 6000))
        r = int(g.choice([8, 16, 40, 64, 128, 256]))
        T = float(g.choice([0.0, 0.7, 1.0, 1.5]))
        out.append((i, B, K, H, V, r, T))
    return out


@pytest.mark.parametrize("i,B,K,H,V,r,T", _shapes())
@pytest.mark.parametrize("e4m3", [False, True])
def test_fuzz_fused_draft(lib, i, B, K, H, V, r, T, e4m3):
    from test_gpu_e4m3 import run_e4m3
    from test_gpu_parity import run_fused
    w = synth.Workload(f"fuzz{i}", B=B, K=K, V=V, H=H, r=r, dtype="bf16",
                       T=T, seed=100 + i, w_lm_sd=0.1, conv_sd=0.05,
                       sel_sd=0.1, target=("affine", 0.9, 1.0))
    x = synth.make_inputs(w)
    L = synth.target_logits(w, draft_logits_oracle(x, w))
    if e4m3:
        run_e4m3(lib, w, x, L, seed=11 + i, cycle=i)
    else:
        run_fused(lib, w, x, L, seed=11 + i, cycle=i)
