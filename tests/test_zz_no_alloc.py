"""dflash_verify_noalloc: verify for callers that cannot allocate device
memory (serving loops whose memory belongs to another engine's allocator,
code where allocating is not allowed, C callers without an allocator).  It
keeps its scratch in the library's own fixed device array; its results must
equal dflash_verify's, call after call, since every call reuses (and must
re-clear) that array.  This file is collected last."""
import numpy as np
import pytest
import torch

import synth
from parity import draft_logits_oracle, np_, to_dev

pytestmark = pytest.mark.gpu
C = 16


def _drafts(lib, w, x):
    """Candidates, drafts and q from the library's own first three steps."""
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r,
                         {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate",
                                                    "e_in", "e_out")})
    h = to_dev(x["h"][:, :w.K])
    dv.lmhead(h)
    dv.pair_score(h, to_dev(x["anchor"]))
    dv.walk(w.T, 17, 4)
    return dv


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_noalloc_verify_matches_verify_on_consecutive_calls(lib, T):
    w = synth.Workload("noalloc", B=6, K=5, V=4099, H=128, r=32, dtype="bf16",
                       T=T, seed=21, w_lm_sd=0.2, conv_sd=0.05, sel_sd=0.1,
                       target=("affine", 0.9, 0.7))
    x = synth.make_inputs(w)
    L = to_dev(synth.target_logits(w, draft_logits_oracle(x, w)))
    dv = _drafts(lib, w, x)
    topi = dv.topi.view(w.B, w.K, C)
    i32 = dict(dtype=torch.int32, device="cuda")
    for call in range(2):                       # two calls in a row
        cyc = 100 + call
        n_ref = torch.empty(w.B, **i32)
        out_ref = torch.empty(w.B, w.K + 1, **i32)
        ws = torch.empty(lib.dflash_workspace_bytes(1, w.B, w.K, w.H, w.V),
                         dtype=torch.uint8, device="cuda")
        lib.dflash_verify(L, dv.draft, topi, dv.q, T, 7, cyc, n_ref, out_ref,
                          ws)
        n = torch.full((w.B,), -7, **i32)
        out = torch.full((w.B, w.K + 1), -7, **i32)
        lib.dflash_verify_noalloc(L, dv.draft, topi, dv.q, T, 7, cyc, n, out)
        torch.cuda.synchronize()
        lib.dflash_check()
        assert np.array_equal(np_(n), np_(n_ref))
        assert np.array_equal(np_(out), np_(out_ref))


def _valid_inputs(B, K, V, seed):
    """Target logits and drafts of the right shapes on the device (drafts
    among their candidates, q a distribution over them)."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    L = torch.randn(B, K + 1, V, generator=g, device="cuda")
    topi = torch.randint(0, V, (B, K, C), generator=g, device="cuda",
                         dtype=torch.int32)
    q = torch.rand(B, K, C, generator=g, device="cuda") + 0.01
    q /= q.sum(-1, keepdim=True)
    draft = topi[:, :, 0].contiguous()
    return L, draft, topi, q


LIMIT = 4 << 20


@pytest.mark.parametrize("V,K,B", [
    (151936, 16, 405),     # the largest batch whose scratch fits, K = 16
    (151936, 16, 406),     # one sequence more: over the limit
    (262144, 14, 256),     # B = 256 fits up to K = 14 at V = 262144
    (262144, 15, 256),     # ... and not at K = 15
])
def test_noalloc_verify_at_the_scratch_limit(lib, V, K, B):
    """Just inside the 4 MiB limit the call runs and matches dflash_verify;
    just outside it is refused with DFLASH_ERR_UNSUPPORTED."""
    need = lib.dflash_workspace_bytes(1, B, K, 0, V)
    L, draft, topi, q = _valid_inputs(B, K, V, seed=B + K)
    i32 = dict(dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, **i32)
    out = torch.full((B, K + 1), -7, **i32)
    if need > LIMIT:
        with pytest.raises(lib.DFlashError) as e:
            lib.dflash_verify_noalloc(L, draft, topi, q, 1.0, 3, 1, n, out)
        assert e.value.status == 2      # DFLASH_ERR_UNSUPPORTED
        assert int(n.min()) == -7       # nothing launched
        return
    n_ref = torch.empty(B, **i32)
    out_ref = torch.empty(B, K + 1, **i32)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    lib.dflash_verify(L, draft, topi, q, 1.0, 3, 1, n_ref, out_ref, ws)
    lib.dflash_verify_noalloc(L, draft, topi, q, 1.0, 3, 1, n, out)
    torch.cuda.synchronize()
    lib.dflash_check()
    assert torch.equal(n, n_ref) and torch.equal(out, out_ref)


def test_noalloc_verify_refuses_sizes_beyond_its_scratch(lib):
    # 278,528 target rows: their per-row results and tickets alone outgrow
    # the 4 MiB array
    B, K, V = 16384, 16, 64
    assert lib.dflash_workspace_bytes(1, B, K, 0, V) > 4 << 20
    L = torch.zeros(B, K + 1, V, device="cuda")
    draft = torch.zeros(B, K, dtype=torch.int32, device="cuda")
    topi = torch.zeros(B, K, C, dtype=torch.int32, device="cuda")
    q = torch.zeros(B, K, C, device="cuda")
    n = torch.empty(B, dtype=torch.int32, device="cuda")
    out = torch.empty(B, K + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(lib.DFlashError) as e:
        lib.dflash_verify_noalloc(L, draft, topi, q, 1.0, 0, 0, n, out)
    assert e.value.status == 2      # DFLASH_ERR_UNSUPPORTED
