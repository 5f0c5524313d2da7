"""dflash_cycle (draft and verify in one call; on the tensor-core paths the
conv launch zeroes the verify's tickets) against dflash_draft followed by
dflash_verify: every output equal bit for bit, with the verify workspace
holding garbage before the call, and again on a second call."""
import pytest
import torch

import synth
from parity import to_dev

pytestmark = pytest.mark.gpu

CASES = [
    ("b32k8", dict(V=30011)),                # CTA-pair LM head, T = 1
    ("b32k8", dict(B=4, V=30011, T=0.0)),    # single-CTA LM head, greedy
    ("b32k8e4m3", dict(V=30016)),            # 8-bit LM head
    ("tiny_conv", dict(B=3, T=1.0)),         # fp32: the separate calls
]


def _dv(lib, w, x):
    weights = {k: (None if x[k] is None else to_dev(x[k]))
               for k in ("w_conv", "w_lm", "w_gate", "e_in", "e_out")}
    return lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, weights,
                           lm_e4m3=w.lm_e4m3)


OUTS = ("topv", "topi", "lse", "scores", "slot", "draft", "q", "n", "out")


@pytest.mark.parametrize("name,over", CASES)
def test_cycle_equals_draft_then_verify(lib, name, over):
    w = synth.get(name, **over)
    x = synth.make_inputs(w)
    h = to_dev(x["h"][:, :w.K])
    anchor = to_dev(x["anchor"])
    g = torch.Generator(device="cuda").manual_seed(w.B * 131 + w.V)
    L = torch.randn(w.B, w.K + 1, w.V, generator=g, device="cuda") * 3.0
    ref = _dv(lib, w, x)
    ref.draft_all(h, anchor, w.T, 11, 4)
    ref.verify(L, w.T, 11, 4)
    got = _dv(lib, w, x)
    for rep in range(2):
        got.ws_v.fill_(0xFF)                # tickets must not be trusted
        got.cycle(h, anchor, L, w.T, 11, 4)
        torch.cuda.synchronize()
        lib.dflash_check()
        for k in OUTS:
            a, b = getattr(ref, k), getattr(got, k)
            assert torch.equal(a, b), f"{name} {over}: {k} differs (call {rep})"
    assert int(got.n.min()) >= 0 and int(got.n.max()) <= w.K
