"""Failure detection on the device without a GPU fault: a bounded wait
inside the tensor-core kernels gives up, the kernel drains and exits, and
the host reads DFLASH_ERR_DEVICE_TIMEOUT from the error word; the context
stays usable and the next call is correct."""
import numpy as np
import pytest
import torch

import oracle
import synth
from parity import ERR_C, check_topk, check_y, f64, to_dev

pytestmark = pytest.mark.gpu


def _workload():
    # one row tile (B*K = 32): single-CTA LM head; 32 k-steps per tile, so
    # the epilogue's accumulator waits last microseconds
    return synth.Workload("timeout", B=4, K=8, V=151936, H=2048, r=32,
                          dtype="bf16", T=1.0, seed=51, w_lm_sd=0.02,
                          conv_sd=0.05, sel_sd=0.1,
                          target=("affine", 0.9, 1.0))


def test_wait_limit_gives_up_and_the_next_call_is_correct(lib):
    w = _workload()
    x = synth.make_inputs(w)
    weights = {k: to_dev(x[k]) for k in ("w_conv", "w_lm", "w_gate", "e_in",
                                         "e_out")}
    dv = lib.DraftVerify(w.B, w.K, w.H, w.V, w.r, weights)
    h = to_dev(x["h"][:, :w.K])
    lib.dflash_check()                       # nothing pending
    try:
        lib.dflash_set_wait_limit_ns(100)    # far below any wait here
        dv.lmhead(h)                         # conv + LM head + merge
        with pytest.raises(lib.DFlashError) as e:
            lib.dflash_check()
        assert e.value.status == 5           # DFLASH_ERR_DEVICE_TIMEOUT
    finally:
        lib.dflash_set_wait_limit_ns(0)      # back to the default (2 s)
    lib.dflash_check()                       # the word was cleared
    dv.lmhead(h)
    torch.cuda.synchronize()
    lib.dflash_check()
    h64 = f64(h)
    W = f64(x["w_conv"])
    y = dv.y()
    check_y(y, oracle.conv2tap(h64, W), oracle.conv2tap(np.abs(h64),
                                                        np.abs(W)), w.dtype)
    y64 = f64(y).reshape(-1, w.H)
    W_lm = f64(x["w_lm"])
    ref = oracle.lmhead_topk(y64, W_lm, want_logits=True)
    A = np.abs(y64) @ np.abs(W_lm).T
    check_topk(dv.topv, dv.topi, dv.lse, ref, A, ERR_C[w.dtype])
