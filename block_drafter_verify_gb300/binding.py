"""ctypes binding of libdflash: the C ABI of include/dflash.h under the same
names, taking torch CUDA tensors.  Argument marshalling only — every step of
the path runs in the library's CUDA kernels.  Importing works without a GPU;
calling needs the built library and a CUDA device, and fails loudly if
either is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

BF16, FP32 = 0, 1
C = 16
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported",
          3: "CUDA runtime error", 4: "non-finite target logit",
          5: "device wait timed out", 6: "token index out of range"}

EXPORTS = ("dflash_workspace_bytes", "dflash_lmhead_topk", "dflash_pair_score",
           "dflash_path_walk", "dflash_draft", "dflash_verify", "dflash_cycle",
           "dflash_verify_noalloc", "dflash_commit", "dflash_path_viterbi",
           "dflash_top16_recall", "dflash_quantize_e4m3_rows",
           "dflash_draft_e4m3", "dflash_philox4x32", "dflash_profile_stage",
           "dflash_set_wait_limit_ns", "dflash_lmhead_topk_shard",
           "dflash_topk_merge_shards", "dflash_verify_shard_stats",
           "dflash_verify_shard_decide", "dflash_verify_shard_draw",
           "dflash_check", "dflash_status_string")
STAGES = ("conv", "lmhead", "merge", "pair_score", "walk", "verify",
          "quant")


class DFlashError(RuntimeError):
    def __init__(self, fn, status):
        self.status = int(status)
        super().__init__(f"{fn}: {STATUS.get(self.status, self.status)}")


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libdflash.so (built by ``build.build()``) and declare its ABI."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(
            f"{p} is missing: build it with block_drafter_verify_gb300.build"
            ".build() (or __graft_entry__.build()); there is no fallback")
    L = ctypes.CDLL(p)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    u64, sz, i64 = ctypes.c_uint64, ctypes.c_size_t, ctypes.c_int64
    sig = {
        "dflash_workspace_bytes": (sz, [i32, i32, i32, i32, i32]),
        "dflash_lmhead_topk": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp,
                                     vp, vp, vp, sz, vp]),
        "dflash_pair_score": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32,
                                    i32, i32, i32, vp, vp]),
        "dflash_path_walk": (i32, [vp, vp, i32, i32, f32, u64, u64, vp, vp,
                                   vp, vp]),
        "dflash_draft": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                               i32, i32, f32, u64, u64, vp, vp, vp, vp, vp,
                               vp, vp, vp, sz, vp]),
        "dflash_verify": (i32, [vp, vp, vp, vp, i32, i32, i32, f32, u64, u64,
                                vp, vp, vp, sz, vp]),
        "dflash_cycle": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                               i32, i32, i32, i32, f32, u64, u64, vp, vp, vp,
                               vp, vp, vp, vp, vp, vp, vp, sz, vp, sz, vp]),
        "dflash_verify_noalloc": (i32, [vp, vp, vp, vp, i32, i32, i32, f32,
                                        u64, u64, vp, vp, vp]),
        "dflash_philox4x32": (i32, [vp, u64, vp, i64, vp]),
        "dflash_commit": (i32, [vp, vp, i32, i32, vp, vp, vp, i32, vp, vp]),
        "dflash_path_viterbi": (i32, [vp, vp, i32, i32, vp, vp, vp, vp]),
        "dflash_top16_recall": (i32, [vp, vp, i32, i32, i32, vp, vp, vp]),
        "dflash_quantize_e4m3_rows": (i32, [vp, i32, i32, vp, vp, vp]),
        "dflash_draft_e4m3": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32,
                                    i32, i32, i32, f32, u64, u64, vp, vp, vp,
                                    vp, vp, vp, vp, vp, sz, vp]),
        "dflash_profile_stage": (i32, [i32, vp, vp]),
        "dflash_set_wait_limit_ns": (i32, [u64]),
        "dflash_lmhead_topk_shard": (i32, [vp, vp, vp, i32, i32, i32, i32,
                                           i32, i32, vp, vp, vp, vp, vp, sz,
                                           vp]),
        "dflash_topk_merge_shards": (i32, [vp, vp, vp, vp, i32, i32, vp, vp,
                                           vp, vp]),
        "dflash_verify_shard_stats": (i32, [vp, vp, vp, i32, i32, i32, i32,
                                            i32, f32, vp, vp, sz, vp]),
        "dflash_verify_shard_decide": (i32, [vp, i32, vp, vp, vp, i32, i32,
                                             i32, f32, u64, u64, vp, vp, vp,
                                             vp]),
        "dflash_verify_shard_draw": (i32, [vp, vp, vp, vp, i32, i32, i32,
                                           i32, i32, f32, vp, vp, sz, vp]),
        "dflash_check": (i32, [vp]),
        "dflash_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = L
    return L


# --------------------------------------------------------------------------
# marshalling helpers
# --------------------------------------------------------------------------
def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype(t):
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return FP32
    raise ValueError(f"unsupported storage dtype {t.dtype}")


def _want(t, dtype, name):
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _call(name, *args):
    st = getattr(load(), name)(*args)
    if st != 0:
        raise DFlashError(name, st)


# --------------------------------------------------------------------------
# the ABI, one function per entry point
# --------------------------------------------------------------------------
def dflash_workspace_bytes(which: int, B: int, K: int, H: int, V: int) -> int:
    return int(load().dflash_workspace_bytes(which, B, K, H, V))


def dflash_lmhead_topk(h, conv_w, w_lm, topv, topi, lse, ws, stream=None):
    """h [B,K,H]; conv_w [2H,H] or None; w_lm [V,H] (same dtype);
    topv [B*K,16] f32, topi [B*K,16] i32, lse [B*K] f32 outputs; ws uint8."""
    B, K, H = h.shape
    V = w_lm.shape[0]
    dt = _dtype(h)
    for t, n in ((w_lm, "w_lm"), (conv_w, "conv_w")):
        if t is not None:
            _want(t, h.dtype, n)
    _want(topv, torch.float32, "topv")
    _want(topi, torch.int32, "topi")
    _want(lse, torch.float32, "lse")
    _call("dflash_lmhead_topk", _ptr(h), _ptr(conv_w), _ptr(w_lm), B, K, H, V,
          dt, _ptr(topv), _ptr(topi), _ptr(lse), _ptr(ws), ws.numel(),
          _stream(stream))


def dflash_pair_score(topv, topi, anchor, h, w_gate, e_in, e_out, scores,
                      stream=None):
    """topv/topi [B,K,16]; anchor [B] i32; h [B,K,H]; w_gate [r,H];
    e_in/e_out [V,r]; scores [B,K,16,16] f32 output."""
    B, K, H = h.shape
    V, r = e_in.shape
    _want(anchor, torch.int32, "anchor")
    _want(scores, torch.float32, "scores")
    _call("dflash_pair_score", _ptr(topv), _ptr(topi), _ptr(anchor), _ptr(h),
          _ptr(w_gate), _ptr(e_in), _ptr(e_out), B, K, H, V, r, _dtype(h),
          _ptr(scores), _stream(stream))


def dflash_path_walk(scores, topi, T, seed, cycle, slot, draft, q,
                     stream=None):
    """scores [B,K,16,16]; topi [B,K,16]; slot/draft [B,K] i32 and
    q [B,K,16] f32 outputs."""
    B, K = scores.shape[:2]
    _call("dflash_path_walk", _ptr(scores), _ptr(topi), B, K, float(T),
          int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1), _ptr(slot),
          _ptr(draft), _ptr(q), _stream(stream))


def dflash_draft(h, conv_w, w_lm, w_gate, e_in, e_out, anchor, T, seed,
                 cycle, topv, topi, lse, scores, slot, draft, q, ws,
                 stream=None):
    """Steps a1-a4 in one call: h [B,K,H]; conv_w [2H,H] or None; w_lm
    [V,H]; w_gate [r,H]; e_in/e_out [V,r] (one storage dtype); anchor [B]
    i32; outputs topv/topi [B*K,16], lse [B*K], scores [B,K,16,16], slot and
    draft [B,K] i32, q [B,K,16]; ws uint8 (workspace kind 2)."""
    B, K, H = h.shape
    V = w_lm.shape[0]
    r = w_gate.shape[0]
    _call("dflash_draft", _ptr(h), _ptr(conv_w), _ptr(w_lm), _ptr(w_gate),
          _ptr(e_in), _ptr(e_out), _ptr(anchor), B, K, H, V, r, _dtype(h),
          float(T), int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1),
          _ptr(topv), _ptr(topi), _ptr(lse), _ptr(scores), _ptr(slot),
          _ptr(draft), _ptr(q), _ptr(ws), ws.numel(), _stream(stream))


def dflash_quantize_e4m3_rows(x, codes, scale, stream=None):
    """x [R,H] bf16 -> codes [R,H] uint8 (E4M3) and scale [R] f32."""
    R, H = x.shape
    _want(x, torch.bfloat16, "x")
    _want(codes, torch.uint8, "codes")
    _want(scale, torch.float32, "scale")
    _call("dflash_quantize_e4m3_rows", _ptr(x), R, H, _ptr(codes),
          _ptr(scale), _stream(stream))


def dflash_draft_e4m3(h, conv_w, w_codes, w_scale, w_gate, e_in, e_out,
                      anchor, T, seed, cycle, topv, topi, lse, scores, slot,
                      draft, q, ws, stream=None):
    """dflash_draft (bf16, with a conv) with the LM head on E4M3 codes:
    w_codes [V,H] uint8 and w_scale [V] f32 from dflash_quantize_e4m3_rows;
    ws uint8 (workspace kind 3)."""
    B, K, H = h.shape
    V = w_codes.shape[0]
    r = w_gate.shape[0]
    _want(h, torch.bfloat16, "h")
    _want(w_codes, torch.uint8, "w_codes")
    _call("dflash_draft_e4m3", _ptr(h), _ptr(conv_w), _ptr(w_codes),
          _ptr(w_scale), _ptr(w_gate), _ptr(e_in), _ptr(e_out), _ptr(anchor),
          B, K, H, V, r, float(T), int(seed) & (2**64 - 1),
          int(cycle) & (2**64 - 1), _ptr(topv), _ptr(topi), _ptr(lse),
          _ptr(scores), _ptr(slot), _ptr(draft), _ptr(q), _ptr(ws),
          ws.numel(), _stream(stream))


def dflash_verify(target_logits, draft, topi, q, T, seed, cycle, n_accepted,
                  out_tok, ws, stream=None):
    """target_logits [B,K+1,V] f32; draft [B,K]; topi/q [B,K,16];
    n_accepted [B] and out_tok [B,K+1] i32 outputs; ws uint8."""
    B, K1, V = target_logits.shape
    _want(target_logits, torch.float32, "target_logits")
    _call("dflash_verify", _ptr(target_logits), _ptr(draft), _ptr(topi),
          _ptr(q), B, K1 - 1, V, float(T), int(seed) & (2**64 - 1),
          int(cycle) & (2**64 - 1), _ptr(n_accepted), _ptr(out_tok),
          _ptr(ws), ws.numel(), _stream(stream))


def dflash_cycle(h, conv_w, w_lm, w_scale, w_gate, e_in, e_out, anchor,
                 target_logits, T, seed, cycle, topv, topi, lse, scores, slot,
                 draft, q, n_accepted, out_tok, ws_draft, ws_verify,
                 stream=None):
    """One whole cycle: dflash_draft (w_scale None; else dflash_draft_e4m3
    with w_lm the E4M3 codes [V,H] uint8 and w_scale [V] f32) and
    dflash_verify of its draft; the arguments and outputs of the two calls,
    ws_draft (workspace kind 2, or 3 with w_scale) and ws_verify (kind 1)."""
    B, K, H = h.shape
    V = w_lm.shape[0]
    r = w_gate.shape[0]
    _want(target_logits, torch.float32, "target_logits")
    if w_scale is not None:
        _want(h, torch.bfloat16, "h")
        _want(w_lm, torch.uint8, "w_lm")
    _call("dflash_cycle", _ptr(h), _ptr(conv_w), _ptr(w_lm), _ptr(w_scale),
          _ptr(w_gate), _ptr(e_in), _ptr(e_out), _ptr(anchor),
          _ptr(target_logits), B, K, H, V, r, _dtype(h), float(T),
          int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1), _ptr(topv),
          _ptr(topi), _ptr(lse), _ptr(scores), _ptr(slot), _ptr(draft),
          _ptr(q), _ptr(n_accepted), _ptr(out_tok), _ptr(ws_draft),
          ws_draft.numel(), _ptr(ws_verify), ws_verify.numel(),
          _stream(stream))


def dflash_verify_noalloc(target_logits, draft, topi, q, T, seed, cycle,
                          n_accepted, out_tok, stream=None):
    """dflash_verify with the library's own fixed scratch, for callers that
    cannot allocate device memory; same arguments minus the workspace."""
    B, K1, V = target_logits.shape
    _want(target_logits, torch.float32, "target_logits")
    _call("dflash_verify_noalloc", _ptr(target_logits), _ptr(draft),
          _ptr(topi), _ptr(q), B, K1 - 1, V, float(T),
          int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1),
          _ptr(n_accepted), _ptr(out_tok), _stream(stream))


def dflash_path_viterbi(scores, topi, slot, draft, q, stream=None):
    """scores [B,K,16,16] f32, topi [B,K,16] i32 -> slot, draft [B,K] i32,
    q [B,K,16] f32 (one-hot): the global max-sum path (T = 0)."""
    B, K = scores.shape[:2]
    _call("dflash_path_viterbi", _ptr(scores), _ptr(topi), B, K, _ptr(slot),
          _ptr(draft), _ptr(q), _stream(stream))


def dflash_top16_recall(target_logits, topi, target_argmax, in_top16,
                        stream=None):
    """target_logits [B,K+1,V] f32, topi [B,K,16] -> target_argmax and
    in_top16 [B,K] i32 for the K drafted positions."""
    B, K1, V = target_logits.shape
    _want(target_logits, torch.float32, "target_logits")
    _call("dflash_top16_recall", _ptr(target_logits), _ptr(topi), B, K1 - 1,
          V, _ptr(target_argmax), _ptr(in_top16), _stream(stream))


COMMIT_STATS = 3 + 16 + 1


def dflash_commit(n_accepted, out_tok, anchor, tokens, length, stats,
                  stream=None):
    """n_accepted [B], out_tok [B,K+1] i32 (from dflash_verify); anchor [B]
    i32 in/out; tokens [B,capacity] and length [B] i32 in/out; stats
    [COMMIT_STATS] int64 in/out (accepted, passes, emitted, histogram)."""
    B, K1 = out_tok.shape
    _call("dflash_commit", _ptr(n_accepted), _ptr(out_tok), B, K1 - 1,
          _ptr(anchor), _ptr(tokens), _ptr(length), tokens.shape[1],
          _ptr(stats), _stream(stream))


def dflash_philox4x32(ctr, seed, out, stream=None):
    """ctr [n,4] and out [n,4] int32 tensors holding uint32 words."""
    _call("dflash_philox4x32", _ptr(ctr), int(seed) & (2**64 - 1), _ptr(out),
          ctr.shape[0], _stream(stream))


def dflash_profile_stage(stage, begin=None, end=None):
    """Record torch.cuda.Event ``begin``/``end`` around the kernel of
    ``stage`` (index or name in STAGES) on every later call; None stops.
    The events must already exist on the device (record them once)."""
    if isinstance(stage, str):
        stage = STAGES.index(stage)
    b = None if begin is None else ctypes.c_void_p(begin.cuda_event)
    e = None if end is None else ctypes.c_void_p(end.cuda_event)
    _call("dflash_profile_stage", int(stage), b, e)


def dflash_set_wait_limit_ns(ns):
    """Limit of the tensor-core kernels' bounded waits in later launches
    (0 = the default 2 s); for tests of the timeout path."""
    _call("dflash_set_wait_limit_ns", int(ns))


SHARD_STATS, SHARD_PLAN = 20, 8


def dflash_lmhead_topk_shard(h, conv_w, w_lm_shard, v0, part_v, part_i,
                             part_m, part_s, ws, stream=None):
    """h [B,K,H]; conv_w [2H,H] or None; w_lm_shard [V_shard,H] (rows of
    the vocabulary from v0); outputs part_v [B*K,16] f32, part_i [B*K,16]
    i32 (global ids), part_m, part_s [B*K] f32; ws uint8 (kind 0 for
    V_shard)."""
    B, K, H = h.shape
    Vs = w_lm_shard.shape[0]
    _want(part_i, torch.int32, "part_i")
    _call("dflash_lmhead_topk_shard", _ptr(h), _ptr(conv_w), _ptr(w_lm_shard),
          B, K, H, Vs, int(v0), _dtype(h), _ptr(part_v), _ptr(part_i),
          _ptr(part_m), _ptr(part_s), _ptr(ws), ws.numel(), _stream(stream))


def dflash_topk_merge_shards(part_v, part_i, part_m, part_s, topv, topi, lse,
                             stream=None):
    """part_v, part_i [S,M,16]; part_m, part_s [S,M] -> topv, topi [M,16],
    lse [M]."""
    S, M = part_m.shape
    _call("dflash_topk_merge_shards", _ptr(part_v), _ptr(part_i),
          _ptr(part_m), _ptr(part_s), S, M, _ptr(topv), _ptr(topi), _ptr(lse),
          _stream(stream))


def dflash_verify_shard_stats(target_shard, draft, topi, v0, V, T, stats, ws,
                              stream=None):
    """target_shard [B,K+1,V_shard] f32 (ids from v0 of V); draft [B,K];
    topi [B,K,16] -> stats [B*(K+1), SHARD_STATS] f32; ws uint8 (kind 1
    for V_shard), kept for dflash_verify_shard_draw."""
    B, K1, Vs = target_shard.shape
    _want(target_shard, torch.float32, "target_shard")
    _call("dflash_verify_shard_stats", _ptr(target_shard), _ptr(draft),
          _ptr(topi), B, K1 - 1, Vs, int(v0), int(V), float(T), _ptr(stats),
          _ptr(ws), ws.numel(), _stream(stream))


def dflash_verify_shard_decide(stats, draft, topi, q, V, T, seed, cycle,
                               n_accepted, out_tok, plan, stream=None):
    """stats [S, B*(K+1), SHARD_STATS] -> n_accepted [B], out_tok [B,K+1],
    plan [B, SHARD_PLAN] f32."""
    S = stats.shape[0]
    B, K = draft.shape
    _call("dflash_verify_shard_decide", _ptr(stats), S, _ptr(draft),
          _ptr(topi), _ptr(q), B, K, int(V), float(T),
          int(seed) & (2**64 - 1), int(cycle) & (2**64 - 1),
          _ptr(n_accepted), _ptr(out_tok), _ptr(plan), _stream(stream))


def dflash_verify_shard_draw(target_shard, plan, topi, q, shard, v0, T,
                             out_tok, ws, stream=None):
    """The draws the plan gives to shard `shard` (its target_shard and the
    ws of its stats call) into out_tok."""
    B, K1, Vs = target_shard.shape
    _call("dflash_verify_shard_draw", _ptr(target_shard), _ptr(plan),
          _ptr(topi), _ptr(q), int(shard), B, K1 - 1, Vs, int(v0), float(T),
          _ptr(out_tok), _ptr(ws), ws.numel(), _stream(stream))


def dflash_check(stream=None):
    """Synchronise and raise if a kernel flagged a problem."""
    _call("dflash_check", _stream(stream))


# --------------------------------------------------------------------------
# one cycle with its buffers (still marshalling: four ABI calls)
# --------------------------------------------------------------------------
class DraftVerify:
    """Device buffers for one workload shape plus the four calls of a cycle.

    weights: dict with w_conv (or None), w_lm, w_gate, e_in, e_out as CUDA
    tensors of one storage dtype.  ``cycle(h, anchor, L, T, seed, c)`` runs
    conv + LM head + top-16, pair scores, walk and verify on the current
    stream and returns the (device) n_accepted and out_tok tensors.
    With ``lm_e4m3`` (bf16 with a conv) W_lm is quantized once to E4M3
    codes and row scales, and draft_all runs dflash_draft_e4m3.
    """

    def __init__(self, B, K, H, V, r, weights, device="cuda", lm_e4m3=False):
        self.B, self.K, self.H, self.V, self.r = B, K, H, V, r
        self.w = weights
        self.lm_e4m3 = bool(lm_e4m3)
        dev = torch.device(device)
        M = B * K
        f32, i32 = torch.float32, torch.int32
        self.topv = torch.empty(M, C, dtype=f32, device=dev)
        self.topi = torch.empty(M, C, dtype=i32, device=dev)
        self.lse = torch.empty(M, dtype=f32, device=dev)
        self.scores = torch.empty(B, K, C, C, dtype=f32, device=dev)
        self.slot = torch.empty(B, K, dtype=i32, device=dev)
        self.draft = torch.empty(B, K, dtype=i32, device=dev)
        self.q = torch.empty(B, K, C, dtype=f32, device=dev)
        self.n = torch.empty(B, dtype=i32, device=dev)
        self.out = torch.empty(B, K + 1, dtype=i32, device=dev)
        self.ws_lm = torch.empty(dflash_workspace_bytes(0, B, K, H, V),
                                 dtype=torch.uint8, device=dev)
        self.ws_v = torch.empty(dflash_workspace_bytes(1, B, K, H, V),
                                dtype=torch.uint8, device=dev)
        self.ws_d = torch.empty(
            dflash_workspace_bytes(3 if self.lm_e4m3 else 2, B, K, H, V),
            dtype=torch.uint8, device=dev)
        if self.lm_e4m3:
            self.w_codes = torch.empty(V, H, dtype=torch.uint8, device=dev)
            self.w_scale = torch.empty(V, dtype=f32, device=dev)
            dflash_quantize_e4m3_rows(weights["w_lm"], self.w_codes,
                                      self.w_scale)

    def lmhead(self, h, stream=None):
        dflash_lmhead_topk(h, self.w["w_conv"], self.w["w_lm"], self.topv,
                           self.topi, self.lse, self.ws_lm, stream)

    def pair_score(self, h, anchor, stream=None):
        B, K = self.B, self.K
        dflash_pair_score(self.topv.view(B, K, C), self.topi.view(B, K, C),
                          anchor, h, self.w["w_gate"], self.w["e_in"],
                          self.w["e_out"], self.scores, stream)

    def walk(self, T, seed, cycle, stream=None):
        dflash_path_walk(self.scores, self.topi.view(self.B, self.K, C), T,
                         seed, cycle, self.slot, self.draft, self.q, stream)

    def verify(self, L, T, seed, cycle, stream=None):
        dflash_verify(L, self.draft, self.topi.view(self.B, self.K, C),
                      self.q, T, seed, cycle, self.n, self.out, self.ws_v,
                      stream)

    def draft_all(self, h, anchor, T, seed, cycle, stream=None):
        """Steps a1-a4 in one dflash_draft call (gate inside the conv)."""
        if self.lm_e4m3:
            dflash_draft_e4m3(h, self.w["w_conv"], self.w_codes, self.w_scale,
                              self.w["w_gate"], self.w["e_in"],
                              self.w["e_out"], anchor, T, seed, cycle,
                              self.topv, self.topi, self.lse, self.scores,
                              self.slot, self.draft, self.q, self.ws_d, stream)
            return
        dflash_draft(h, self.w["w_conv"], self.w["w_lm"], self.w["w_gate"],
                     self.w["e_in"], self.w["e_out"], anchor, T, seed, cycle,
                     self.topv, self.topi, self.lse, self.scores, self.slot,
                     self.draft, self.q, self.ws_d, stream)

    def cycle(self, h, anchor, L, T, seed, cycle, stream=None):
        """One draft-verify cycle in one dflash_cycle call (dflash_draft +
        dflash_verify, the verify's tickets zeroed by the conv launch)."""
        e4 = self.lm_e4m3
        dflash_cycle(h, self.w["w_conv"],
                     self.w_codes if e4 else self.w["w_lm"],
                     self.w_scale if e4 else None, self.w["w_gate"],
                     self.w["e_in"], self.w["e_out"], anchor, L, T, seed,
                     cycle, self.topv, self.topi, self.lse, self.scores,
                     self.slot, self.draft, self.q, self.n, self.out,
                     self.ws_d, self.ws_v, stream)
        return self.n, self.out

    def commit(self, anchor, tokens, length, stats, stream=None):
        """Commit the last verify's tokens; the anchor moves to the last
        emitted token of each sequence."""
        dflash_commit(self.n, self.out, anchor, tokens, length, stats, stream)

    def y(self, fused=False):
        """y written by the last lmhead (or, fused=True, draft_all) call:
        the conv output in the storage dtype."""
        dt = self.w["w_lm"].dtype
        n = self.B * self.K * self.H
        ws = self.ws_d if fused else self.ws_lm
        return ws[: n * (2 if dt == torch.bfloat16 else 4)].view(
            dt).view(self.B, self.K, self.H)

    def y_e4m3(self):
        """y's E4M3 codes [B*K, H] and row scales [B*K] written by the last
        draft_all with lm_e4m3: the workspace of kind 3 holds them after
        the first dflash_workspace_bytes(2, ...) bytes, the scales from the
        next 256-byte boundary after the codes."""
        M, H = self.B * self.K, self.H
        off = dflash_workspace_bytes(2, self.B, self.K, H, self.V)
        off2 = off + (M * H + 255) // 256 * 256
        codes = self.ws_d[off: off + M * H].view(M, H)
        scale = self.ws_d[off2: off2 + 4 * M].view(torch.float32)
        return codes, scale
