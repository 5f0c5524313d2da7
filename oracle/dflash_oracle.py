"""Plain CPU oracle of the DFlash 2 draft-verify hot path.

TEST INFRASTRUCTURE ONLY.  This module is imported by tests/, by
``__graft_entry__.smoke()`` and by the CPU-baseline / reference legs of
``bench.py``, nowhere else.  It shares no code with the CUDA library and
never imports it.  It is deliberately slow: float64 numpy, one library
primitive per step (a matmul, a sort, a cumulative sum), loops over
sequences and positions written out.

Sources (page title, section):
  [DC]  "DFlash 2: Block diffusion, wearing a drafter's coat"
  [2B]  "A 2B Drafter Made a 27B Model 3.4x Faster. Same Exact Output."
  [KP]  "DFlash 2: Keep Drafting Parallel"
  [QW]  "Qwen3.8-27B-DFlash2" (aiany.app item page)

Readings where the pages are silent or garbled (each also listed in the
design notes):
  * conv: ``w_j(h) = W_j h`` (linear, no bias), ``x_t = h_t``, causal zero
    pad ``h_{-1} = 0``, no residual; y rounded to the storage dtype.
  * pair score: ``S_t(a, b) = U_t(b) + <E_in(a), G(h_t) * E_out(b)>`` with
    ``G(h) = sigmoid(W_g h)``; the page's own equation did not survive
    extraction, only its description ([KP] "A Lightweight Path Selector").
  * U_t(b) is the raw drafter logit of candidate b (not the log-prob).
  * the walk starts from the verified (anchor) token; greedy takes the best
    successor, sampling draws from softmax(S_t(prev, .)/T) over the 16
    candidates, and that conditional is the draft distribution q_t used by
    the verifier (zero off the candidates).
  * inverse CDF: the smallest index whose running sum is strictly greater
    than u * total.
  * accept test ``u * q(x) < p(x)`` (= ``u < min(1, p/q)``).
  * degenerate residual (all weights zero): sample from p instead.
  * bonus token when all K drafts are accepted: drawn from target row K.
  * T = 0: greedy walk, accept iff the draft equals the target argmax, emit
    the target argmax at the first mismatch / bonus slot.
  * decisions (ranking, argmax, accept, inverse CDF) compare their operands
    rounded to fp32, the precision the CUDA kernels decide in; the operands
    themselves are computed in float64 from the exact input values.
  * 8-bit LM head (the pages name quantized drafter builds, not a format):
    OCP FP8 E4M3 codes with one fp32 scale per row for y and W_lm, scale =
    max|x| / 448, codes rounded to nearest even and saturated, both
    divisions in fp32 (the codes are decisions taken in fp32); the logits
    are the exact products of the dequantized operands.
  * selector variants (beyond the pages' greedy and sampled walks): the
    Viterbi walk maximises the sum of pair scores along the path, ties to
    the lowest slot; recall@16 is measured against the target's first
    argmax.
"""
from __future__ import annotations

import numpy as np

from . import philox

C = 16  # candidates per position ([DC] "Sixteen candidates per position")


# --------------------------------------------------------------------------
# storage rounding
# --------------------------------------------------------------------------
def round_bf16(x) -> np.ndarray:
    """Round to the nearest bfloat16 (ties to even), via float32.

    bfloat16 is the upper 16 bits of an IEEE float32; rounding adds
    0x7FFF plus the lowest kept bit before truncating the low half.
    Returns float32 values that are exactly representable in bf16.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) \
        & np.uint64(0xFFFF0000)
    return u.astype(np.uint32).view(np.float32)


def to_storage(x, dtype: str) -> np.ndarray:
    """float64 -> the storage dtype's values (float32 array)."""
    return round_bf16(x) if dtype == "bf16" else np.asarray(x, np.float32)


# --------------------------------------------------------------------------
# a1: two-tap dynamic depthwise convolution
# --------------------------------------------------------------------------
def conv2tap(h: np.ndarray, w_conv) -> np.ndarray:
    """y_t = w0(h_t) * x_t + w1(h_t) * x_{t-1}, per channel, in float64.

    [DC] "Suffix-decay convolution": a two-tap dynamic depthwise conv that
    mixes each position with its predecessor; [2B] "The two fixes": "mixes
    each position's representation with its immediate predecessor's".
    h: [B, K, H]; w_conv: [2H, H] (rows 0..H-1 = W0, H..2H-1 = W1) or None,
    in which case y = h.  The predecessor of the first block position is
    zero (causal pad); positions never mix across sequences.
    """
    h = np.asarray(h, dtype=np.float64)
    if w_conv is None:
        return h.copy()
    B, K, H = h.shape
    W = np.asarray(w_conv, dtype=np.float64)
    W0, W1 = W[:H], W[H:]
    y = np.empty_like(h)
    for b in range(B):
        # the dynamic tap weights of every position of the sequence at once:
        # row t of w0 is W0 h_t, row t of w1 is W1 h_t
        w0 = h[b] @ W0.T
        w1 = h[b] @ W1.T
        prev = np.zeros((K, H))          # h_{t-1}, zero before the block
        prev[1:] = h[b, :-1]
        y[b] = w0 * h[b] + w1 * prev
    return y


# --------------------------------------------------------------------------
# a2: LM head, logsumexp, top-16
# --------------------------------------------------------------------------
def lmhead_topk(y: np.ndarray, w_lm: np.ndarray, want_logits=False):
    """Drafter logits U = y W^T, their logsumexp and the top-16 per row.

    [DC] "Sixteen candidates per position"; [2B] "What a block-diffusion
    drafter is": the drafter keeps its 16 best tokens per block slot;
    [KP] "A Lightweight Path Selector": U_t is the drafter's own logit.
    y: [M, H]; w_lm: [V, H].  Returns topv f32 [M,16], topi i32 [M,16]
    (descending value, ties to the lower token id, padding -inf / -1 when
    V < 16), lse f64 [M]; with want_logits also U f64 [M, V].
    """
    y = np.asarray(y, dtype=np.float64)
    W = np.asarray(w_lm, dtype=np.float64)
    U = y @ W.T                                   # [M, V] float64
    M, V = U.shape
    m = U.max(axis=1, keepdims=True)
    lse = (m + np.log(np.exp(U - m).sum(axis=1, keepdims=True)))[:, 0]
    U32 = U.astype(np.float32)                    # ranking precision
    order = np.argsort(-U32, axis=1, kind="stable")[:, :C]
    n = min(C, V)
    topi = np.full((M, C), -1, np.int32)
    topv = np.full((M, C), -np.inf, np.float32)
    topi[:, :n] = order[:, :n]
    topv[:, :n] = np.take_along_axis(U32, order[:, :n], axis=1)
    out = (topv, topi, lse)
    return out + (U,) if want_logits else out


# --------------------------------------------------------------------------
# a2 with 8-bit LM-head operands (quantized drafters: [2B] "What a
# block-diffusion drafter is" and [KP] "What Comes Next" ship GGUF Q4_K_M
# drafter builds and note that quantized kernels may prefer other block
# sizes).  The format is OCP FP8 E4M3 ("e4m3fn"): 1 sign bit, 4 exponent
# bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, the
# largest finite magnitude is 448, subnormals are m/8 * 2^-6.
# --------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_decode(codes) -> np.ndarray:
    """Values (float64) of E4M3 codes, NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6,
                   (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Nearest E4M3 code of each finite float32 value (ties to the even
    mantissa), magnitudes beyond 448 saturated to 448; the sign of zero is
    kept.  Works on the exact float64 value of the float32 input: the
    quantum at magnitude a is 2^(max(floor(log2 a), -6) - 3)."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e4m3_encode: non-finite input")
    neg = np.signbit(x)
    a = np.abs(x)
    _, E = np.frexp(np.where(a > 0, a, 1.0))     # a = f * 2^E, f in [0.5, 1)
    e = np.maximum(E - 1, -6)                     # floor(log2 a), clamped
    quantum = np.exp2((e - 3).astype(np.float64))
    r = np.rint(a / quantum) * quantum            # rint: ties to even
    r = np.minimum(np.where(a > 0, r, 0.0), E4M3_MAX)
    # the code of the (representable) magnitude r
    _, Er = np.frexp(np.where(r > 0, r, 1.0))
    er = Er - 1
    normal = r >= 2.0 ** -6
    exp_field = np.where(normal, er + 7, 0)
    mant = np.where(normal, r / np.exp2(er.astype(np.float64)) * 8 - 8,
                    r / 2.0 ** -9)
    code = (exp_field.astype(np.int64) << 3) | np.rint(mant).astype(np.int64)
    code = np.where(r > 0, code, 0) | np.where(neg, 0x80, 0)
    return code.astype(np.uint8)


def quantize_e4m3_rows(X):
    """Per-row scaled E4M3 codes of a matrix: X[i] ~ scale[i] * code[i].

    In float32 arithmetic, as the CUDA kernel decides the codes:
    amax = max |x| over the row, scale = amax / 448 (1 for an all-zero
    row), code = e4m3(x / scale) with both divisions correctly rounded.
    X: [R, H] (values of the storage dtype).  Returns codes uint8 [R, H]
    and scale float32 [R]."""
    X = np.asarray(X, dtype=np.float32)
    amax = np.abs(X).max(axis=1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX),
                     np.float32(1.0)).astype(np.float32)
    codes = np.empty(X.shape, np.uint8)
    for i in range(0, X.shape[0], 4096):        # row blocks: bounded memory
        codes[i:i + 4096] = e4m3_encode(X[i:i + 4096] /
                                        scale[i:i + 4096, None])
    return codes, scale


def dequantize_e4m3_rows(codes, scale) -> np.ndarray:
    """scale[i] * value(code[i, k]) in float64."""
    return e4m3_decode(codes) * np.asarray(scale, np.float64)[:, None]


def lmhead_topk_e4m3(y, w_codes, w_scale, want_logits=False, w_deq=None):
    """The LM head with 8-bit operands: y (the conv output, storage
    values) is quantized per row, W_lm is given as per-row codes and
    scales; U = (s_y q_y)(s_W q_W)^T exactly (float64), then logsumexp and
    top-16 as in :func:`lmhead_topk`.  Also returns the y codes/scales.
    ``w_deq``: dequantize_e4m3_rows(w_codes, w_scale), if the caller keeps
    it (weight preparation done once)."""
    yc, ys = quantize_e4m3_rows(y)
    if w_deq is None:
        w_deq = dequantize_e4m3_rows(w_codes, w_scale)
    out = lmhead_topk(dequantize_e4m3_rows(yc, ys), w_deq, want_logits)
    return out + (yc, ys)


# --------------------------------------------------------------------------
# a2 with 4-bit LM-head operands (NVFP4 reading; the CUDA kernel is not
# built yet).  Elements are E2M1 (1 sign, 2 exponent, 1 mantissa bit:
# magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6); each block of 16 consecutive
# elements of a row carries an E4M3 scale, and the whole matrix one fp32
# scale, so that x ~ g * value(block scale) * value(code).
# --------------------------------------------------------------------------
E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
NVFP4_BLOCK = 16


def e2m1_decode(codes) -> np.ndarray:
    """Values (float64) of 4-bit E2M1 codes (bit 3 = sign)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    return np.where(c & 8, -1.0, 1.0) * E2M1_MAG[c & 7]


def e2m1_encode(x) -> np.ndarray:
    """Nearest E2M1 code of each finite value, ties to the even code (the
    one whose mantissa bit is 0), magnitudes beyond 6 saturated to 6, the
    sign of zero kept."""
    x = np.asarray(x, dtype=np.float64)
    if not np.all(np.isfinite(x)):
        raise ValueError("e2m1_encode: non-finite input")
    a = np.minimum(np.abs(x), 6.0)
    d = np.abs(a[..., None] - E2M1_MAG)              # distance to each
    best = d.min(axis=-1, keepdims=True)
    tie = np.isclose(d, best, rtol=0, atol=0)        # exact ties only
    # among equally near codes take the even one (lowest bit 0)
    pref = np.where(tie, (np.arange(8) & 1) * 8 + np.arange(8), 99)
    code = np.argmin(pref, axis=-1)
    return (code | np.where(np.signbit(x), 8, 0)).astype(np.uint8)


def quantize_nvfp4_rows(X):
    """Two-level 4-bit quantization of a matrix [R, H] (H % 16 == 0), in
    float32 arithmetic: g = max|X| / (448 * 6) (1 for a zero matrix);
    per block of 16 elements b: scale code s_b = E4M3(max|x_b| / (6 g)),
    d_b its value; element codes E2M1(x / (d_b * g)) (0 where d_b = 0).
    Returns (codes uint8 [R, H], block scale codes uint8 [R, H/16], g)."""
    X = np.asarray(X, dtype=np.float32)
    R, H = X.shape
    if H % NVFP4_BLOCK:
        raise ValueError("H must be a multiple of 16")
    amax = np.float32(np.abs(X).max()) if X.size else np.float32(0)
    g = np.float32(amax / np.float32(448.0 * 6.0)) if amax > 0 else \
        np.float32(1.0)
    Xb = X.reshape(R, H // NVFP4_BLOCK, NVFP4_BLOCK)
    bmax = np.abs(Xb).max(axis=2).astype(np.float32)
    sc = e4m3_encode((bmax / (np.float32(6.0) * g)).astype(np.float32))
    d = e4m3_decode(sc).astype(np.float32)
    den = (d * g).astype(np.float32)[..., None]
    safe = np.where(den > 0, den, np.float32(1.0))
    q = np.where(den > 0, (Xb / safe).astype(np.float32), np.float32(0.0))
    codes = e2m1_encode(q).reshape(R, H)
    return codes, sc, g


def dequantize_nvfp4_rows(codes, scale_codes, g) -> np.ndarray:
    """value(code) * value(block scale) * g in float64."""
    codes = np.asarray(codes)
    R, H = codes.shape
    d = e4m3_decode(scale_codes) * np.float64(g)
    return (e2m1_decode(codes).reshape(R, H // NVFP4_BLOCK, NVFP4_BLOCK) *
            d[..., None]).reshape(R, H)


def lmhead_topk_nvfp4(y, w_codes, w_scale_codes, w_g, want_logits=False):
    """The LM head with 4-bit operands: y (the conv output) quantized by
    :func:`quantize_nvfp4_rows`, W_lm given in the same form; U is the
    exact product of the dequantized operands (float64), then logsumexp
    and top-16 as in :func:`lmhead_topk`.  Also returns y's codes, block
    scale codes and matrix scale."""
    yc, ysc, yg = quantize_nvfp4_rows(y)
    out = lmhead_topk(dequantize_nvfp4_rows(yc, ysc, yg),
                      dequantize_nvfp4_rows(w_codes, w_scale_codes, w_g),
                      want_logits)
    return out + (yc, ysc, yg)


# --------------------------------------------------------------------------
# a3: context gate + low-rank bilinear pair scores
# --------------------------------------------------------------------------
def gate(h: np.ndarray, w_gate: np.ndarray) -> np.ndarray:
    """G(h_t) = sigmoid(W_g h_t) in float64.  h: [..., H]; w_gate [r, H].

    [KP] "A Lightweight Path Selector": embeddings are matched under a
    context gate of h_t.
    """
    z = np.asarray(h, np.float64) @ np.asarray(w_gate, np.float64).T
    return 1.0 / (1.0 + np.exp(-z))


def pair_score(topv, topi, anchor, g, e_in, e_out) -> np.ndarray:
    """S[b,t,i,j] = U_t(c_j) + sum_k E_in[a_i,k] G_t[k] E_out[c_j,k].

    [KP] "A Lightweight Path Selector" (every adjacent pair of candidates is
    scored, predecessor a and current candidate b, low-rank bilinear over a
    256-dim embedding, no backbone or LM-head pass); [DC] "A path selector".
    Position 0's predecessor is the anchor (last verified) token for every
    row i; position t >= 1 uses the candidates of position t-1.  Invalid
    (-1) candidates or predecessors give -inf.
    topv/topi: [B,K,16]; anchor [B]; g [B,K,r]; e_in/e_out [V,r].
    Returns float64 [B,K,16,16].
    """
    topv = np.asarray(topv, np.float64)
    topi = np.asarray(topi)
    Ein = np.asarray(e_in, np.float64)
    Eout = np.asarray(e_out, np.float64)
    B, K, _ = topv.shape
    S = np.full((B, K, C, C), -np.inf)
    for b in range(B):
        for t in range(K):
            preds = (np.full(C, int(anchor[b])) if t == 0
                     else topi[b, t - 1])
            cands = topi[b, t]
            for i in range(C):
                if preds[i] < 0:
                    continue
                ein = Ein[preds[i]]
                for j in range(C):
                    if cands[j] < 0:
                        continue
                    S[b, t, i, j] = topv[b, t, j] + np.dot(
                        ein * g[b, t], Eout[cands[j]])
    return S


# --------------------------------------------------------------------------
# a4: walk through the K x 16 lattice
# --------------------------------------------------------------------------
def _inverse_cdf(w: np.ndarray, u: float):
    """Smallest index whose running sum is strictly greater than u*total,
    decided on fp32-rounded operands.  Returns (index, relative margin)."""
    cum = np.cumsum(w)
    tot = cum[-1]
    thr32 = np.float32(u) * np.float32(tot)
    above = np.nonzero(cum.astype(np.float32) > thr32)[0]
    j = int(above[0]) if above.size else int(np.nonzero(w > 0)[0][-1])
    thr = u * tot
    lo = cum[j - 1] if j > 0 else 0.0
    margin = min(abs(cum[j] - thr), abs(thr - lo)) / tot
    return j, margin


def path_walk(S, topi, T: float, u_walk):
    """Walk one path through the candidate lattice per sequence.

    [KP] "A Lightweight Path Selector": starting from the verified token,
    greedy follows the best successor and sampling draws from the scores;
    [2B] "The two fixes": one coherent route through the grid.
    S: [B,K,16,16] (row = predecessor slot, column = candidate slot);
    topi [B,K,16]; u_walk [B,K] uniforms (unused at T = 0).
    Returns slot [B,K] i32, draft [B,K] i32, q [B,K,16] f64 and the
    per-step decision margin [B,K] (score gap at T=0, CDF distance at T>0).
    """
    S = np.asarray(S, np.float64)
    B, K = S.shape[:2]
    slot = np.zeros((B, K), np.int32)
    draft = np.zeros((B, K), np.int32)
    q = np.zeros((B, K, C))
    margin = np.zeros((B, K))
    for b in range(B):
        prev = 0            # every row of position 0 is the anchor's row
        for t in range(K):
            row = S[b, t, prev]
            if T == 0.0:
                r32 = row.astype(np.float32)
                j = int(np.argmax(r32))           # first maximum
                others = np.delete(row, j)
                fin = others[np.isfinite(others)]
                margin[b, t] = row[j] - fin.max() if fin.size else np.inf
                q[b, t, j] = 1.0
            else:
                mx = row.max()
                w = np.where(np.isfinite(row), np.exp((row - mx) / T), 0.0)
                j, margin[b, t] = _inverse_cdf(w, u_walk[b, t])
                q[b, t] = w / w.sum()
            slot[b, t] = j
            draft[b, t] = topi[b, t, j]
            prev = j
    return slot, draft, q, margin


# --------------------------------------------------------------------------
# a5 + a6: rejection-sampling verify with residual / bonus resample
# --------------------------------------------------------------------------
def _softmax(z: np.ndarray):
    m = z.max()
    lse = m + np.log(np.exp(z - m).sum())
    return np.exp(z - lse), lse


def verify(L, draft, topi, q, T: float, u_acc, u_res):
    """Verify K drafts per sequence against the target's K+1 logit rows.

    [DC] "Lossless, with conditions I did not used to state": accept a
    draft token with probability min(1, p/q) and resample from the residual
    on rejection; [KP] "A Lightweight Path Selector": rejection sampling
    restores the exact target distribution; [2B] "Caveats": greedy output
    matches the target exactly.
    L: [B,K+1,V] target logits; draft [B,K]; topi/q [B,K,16] (q = the
    walk's draft distribution, zero off the candidates); u_acc [B,K];
    u_res [B].  Returns n [B] (accepted drafts), out [B,K+1] (accepted
    drafts, then the resampled / bonus token, then -1) and a dict of
    decision margins.
    """
    L = np.asarray(L, np.float64)
    B, K1, V = L.shape
    K = K1 - 1
    n_acc = np.zeros(B, np.int32)
    out = np.full((B, K1), -1, np.int32)
    acc_margin = np.full((B, K), np.inf)
    res_margin = np.full(B, np.inf)
    degenerate = np.zeros(B, bool)
    for b in range(B):
        n = K
        for t in range(K):
            d = int(draft[b, t])
            if T == 0.0:
                a = int(np.argmax(L[b, t].astype(np.float32)))
                ok = (d == a)
            else:
                p, _ = _softmax(L[b, t] / T)
                js = np.nonzero(topi[b, t] == d)[0]
                qd = float(q[b, t, js[0]]) if js.size else 0.0
                ok = bool(np.float32(u_acc[b, t]) * np.float32(qd)
                          < np.float32(p[d]))
                acc_margin[b, t] = abs(p[d] - u_acc[b, t] * qd) / max(p[d],
                                                                      1e-300)
            if not ok:
                n = t
                break
        n_acc[b] = n
        out[b, :n] = draft[b, :n]
        if T == 0.0:
            out[b, n] = int(np.argmax(L[b, n].astype(np.float32)))
            continue
        p, _ = _softmax(L[b, n] / T)
        if n < K:
            qf = np.zeros(V)
            ok = topi[b, n] >= 0
            qf[topi[b, n][ok]] = q[b, n][ok]
            r = np.maximum(0.0, p - qf)
        else:
            r = p
        if not r.sum() > 0.0:
            r = p
            degenerate[b] = True
        v, res_margin[b] = _inverse_cdf(r, u_res[b])
        out[b, n] = v
    return n_acc, out, {"accept": acc_margin, "resample": res_margin,
                        "degenerate": degenerate}


# --------------------------------------------------------------------------
# one whole draft-verify cycle
# --------------------------------------------------------------------------
def draft_verify_cycle(h, w_conv, w_lm, w_gate, e_in, e_out, anchor, L,
                       T: float, seed: int, cycle: int, dtype: str,
                       w_lm_e4m3=None):
    """All five steps for B sequences, each stage fed by the previous one.

    h: [B,K,H] drafter hidden states (values of the storage dtype);
    L: [B,K+1,V] target logits.  With ``w_lm_e4m3 = (codes, scale)`` the
    LM head runs on 8-bit operands (:func:`lmhead_topk_e4m3`) and w_lm is
    unused; a third element, if present, is their dequantized matrix.
    Returns a dict of every intermediate.
    """
    h = np.asarray(h, np.float64)
    B, K, H = h.shape
    y = to_storage(conv2tap(h, w_conv), dtype).astype(np.float64)
    if w_lm_e4m3 is not None:
        topv, topi, lse, _, _ = lmhead_topk_e4m3(
            y.reshape(B * K, H), w_lm_e4m3[0], w_lm_e4m3[1],
            w_deq=w_lm_e4m3[2] if len(w_lm_e4m3) > 2 else None)
    else:
        topv, topi, lse = lmhead_topk(y.reshape(B * K, H), w_lm)
    topv = topv.reshape(B, K, C)
    topi = topi.reshape(B, K, C)
    g = gate(h, w_gate)
    S = pair_score(topv, topi, anchor, g, e_in, e_out)
    S32 = S.astype(np.float32)
    slot, draft, q, _ = path_walk(S32, topi, T,
                                  philox.walk_uniforms(seed, cycle, B, K))
    q32 = q.astype(np.float32)
    n, out, _ = verify(L, draft, topi, q32, T,
                       philox.accept_uniforms(seed, cycle, B, K),
                       philox.resample_uniforms(seed, cycle, B, K))
    return {"y": y, "topv": topv, "topi": topi, "lse": lse.reshape(B, K),
            "g": g, "S": S32, "slot": slot, "draft": draft, "q": q32,
            "n": n, "out": out}


def commit(n, out, anchor, tokens, length, stats):
    """Commit each sequence's emitted tokens and hand the last one over as
    the next anchor (in place; numpy arrays).

    [2B] "What a block-diffusion drafter is": the target verifies the run
    and the matching prefix is kept; "How many tokens survive": acceptance
    length is the mean number of draft tokens kept per verification pass.
    n [B] accepted drafts and out [B,K+1] from verify; anchor [B];
    tokens [B,capacity] and length [B] the committed tokens; stats
    [3+17]: accepted drafts, passes, emitted tokens, histogram of n.
    Tokens past a sequence's capacity are dropped (its length still
    advances).
    """
    B, cap = tokens.shape
    for b in range(B):
        nb = int(n[b])
        for i in range(nb + 1):
            pos = int(length[b]) + i
            if pos < cap:
                tokens[b, pos] = out[b, i]
        length[b] += nb + 1
        anchor[b] = out[b, nb]
        stats[0] += nb
        stats[1] += 1
        stats[2] += nb + 1
        stats[3 + nb] += 1


def path_viterbi(S, topi):
    """Global max-sum path through the candidate lattice (T = 0 selector
    variant; [KP] "What Comes Next": pairwise scoring is the simplest
    selector, there is room to explore).

    best_0(j) = S[b,0,0,j]; best_t(j) = max_i best_{t-1}(i) + S[b,t,i,j];
    the path ends in the lowest j of maximal total and takes the lowest
    predecessor i on ties (the sums in float64 of the given values).
    Returns slot [B,K], draft [B,K], q one-hot [B,K,16] and the path's
    total [B].
    """
    S = np.asarray(S, np.float64)
    B, K = S.shape[:2]
    slot = np.zeros((B, K), np.int32)
    draft = np.zeros((B, K), np.int32)
    q = np.zeros((B, K, C))
    total = np.zeros(B)
    for b in range(B):
        best = S[b, 0, 0].copy()
        back = np.zeros((K, C), np.int64)
        for t in range(1, K):
            cand = best[:, None] + S[b, t]          # [i, j]
            back[t] = np.argmax(cand, axis=0)       # first maximum: lowest i
            best = cand[back[t], np.arange(C)]
        j = int(np.argmax(best))
        total[b] = best[j]
        for t in range(K - 1, -1, -1):
            slot[b, t] = j
            draft[b, t] = topi[b, t, j]
            q[b, t, j] = 1.0
            if t > 0:
                j = int(back[t, j])
    return slot, draft, q, total


def path_total(S, slot):
    """Sum of the scores along each sequence's path (float64)."""
    S = np.asarray(S, np.float64)
    B, K = slot.shape
    tot = np.zeros(B)
    for b in range(B):
        prev = 0
        for t in range(K):
            tot[b] += S[b, t, prev, slot[b, t]]
            prev = slot[b, t]
    return tot


def top16_recall(L, topi):
    """For each drafted position (b, t), t < K: the target's first argmax
    and whether it is among the 16 candidates ([KP] "What Comes Next":
    recall of the candidate lists by position, and the oracle selector).
    L [B,K+1,V]; topi [B,K,16].  Returns target_argmax [B,K], in_top16
    [B,K] (0/1)."""
    L = np.asarray(L)
    B, K = topi.shape[:2]
    arg = np.zeros((B, K), np.int64)
    hit = np.zeros((B, K), np.int64)
    for b in range(B):
        for t in range(K):
            a = int(np.argmax(L[b, t]))             # first maximum
            arg[b, t] = a
            hit[b, t] = int(a in set(int(v) for v in topi[b, t]))
    return arg, hit
