/*
 * dflash.h — C ABI of the DFlash 2 draft-verify hot path on one GB300 GPU.
 *
 * One draft-verify cycle is four calls, in this order, on one stream:
 *
 *   dflash_lmhead_topk  two-tap conv + drafter LM head + logsumexp + top-16
 *   dflash_pair_score   context gate + low-rank bilinear scores of the
 *                       16 x 16 candidate pairs of adjacent positions
 *   dflash_path_walk    greedy or sampled walk through the K x 16 lattice
 *   dflash_verify       rejection-sampling verify, residual / bonus draw
 *
 * or two: dflash_draft (the first three in one call, with the context gate
 * computed inside the conv launch) and dflash_verify.
 *
 * Sources (page title, section):
 *   "DFlash 2: Block diffusion, wearing a drafter's coat" — "Sixteen
 *     candidates per position", "A path selector", "Suffix-decay
 *     convolution", "Lossless, with conditions I did not used to state".
 *   "A 2B Drafter Made a 27B Model 3.4x Faster. Same Exact Output." —
 *     "The two fixes", "Running it", "Caveats before you rebuild your
 *     serving stack".
 *   "DFlash 2: Keep Drafting Parallel" — "What Comes Next", "A Lightweight
 *     Path Selector".
 *
 * Conventions shared by every call:
 *   - Shapes: B sequences, K drafted positions per sequence (1..16), V
 *     vocabulary, H drafter hidden size, r selector rank (1..256), C = 16
 *     candidates per position.  M = B*K rows.  All arrays are row-major and
 *     contiguous.
 *   - Every pointer argument except `seed`-like scalars is DEVICE memory
 *     owned by the caller (for example a torch CUDA tensor).  The library
 *     allocates nothing on these paths; scratch comes from the caller's
 *     workspace `ws` of at least dflash_workspace_bytes(...) bytes.
 *   - Calls are asynchronous on stream `s` (NULL = legacy default stream).
 *     Arguments are checked on the host before anything is launched; a bad
 *     argument returns DFLASH_ERR_INVALID_ARG (or _UNSUPPORTED) and
 *     launches nothing.
 *   - Problems found on the device (an index out of range, a non-finite
 *     target logit, a draft that is not among its candidates) set a sticky
 *     device error word; kernels never trap.  dflash_check() synchronises
 *     the stream, reads and clears that word and returns the matching
 *     status.
 *   - dtype (DFLASH_BF16 or DFLASH_FP32) is the storage type of the
 *     drafter-side tensors (hidden states, weights, embeddings).  All
 *     accumulation is fp32.  Scores, probabilities and target logits are
 *     fp32 whatever dtype is.
 *   - When V < 16 the candidate lists are padded with index -1 and value
 *     -inf (q = 0).
 *   - Randomness: uniforms are Philox4x32-10 (Salmon et al., SC'11) with
 *     key (seed lo, seed hi) and counter (b, t, purpose, cycle mod 2^32);
 *     purpose 0 = walk draw of position t, 1 = accept draw of position t,
 *     2 = residual / bonus draw (t = K); u = (word0 >> 8) * 2^-24.  Give
 *     each cycle a new `cycle` value.  T = 0 selects the greedy forms and
 *     ignores seed and cycle.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream. */
typedef struct CUstream_st* dflash_stream_t;

typedef enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,    /* bad pointer, size, alignment or value */
  DFLASH_ERR_UNSUPPORTED = 2,    /* valid request this build cannot run  */
  DFLASH_ERR_CUDA = 3,           /* a CUDA runtime call failed           */
  DFLASH_ERR_NONFINITE = 4,      /* device: NaN or +inf target logit     */
  DFLASH_ERR_DEVICE_TIMEOUT = 5, /* device: a bounded wait ran out       */
  DFLASH_ERR_BAD_INDEX = 6       /* device: token id outside [0, V), or a
                                    draft not among its candidates        */
} dflash_status;

typedef enum { DFLASH_BF16 = 0, DFLASH_FP32 = 1 } dflash_dtype;

#define DFLASH_CANDIDATES 16
#define DFLASH_MAX_K 16
#define DFLASH_MAX_RANK 256
#define DFLASH_MAX_SHARDS 64   /* vocabulary shards of one merge / decide */
#define DFLASH_SHARD_STATS 20  /* words per target row of shard statistics */
#define DFLASH_SHARD_PLAN 8    /* words per sequence of a shard draw plan */

/* Workspace needed by dflash_lmhead_topk (which = 0), dflash_verify
 * (which = 1), dflash_draft (which = 2) or dflash_draft_e4m3 (which = 3)
 * for these sizes, in bytes; an upper bound over both dtypes and every r.
 * Returns 0 for invalid sizes. */
size_t dflash_workspace_bytes(int which, int B, int K, int H, int V);

/*
 * Steps a1 + a2: two-tap dynamic depthwise conv, drafter LM head, online
 * logsumexp and per-position top-16.
 *
 * "Suffix-decay convolution" (drafter's coat page) and "The two fixes"
 * (2B-drafter page): each position is mixed with its predecessor,
 *     w0_t = W0 h_t,  w1_t = W1 h_t,  y_t = w0_t * h_t + w1_t * h_{t-1},
 * per channel, h_{-1} = 0 at the first block position of every sequence,
 * y rounded to dtype.  "Sixteen candidates per position" and "A Lightweight
 * Path Selector": U_t = y_t W_lm^T is the drafter's own logit; the call
 * keeps its 16 largest entries and log(sum_v exp U_t(v)) without writing
 * U_t to memory.
 *
 *   h      [B, K, H] dtype        drafter final hidden states
 *   conv_w [2H, H]   dtype        rows 0..H-1 = W0, rows H..2H-1 = W1;
 *                                 NULL skips the conv (y = h)
 *   w_lm   [V, H]    dtype        LM head
 *   topv   [B*K, 16] fp32  out    U_t of the candidates, descending
 *   topi   [B*K, 16] int32 out    their token ids (ties: lower id first)
 *   lse    [B*K]     fp32  out    logsumexp of U_t over the vocabulary
 *   ws     >= dflash_workspace_bytes(0, B, K, H, V) bytes, 256-B aligned.
 *          On return its first B*K*H elements (dtype) hold y when conv_w
 *          is not NULL.
 * Requirements: 1 <= K <= 16, B >= 1, H % 8 == 0, V >= 1; bf16 operand
 * pointers 16-byte aligned.
 */
dflash_status dflash_lmhead_topk(const void* h, const void* conv_w,
                                 const void* w_lm, int B, int K, int H,
                                 int V, dflash_dtype dt, float* topv,
                                 int32_t* topi, float* lse, void* ws,
                                 size_t ws_bytes, dflash_stream_t s);

/*
 * Step a3: context gate and low-rank bilinear pair scores.
 *
 * "A Lightweight Path Selector" (Keep Drafting Parallel page) and "A path
 * selector" (drafter's coat page): for predecessor a and current candidate
 * b of adjacent positions,
 *     S_t(a, b) = U_t(b) + < E_in(a), G(h_t) * E_out(b) >,
 *     G(h_t) = sigmoid(W_g h_t)   (gate form: this library's reading),
 * every pair scored at once, with no backbone or LM-head pass.  The
 * predecessor of position 0 is the anchor (last verified) token, so all 16
 * rows of S[b, 0] are equal.
 *
 *   topv, topi [B, K, 16]  from dflash_lmhead_topk
 *   anchor     [B] int32   last verified token of each sequence
 *   h          [B, K, H] dtype   (the same hidden states, pre-conv)
 *   w_gate     [r, H] dtype;  e_in, e_out [V, r] dtype
 *   scores     [B, K, 16, 16] fp32 out: scores[b,t,i,j] = S_t(pred_i,
 *              cand_j); -inf where either index is -1.
 * Requirements: 1 <= r <= 256, 1 <= K <= 16, H % 8 == 0; h, w_gate, e_in
 * and e_out 16-byte aligned.
 */
dflash_status dflash_pair_score(const float* topv, const int32_t* topi,
                                const int32_t* anchor, const void* h,
                                const void* w_gate, const void* e_in,
                                const void* e_out, int B, int K, int H, int V,
                                int r, dflash_dtype dt, float* scores,
                                dflash_stream_t s);

/*
 * Step a4: walk one path through the K x 16 candidate lattice.
 *
 * "A Lightweight Path Selector": starting from the verified token, greedy
 * follows the best successor; sampling draws from the scores.  With
 * prev = 0 (the anchor row) and for t = 0..K-1:
 *   T == 0: j = argmax_j scores[b,t,prev,j] (lowest j on ties), q one-hot;
 *   T >  0: w_j = exp((scores[b,t,prev,j] - max) / T), q = w / sum(w),
 *           j = the smallest j with w_0 + .. + w_j > u * sum(w),
 *           u = walk uniform (b, t);
 *   prev = j.
 *   slot  [B, K] int32 out   chosen candidate slot
 *   draft [B, K] int32 out   topi[b, t, slot]
 *   q     [B, K, 16] fp32 out the draft distribution the verifier needs
 */
dflash_status dflash_path_walk(const float* scores, const int32_t* topi,
                               int B, int K, float T, uint64_t seed,
                               uint64_t cycle, int32_t* slot, int32_t* draft,
                               float* q, dflash_stream_t s);

/*
 * Steps a1-a4 in one call: dflash_lmhead_topk, dflash_pair_score and
 * dflash_path_walk with the same arguments and outputs as those three
 * calls, in that order ("Suffix-decay convolution" and "Sixteen candidates
 * per position" of "DFlash 2: Block diffusion, wearing a drafter's coat";
 * "A Lightweight Path Selector" of "DFlash 2: Keep Drafting Parallel").
 * For bf16 storage with a conv, the context gate g_t = sigmoid(W_g h_t)
 * reads the same h tiles as the conv, so it is computed by the conv launch
 * on the tensor cores and kept in the workspace; after the LM head, one
 * launch merges its partials, scores the pairs of each position (only
 * gathering embedding rows) and walks each sequence.  Otherwise the three
 * steps run as the separate calls do.
 *   inputs   h, conv_w (may be NULL: no conv), w_lm, w_gate, e_in, e_out,
 *            anchor, sizes, dt, T, seed, cycle: as in the three calls
 *   outputs  topv, topi, lse (dflash_lmhead_topk), scores
 *            (dflash_pair_score), slot, draft, q (dflash_path_walk)
 *   ws       >= dflash_workspace_bytes(2, B, K, H, V) bytes, 256-byte
 *            aligned, caller-owned; holds y, the LM-head partials, the
 *            gate and one walk ticket per sequence.
 * Requirements: the union of the three calls' (h, w_lm, w_gate, e_in,
 * e_out, scores 16-byte aligned; H % 8 == 0; 1 <= r <= 256; T >= 0).
 * Results equal the three calls' up to the order of fp32 accumulation in
 * the gate and in the logsumexp fold: the same candidates, lse and scores
 * within fp32 rounding.
 */
dflash_status dflash_draft(const void* h, const void* conv_w, const void* w_lm,
                           const void* w_gate, const void* e_in,
                           const void* e_out, const int32_t* anchor, int B,
                           int K, int H, int V, int r, dflash_dtype dt,
                           float T, uint64_t seed, uint64_t cycle, float* topv,
                           int32_t* topi, float* lse, float* scores,
                           int32_t* slot, int32_t* draft, float* q, void* ws,
                           size_t ws_bytes, dflash_stream_t s);

/*
 * 8-bit LM head (quantized drafters: "What a block-diffusion drafter is"
 * of the 2B-drafter page and "What Comes Next" of "DFlash 2: Keep Drafting
 * Parallel" ship GGUF-quantized drafter builds; this library's 8-bit form
 * is OCP FP8 E4M3 with one fp32 scale per row, the operand type of the
 * tensor cores' kind::f8f6f4 MMA).
 *
 * dflash_quantize_e4m3_rows: x [R, H] bf16 -> codes [R, H] uint8 (E4M3:
 * bias 7, 3 mantissa bits, no infinities, 448 largest) and scale [R] fp32:
 *     scale_i = max_k |x_ik| / 448 (1 for an all-zero row),
 *     codes_ik = E4M3(x_ik / scale_i), nearest with ties to even, saturated,
 * both divisions correctly rounded fp32.  Used once on W_lm when it is
 * loaded; dflash_draft_e4m3 applies it to y every call.
 * Requirements: H % 16 == 0; x and codes 16-byte aligned.  A non-finite
 * input sets DFLASH_ERR_NONFINITE in the device error word.
 */
dflash_status dflash_quantize_e4m3_rows(const void* x, int R, int H,
                                        uint8_t* codes, float* scale,
                                        dflash_stream_t s);

/*
 * dflash_draft for bf16 storage with a conv, with the LM head on 8-bit
 * operands: the conv output y is quantized per row
 * (dflash_quantize_e4m3_rows) and U_t(v) = s_y[t] s_W[v] sum_k
 * code_y[t,k] code_W[v,k] (fp32 accumulation; the codes' products are
 * exact).  W_lm is given as codes [V, H] uint8 and row scales [V] fp32.
 * Everything else (gate, candidates, lse, scores, walk, outputs) is as in
 * dflash_draft with dt = DFLASH_BF16.
 *   ws >= dflash_workspace_bytes(3, B, K, H, V) bytes, 256-byte aligned;
 *        holds dflash_draft's workspace (its first
 *        dflash_workspace_bytes(2, B, K, H, V) bytes, with y in bf16 at
 *        offset 0), then y's codes [B*K, H] uint8, then from the next
 *        256-byte boundary y's scales [B*K] fp32.
 * Requirements: conv_w not NULL; H % 16 == 0; w_lm_codes 16-byte aligned;
 * the rest as dflash_draft.
 */
dflash_status dflash_draft_e4m3(
    const void* h, const void* conv_w, const uint8_t* w_lm_codes,
    const float* w_lm_scale, const void* w_gate, const void* e_in,
    const void* e_out, const int32_t* anchor, int B, int K, int H, int V,
    int r, float T, uint64_t seed, uint64_t cycle, float* topv,
    int32_t* topi, float* lse, float* scores, int32_t* slot, int32_t* draft,
    float* q, void* ws, size_t ws_bytes, dflash_stream_t s);

/*
 * Steps a5 + a6: rejection-sampling verify with residual or bonus draw.
 *
 * "Lossless, with conditions I did not used to state" (drafter's coat
 * page): accept a draft token x with probability min(1, p(x)/q(x)), and on
 * the first rejection resample from normalize(max(0, p - q)); the emitted
 * tokens then follow the target distribution exactly.  p_t =
 * softmax(L[b,t] / T).  For t = 0..K-1 in order, draft t is accepted iff
 * u_t * q_t(x) < p_t(x) (u_t = accept uniform (b, t)); n = the number
 * accepted before the first rejection.  If n < K the token at n is drawn
 * from max(0, p_n - q_n) (q_n zero off the candidates; p_n if that is all
 * zero); if n = K a bonus token is drawn from p_K.  A draw takes the
 * smallest token v whose running weight sum exceeds u * total (u =
 * residual uniform (b, K)).  T == 0: accept iff the draft equals
 * argmax L[b,t] (lowest id on ties) and emit argmax L[b,n].
 *
 *   target_logits [B, K+1, V] fp32   target model logits, rows 0..K
 *   draft [B, K], topi [B, K, 16], q [B, K, 16]   from the walk
 *   n_accepted [B] int32 out
 *   out_tok [B, K+1] int32 out   draft[0..n-1], the drawn token, then -1
 *   ws >= dflash_workspace_bytes(1, B, K, 0, V) bytes, 256-B aligned
 * Requirements: target_logits 16-byte aligned; T >= 0.  A NaN or +inf
 * target logit sets DFLASH_ERR_NONFINITE in the device error word.
 * Rows are read in position order, and a row after its sequence's first
 * rejection (which no result depends on) stops being read once that
 * rejection is known: a non-finite logit there may go unreported.  Rows
 * 0..n of every sequence are always read in full.
 */
dflash_status dflash_verify(const float* target_logits, const int32_t* draft,
                            const int32_t* topi, const float* q, int B, int K,
                            int V, float T, uint64_t seed, uint64_t cycle,
                            int32_t* n_accepted, int32_t* out_tok, void* ws,
                            size_t ws_bytes, dflash_stream_t s);

/*
 * One whole cycle, steps a1-a6: dflash_draft (or, with w_lm_scale,
 * dflash_draft_e4m3 with w_lm as the E4M3 codes) followed by dflash_verify
 * of its draft, topi and q, with the same arguments, outputs and results
 * as those two calls.  On the tensor-core paths (bf16 storage with a conv)
 * the conv launch also zeroes the verify's tickets, which dflash_verify
 * otherwise zeroes with a copy-engine fill of its own before its launch;
 * that fill and its gap before the verify launch cost about 4.5 us of a
 * b32k8 cycle (B = 32, K = 8, V = 151936).
 *   inputs   h, conv_w, w_lm, w_lm_scale (NULL: bf16 LM head; else w_lm
 *            holds [V, H] uint8 codes and w_lm_scale [V] fp32 scales from
 *            dflash_quantize_e4m3_rows), w_gate, e_in, e_out, anchor, the
 *            sizes, dt, T, seed, cycle: as in dflash_draft(_e4m3);
 *            target_logits [B, K+1, V] fp32 as in dflash_verify
 *   outputs  topv, topi, lse, scores, slot, draft, q (the draft call's),
 *            n_accepted, out_tok (the verify's)
 *   ws_draft >= dflash_workspace_bytes(2, ...) bytes (3 with w_lm_scale),
 *            ws_verify >= dflash_workspace_bytes(1, B, K, 0, V) bytes, both
 *            256-byte aligned and caller-owned; ws_verify's contents need
 *            no zeroing by the caller.
 * Requirements: the union of the two calls'; w_lm_scale only with
 * dt == DFLASH_BF16.  Every argument is checked before anything is
 * launched.
 */
dflash_status dflash_cycle(
    const void* h, const void* conv_w, const void* w_lm,
    const float* w_lm_scale, const void* w_gate, const void* e_in,
    const void* e_out, const int32_t* anchor, const float* target_logits,
    int B, int K, int H, int V, int r, dflash_dtype dt, float T,
    uint64_t seed, uint64_t cycle, float* topv, int32_t* topi, float* lse,
    float* scores, int32_t* slot, int32_t* draft, float* q,
    int32_t* n_accepted, int32_t* out_tok, void* ws_draft,
    size_t ws_draft_bytes, void* ws_verify, size_t ws_verify_bytes,
    dflash_stream_t s);

/*
 * dflash_verify without any caller-provided scratch, for callers that
 * cannot allocate device memory at the time they verify: serving loops whose
 * device memory belongs to another engine's allocator, code running where
 * allocation (and the synchronisation it can bring) is not allowed, and C
 * callers with no allocator of their own.  This entry point has no
 * counterpart in the pages; it exists for those callers only.
 *
 * Same arguments, checks, semantics, results and profiling stage as
 * dflash_verify, minus ws and ws_bytes.  The scratch is a fixed 4 MiB array
 * the library holds in device memory on every GPU that loads it, until the
 * process exits; sizes whose scratch, dflash_workspace_bytes(1, B, K, 0, V)
 * (about B*(K+1)*ceil(V/2048)*8 bytes), exceeds 4 MiB are refused with
 * DFLASH_ERR_UNSUPPORTED.  At V = 151936, B = 256 with K = 16 fits (2.7 MB)
 * and K = 16 fits up to B = 405; at V = 262144, B = 256 fits up to K = 14.
 * The first call on a device looks up the array's device address (so make
 * that first call before any stream capture).  All calls share the
 * array: each clears what must start at zero itself, and calls whose
 * kernels overlap on the GPU (several streams or threads on one device)
 * race on it and must be serialised by the caller.  Allocates nothing.
 */
dflash_status dflash_verify_noalloc(const float* target_logits,
                                   const int32_t* draft, const int32_t* topi,
                                   const float* q, int B, int K, int V,
                                   float T, uint64_t seed, uint64_t cycle,
                                   int32_t* n_accepted, int32_t* out_tok,
                                   dflash_stream_t s);

/*
 * The step after verify in a draft-verify loop: commit each sequence's
 * emitted tokens and hand the last one over as the next cycle's anchor.
 *
 * "What a block-diffusion drafter is" (2B-drafter page): the target
 * verifies the whole run and the matching prefix is kept; "How many tokens
 * survive": acceptance length is the mean number of draft tokens kept per
 * verification pass.  For every sequence b, with n = n_accepted[b]:
 *   tokens[b, length[b] .. length[b] + n] = out_tok[b, 0 .. n]
 *   (the n accepted drafts, then the resampled or bonus token),
 *   length[b] += n + 1, anchor[b] = out_tok[b, n];
 *   stats[0] += n (accepted drafts), stats[1] += 1 (verification passes),
 *   stats[2] += n + 1 (emitted tokens), stats[3 + n] += 1 (histogram).
 * Mean acceptance length = stats[0] / stats[1].
 *   n_accepted [B] int32, out_tok [B, K+1] int32   from dflash_verify
 *   anchor     [B] int32 in/out      the next cycle's anchor
 *   tokens     [B, capacity] int32 in/out, length [B] int32 in/out:
 *              each sequence's committed tokens; a sequence whose buffer
 *              is full keeps the tokens that fit, and the call flags
 *              DFLASH_ERR_BAD_INDEX in the device error word (length still
 *              advances, so a caller can tell how many were dropped)
 *   stats      [DFLASH_COMMIT_STATS] int64 in/out, accumulated over calls
 * All device memory, caller-owned; no workspace.  Requires 1 <= K <= 16,
 * capacity >= 1.  An n_accepted outside [0, K] is flagged as
 * DFLASH_ERR_BAD_INDEX and that sequence is left unchanged.
 */
#define DFLASH_COMMIT_STATS (3 + DFLASH_MAX_K + 1)
dflash_status dflash_commit(const int32_t* n_accepted, const int32_t* out_tok,
                            int B, int K, int32_t* anchor, int32_t* tokens,
                            int32_t* length, int capacity, int64_t* stats,
                            dflash_stream_t s);

/*
 * Selector variant: the global max-sum path through the K x 16 lattice
 * (a Viterbi walk), for T = 0.  "What Comes Next" (Keep Drafting Parallel
 * page): pairwise scoring is the simplest selector and there is room to
 * explore; the pages' own greedy walk follows the best successor instead.
 *   best_0(j) = scores[b,0,0,j],
 *   best_t(j) = max_i best_{t-1}(i) + scores[b,t,i,j]  (t = 1..K-1),
 * the path ends in the lowest j of maximal best_{K-1}(j), predecessors on
 * ties are the lowest i, sums in fp32.  Outputs as dflash_path_walk: slot,
 * draft = topi[b,t,slot], q one-hot.  scores 16-byte aligned; 1 <= K <= 16.
 * A sequence with no path of finite score flags DFLASH_ERR_BAD_INDEX.
 */
dflash_status dflash_path_viterbi(const float* scores, const int32_t* topi,
                                  int B, int K, int32_t* slot, int32_t* draft,
                                  float* q, dflash_stream_t s);

/*
 * Diagnostic of the candidate lists ("What Comes Next", Keep Drafting
 * Parallel page: recall of the 16 candidates by position, and the
 * acceptance length an oracle that always picks the right candidate among
 * them would reach).  For every drafted position (b, t), t < K:
 *   target_argmax[b,t] = the first argmax over v of target_logits[b,t,v],
 *   in_top16[b,t]      = 1 if that token is among topi[b,t,:], else 0.
 * Recall@16 at position t is the mean of in_top16[:, t]; with greedy
 * verification a perfect selector is accepted up to the first position
 * whose in_top16 is 0.  Reads the K target rows once (B*K*V*4 bytes).
 * target_logits [B, K+1, V] fp32; topi [B*K, 16]; outputs [B*K] int32.
 * A NaN / +inf logit flags DFLASH_ERR_NONFINITE.
 */
dflash_status dflash_top16_recall(const float* target_logits,
                                  const int32_t* topi, int B, int K, int V,
                                  int32_t* target_argmax, int32_t* in_top16,
                                  dflash_stream_t s);

/*
 * Vocabulary shards.  With the vocabulary split into S contiguous ranges
 * [v0, v0 + V_shard) (an LM head and target logits too large for one
 * device, or a target that is itself split by vocabulary), each shard
 * computes what depends on its range only, the shards' small summaries are
 * gathered (S x a few words per row), and a merge gives exactly what the
 * whole-vocabulary calls give: the same candidates and tokens, logsumexp
 * and probabilities within fp32 rounding of another summation order.  The
 * pages have no sharded form; the decomposition follows from the
 * definitions of the top-16, the logsumexp, the accept test and the
 * inverse CDF (each a fold over the vocabulary).  Every call runs on the
 * caller's device and stream; moving the summaries between devices (an
 * all-gather) is the caller's, and one device can run all shards in turn.
 *
 * dflash_lmhead_topk_shard: steps a1 + a2 of dflash_lmhead_topk on the
 * shard's LM-head rows w_lm_shard [V_shard, H] (the conv is recomputed on
 * every shard; it is small).  Writes the shard's partial of every row:
 *   part_v, part_i [B*K, 16]  the shard's 16 best logits and their global
 *                             ids (v0 + row of w_lm_shard), descending,
 *                             ties to the lower id, padding (-inf, -1)
 *   part_m, part_s [B*K]      the shard's max of U_t and sum exp(U_t - max)
 *   ws >= dflash_workspace_bytes(0, B, K, H, V_shard) bytes.
 * Requirements as dflash_lmhead_topk; v0 >= 0.
 */
dflash_status dflash_lmhead_topk_shard(const void* h, const void* conv_w,
                                       const void* w_lm_shard, int B, int K,
                                       int H, int V_shard, int v0,
                                       dflash_dtype dt, float* part_v,
                                       int32_t* part_i, float* part_m,
                                       float* part_s, void* ws,
                                       size_t ws_bytes, dflash_stream_t s);

/* The S shards' partials gathered in shard order (part_v, part_i
 * [S, M, 16]; part_m, part_s [S, M]; M = B*K) merged into topv, topi
 * [M, 16] and lse [M], as dflash_lmhead_topk writes them.  1 <= S <= 64. */
dflash_status dflash_topk_merge_shards(const float* part_v,
                                       const int32_t* part_i,
                                       const float* part_m,
                                       const float* part_s, int S, int M,
                                       float* topv, int32_t* topi, float* lse,
                                       dflash_stream_t s);

/*
 * Steps a5 + a6 by vocabulary shard, in three calls.
 *
 * 1. dflash_verify_shard_stats, on each shard: the shard's target logits
 *    target_shard [B, K+1, V_shard] (ids v0 .. v0 + V_shard - 1 of a
 *    vocabulary of V) -> stats [B*(K+1), DFLASH_SHARD_STATS] fp32 words,
 *    per target row: [0] the shard's max logit, [1] at T > 0 its sum of
 *    exp((x - max) / T), at T = 0 its first argmax (global id, int bits),
 *    [2..17] the logits of the row's 16 candidates the shard holds,
 *    [18] that of the draft, [19] a mask (uint bits) of which it holds
 *    (bit j: candidate j, bit 16: the draft).  The shard's segment sums
 *    stay in ws (>= dflash_workspace_bytes(1, B, K, 0, V_shard) bytes) for
 *    step 3.
 * 2. dflash_verify_shard_decide, with every shard's stats gathered in
 *    shard order ([S, B*(K+1), DFLASH_SHARD_STATS]): each row's max and Z
 *    (or argmax), the accept tests as dflash_verify takes them, n_accepted
 *    and out_tok; at T = 0 out_tok is final.  At T > 0 the token at n is
 *    drawn in step 3 (out_tok holds -1 there until then) from the plan
 *    [B, DFLASH_SHARD_PLAN]: the shard whose part of the residual (or of p)
 *    holds the draw, and the remaining mass within it.
 * 3. dflash_verify_shard_draw, on each shard (index `shard`, with its ws
 *    from step 1): the draws the plan gives to that shard, written to
 *    out_tok.  Nothing to do at T = 0.
 * Same uniforms, tests and draws as dflash_verify ("Lossless, with
 * conditions I did not used to state", drafter's coat page); the sums are
 * folded per shard, then over shards in shard order.
 */
dflash_status dflash_verify_shard_stats(const float* target_shard,
                                        const int32_t* draft,
                                        const int32_t* topi, int B, int K,
                                        int V_shard, int v0, int V, float T,
                                        float* stats, void* ws,
                                        size_t ws_bytes, dflash_stream_t s);
dflash_status dflash_verify_shard_decide(
    const float* stats, int S, const int32_t* draft, const int32_t* topi,
    const float* q, int B, int K, int V, float T, uint64_t seed,
    uint64_t cycle, int32_t* n_accepted, int32_t* out_tok, float* plan,
    dflash_stream_t s);
dflash_status dflash_verify_shard_draw(const float* target_shard,
                                       const float* plan,
                                       const int32_t* topi, const float* q,
                                       int shard, int B, int K, int V_shard,
                                       int v0, float T, int32_t* out_tok,
                                       void* ws, size_t ws_bytes,
                                       dflash_stream_t s);

/* Philox4x32-10 of n counters (ctr [n, 4] uint32, device) under key
 * (seed lo, seed hi) into out [n, 4] uint32 (device): the generator the
 * walk and verify draw from, exposed so callers can reproduce draws. */
dflash_status dflash_philox4x32(const uint32_t* ctr, uint64_t seed,
                                uint32_t* out, int64_t n, dflash_stream_t s);

/* Per-stage timing.  While set, the library records the caller's CUDA
 * events `begin` and `end` (cudaEvent_t, created by the caller) on the
 * call's stream right before and right after it launches the kernel of
 * `stage`:
 *   0 conv, 1 LM head with top-16 / logsumexp epilogue, 2 top-16 merge,
 *   3 pair score, 4 walk, 5 verify (row pass, accept tests and draw),
 *   6 E4M3 quantization of y (dflash_draft_e4m3).
 * In dflash_draft with bf16 storage and a conv, stage 0 is the conv with
 * the context gate and stage 3 the one launch that merges, scores and
 * walks (stages 2 and 4 are not recorded).
 * Calls captured into a CUDA graph record the events as event-record
 * nodes (cudaEventRecordExternal), stamped at every replay.
 * Pass NULL for both to stop.  Process-wide host state; set it from the
 * thread that makes the calls, not while other threads call the library.
 * Returns DFLASH_ERR_INVALID_ARG for an unknown stage or a lone NULL. */
dflash_status dflash_profile_stage(int stage, void* begin, void* end);

/* Limit, in nanoseconds, of the bounded waits inside the tensor-core
 * kernels of later launches: the conv and the single-CTA LM head (one row
 * tile, B*K <= 128) give up on a wait that runs longer, stop issuing work,
 * let their copies and MMAs in flight complete, free their TMEM and set
 * DFLASH_ERR_DEVICE_TIMEOUT in the device error word (their results are
 * then invalid).  0 restores the default of 2 s, far beyond any real wait;
 * the CTA-pair LM head always uses it.  Process-wide host state,
 * meant for tests of that failure path ("Failure detection": a wait that
 * never completes must end in a status the host reads, not a hang).
 * Always returns DFLASH_OK. */
dflash_status dflash_set_wait_limit_ns(uint64_t ns);

/* Synchronise `s`, read and clear the device error word of the current
 * device; DFLASH_OK if no kernel reported a problem since the last call. */
dflash_status dflash_check(dflash_stream_t s);

/* Static, human-readable name of a status. */
const char* dflash_status_string(dflash_status st);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */
