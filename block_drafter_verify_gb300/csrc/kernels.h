// Host-side launchers of every kernel; the C ABI in api.cu calls these.
// Each returns the cudaError_t of its launch(es).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace dflash {

// Default limit of the tensor-core kernels' bounded waits (2 s, far beyond
// any real wait); dflash_set_wait_limit_ns changes it for later launches of
// the conv and of the single-CTA LM head.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// conv.cu -----------------------------------------------------------------
template <typename T>
cudaError_t launch_conv_simt(const T* h, const T* w_conv, int B, int K, int H,
                             T* y, cudaStream_t s);

// conv_tc.cu / lmhead_tc.cu: tensor-core (tcgen05) kernels for bf16 ------
// TMA descriptor of a row-major bf16 [rows, inner] matrix, 128-byte swizzle.
bool make_tmap_bf16_2d(CUtensorMap* map, const void* base, uint64_t inner,
                       uint64_t rows, uint32_t box_inner, uint32_t box_rows);
// map_h: h [B*K, H] box {64, 128}; map_wc: conv_w [2H, H] box {64, BC}
// with BC = conv_tc_bc(B*K, H) channels per tile (map_wg likewise).
// With map_wg (w_gate [r, H], box {64, 32}) the launch also writes the pair
// selector's gate g = sigmoid(W_g h) as gate [B*K, r] fp32.  tickets (B
// words, may be NULL) are zeroed and row_bound (nbound floats, may be NULL)
// set to -inf for later launches of the same call; so are tickets2
// (ntickets2 words, may be NULL: the tickets of the cycle's verify).
int conv_tc_bc(int M, int H);
cudaError_t launch_conv_tc(const CUtensorMap& map_h, const CUtensorMap& map_wc,
                           const CUtensorMap* map_wg, const __nv_bfloat16* h,
                           int B, int K, int H, int r, __nv_bfloat16* y,
                           float* gate, unsigned* tickets, float* row_bound,
                           int nbound, int* err, cudaStream_t s,
                           uint64_t wait_ns = kWaitLimitNs,
                           unsigned* tickets2 = nullptr, int ntickets2 = 0);
// TMA descriptor of a row-major 8-bit [rows, inner] matrix, 128-byte
// swizzle (inner a multiple of 16).
bool make_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t inner,
                     uint64_t rows, uint32_t box_inner, uint32_t box_rows);
// map_y: y [M, H] box {64, 128}; map_w: w_lm [V, H] box {64, 256}, or
// {64, 128} when lmhead_tc_pairs(M) (CTA pairs, two or more row tiles).
// Writes `*strips` partial lists per row.  With y_scale and w_scale the
// operands are E4M3 codes (maps from make_tmap_u8_2d, boxes of 128 codes
// along H) and logit (m, v) = y_scale[m] * w_scale[v] * (codes' dot).
// row_bound (M * kBoundSlots floats set to -inf by an earlier launch of
// the same stream, may be NULL) is where units share their rows' running
// maxima, from which every unit prunes values that cannot reach a row's
// top 16 (room for 32 slots per row; 16 per row, rows 16 floats apart,
// except for at most 8 rows).
constexpr int kBoundSlots = 32;
cudaError_t launch_lmhead_tc(const CUtensorMap& map_y, const CUtensorMap& map_w,
                             int M, int H, int V, int num_sms, TopkPartials P,
                             int* err, int* strips, cudaStream_t s,
                             const float* y_scale = nullptr,
                             const float* w_scale = nullptr,
                             float* row_bound = nullptr,
                             uint64_t wait_ns = kWaitLimitNs);

// quant_e4m3.cu: per-row E4M3 quantization of a bf16 [R, H] matrix
// (H % 8 == 0): scale[i] = max_k |x_ik| / 448 (1 for a zero row), code =
// e4m3(x / scale), round to nearest even, saturated.  Non-finite input
// sets kErrNonfinite.  Launched with programmatic dependent launch.
cudaError_t launch_quantize_e4m3_rows(const __nv_bfloat16* x, int R, int H,
                                      uint8_t* codes, float* scale, int* err,
                                      cudaStream_t s);
bool lmhead_tc_pairs(int M);
int lmhead_tc_grid(int M, int V, int num_sms, int* row_groups, int* strips,
                   bool fp8 = false);

// lmhead_simt.cu ----------------------------------------------------------
template <typename T>
cudaError_t launch_lmhead_simt(const T* y, const T* w_lm, int M, int H, int V,
                               int nstrip, TopkPartials P, cudaStream_t s);
int lmhead_simt_strips(int M, int V, int num_sms);
// With out_m / out_s (a vocabulary shard whose ids start at id_off): ids
// offset by id_off, the rows' (max, sum) pairs instead of lse.
cudaError_t launch_topk_merge(TopkPartials P, int nstrip, int M, float* topv,
                              int* topi, float* lse, cudaStream_t s,
                              int id_off = 0, float* out_m = nullptr,
                              float* out_s = nullptr);
// S shards' partials [S][M][16] + [S][M] pairs -> topv, topi, lse.
cudaError_t launch_shard_merge(const float* pv, const int* pi, const float* pm,
                               const float* ps, int S, int M, float* topv,
                               int* topi, float* lse, cudaStream_t s);

// pair_score.cu -----------------------------------------------------------
// After the LM head, for a precomputed gate [B*K, r] fp32: merge of the
// strip partials, pair scores and walk in one launch (tickets [B], zeroed
// by the conv launch, pick each sequence's walker; walk_j [B*K, 16] and
// walk_q [B*K, 16, 16] hold every row's step from each predecessor slot).
template <typename T>
cudaError_t launch_draft_tail(TopkPartials P, int nstrip, const int* anchor,
                              const float* gate, const T* e_in,
                              const T* e_out, int B, int K, int V, int r,
                              float T_, uint64_t seed, uint64_t cycle,
                              float* topv, int* topi, float* lse,
                              float* scores, int* slot, int* draft, float* q,
                              unsigned* tickets, int* walk_j, float* walk_q,
                              int* err, cudaStream_t s);
// Pair scores from a precomputed gate [B*K, r] fp32 (gathers + bilinear).
template <typename T>
cudaError_t launch_pair_score_gated(const float* topv, const int* topi,
                                    const int* anchor, const float* gate,
                                    const T* e_in, const T* e_out, int B,
                                    int K, int V, int r, float* scores,
                                    int* err, cudaStream_t s);
template <typename T>
cudaError_t launch_pair_score(const float* topv, const int* topi,
                              const int* anchor, const T* h, const T* w_gate,
                              const T* e_in, const T* e_out, int B, int K,
                              int H, int V, int r, float* scores, int* err,
                              cudaStream_t s);

// walk.cu -----------------------------------------------------------------
cudaError_t launch_path_walk(const float* scores, const int* topi, int B,
                             int K, float T, uint64_t seed, uint64_t cycle,
                             int* slot, int* draft, float* q, int* err,
                             cudaStream_t s);

// verify.cu ---------------------------------------------------------------
struct VerifyWs {
  float2* part;        // [rows][segments]: segment (max, sum) pairs at
                       // T > 0, chunk (max, argmax) at T = 0
  int* row_tok;        // [rows] token emitted if t is the first rejection
                       // (t = K: the bonus token)
  unsigned* counters;  // zeroed before every launch: the sequences' words,
                       // then the rows' tickets
  unsigned long long* seq;  // [B] (in counters): bit t (t < K) position t
                            // rejected, bit 32 + t row t decided
  unsigned* tickets;   // [rows] (in counters): chunks of the row done
  size_t counter_bytes;
};
constexpr int kVerifyMaxChunks = 64;  // row chunks (CTAs) per target row
// The verify grid: positions t < t_split in nchunk0 chunks of bpc0 blocks
// per row, later positions in nchunk1 chunks of bpc1 blocks.
struct VerifyGrid {
  int nchunk0, bpc0, nchunk1, bpc1, t_split;
};
size_t verify_ws_layout(int B, int K, int V, void* base, VerifyWs* out);
// The caller zeroes ws.counters on stream s first.  With `stats` (a
// vocabulary shard [v0, v0 + V) of the rows): the rows' shard statistics
// (kShardStats words per row) instead of the accept tests and draws, and
// the segment pairs kept in ws for the shard's draw.
constexpr int kShardStats = DFLASH_SHARD_STATS;
constexpr int kShardPlan = DFLASH_SHARD_PLAN;
cudaError_t launch_verify(const float* L, const int* draft, const int* topi,
                          const float* q, int B, int K, int V, float T,
                          uint64_t seed, uint64_t cycle, int* n_accepted,
                          int* out_tok, const VerifyWs& ws, int num_sms,
                          int* err, cudaStream_t s, int v0 = 0,
                          float* stats = nullptr);
// Every shard's statistics [S][B*(K+1)][kShardStats] -> n, the emitted
// tokens (at T > 0 the drawn one is left -1 for the owner shard's draw) and
// each sequence's draw plan [B][kShardPlan].
cudaError_t launch_verify_shard_decide(const float* stats, int S,
                                       const int* draft, const int* topi,
                                       const float* q, int B, int K, int V,
                                       float T, uint64_t seed, uint64_t cycle,
                                       int* n_accepted, int* out_tok,
                                       float* plan, int* err, cudaStream_t s);
// The draws the plan gives to shard `shard` (its logits L [B*(K+1), V],
// ids v0..v0+V-1, ws from its statistics launch).
cudaError_t launch_verify_shard_draw(const float* L, const float* plan,
                                     const int* topi, const float* q,
                                     int shard, int B, int K, int V, int v0,
                                     float T, int* out_tok,
                                     const VerifyWs& ws, int* err,
                                     cudaStream_t s);

// philox --------------------------------------------------------------------
cudaError_t launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out,
                          int64_t n, cudaStream_t s);

}  // namespace dflash
