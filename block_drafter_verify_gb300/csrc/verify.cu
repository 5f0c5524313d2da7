// Steps a5 + a6: rejection-sampling verify with residual / bonus draw.
//
// "Lossless, with conditions I did not used to state" (DFlash 2: Block
// diffusion, wearing a drafter's coat): accept a draft token with
// probability min(1, p/q) and resample from the residual on rejection.
//
// One launch over the B*(K+1) target rows, each in chunks, 256 threads:
//   order       the CTAs go in position order (all sequences' chunks of
//               position 0, then position 1, ...).  The first positions,
//               as many as fill the GPU, get chunks sized so that position
//               0 alone makes about two CTAs per SM; the later ones get
//               chunks sized over all their rows, so that few CTAs start.
//               Only rows 0..n of a sequence matter (n its first
//               rejection): once the sequence's word shows a rejection
//               before t, the chunks of row t stop reading and leave
//               without arriving anywhere (a chunk that starts after it
//               reads nothing).  At low acceptance most of the later rows
//               are never read; at high acceptance every row is needed and
//               read, as before.
//   main pass   a CTA walks its chunk in blocks of 16384 tokens; warp w of
//               the CTA owns the contiguous 2048-token segment w of each
//               block and reads it with 16-byte loads straight into
//               registers (lane l holds the words 4l + 128u, u < 16), with
//               no shared-memory staging.  Before each segment a warp
//               checks the sequence's word (rejected positions), read at
//               the CTA's start and then one segment ahead.  At
//               T > 0 a warp reduces a segment to (max, sum
//               2^((x-max)/T log2 e)); at T = 0 the CTA keeps the first
//               argmax.
//   row work    the last CTA to finish row (b, t) (atomic ticket) folds the
//               row in a fixed tree (row max, Z, argmax) and then settles
//               everything that depends on that row alone: the accept test
//               of position t, and at T > 0 the token to emit if position t
//               turns out to be the first rejection (a draw from the
//               residual max(0, p - q) over the <= 16 candidates) or, for
//               t = K, the bonus draw from p.  All draws of sequence b share
//               its one resample uniform, so drawing every row ahead of time
//               gives the same token as drawing only the rejected one.  A
//               row that cannot be emitted skips its draw: its draft was
//               accepted, or an earlier position of the sequence had already
//               recorded a rejection in the sequence's word when the row
//               read it (for t = K: any rejection).  The drafter's inputs of
//               row t (draft, candidates, q and the target logits at those
//               tokens) are fetched at the start of the CTA, and the row's
//               uniforms drawn then, so none of this waits on another launch
//               or row.
//   sequence    a rejected row sets its position's bit in the sequence's
//               64-bit word right after its test; every tested row then
//               sets its decided bit (after its draw).  The row whose bit
//               completes rows 0..n, n the lowest rejected position (K if
//               none), keeps the prefix before n and emits row n's token.
//               A row that stopped early is never among rows 0..n: it
//               stopped on a rejection before it.
// "Last CTA" is an atomic ticket; nothing ever waits.  All folds and sums
// run in a fixed order, so results are identical run to run.
#include <algorithm>

#include "kernels.h"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSegTokens = 2048;                   // one warp's segment
constexpr int kBlockTokens = kWarps * kSegTokens;  // 16384
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// A sequence's result is known once rows 0..n are decided, n its first
// rejected position (K if none): w holds the rejected positions in its low
// word and the decided rows in its high word.  A row's rejection bit goes
// in before its decided bit, so once rows 0..n are decided no bit below n
// can still appear, and the state never turns back.
__device__ __forceinline__ bool seq_settled(unsigned long long w, int K) {
  const unsigned rej = (unsigned)w;
  const int n = rej ? __ffs(rej) - 1 : K;
  const unsigned need = (2u << n) - 1u;  // rows 0..n (n <= 16)
  return ((unsigned)(w >> 32) & need) == need;
}

__device__ __forceinline__ bool arg_better(float v1, int i1, float v2,
                                           int i2) {
  return v1 > v2 || (v1 == v2 && (unsigned)i1 < (unsigned)i2);
}

// exp((x - m) / T) written as 2^(x*s2 + nb) with s2 = log2(e)/T and
// nb = -m*s2: the single weight formula of this file.
__device__ __forceinline__ float weight(float x, float s2, float nb) {
  return ex2f(fmaf(x, s2, nb));
}

// Fold (m2, s2v) into (m, s): pairs of (max, sum of 2^((x-max) s2)).
__device__ __forceinline__ void fold_lse(float& m, float& s, float m2,
                                         float s2v, float s2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2v; return; }
  const float mx = fmaxf(m, m2);
  s = s * ex2f((m - mx) * s2) + s2v * ex2f((m2 - mx) * s2);
  m = mx;
}

__device__ __forceinline__ float max4(const float4& f) {
  return fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w));
}

// The 64 tokens lane `lane` owns in the segment starting at `base`:
// 16-byte loads at base + 4*lane + 128*u (u < 16), -inf past V.
__device__ __forceinline__ void load_segment(const float* x, int base, int V,
                                             int lane, int vec4,
                                             float4 (&f)[16]) {
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const int v = base + 4 * lane + 128 * u;
    if (vec4) {
      f[u] = v < V ? *reinterpret_cast<const float4*>(x + v)
                   : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    } else {
      f[u] = make_float4(v < V ? x[v] : -INFINITY,
                         v + 1 < V ? x[v + 1] : -INFINITY,
                         v + 2 < V ? x[v + 2] : -INFINITY,
                         v + 3 < V ? x[v + 3] : -INFINITY);
    }
  }
}

// Shared memory of one row's draw (row_draw).
struct DrawSmem {
  int seg, use_raw, pick, last;
  float rem;
  float W[kWarps];
};

// The inverse-CDF draw inside one target row x[0, V), by every thread of
// the CTA.  Token v weighs w(v) = 2^((x_v - m) s2) minus, unless raw, the
// correction of the candidate it is (s_ci / s_qz: w = max(0, w - q Z));
// the row's 2048-token segments weigh their (max, sum) pair (s_pair)
// rescaled to m plus the corrections of the candidates inside them
// (s_corr), clamped at zero; every thread computes some segments' two
// weights (residual, raw), which replace their pairs in s_pair.  Target
// theta: u * (the row's total) when theta_abs < 0, where a zero residual
// total switches to raw weights; else theta_abs with raw = raw_given.
// Warp 0 locates the segment (lane l owns segments l*per .. l*per+per-1:
// one inclusive scan of the lane totals and a ballot); the CTA then takes
// the smallest token of the
// segment whose running sum exceeds theta (8 contiguous tokens per thread,
// block scan in a fixed tree).  Returns the token on every thread (the
// segment's last token of positive weight if rounding leaves the target at
// the segment's end), or -1 if no segment has weight.
__device__ __forceinline__ int row_draw(
    const float* __restrict__ x, int V, int nseg, float2* s_pair,
    const int* s_ci, const float* s_qz, const float* s_corr, float m,
    float s2, float u, float theta_abs, bool raw_given, DrawSmem& sm,
    int* err) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const float nb = -m * s2;
  for (int k = tid; k < nseg; k += kThreads) {
    const float2 p = s_pair[k];
    const float wr = (p.x == -INFINITY) ? 0.f : p.y * ex2f((p.x - m) * s2);
    float w = wr;
#pragma unroll
    for (int j = 0; j < kC; ++j)
      if (s_ci[j] >= 0 && s_ci[j] / kSegTokens == k) w += s_corr[j];
    s_pair[k] = make_float2(fmaxf(w, 0.f), fmaxf(wr, 0.f));
  }
  __syncthreads();
  if (wid == 0) {
    const int per = (nseg + 31) / 32;
    auto seg_weight = [&](int k, bool raw) -> float {
      if (k >= nseg) return 0.f;
      return raw ? s_pair[k].y : s_pair[k].x;
    };
    int f_seg = -1, f_raw = 0;
    float f_rem = 0.f;
    const int raw0 = theta_abs >= 0.f ? (raw_given ? 1 : 0) : 0;
    const int raw1 = theta_abs >= 0.f ? raw0 : 1;
    for (int raw = raw0; raw <= raw1 && f_seg < 0; ++raw) {
      float ltot = 0.f;
      for (int i = 0; i < per; ++i) ltot += seg_weight(lane * per + i, raw);
      float incl = ltot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float tt = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += tt;
      }
      const float total = __shfl_sync(0xffffffffu, incl, 31);
      if (!(total > 0.f)) continue;  // degenerate residual: draw from p
      const float theta = theta_abs >= 0.f ? theta_abs : u * total;
      const unsigned hit = __ballot_sync(0xffffffffu, ltot > 0.f && incl > theta);
      const unsigned live = __ballot_sync(0xffffffffu, ltot > 0.f);
      // theta rounded up to the total: the last lane with weight
      const int Ls = hit ? __ffs(hit) - 1 : 31 - __clz(live);
      if (lane == Ls) {
        float a = incl - ltot;
        int last = -1;
        for (int i = 0; i < per; ++i) {
          const float w = seg_weight(lane * per + i, raw);
          if (w > 0.f) last = lane * per + i;
          if (w > 0.f && a + w > theta) {
            f_seg = lane * per + i;
            f_rem = theta - a;
            break;
          }
          a += w;
        }
        if (f_seg < 0) {
          f_seg = last;
          f_rem = INFINITY;
        }
      }
      f_seg = __shfl_sync(0xffffffffu, f_seg, Ls);
      f_rem = __shfl_sync(0xffffffffu, f_rem, Ls);
      f_raw = raw;
    }
    if (lane == 0) {
      sm.seg = f_seg;
      sm.rem = f_rem;
      sm.use_raw = f_raw;
      sm.pick = -1;
      sm.last = -1;
    }
  }
  __syncthreads();
  const int seg = sm.seg;
  if (seg < 0) {  // no weight anywhere (the row maximum has weight 1)
    if (tid == 0) raise_error(err, kErrBadIndex);
    return -1;
  }
  // the 2048 tokens of the segment: 8 contiguous tokens per thread
  const bool use_raw = sm.use_raw;
  const int t0 = seg * kSegTokens + tid * 8;
  unsigned own = 0;  // the candidates among this thread's tokens
  if (!use_raw) {
#pragma unroll
    for (int j = 0; j < kC; ++j)
      if ((unsigned)(s_ci[j] - t0) < 8u) own |= 1u << j;
  }
  float w8[8];
  float tsum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int v = t0 + i;
    float wv = 0.f;
    if (v < V) {
      wv = weight(x[v], s2, nb);
      for (unsigned mm = own; mm; mm &= mm - 1) {
        const int j = __ffs(mm) - 1;  // candidate order, as in the weights
        if (s_ci[j] == v) wv = fmaxf(wv - s_qz[j], 0.f);
      }
    }
    w8[i] = wv;
    tsum += wv;
  }
  // block exclusive scan of tsum (fixed tree)
  float incl = tsum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float tt = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += tt;
  }
  if (lane == 31) sm.W[wid] = incl;
  __syncthreads();
  float pre = 0.f, segtot = 0.f;
  for (int w = 0; w < kWarps; ++w) {
    if (w < wid) pre += sm.W[w];
    segtot += sm.W[w];
  }
  const float excl = pre + incl - tsum;
  // rounding may leave the target at or past the recomputed total
  const float rem = fminf(sm.rem, segtot * (1.f - 0x1p-22f));
  int last = -1;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (w8[i] > 0.f) last = t0 + i;
  if (last >= 0) atomicMax(&sm.last, last);
  if (tsum > 0.f && excl <= rem && rem < excl + tsum) {
    float a = excl;
    int pick = -1;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      a += w8[i];
      if (pick < 0 && a > rem) pick = t0 + i;
    }
    atomicMax(&sm.pick, pick >= 0 ? pick : last);
  }
  __syncthreads();
  return sm.pick >= 0 ? sm.pick : sm.last;
}

// kStats: the row statistics of one vocabulary shard [v0, v0 + V) (the
// rows hold the shard's V logits; token ids are global): the main pass
// keeps its segment pairs in the workspace for the shard's later draw, and
// the row's last CTA writes the row's entry of `stats` (kShardStats words:
// max and sum, or max and argmax at T = 0; the logits of the candidates
// and of the draft the shard holds; a mask of which it holds) instead of
// the accept test and draw.
template <bool kStats>
__global__ void __launch_bounds__(kThreads, 2)  // two CTAs per SM
    verify_kernel(const float* __restrict__ L, const int* __restrict__ draft,
                  const int* __restrict__ topi, const float* __restrict__ q,
                  int B, int K, int V, VerifyGrid g, float T, float s2,
                  uint64_t seed, uint64_t cycle, int* __restrict__ n_accepted,
                  int* __restrict__ out_tok, VerifyWs ws, int* err, int vec4,
                  int v0, float* __restrict__ stats) {
  // CTAs in position order: the rows of positions t < g.t_split (enough to
  // fill the GPU) in g.nchunk0 chunks each, chunk c of row (b, t) being CTA
  // (t B + b) nchunk0 + c; after them the later positions' rows, in
  // g.nchunk1 chunks each, in the same order
  const int tid = threadIdx.x;
  const int lane = tid & 31, wid = tid >> 5;
  const int K1 = K + 1;
  const unsigned n_early = (unsigned)(g.t_split * B * g.nchunk0);
  const bool early = blockIdx.x < n_early;
  const int nchunk = early ? g.nchunk0 : g.nchunk1;
  const int bpc = early ? g.bpc0 : g.bpc1;
  const unsigned xi = early ? blockIdx.x : blockIdx.x - n_early;
  const int c = (int)(xi % (unsigned)nchunk);
  const int rt = (int)(xi / (unsigned)nchunk);
  const int t = (early ? 0 : g.t_split) + rt / B, b = rt % B;
  const int row = b * K1 + t;
  const int nseg = (V + kSegTokens - 1) / kSegTokens;
  const float* x = L + (size_t)row * V;
  const bool greedy = (T == 0.f);
  // the row's pairs: written here when one CTA covers the row, else loaded
  extern __shared__ float2 s_pair[];

  __shared__ float s_a[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_flag, s_acc, s_need;
  __shared__ unsigned s_rej;
  __shared__ float s_m;
  __shared__ DrawSmem s_draw;
  __shared__ int s_ci[kC];
  __shared__ float s_qz[kC], s_corr[kC];

  // A row after its sequence's first rejection is never emitted: once the
  // sequence's word shows a rejection before t, a warp stops reading.  The
  // word is read first (a CTA that starts after such a rejection reads no
  // segment; the inputs below cover the read's latency), then one segment
  // ahead.
  const bool may_skip = !kStats && t > 0;
  const unsigned before = (1u << t) - 1u;
  unsigned mk = 0;
  if (may_skip && lane == 0) mk = (unsigned)__ldcg(&ws.seq[b]);

  // ---- the drafter's inputs of this row, in flight during the main pass --
  // lanes 0-15 of warp 0: candidate j (token, q, target logit); lane 16:
  // the draft token.  Loaded into registers now, stored after the pass.
  const bool has_draft = t < K;
  int r_tok = -1;
  float r_q = 0.f;
  if (wid == 0 && has_draft) {
    if (lane < kC) {
      r_tok = topi[(b * K + t) * kC + lane];
      r_q = kStats ? 0.f : q[(b * K + t) * kC + lane];
    } else if (lane == kC) {
      r_tok = draft[b * K + t];
    }
  }
  // the row's accept uniform and the sequence's resample uniform, computed
  // now rather than after the pass, where the row's work waits on them
  const bool draws = !kStats && !greedy;
  const float u_acc =
      draws && has_draft ? philox_uniform(seed, b, t, kPurposeAccept, cycle)
                         : 0.f;
  const float u_res =
      draws ? philox_uniform(seed, b, K, kPurposeResample, cycle) : 0.f;

  // ---- main pass ------------------------------------------------------
  // Segments of this chunk: sc0 .. sc1-1; warp w takes sc0 + w + 8 j.
  bool skipped = false;
  bool bad = false;
  float ga = -INFINITY;   // T = 0: this thread's best value ...
  int gi = 0x7fffffff;    // ... and its (first) index
  const int sc0 = c * bpc * kWarps;
  const int sc1 = min(nseg, (c + 1) * bpc * kWarps);
  const int nmine = sc0 + wid < sc1 ? (sc1 - (sc0 + wid) + kWarps - 1) / kWarps : 0;
  float r_x = 0.f;  // target logit at r_tok (fetched after the first segment)
  // the row holds r_tok (a shard holds ids v0 .. v0 + V - 1)
  const bool r_own = r_tok >= v0 && r_tok - v0 < V;
  for (int j = 0; j < nmine; ++j) {
    if (may_skip && (__shfl_sync(0xffffffffu, mk, 0) & before)) {
      skipped = true;
      break;
    }
    const int seg = sc0 + wid + kWarps * j;
    const int base = seg * kSegTokens;
    float4 f[16];
    load_segment(x, base, V, lane, vec4, f);
    if (may_skip && lane == 0) mk = (unsigned)__ldcg(&ws.seq[b]);
    if (j == 0 && wid == 0 && r_own) r_x = x[r_tok - v0];
    if (greedy) {
      float chk = 0.f;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int v = base + 4 * lane + 128 * u;
        chk += (f[u].x + f[u].y) + (f[u].z + f[u].w);
        if (f[u].x > ga) { ga = f[u].x; gi = v; }
        if (f[u].y > ga) { ga = f[u].y; gi = v + 1; }
        if (f[u].z > ga) { ga = f[u].z; gi = v + 2; }
        if (f[u].w > ga) { ga = f[u].w; gi = v + 3; }
      }
      bad |= (chk != chk) || ga == INFINITY;
    } else {
      float mx = max4(f[0]);
#pragma unroll
      for (int u = 1; u < 16; ++u) mx = fmaxf(mx, max4(f[u]));
#pragma unroll
      for (int o = 16; o; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      float sum = 0.f;
      if (mx != -INFINITY) {
        const float nb = -mx * s2;
        float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          p[u & 3] += weight(f[u].x, s2, nb) + weight(f[u].y, s2, nb) +
                      weight(f[u].z, s2, nb) + weight(f[u].w, s2, nb);
        }
        sum = (p[0] + p[1]) + (p[2] + p[3]);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      bad |= (sum != sum) || mx == INFINITY;
      if (lane == 0) {
        const float2 pr = make_float2(mx, sum);
        if (nchunk == 1) s_pair[seg] = pr;
        if (nchunk > 1 || kStats) ws.part[(size_t)row * nseg + seg] = pr;
      }
    }
  }
  if (wid == 0 && nmine == 0 && r_own) r_x = x[r_tok - v0];
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(err, kErrNonfinite);
  if (greedy) {  // chunk argmax: lanes, then warps, in a fixed tree
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float oa = __shfl_xor_sync(0xffffffffu, ga, o);
      const int oi = __shfl_xor_sync(0xffffffffu, gi, o);
      if (arg_better(oa, oi, ga, gi)) { ga = oa; gi = oi; }
    }
    if (lane == 0) { s_a[wid] = ga; s_i[wid] = gi; }
  }
  // a CTA that stopped early leaves without arriving: its row is after the
  // sequence's first rejection, and no result depends on it
  if (__syncthreads_or(skipped)) return;
  if (tid == 0) {
    if (greedy) {
      float ra = s_a[0];
      int ri = s_i[0];
      for (int w = 1; w < kWarps; ++w)
        if (arg_better(s_a[w], s_i[w], ra, ri)) { ra = s_a[w]; ri = s_i[w]; }
      s_a[0] = ra;
      s_i[0] = ri;
      if (nchunk > 1)
        ws.part[(size_t)row * nseg + c] = make_float2(ra, __int_as_float(ri));
    }
    if (nchunk > 1) {
      __threadfence();
      s_flag = (atomicAdd(&ws.tickets[row], 1u) == (unsigned)(nchunk - 1));
    } else {
      s_flag = 1;
    }
  }
  __syncthreads();
  if (!s_flag) return;

  // ---- last CTA of row (b, t): fold it ----------------------------------
  if (nchunk > 1) {
    __threadfence();
    const int nparts = greedy ? nchunk : nseg;
    for (int k = tid; k < nparts; k += kThreads)
      s_pair[k] = __ldcg(&ws.part[(size_t)row * nseg + k]);
    __syncthreads();
  }
  if (wid == 0) {
    // the sequence's rejections so far, in flight during the fold
    unsigned seen = 0;
    if (!kStats && !greedy && lane == 0) seen = (unsigned)__ldcg(&ws.seq[b]);
    float ra = -INFINITY, rs = 0.f;
    int ri = 0x7fffffff;
    if (greedy) {
      if (nchunk == 1) {
        ra = s_a[0];
        ri = s_i[0];
      } else {
        for (int k = lane; k < nchunk; k += 32) {
          const float2 p = s_pair[k];
          if (arg_better(p.x, __float_as_int(p.y), ra, ri)) {
            ra = p.x;
            ri = __float_as_int(p.y);
          }
        }
      }
    } else {
      for (int k = lane; k < nseg; k += 32) {
        const float2 p = s_pair[k];
        fold_lse(ra, rs, p.x, p.y, s2);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float oa = __shfl_xor_sync(0xffffffffu, ra, o);
      const float os = __shfl_xor_sync(0xffffffffu, rs, o);
      const int oi = __shfl_xor_sync(0xffffffffu, ri, o);
      if (greedy) {
        if (arg_better(oa, oi, ra, ri)) { ra = oa; ri = oi; }
      } else {
        fold_lse(ra, rs, oa, os, s2);
      }
    }
    if constexpr (kStats) {
      // a shard may hold no mass of a row: (-inf, 0) folds to nothing
      float* st = stats + (size_t)row * kShardStats;
      const unsigned own = __ballot_sync(0xffffffffu, lane <= kC && r_own);
      if (lane == 0) {
        st[0] = ra;
        st[1] = greedy ? __int_as_float(ri == 0x7fffffff ? -1 : v0 + ri) : rs;
        st[kShardStats - 1] = __uint_as_float(own);
      }
      if (lane < kC) st[2 + lane] = r_own ? r_x : 0.f;
      if (lane == kC) st[2 + kC] = r_own ? r_x : 0.f;
      return;
    }
    if (ra == -INFINITY) {  // every logit of the row is -inf
      if (lane == 0) raise_error(err, kErrNonfinite);
      ri = 0; ra = 0.f; rs = 1.f;
    }
    // accept test of position t (t < K), lane 16 holding the draft token
    const int d = __shfl_sync(0xffffffffu, r_tok, kC);
    const float xd = __shfl_sync(0xffffffffu, r_x, kC);
    int acc = 1;
    if (has_draft) {
      if (d < 0 || d >= V) {
        if (lane == 0) raise_error(err, kErrBadIndex);
        acc = 0;
      } else if (greedy) {
        acc = (d == ri);
      } else {
        // q of the draft: its first match among the candidates
        const unsigned hit = __ballot_sync(0xffffffffu, lane < kC && r_tok == d);
        const float qd = hit ? __shfl_sync(0xffffffffu, r_q, __ffs(hit) - 1) : 0.f;
        if (!hit && lane == 0) raise_error(err, kErrBadIndex);
        const float pd = weight(xd, s2, -ra * s2) / rs;
        acc = (u_acc * qd < pd);
      }
    }
    if (greedy) {
      if (lane == 0) {
        s_acc = acc;
        ws.row_tok[row] = ri;
        if (has_draft && !acc) atomicOr(&ws.seq[b], 1ull << t);
      }
    } else {
      // residual corrections of the candidates: -min(p_j Z, q_j Z)
      if (lane < kC) {
        int cj = has_draft ? r_tok : -1;
        float qz = 0.f, corr = 0.f;
        if (cj >= 0 && cj < V) {
          qz = r_q * rs;
          corr = -fminf(weight(r_x, s2, -ra * s2), qz);
        } else {
          cj = -1;
        }
        s_ci[lane] = cj;
        s_qz[lane] = qz;
        s_corr[lane] = corr;
      }
      if (lane == 0) {
        s_m = ra;
        s_acc = acc;
        // Row t's token is emitted only if t is the first rejection (t < K)
        // or nothing is rejected (t = K): a row whose draft was accepted,
        // or that follows a rejection already in the sequence's word (read
        // before the fold), skips its draw.  A stale word only costs a
        // draw.  The row's own rejection is added without waiting.
        const unsigned below = (1u << t) - 1u;
        if (has_draft) {
          s_need = !acc && !(seen & below);
          if (!acc) atomicOr(&ws.seq[b], 1ull << t);
        } else {
          s_need = seen == 0u;
        }
      }
    }
  }
  if constexpr (kStats) return;  // warp 0 wrote the row's statistics
  if (!greedy) {
    __syncthreads();
  }
  if (!greedy && s_need) {
    // ---- draw of row (b, t): residual max(0, p - q), or p for t = K ------
    const int tok = row_draw(x, V, nseg, s_pair, s_ci, s_qz, s_corr, s_m, s2,
                             u_res, -1.f, false, s_draw, err);
    if (tid == 0) ws.row_tok[row] = tok;
  }

  // ---- the sequence's word: the row is decided (and, rejected, its
  // position's bit); the row whose bit completes rows 0..n (n the first
  // rejection) emits the tokens ------------------------------------------
  __syncthreads();
  if (tid == 0) {
    const unsigned long long mine =
        (1ull << (32 + t)) | (has_draft && !s_acc ? 1ull << t : 0ull);
    __threadfence();  // the row's token before its bit
    const unsigned long long old = atomicOr(&ws.seq[b], mine);
    s_flag = !seq_settled(old, K) && seq_settled(old | mine, K);
    s_rej = (unsigned)(old | mine);
  }
  __syncthreads();
  if (!s_flag || wid != 0) return;
  __threadfence();
  const unsigned rej = s_rej;
  const int n = rej ? __ffs(rej) - 1 : K;
  if (lane == 0) n_accepted[b] = n;
  if (lane <= K) {
    int tok = -1;
    if (lane < n) tok = draft[b * K + lane];
    else if (lane == n) tok = __ldcg(&ws.row_tok[b * K1 + n]);
    out_tok[b * K1 + lane] = tok;
  }
}

// ---- vocabulary shards: decide and draw ----------------------------------
// Plan of one sequence's draw (kShardPlan words): [0] owner shard (int,
// -1: none), [1] target theta within the owner's residual (or p) weights,
// [2] the row's global max m, [3] its Z = sum 2^((x - m) s2), [4] raw
// weights (int), [5] the row n (int).

// One warp per sequence, lane t = row t (t <= K): the rows' shard
// statistics folded in shard order (global max and Z, or the argmax), the
// accept tests with the draft's logit from the shard that holds it, n, the
// emitted prefix, and for T > 0 the draw plan of row n: each shard's
// residual mass (its rescaled sum plus the corrections of the candidates it
// holds, clamped at zero; raw sums when the total residual is zero or
// n = K), theta = u * total, the first shard whose running mass exceeds
// theta and the remainder within it.
__global__ void verify_shard_decide_kernel(
    const float* __restrict__ stats, int S, const int* __restrict__ draft,
    const int* __restrict__ topi, const float* __restrict__ q, int B, int K,
    int V, float T, float s2, uint64_t seed, uint64_t cycle,
    int* __restrict__ n_accepted, int* __restrict__ out_tok,
    float* __restrict__ plan, int* err) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (b >= B) return;
  const int K1 = K + 1, rows = B * K1;
  const bool greedy = T == 0.f;
  const int t = lane;
  const int row = b * K1 + min(t, K);
  float m = -INFINITY, Z = 0.f, xd = 0.f;
  int bi = 0x7fffffff;
  bool have_d = false;
  for (int sh = 0; sh < S; ++sh) {
    const float* st = stats + ((size_t)sh * rows + row) * kShardStats;
    if (greedy) {
      const int id = __float_as_int(st[1]);
      if (id >= 0 && arg_better(st[0], id, m, bi)) { m = st[0]; bi = id; }
    } else {
      fold_lse(m, Z, st[0], st[1], s2);
    }
    if ((__float_as_uint(st[kShardStats - 1]) >> kC) & 1u) {
      xd = st[2 + kC];
      have_d = true;
    }
  }
  if (t <= K && (m == -INFINITY || (greedy && bi == 0x7fffffff))) {
    raise_error(err, kErrNonfinite);  // every logit of the row is -inf
    m = 0.f; Z = 1.f; bi = 0;
  }
  int acc = 1;
  int d = -1;
  if (t < K) {
    d = draft[b * K + t];
    if (d < 0 || d >= V || !have_d) {
      raise_error(err, kErrBadIndex);
      acc = 0;
    } else if (greedy) {
      acc = d == bi;
    } else {
      float qd = 0.f;
      int j = 0;
      for (; j < kC; ++j)
        if (topi[(b * K + t) * kC + j] == d) { qd = q[(b * K + t) * kC + j]; break; }
      if (j == kC) raise_error(err, kErrBadIndex);
      const float pd = weight(xd, s2, -m * s2) / Z;
      const float u = philox_uniform(seed, b, t, kPurposeAccept, cycle);
      acc = u * qd < pd;
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, t < K && !acc);
  const int n = rej ? __ffs(rej) - 1 : K;
  if (lane == 0) n_accepted[b] = n;
  if (t <= K) out_tok[b * K1 + t] = t < n ? d : (t == n && greedy ? bi : -1);
  if (t != n) return;
  float* pl = plan + (size_t)b * kShardPlan;
  pl[0] = __int_as_float(-1);
  pl[5] = __int_as_float(n);
  if (greedy) return;
  // row n's draw: residual masses per shard (raw for the bonus row)
  const float u = philox_uniform(seed, b, K, kPurposeResample, cycle);
  float tot_res = 0.f, tot_raw = 0.f;
  auto shard_mass = [&](int sh, bool raw) -> float {
    const float* st = stats + ((size_t)sh * rows + row) * kShardStats;
    float w = st[0] == -INFINITY ? 0.f : st[1] * ex2f((st[0] - m) * s2);
    if (!raw && n < K) {
      const unsigned own = __float_as_uint(st[kShardStats - 1]);
      for (int j = 0; j < kC; ++j)
        if ((own >> j) & 1u) {
          const float qz = q[(b * K + n) * kC + j] * Z;
          w -= fminf(weight(st[2 + j], s2, -m * s2), qz);
        }
    }
    return fmaxf(w, 0.f);
  };
  for (int sh = 0; sh < S; ++sh) {
    tot_res += shard_mass(sh, false);
    tot_raw += shard_mass(sh, true);
  }
  const bool raw = !(tot_res > 0.f) || n == K;
  const float total = raw ? tot_raw : tot_res;
  const float theta = u * total;
  int owner = -1, last = -1;
  float a = 0.f, rem = 0.f;
  for (int sh = 0; sh < S; ++sh) {
    const float w = shard_mass(sh, raw);
    if (w > 0.f) last = sh;
    if (w > 0.f && a + w > theta) { owner = sh; rem = theta - a; break; }
    a += w;
  }
  if (owner < 0) {  // theta rounded up to the total: the last shard's end
    owner = last;
    rem = INFINITY;
  }
  if (owner < 0) raise_error(err, kErrBadIndex);  // no mass anywhere
  pl[0] = __int_as_float(owner);
  pl[1] = rem;
  pl[2] = m;
  pl[3] = Z;
  pl[4] = __int_as_float(raw ? 1 : 0);
}

// The draw of each sequence whose plan names this shard, one CTA per
// sequence: the shard's segment pairs of row n (left in its workspace by
// the statistics launch), the corrections of the candidates it holds, and
// row_draw with the plan's target, max, Z and weights.
__global__ void __launch_bounds__(kThreads)
    verify_shard_draw_kernel(const float* __restrict__ L,
                             const float* __restrict__ plan,
                             const int* __restrict__ topi,
                             const float* __restrict__ q, int shard, int B,
                             int K, int V, int v0, float s2,
                             int* __restrict__ out_tok, VerifyWs ws,
                             int* err) {
  const int b = blockIdx.x, tid = threadIdx.x;
  const int K1 = K + 1;
  const int nseg = (V + kSegTokens - 1) / kSegTokens;
  const float* pl = plan + (size_t)b * kShardPlan;
  if (__float_as_int(pl[0]) != shard) return;
  const int n = __float_as_int(pl[5]);
  const float theta = pl[1], m = pl[2], Z = pl[3];
  const bool raw = __float_as_int(pl[4]) != 0;
  const int row = b * K1 + n;
  const float* x = L + (size_t)row * V;
  extern __shared__ float2 s_pair[];
  __shared__ int s_ci[kC];
  __shared__ float s_qz[kC], s_corr[kC];
  __shared__ DrawSmem s_draw;
  for (int k = tid; k < nseg; k += kThreads)
    s_pair[k] = __ldcg(&ws.part[(size_t)row * nseg + k]);
  if (tid < kC) {
    int ci = -1;
    float qz = 0.f, corr = 0.f;
    if (n < K) {
      const int c = topi[(b * K + n) * kC + tid];
      if (c >= v0 && c - v0 < V) {
        ci = c - v0;
        qz = q[(b * K + n) * kC + tid] * Z;
        corr = -fminf(weight(x[ci], s2, -m * s2), qz);
      }
    }
    s_ci[tid] = ci;
    s_qz[tid] = qz;
    s_corr[tid] = corr;
  }
  __syncthreads();
  const int tok = row_draw(x, V, nseg, s_pair, s_ci, s_qz, s_corr, m, s2,
                           0.f, fmaxf(theta, 0.f), raw, s_draw, err);
  if (tid == 0) out_tok[b * K1 + n] = tok >= 0 ? v0 + tok : -1;
}

__global__ void philox_kernel(const uint32_t* __restrict__ ctr, uint64_t seed,
                              uint32_t* __restrict__ out, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = reinterpret_cast<const uint4*>(ctr)[i];
  const U32x4 r = philox4x32_10(U32x4{c.x, c.y, c.z, c.w}, (uint32_t)seed,
                                (uint32_t)(seed >> 32));
  reinterpret_cast<uint4*>(out)[i] = make_uint4(r.x, r.y, r.z, r.w);
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

size_t verify_ws_layout(int B, int K, int V, void* base, VerifyWs* o) {
  const size_t rows = (size_t)B * (K + 1);
  const size_t nseg = ((size_t)V + kSegTokens - 1) / kSegTokens;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = align256(off);
    char* r = p ? p + off : nullptr;
    off += bytes;
    return r;
  };
  VerifyWs w{};
  // per row: segment pairs (T > 0) or chunk argmaxes (T = 0, <= nseg)
  w.part = reinterpret_cast<float2*>(take(rows * nseg * sizeof(float2)));
  w.row_tok = reinterpret_cast<int*>(take(rows * sizeof(int)));
  // the sequences' 64-bit words (rejected positions, decided rows; first,
  // so they are 8-byte aligned), then the rows' tickets (chunks done), all
  // zeroed together before a launch
  w.counter_bytes = (2 * (size_t)B + rows) * sizeof(unsigned);
  w.counters = reinterpret_cast<unsigned*>(take(w.counter_bytes));
  w.seq = reinterpret_cast<unsigned long long*>(w.counters);
  w.tickets = w.counters ? w.counters + 2 * B : nullptr;
  if (o) *o = w;
  return align256(off);
}

// The caller zeroes ws.counters on the stream before this launch.
cudaError_t launch_verify(const float* L, const int* draft, const int* topi,
                          const float* q, int B, int K, int V, float T,
                          uint64_t seed, uint64_t cycle, int* n_accepted,
                          int* out_tok, const VerifyWs& ws, int num_sms,
                          int* err, cudaStream_t s, int v0, float* stats) {
  const int rows = B * (K + 1);
  const int nseg = (V + kSegTokens - 1) / kSegTokens;
  const int blocks_per_row = (V + kBlockTokens - 1) / kBlockTokens;
  const int vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(L) & 15) == 0);
  // Chunks of whole 16384-token blocks, at most kVerifyMaxChunks per row,
  // equal to within a block: for `nrows` rows, about two CTAs per SM.
  const long long per_sm = 2, slots = per_sm * num_sms;
  auto chunking = [&](long long nrows, int* nchunk, int* bpc) {
    const long long blocks = nrows * blocks_per_row;
    int b = (int)std::max<long long>(1, (blocks + slots - 1) / slots);
    b = std::max(b, (blocks_per_row + kVerifyMaxChunks - 1) / kVerifyMaxChunks);
    b = std::min(b, blocks_per_row);
    *nchunk = (blocks_per_row + b - 1) / b;
    *bpc = (blocks_per_row + *nchunk - 1) / *nchunk;
  };
  // The CTAs run in position order and rows after a sequence's first
  // rejection stop early.  The first positions (enough to fill the GPU)
  // get chunks sized so that position 0 alone makes about two CTAs per SM;
  // the later positions get chunks sized over all their rows, so that few
  // CTAs have to start (and, at low acceptance, leave at once).  Shard
  // statistics read every row: one chunking over all rows.
  VerifyGrid g{};
  const int K1 = K + 1;
  if (stats) {
    chunking(rows, &g.nchunk0, &g.bpc0);
    g.t_split = K1;
  } else {
    chunking(B, &g.nchunk0, &g.bpc0);
    const long long per_pos = (long long)B * g.nchunk0;
    g.t_split = (int)std::min<long long>(K1, (slots + per_pos - 1) / per_pos);
  }
  g.nchunk1 = g.nchunk0;
  g.bpc1 = g.bpc0;
  if (g.t_split < K1) chunking((long long)(K1 - g.t_split) * B, &g.nchunk1, &g.bpc1);
  const long long ctas = (long long)g.t_split * B * g.nchunk0 +
                         (long long)(K1 - g.t_split) * B * g.nchunk1;
  const float s2 = T > 0.f ? kLog2e / T : 0.f;
  const size_t smem = (size_t)nseg * sizeof(float2);
  auto kern = stats ? verify_kernel<true> : verify_kernel<false>;
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)ctas, kThreads, smem, s>>>(
      L, draft, topi, q, B, K, V, g, T, s2, seed, cycle, n_accepted,
      out_tok, ws, err, vec4, v0, stats);
  return cudaGetLastError();
}

cudaError_t launch_verify_shard_decide(const float* stats, int S,
                                       const int* draft, const int* topi,
                                       const float* q, int B, int K, int V,
                                       float T, uint64_t seed, uint64_t cycle,
                                       int* n_accepted, int* out_tok,
                                       float* plan, int* err, cudaStream_t s) {
  const float s2 = T > 0.f ? kLog2e / T : 0.f;
  const int per_cta = 4;  // warps (sequences) per CTA
  verify_shard_decide_kernel<<<(B + per_cta - 1) / per_cta, 32 * per_cta, 0,
                               s>>>(stats, S, draft, topi, q, B, K, V, T, s2,
                                    seed, cycle, n_accepted, out_tok, plan,
                                    err);
  return cudaGetLastError();
}

cudaError_t launch_verify_shard_draw(const float* L, const float* plan,
                                     const int* topi, const float* q,
                                     int shard, int B, int K, int V, int v0,
                                     float T, int* out_tok,
                                     const VerifyWs& ws, int* err,
                                     cudaStream_t s) {
  if (!(T > 0.f)) return cudaSuccess;  // T = 0: decided with the argmax
  const float s2 = kLog2e / T;
  const int nseg = (V + kSegTokens - 1) / kSegTokens;
  const size_t smem = (size_t)nseg * sizeof(float2);
  if (smem > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(
        verify_shard_draw_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem);
    if (e != cudaSuccess) return e;
  }
  verify_shard_draw_kernel<<<B, kThreads, smem, s>>>(
      L, plan, topi, q, shard, B, K, V, v0, s2, out_tok, ws, err);
  return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out,
                          int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  philox_kernel<<<(unsigned)blocks, threads, 0, s>>>(ctr, seed, out, n);
  return cudaGetLastError();
}

}  // namespace dflash
