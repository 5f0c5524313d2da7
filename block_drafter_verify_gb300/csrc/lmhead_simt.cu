// Step a2 on CUDA cores: LM head + online logsumexp + per-row top-16, for
// fp32 storage (exact fp32 products), plus the merge of per-strip partials
// that every LM-head kernel shares.
//
// "Sixteen candidates per position" (DFlash 2: Block diffusion, wearing a
// drafter's coat): the drafter keeps its 16 best tokens per block slot.
//
// lmhead_simt: grid (row groups of 8, vocab strips).  Warp w owns row w of
// its group and walks the strip 32 columns at a time: lane l computes the
// logit of column v0 + l, the warp folds the 32 logits into its running
// (max, sum exp) and into a top-16 list held by lanes 0..15, sorted by
// (value desc, id asc).  Logits never leave registers.
// topk_merge: one CTA per row merges the strips' lists and (max, sum)
// pairs and writes topv / topi / lse.
#include <algorithm>
#include <climits>

#include "kernels.h"
#include "merge.cuh"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = kThreads / 32;

// Insert (xv, xi) into the lane-distributed sorted list (lanes 0..15).
// `pos` lanes hold entries that rank ahead of the new one.
__device__ __forceinline__ void list_insert(float& tv, int& ti, float xv,
                                            int xi, int pos, int lane) {
  const float pv = __shfl_up_sync(0xffffffffu, tv, 1);
  const int pi = __shfl_up_sync(0xffffffffu, ti, 1);
  if (lane < kC) {
    if (lane > pos) { tv = pv; ti = pi; }
    else if (lane == pos) { tv = xv; ti = xi; }
  }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
    lmhead_simt_kernel(const T* __restrict__ y, const T* __restrict__ w,
                       int M, int H, int V, int strip_w, TopkPartials P) {
  extern __shared__ float4 smem4[];
  float* ys = reinterpret_cast<float*>(smem4);  // [8][H]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int strip = blockIdx.y;
  const int m0 = blockIdx.x * kRowsPerCta;
  for (int i = tid; i < kRowsPerCta * H; i += kThreads) {
    const int rr = i / H, k = i % H;
    ys[i] = (m0 + rr < M) ? to_f32(y[(size_t)(m0 + rr) * H + k]) : 0.f;
  }
  __syncthreads();
  const int m = m0 + warp;
  if (m >= M) return;
  const float* yr = ys + warp * H;

  float tv = -INFINITY;
  int ti = -1;
  float run_m = -INFINITY, run_s = 0.f;
  const int vb = strip * strip_w, ve = min(V, vb + strip_w);
  for (int v0 = vb; v0 < ve; v0 += 32) {
    const int v = v0 + lane;
    float x = -INFINITY;
    if (v < ve) {
      const T* wr = w + (size_t)v * H;
      float acc = 0.f;
      for (int k = 0; k < H; ++k) acc = fmaf(to_f32(wr[k]), yr[k], acc);
      x = acc;
    }
    // running logsumexp
    const float cmax = warp_max(x);
    if (cmax > run_m) {
      run_s *= __expf(run_m - cmax);
      run_m = cmax;
    }
    run_s += warp_sum(x != -INFINITY ? __expf(x - run_m) : 0.f);
    // top-16: columns arrive in increasing id, so a new entry never ranks
    // ahead of an equal value already held
    unsigned ball = __ballot_sync(0xffffffffu, x > __shfl_sync(0xffffffffu, tv, 15));
    while (ball) {
      const int src = __ffs(ball) - 1;
      ball &= ball - 1;
      const float xv = __shfl_sync(0xffffffffu, x, src);
      const int xi = __shfl_sync(0xffffffffu, v, src);
      if (!(xv > __shfl_sync(0xffffffffu, tv, 15))) continue;
      const int pos = __popc(__ballot_sync(0xffffffffu, lane < kC && tv >= xv));
      list_insert(tv, ti, xv, xi, pos, lane);
    }
  }
  const size_t pr = (size_t)m * gridDim.y + strip;
  if (lane < kC) {
    P.v[pr * kC + lane] = tv;
    P.i[pr * kC + lane] = ti;
  }
  if (lane == 0) {
    P.m[pr] = run_m;
    P.s[pr] = run_s;
  }
}

// One CTA of eight warps per row: the merge of merge.cuh.  With out_m
// (a vocabulary shard whose first id is id_off): ids offset by id_off and
// the row's (max, sum) pair written to out_m / out_s instead of lse.
__global__ void __launch_bounds__(kMergeWarps * 32)
    topk_merge_kernel(TopkPartials P, int nstrip, int M, float* topv,
                      int* topi, float* lse, int id_off, float* out_m,
                      float* out_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  __shared__ float s_v[kMergeWarps][kC], s_m[kMergeWarps], s_s[kMergeWarps];
  __shared__ int s_i[kMergeWarps][kC];
  float tv, rm, rs;
  int ti;
  merge_fold_warp(P, nstrip, m, warp, lane, tv, ti, rm, rs);
  if (lane < kC) { s_v[warp][lane] = tv; s_i[warp][lane] = ti; }
  if (lane == 0) { s_m[warp] = rm; s_s[warp] = rs; }
  __syncthreads();
  if (warp != 0) return;
  merge_combine(s_v, s_i, s_m, s_s, lane, tv, ti, rm, rs);
  if (lane < kC) {
    topv[(size_t)m * kC + lane] = tv;
    topi[(size_t)m * kC + lane] = ti >= 0 ? ti + id_off : -1;
  }
  if (lane == 0) {
    if (out_m) {
      out_m[m] = rm;
      out_s[m] = rs;
    } else {
      lse[m] = rm + logf(rs);
    }
  }
}

// Merge of S shards' partials [S][M][16] (global ids) and [S][M] pairs into
// the rows' top-16 and logsumexp: one warp per row, shards in order, each
// list folded by one bitonic merge (skipped when its best entry cannot
// enter the top 16).
__global__ void shard_merge_kernel(const float* __restrict__ pv,
                                   const int* __restrict__ pi,
                                   const float* __restrict__ pm,
                                   const float* __restrict__ ps, int S,
                                   int M, float* __restrict__ topv,
                                   int* __restrict__ topi,
                                   float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int m = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (m >= M) return;
  const int k = lane < kC ? lane : 31 - lane;  // lanes 16..31: reversed
  float tv = -INFINITY, rm = -INFINITY, rs = 0.f;
  int ti = -1;
  for (int sh = 0; sh < S; ++sh) {
    const size_t r = (size_t)sh * M + m;
    lse_combine(rm, rs, pm[r], ps[r], 1.f);
    const float bv = pv[r * kC];
    const int bi = pi[r * kC];
    if (!ranks_ahead(bv, bi, __shfl_sync(0xffffffffu, tv, kC - 1),
                     __shfl_sync(0xffffffffu, ti, kC - 1)))
      continue;
    float v = lane < kC ? tv : pv[r * kC + k];
    int i = lane < kC ? ti : pi[r * kC + k];
    bitonic_merge32(v, i, lane);
    tv = v;
    ti = i;
  }
  if (lane < kC) {
    topv[(size_t)m * kC + lane] = tv;
    topi[(size_t)m * kC + lane] = ti;
  }
  if (lane == 0) lse[m] = rm + logf(rs);
}

}  // namespace

int lmhead_simt_strips(int M, int V, int num_sms) {
  const int groups = (M + kRowsPerCta - 1) / kRowsPerCta;
  int ns = std::max(1, (4 * num_sms + groups - 1) / groups);
  ns = std::min(ns, std::max(1, (V + 255) / 256));
  return std::min(ns, kMaxStrips);
}

template <typename T>
cudaError_t launch_lmhead_simt(const T* y, const T* w_lm, int M, int H, int V,
                               int nstrip, TopkPartials P, cudaStream_t s) {
  int strip_w = (V + nstrip - 1) / nstrip;
  strip_w = (strip_w + 31) & ~31;
  const size_t smem = (size_t)kRowsPerCta * H * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(
      lmhead_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((M + kRowsPerCta - 1) / kRowsPerCta, nstrip);
  lmhead_simt_kernel<T><<<grid, kThreads, smem, s>>>(y, w_lm, M, H, V,
                                                     strip_w, P);
  return cudaGetLastError();
}

cudaError_t launch_topk_merge(TopkPartials P, int nstrip, int M, float* topv,
                              int* topi, float* lse, cudaStream_t s,
                              int id_off, float* out_m, float* out_s) {
  topk_merge_kernel<<<M, kMergeWarps * 32, 0, s>>>(P, nstrip, M, topv, topi,
                                                   lse, id_off, out_m, out_s);
  return cudaGetLastError();
}

cudaError_t launch_shard_merge(const float* pv, const int* pi, const float* pm,
                               const float* ps, int S, int M, float* topv,
                               int* topi, float* lse, cudaStream_t s) {
  const int per_cta = 8;
  shard_merge_kernel<<<(M + per_cta - 1) / per_cta, 32 * per_cta, 0, s>>>(
      pv, pi, pm, ps, S, M, topv, topi, lse);
  return cudaGetLastError();
}

template cudaError_t launch_lmhead_simt<float>(const float*, const float*,
                                               int, int, int, int,
                                               TopkPartials, cudaStream_t);
template cudaError_t launch_lmhead_simt<__nv_bfloat16>(
    const __nv_bfloat16*, const __nv_bfloat16*, int, int, int, int,
    TopkPartials, cudaStream_t);

}  // namespace dflash
