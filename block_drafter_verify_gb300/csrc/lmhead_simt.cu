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

__device__ __forceinline__ bool ranks_ahead(float v1, int i1, float v2,
                                            int i2) {
  return v1 > v2 || (v1 == v2 && (unsigned)i1 < (unsigned)i2);
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

// One CTA of eight warps per row.  Warp w prefetches the lists of strips
// w, w+8, ... (all loads in flight at once) and folds each into a sorted
// top-16 held by lanes 0..15 with a bitonic merge: lanes 0..15 hold the
// current list best-first, lanes 16..31 the new list worst-first, and five
// compare-exchange steps (distance 16, 8, 4, 2, 1) sort the 32 entries.  A
// list whose best entry does not beat the current 16th is skipped.  Warp 0
// then merges the eight warp lists in warp order; (max, sum) pairs are
// folded per warp in strip order and then in warp order.  The result does
// not depend on timing.
constexpr int kMergeWarps = 8;
constexpr int kMaxPerWarp = (kMaxStrips + kMergeWarps - 1) / kMergeWarps;

// One bitonic merge: (v, i) on lanes 0..15 = current list, lanes 16..31 =
// candidate list reversed; returns with lanes 0..15 = the best 16, sorted.
__device__ __forceinline__ void bitonic_merge32(float& v, int& i, int lane) {
#pragma unroll
  for (int d = 16; d; d >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, d);
    const int oi = __shfl_xor_sync(0xffffffffu, i, d);
    const bool lower = (lane & d) == 0;
    if (lower == ranks_ahead(ov, oi, v, i)) { v = ov; i = oi; }
  }
}

__global__ void __launch_bounds__(kMergeWarps * 32)
    topk_merge_kernel(TopkPartials P, int nstrip, int M, float* topv,
                      int* topi, float* lse) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x;
  __shared__ float s_v[kMergeWarps][kC], s_m[kMergeWarps], s_s[kMergeWarps];
  __shared__ int s_i[kMergeWarps][kC];
  const size_t base = (size_t)m * nstrip;
  const int k = lane < kC ? lane : 31 - lane;  // lanes 16..31: reversed
  float nv[kMaxPerWarp], pm[kMaxPerWarp], ps[kMaxPerWarp];
  int ni[kMaxPerWarp];
#pragma unroll
  for (int j = 0; j < kMaxPerWarp; ++j) {  // every load in flight at once
    const int st = warp + j * kMergeWarps;
    nv[j] = -INFINITY;
    ni[j] = -1;
    pm[j] = -INFINITY;
    ps[j] = 0.f;
    if (st < nstrip) {
      nv[j] = P.v[(base + st) * kC + k];
      ni[j] = P.i[(base + st) * kC + k];
      pm[j] = P.m[base + st];
      ps[j] = P.s[base + st];
    }
  }
  float tv = -INFINITY;
  int ti = -1;
  float rm = -INFINITY, rs = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerWarp; ++j) {
    const int st = warp + j * kMergeWarps;
    if (st >= nstrip) break;
    lse_combine(rm, rs, pm[j], ps[j], 1.f);
    const float bv = __shfl_sync(0xffffffffu, nv[j], 0);
    const int bi = __shfl_sync(0xffffffffu, ni[j], 0);
    if (!ranks_ahead(bv, bi, __shfl_sync(0xffffffffu, tv, kC - 1),
                     __shfl_sync(0xffffffffu, ti, kC - 1)))
      continue;  // nothing in this list enters the top 16
    float v = lane < kC ? tv : nv[j];
    int i = lane < kC ? ti : ni[j];
    bitonic_merge32(v, i, lane);
    tv = v;
    ti = i;
  }
  if (lane < kC) { s_v[warp][lane] = tv; s_i[warp][lane] = ti; }
  if (lane == 0) { s_m[warp] = rm; s_s[warp] = rs; }
  __syncthreads();
  if (warp != 0) return;
  for (int w2 = 1; w2 < kMergeWarps; ++w2) {
    if (lane == 0) lse_combine(rm, rs, s_m[w2], s_s[w2], 1.f);
    const float cv = s_v[w2][k];
    const int ci = s_i[w2][k];
    float v = lane < kC ? tv : cv;
    int i = lane < kC ? ti : ci;
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
                              int* topi, float* lse, cudaStream_t s) {
  topk_merge_kernel<<<M, kMergeWarps * 32, 0, s>>>(P, nstrip, M, topv, topi,
                                                   lse);
  return cudaGetLastError();
}

template cudaError_t launch_lmhead_simt<float>(const float*, const float*,
                                               int, int, int, int,
                                               TopkPartials, cudaStream_t);
template cudaError_t launch_lmhead_simt<__nv_bfloat16>(
    const __nv_bfloat16*, const __nv_bfloat16*, int, int, int, int,
    TopkPartials, cudaStream_t);

}  // namespace dflash
