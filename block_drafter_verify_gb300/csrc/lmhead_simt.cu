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
// topk_merge: one CTA per row folds the strips' lists and (max, sum) pairs
// in strip order and writes topv / topi / lse.
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

// One warp per row.  The row's strip lists are staged in shared memory;
// (max, sum) pairs are folded per lane in strip order and then across lanes
// in a fixed tree; the top-16 is a 16-round tournament of the strips' list
// heads (lane l owns strips l, l+32, ...), so the result does not depend on
// timing.
constexpr int kMergeWarps = 4;
constexpr int kMaxOwned = (kMaxStrips + 31) / 32;

__global__ void __launch_bounds__(kMergeWarps * 32)
    topk_merge_kernel(TopkPartials P, int nstrip, int M, float* topv,
                      int* topi, float* lse) {
  extern __shared__ float4 msm4[];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int m = blockIdx.x * kMergeWarps + warp;
  if (m >= M) return;
  float* sv = reinterpret_cast<float*>(msm4) + (size_t)warp * nstrip * kC;
  int* si = reinterpret_cast<int*>(reinterpret_cast<float*>(msm4) +
                                   (size_t)kMergeWarps * nstrip * kC) +
            (size_t)warp * nstrip * kC;
  const size_t base = (size_t)m * nstrip * kC;
  const float4* gv = reinterpret_cast<const float4*>(P.v + base);
  const int4* gi = reinterpret_cast<const int4*>(P.i + base);
#pragma unroll 4
  for (int i = lane; i < nstrip * kC / 4; i += 32) {
    const float4 fv = gv[i];
    const int4 iv = gi[i];
    reinterpret_cast<float4*>(sv)[i] = fv;
    reinterpret_cast<int4*>(si)[i] = iv;
  }
  // logsumexp: per-lane fold in strip order, then a fixed butterfly
  float rm = -INFINITY, rs = 0.f;
  for (int st = lane; st < nstrip; st += 32)
    lse_combine(rm, rs, P.m[(size_t)m * nstrip + st],
                P.s[(size_t)m * nstrip + st], 1.f);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, rm, o);
    const float os = __shfl_xor_sync(0xffffffffu, rs, o);
    if (lane & o) {  // the higher lane folds the lower lane's value first
      float am = om, as = os;
      lse_combine(am, as, rm, rs, 1.f);
      rm = am; rs = as;
    } else {
      lse_combine(rm, rs, om, os, 1.f);
    }
  }
  __syncwarp();
  // tournament over list heads
  int head[kMaxOwned];
#pragma unroll
  for (int j = 0; j < kMaxOwned; ++j) head[j] = 0;
  float outv = -INFINITY;
  int outi = -1;
  for (int r = 0; r < kC; ++r) {
    float bv = -INFINITY;
    int bi = -1, bj = -1;
#pragma unroll
    for (int j = 0; j < kMaxOwned; ++j) {
      const int st = lane + 32 * j;
      if (st < nstrip && head[j] < kC) {
        const float v = sv[st * kC + head[j]];
        const int id = si[st * kC + head[j]];
        if (bj < 0 || ranks_ahead(v, id, bv, bi)) { bv = v; bi = id; bj = j; }
      }
    }
    int bl = lane;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      const int ol = __shfl_xor_sync(0xffffffffu, bl, o);
      const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
      const bool take = (oj >= 0) && (bj < 0 || ranks_ahead(ov, oi, bv, bi) ||
                                      (ov == bv && oi == bi && ol < bl));
      if (take) { bv = ov; bi = oi; bl = ol; bj = oj; }
    }
    if (lane == r) { outv = bv; outi = bi; }
    if (lane == bl && bj >= 0) {
#pragma unroll
      for (int j = 0; j < kMaxOwned; ++j)
        if (j == bj) ++head[j];
    }
  }
  if (lane < kC) {
    topv[(size_t)m * kC + lane] = outv;
    topi[(size_t)m * kC + lane] = outi;
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
  const size_t smem = (size_t)kMergeWarps * nstrip * kC * 8;
  cudaError_t e = cudaFuncSetAttribute(
      topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  topk_merge_kernel<<<(M + kMergeWarps - 1) / kMergeWarps, kMergeWarps * 32,
                      smem, s>>>(P, nstrip, M, topv, topi, lse);
  return cudaGetLastError();
}

template cudaError_t launch_lmhead_simt<float>(const float*, const float*,
                                               int, int, int, int,
                                               TopkPartials, cudaStream_t);
template cudaError_t launch_lmhead_simt<__nv_bfloat16>(
    const __nv_bfloat16*, const __nv_bfloat16*, int, int, int, int,
    TopkPartials, cudaStream_t);

}  // namespace dflash
