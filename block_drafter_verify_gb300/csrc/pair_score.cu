// Step a3: context gate and low-rank bilinear pair scores.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): every
// adjacent pair (predecessor a, candidate b) is scored at once as the
// drafter's own logit of b plus a 256-dim embedding match under a context
// gate of h_t — no backbone or LM-head pass.
//
// One launch, no scratch memory: a cluster of 8 CTAs owns 16 rows (b, t).
//   1. gate pre-activations: CTA k of the cluster computes z = W_g h for the
//      16 rows over its eighth of the hidden dimension (W_g staged through
//      shared memory in 64-column panels with 16-byte loads and stores);
//   2. the partial sums are added over the cluster through distributed
//      shared memory, in cluster-rank order, and CTA k keeps the gates
//      g = sigmoid(z) of rows 2k and 2k+1;
//   3. CTA k gathers the 16 predecessor rows of E_in and the 16 candidate
//      rows of E_out (scaled by g) and writes the 16 x 16 scores of each of
//      its two rows.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace dflash {
namespace {

constexpr int kCluster = 8;     // CTAs per cluster (split of the hidden dim)
constexpr int kRows = 16;       // rows (b, t) per cluster
constexpr int kRowsPerCta = kRows / kCluster;
constexpr int kThreads = 256;
constexpr int kPanel = 64;           // W_g columns per staged panel
constexpr int kPanelStride = kPanel + 4;  // 16-byte rows, no bank conflicts

// 16-byte vector of storage elements converted to fp32.
template <typename T>
struct Vec16 {
  static constexpr int N = 16 / sizeof(T);
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f);
};
template <>
__device__ __forceinline__ void Vec16<float>::to_f32(const uint4& u,
                                                     float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void Vec16<__nv_bfloat16>::to_f32(const uint4& u,
                                                             float* f) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <typename T>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    pair_score_kernel(const float* __restrict__ topv,
                      const int* __restrict__ topi,
                      const int* __restrict__ anchor, const T* __restrict__ h,
                      const T* __restrict__ w_gate, const T* __restrict__ e_in,
                      const T* __restrict__ e_out, int B, int K, int H, int V,
                      int r, int hs, float* __restrict__ scores, int* err) {
  constexpr int EPV = Vec16<T>::N;            // elements per 16-byte vector
  constexpr int VPR = kPanel / EPV;           // vectors per panel row
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int M = B * K;
  const int m0 = (blockIdx.x / kCluster) * kRows;
  const int k0 = crank * hs, k1 = min(H, k0 + hs);
  const int klen = max(0, k1 - k0);

  float* part = smem;                           // kRows * 256
  float* hsl = part + kRows * 256;              // kRows * hs
  float* panel = hsl + kRows * hs;              // 256 * kPanelStride
  float* gate = panel + 256 * kPanelStride;     // kRowsPerCta * 256

  // ---- phase 1: partial z[row][k] over this CTA's hidden slice ----------
  {  // h slice of the 16 rows: 16-byte loads, a batch issued before use
    const int vrow = hs / EPV;                 // vectors per row slice
    constexpr int kBatch = 8;                  // loads in flight per thread
    for (int i0 = 0; i0 < kRows * vrow; i0 += kBatch * kThreads) {
      uint4 hv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + tid + u * kThreads;
        const int rr = i / vrow, cv = i % vrow;
        const int m = m0 + rr;
        hv[u] = (rr < kRows && m < M && cv * EPV < klen)
                    ? *reinterpret_cast<const uint4*>(h + (size_t)m * H + k0 +
                                                      cv * EPV)
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + tid + u * kThreads;
        const int rr = i / vrow, cv = i % vrow;
        if (rr < kRows) {
          float f[EPV];
          Vec16<T>::to_f32(hv[u], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) hsl[rr * hs + cv * EPV + e] = f[e];
        }
      }
    }
  }
  float acc[kRows];
#pragma unroll
  for (int rr = 0; rr < kRows; ++rr) acc[rr] = 0.f;
  constexpr int kLoads = 256 * VPR / kThreads;  // 16-byte loads per thread
  for (int p0 = 0; p0 < klen; p0 += kPanel) {
    const int pw = min(kPanel, klen - p0);
    uint4 buf[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = tid + u * kThreads;
      const int g = i / VPR, cv = i % VPR;
      buf[u] = (g < r && cv * EPV < pw)
                   ? *reinterpret_cast<const uint4*>(
                         w_gate + (size_t)g * H + k0 + p0 + cv * EPV)
                   : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();  // previous panel fully consumed
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = tid + u * kThreads;
      const int g = i / VPR, cv = i % VPR;
      float f[EPV];
      Vec16<T>::to_f32(buf[u], f);
      float4* dst = reinterpret_cast<float4*>(panel + g * kPanelStride + cv * EPV);
#pragma unroll
      for (int e = 0; e < EPV / 4; ++e)
        dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
    }
    __syncthreads();
    if (tid < r) {
      // four columns per step: one 16-byte load of W_g, one per row of h
      const float4* wrow = reinterpret_cast<const float4*>(panel + tid * kPanelStride);
      for (int c4 = 0; c4 < pw / 4; ++c4) {
        const float4 w = wrow[c4];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const float4 hv =
              *reinterpret_cast<const float4*>(hsl + rr * hs + p0 + 4 * c4);
          acc[rr] = fmaf(w.x, hv.x, acc[rr]);
          acc[rr] = fmaf(w.y, hv.y, acc[rr]);
          acc[rr] = fmaf(w.z, hv.z, acc[rr]);
          acc[rr] = fmaf(w.w, hv.w, acc[rr]);
        }
      }
    }
  }
  if (tid < r) {
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) part[rr * 256 + tid] = acc[rr];
  }
  cluster.sync();

  // ---- phase 2: add the 8 slices (rank order) for this CTA's two rows ---
  if (tid < r) {
#pragma unroll
    for (int j = 0; j < kRowsPerCta; ++j) {
      const int rr = crank * kRowsPerCta + j;
      float z = 0.f;
      for (int c = 0; c < kCluster; ++c) {
        const float* peer = cluster.map_shared_rank(part, c);
        z += peer[rr * 256 + tid];
      }
      gate[j * 256 + tid] = 1.f / (1.f + __expf(-z));
    }
  }
  cluster.sync();  // peers are done reading this CTA's partials

  for (int j = 0; j < kRowsPerCta; ++j) {
    const int m = m0 + crank * kRowsPerCta + j;
    if (m >= M) break;
    const int b = m / K, t = m % K;
    const float* g_row = gate + j * 256;
    __syncthreads();  // the previous row's tiles are consumed

    // ---- phase 3: 16 x 16 scores of row m ---------------------------------
    __shared__ int s_pred[kC], s_cand[kC];
    if (tid < kC) {
      int cand = topi[(size_t)m * kC + tid];
      int pred = (t == 0) ? anchor[b] : topi[(size_t)(m - 1) * kC + tid];
      if (cand < -1 || cand >= V) { raise_error(err, kErrBadIndex); cand = -1; }
      if (pred < -1 || pred >= V) { raise_error(err, kErrBadIndex); pred = -1; }
      s_cand[tid] = cand;
      s_pred[tid] = pred;
    }
    __syncthreads();
    const int rs = r + 1;  // padded row stride
    float* ein_s = panel;             // [16][rs]
    float* eout_s = panel + kC * rs;  // [16][rs], scaled by the gate
    const int vpr = (r + EPV - 1) / EPV;  // vectors per embedding row
    if (r % EPV == 0) {
      // 2 tables x 16 rows x vpr vectors: every load issued before any use
      constexpr int kMaxE =
          (2 * kC * DFLASH_MAX_RANK / 4 + kThreads - 1) / kThreads;
      uint4 ev[kMaxE];
#pragma unroll
      for (int u = 0; u < kMaxE; ++u) {
        const int i = tid + u * kThreads;
        ev[u] = make_uint4(0, 0, 0, 0);
        if (i < 2 * kC * vpr) {
          const int tab = i / (kC * vpr), rem = i % (kC * vpr);
          const int row = rem / vpr, cv = rem % vpr;
          const int tok = tab == 0 ? s_pred[row] : s_cand[row];
          if (tok >= 0)
            ev[u] = *reinterpret_cast<const uint4*>(
                (tab == 0 ? e_in : e_out) + (size_t)tok * r + cv * EPV);
        }
      }
#pragma unroll
      for (int u = 0; u < kMaxE; ++u) {
        const int i = tid + u * kThreads;
        if (i < 2 * kC * vpr) {
          const int tab = i / (kC * vpr), rem = i % (kC * vpr);
          const int row = rem / vpr, cv = rem % vpr;
          float f[EPV];
          Vec16<T>::to_f32(ev[u], f);
          float* dst = (tab == 0 ? ein_s : eout_s) + row * rs + cv * EPV;
#pragma unroll
          for (int e = 0; e < EPV; ++e)
            dst[e] = tab == 0 ? f[e] : f[e] * g_row[cv * EPV + e];
        }
      }
    } else {
      for (int i = tid; i < kC * r; i += kThreads) {
        const int row = i / r, k = i % r;
        const int a = s_pred[row], c = s_cand[row];
        ein_s[row * rs + k] = a >= 0 ? to_f32(e_in[(size_t)a * r + k]) : 0.f;
        eout_s[row * rs + k] =
            c >= 0 ? to_f32(e_out[(size_t)c * r + k]) * g_row[k] : 0.f;
      }
    }
    __syncthreads();
    const int i = tid / kC, jj = tid % kC;
    float s = 0.f;
    const float* ea = ein_s + i * rs;
    const float* eb = eout_s + jj * rs;
    for (int k = 0; k < r; ++k) s = fmaf(ea[k], eb[k], s);
    const bool valid = s_pred[i] >= 0 && s_cand[jj] >= 0;
    scores[(size_t)m * kC * kC + tid] =
        valid ? topv[(size_t)m * kC + jj] + s : -INFINITY;
  }
}

}  // namespace

template <typename T>
cudaError_t launch_pair_score(const float* topv, const int* topi,
                              const int* anchor, const T* h, const T* w_gate,
                              const T* e_in, const T* e_out, int B, int K,
                              int H, int V, int r, float* scores, int* err,
                              cudaStream_t s) {
  const int M = B * K;
  // hidden slice per cluster rank, a multiple of 8 so 16-byte loads align
  const int hs = ((H + kCluster - 1) / kCluster + 7) & ~7;
  const size_t smem = ((size_t)kRows * 256 + (size_t)kRows * hs +
                       (size_t)256 * kPanelStride + kRowsPerCta * 256) *
                      sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(
      pair_score_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const int clusters = (M + kRows - 1) / kRows;
  pair_score_kernel<T><<<clusters * kCluster, kThreads, smem, s>>>(
      topv, topi, anchor, h, w_gate, e_in, e_out, B, K, H, V, r, hs, scores,
      err);
  return cudaGetLastError();
}

template cudaError_t launch_pair_score<float>(const float*, const int*,
                                              const int*, const float*,
                                              const float*, const float*,
                                              const float*, int, int, int,
                                              int, int, float*, int*,
                                              cudaStream_t);
template cudaError_t launch_pair_score<__nv_bfloat16>(
    const float*, const int*, const int*, const __nv_bfloat16*,
    const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, int,
    int, int, int, int, float*, int*, cudaStream_t);

}  // namespace dflash
