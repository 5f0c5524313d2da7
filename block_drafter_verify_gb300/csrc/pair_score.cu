// Step a3: context gate and low-rank bilinear pair scores.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): every
// adjacent pair (predecessor a, candidate b) is scored at once as the
// drafter's own logit of b plus a 256-dim embedding match under a context
// gate of h_t — no backbone or LM-head pass.
//
// One launch, no scratch memory: a cluster of 8 CTAs owns 8 rows (b, t).
//   1. gate pre-activations: CTA k of the cluster computes z = W_g h for the
//      8 rows over its eighth of the hidden dimension (W_g staged through
//      shared memory in coalesced 32-column panels);
//   2. the partial sums are added over the cluster through distributed
//      shared memory, in cluster-rank order, and CTA k keeps row k's gate
//      g = sigmoid(z);
//   3. CTA k gathers the 16 predecessor rows of E_in and the 16 candidate
//      rows of E_out (scaled by g) and writes the 16 x 16 scores of row k.
#include <cooperative_groups.h>

#include "kernels.h"

namespace cg = cooperative_groups;

namespace dflash {
namespace {

constexpr int kCluster = 8;
constexpr int kThreads = 256;
constexpr int kPanel = 32;  // W_g columns per staged panel

struct PairSmem {
  // phase 1-2 (cluster-visible)
  float* part;   // [kCluster rows][256]
  float* hsl;    // [kCluster rows][hs]
  float* panel;  // [256][kPanel + 1]  (reused as E tiles in phase 3)
  float* gate;   // [256]
};

template <typename T>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    pair_score_kernel(const float* __restrict__ topv,
                      const int* __restrict__ topi,
                      const int* __restrict__ anchor, const T* __restrict__ h,
                      const T* __restrict__ w_gate, const T* __restrict__ e_in,
                      const T* __restrict__ e_out, int B, int K, int H, int V,
                      int r, int hs, float* __restrict__ scores, int* err) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int M = B * K;
  const int m0 = (blockIdx.x / kCluster) * kCluster;
  const int k0 = crank * hs, k1 = min(H, k0 + hs);
  const int klen = max(0, k1 - k0);

  float* part = smem;                          // kCluster * 256
  float* hsl = part + kCluster * 256;          // kCluster * hs
  float* panel = hsl + kCluster * hs;          // 256 * (kPanel + 1)
  float* gate = panel + 256 * (kPanel + 1);    // 256

  // ---- phase 1: partial z[row][k] over this CTA's hidden slice ----------
  for (int i = tid; i < kCluster * hs; i += kThreads) {
    const int rr = i / hs, kk = i % hs;
    const int m = m0 + rr;
    hsl[i] = (m < M && kk < klen) ? to_f32(h[(size_t)m * H + k0 + kk]) : 0.f;
  }
  float acc[kCluster];
#pragma unroll
  for (int rr = 0; rr < kCluster; ++rr) acc[rr] = 0.f;
  for (int p0 = 0; p0 < klen; p0 += kPanel) {
    __syncthreads();
    const int pw = min(kPanel, klen - p0);
    for (int i = tid; i < r * kPanel; i += kThreads) {
      const int g = i / kPanel, cc = i % kPanel;
      panel[g * (kPanel + 1) + cc] =
          cc < pw ? to_f32(w_gate[(size_t)g * H + k0 + p0 + cc]) : 0.f;
    }
    __syncthreads();
    if (tid < r) {
      const float* wrow = panel + tid * (kPanel + 1);
      for (int cc = 0; cc < pw; ++cc) {
        const float w = wrow[cc];
#pragma unroll
        for (int rr = 0; rr < kCluster; ++rr)
          acc[rr] = fmaf(w, hsl[rr * hs + p0 + cc], acc[rr]);
      }
    }
  }
  if (tid < r) {
#pragma unroll
    for (int rr = 0; rr < kCluster; ++rr) part[rr * 256 + tid] = acc[rr];
  }
  cluster.sync();

  // ---- phase 2: add the 8 slices (rank order) for row crank -------------
  if (tid < r) {
    float z = 0.f;
    for (int c = 0; c < kCluster; ++c) {
      const float* peer = cluster.map_shared_rank(part, c);
      z += peer[crank * 256 + tid];
    }
    gate[tid] = 1.f / (1.f + __expf(-z));
  }
  cluster.sync();  // peers are done reading this CTA's partials

  const int m = m0 + crank;
  if (m >= M) return;
  const int b = m / K, t = m % K;

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
  for (int i = tid; i < kC * r; i += kThreads) {
    const int row = i / r, k = i % r;
    const int a = s_pred[row], c = s_cand[row];
    ein_s[row * rs + k] = a >= 0 ? to_f32(e_in[(size_t)a * r + k]) : 0.f;
    eout_s[row * rs + k] =
        c >= 0 ? to_f32(e_out[(size_t)c * r + k]) * gate[k] : 0.f;
  }
  __syncthreads();
  const int i = tid / kC, j = tid % kC;
  float s = 0.f;
  const float* ea = ein_s + i * rs;
  const float* eb = eout_s + j * rs;
  for (int k = 0; k < r; ++k) s = fmaf(ea[k], eb[k], s);
  const bool valid = s_pred[i] >= 0 && s_cand[j] >= 0;
  scores[(size_t)m * kC * kC + tid] =
      valid ? topv[(size_t)m * kC + j] + s : -INFINITY;
}

}  // namespace

template <typename T>
cudaError_t launch_pair_score(const float* topv, const int* topi,
                              const int* anchor, const T* h, const T* w_gate,
                              const T* e_in, const T* e_out, int B, int K,
                              int H, int V, int r, float* scores, int* err,
                              cudaStream_t s) {
  const int M = B * K;
  const int hs = (H + kCluster - 1) / kCluster;
  const size_t floats = (size_t)kCluster * 256 + (size_t)kCluster * hs +
                        (size_t)256 * (kPanel + 1) + 256;
  const size_t smem = std::max(floats, (size_t)kCluster * 256 +
                                           (size_t)kCluster * hs +
                                           2 * kC * (DFLASH_MAX_RANK + 1) + 256) *
                      sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(
      pair_score_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const int clusters = (M + kCluster - 1) / kCluster;
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
