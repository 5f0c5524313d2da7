// Selector variants and diagnostics beyond the pages' greedy and sampled
// walks ("What Comes Next", DFlash 2: Keep Drafting Parallel: pairwise
// scoring is the simplest selector; an oracle that always picks the right
// candidate among the 16 bounds what selection can gain).
//
//   path_viterbi_kernel   the global max-sum path through the K x 16
//                         lattice: one warp per sequence, lane j < 16 holds
//                         the best total of the paths ending in slot j.
//   top16_recall_kernel   per drafted position: the target's argmax and
//                         whether it is among the 16 candidates.
#include "kernels.h"

namespace dflash {

// SM count and device error word of the current device (api.cu).
dflash_status current_device_info(int* sms, int** err);

namespace {

constexpr int kViterbiWarps = 2;  // 32 KB of staged scores per warp at K = 16

// best_t(j) = max_i best_{t-1}(i) + S[t][i][j], best_0(j) = S[0][0][j] (all
// rows of position 0 are the anchor's); ties keep the lowest i, and the
// final slot is the lowest j of maximal total; fp32 sums.
__global__ void __launch_bounds__(kViterbiWarps * 32)
    path_viterbi_kernel(const float* __restrict__ scores,
                        const int* __restrict__ topi, int B, int K,
                        int* __restrict__ slot, int* __restrict__ draft,
                        float* __restrict__ q, int* err) {
  __shared__ float s_sc[kViterbiWarps][DFLASH_MAX_K * kC * kC];
  __shared__ int s_back[kViterbiWarps][DFLASH_MAX_K][kC];
  __shared__ int s_path[kViterbiWarps][DFLASH_MAX_K];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int b = blockIdx.x * kViterbiWarps + w;
  if (b >= B) return;
  float* sc = s_sc[w];
  const float4* src =
      reinterpret_cast<const float4*>(scores + (size_t)b * K * kC * kC);
  for (int i = lane; i < K * kC * kC / 4; i += 32)
    reinterpret_cast<float4*>(sc)[i] = src[i];
  __syncwarp();
  float best = lane < kC ? sc[lane] : -INFINITY;
  for (int t = 1; t < K; ++t) {
    float nb = -INFINITY;
    int bi = 0;
#pragma unroll
    for (int i = 0; i < kC; ++i) {
      const float bi_v = __shfl_sync(0xffffffffu, best, i);
      const float c = lane < kC ? bi_v + sc[(t * kC + i) * kC + lane]
                                : -INFINITY;
      if (c > nb) { nb = c; bi = i; }
    }
    best = nb;
    if (lane < kC) s_back[w][t][lane] = bi;
  }
  float bv = best;
  int bj = lane;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oj = __shfl_xor_sync(0xffffffffu, bj, o);
    if (ov > bv || (ov == bv && oj < bj)) { bv = ov; bj = oj; }
  }
  __syncwarp();
  if (lane == 0) {
    int j = bj;
    for (int t = K - 1; t >= 0; --t) {
      s_path[w][t] = j;
      if (t > 0) j = s_back[w][t][j];
    }
    if (bv == -INFINITY) raise_error(err, kErrBadIndex);  // no valid path
  }
  __syncwarp();
  for (int t = 0; t < K; ++t) {
    const int j = s_path[w][t];
    if (lane < kC) q[((size_t)b * K + t) * kC + lane] = lane == j ? 1.f : 0.f;
    if (lane == 0) {
      const int tok = topi[((size_t)b * K + t) * kC + j];
      slot[b * K + t] = j;
      draft[b * K + t] = tok;
      if (tok < 0) raise_error(err, kErrBadIndex);
    }
  }
}

constexpr int kRecallThreads = 512;
constexpr int kRecallUnroll = 4;  // float4 loads in flight per thread

// Row (b, t), t < K, of the target logits: first argmax, and membership of
// that token among topi[b, t, :].  Each thread visits its indices in
// increasing order and keeps the first maximum; the reductions prefer the
// lower index on equal values.
__global__ void __launch_bounds__(kRecallThreads)
    top16_recall_kernel(const float* __restrict__ L,
                        const int* __restrict__ topi, int K, int V, int vec4,
                        int* __restrict__ target_argmax,
                        int* __restrict__ in_top16, int* err) {
  const int m = blockIdx.x, b = m / K, t = m % K;
  const float* x = L + ((size_t)b * (K + 1) + t) * V;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  bool bad = false;
  auto take = [&](float e, int v) {
    bad |= (e != e) || e == INFINITY;
    if (e > bv) { bv = e; bi = v; }
  };
  if (vec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    const int n4 = V / 4;
    constexpr int kStride = kRecallThreads * kRecallUnroll;
    for (int base = tid; base < n4; base += kStride) {
      float4 f[kRecallUnroll];
#pragma unroll
      for (int u = 0; u < kRecallUnroll; ++u) {
        const int i = base + u * kRecallThreads;
        f[u] = i < n4 ? __ldcs(x4 + i)
                      : make_float4(-INFINITY, -INFINITY, -INFINITY,
                                    -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kRecallUnroll; ++u) {
        const int v = 4 * (base + u * kRecallThreads);
        take(f[u].x, v);
        take(f[u].y, v + 1);
        take(f[u].z, v + 2);
        take(f[u].w, v + 3);
      }
    }
  } else {
    for (int v = tid; v < V; v += kRecallThreads) take(x[v], v);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
  }
  __shared__ float s_v[kRecallThreads / 32];
  __shared__ int s_i[kRecallThreads / 32];
  if (lane == 0) { s_v[wid] = bv; s_i[wid] = bi; }
  if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(err, kErrNonfinite);
  __syncthreads();
  if (tid != 0) return;
  for (int w2 = 1; w2 < kRecallThreads / 32; ++w2)
    if (s_v[w2] > bv || (s_v[w2] == bv && s_i[w2] < bi)) {
      bv = s_v[w2];
      bi = s_i[w2];
    }
  if (bv == -INFINITY) {  // every logit of the row is -inf
    raise_error(err, kErrNonfinite);
    bi = 0;
  }
  int hit = 0;
  for (int j = 0; j < kC; ++j) hit |= topi[(size_t)m * kC + j] == bi;
  target_argmax[m] = bi;
  in_top16[m] = hit;
}

}  // namespace
}  // namespace dflash

extern "C" dflash_status dflash_path_viterbi(const float* scores,
                                             const int32_t* topi, int B,
                                             int K, int32_t* slot,
                                             int32_t* draft, float* q,
                                             dflash_stream_t stream) {
  using namespace dflash;
  if (!(scores && topi && slot && draft && q)) return DFLASH_ERR_INVALID_ARG;
  if (B < 1 || B > (1 << 20) || K < 1 || K > DFLASH_MAX_K)
    return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(scores) & 15) return DFLASH_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  const dflash_status st = current_device_info(&sms, &err);
  if (st != DFLASH_OK) return st;
  const int blocks = (B + kViterbiWarps - 1) / kViterbiWarps;
  path_viterbi_kernel<<<blocks, kViterbiWarps * 32, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(
      scores, topi, B, K, slot, draft, q, err);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

extern "C" dflash_status dflash_top16_recall(const float* target_logits,
                                             const int32_t* topi, int B,
                                             int K, int V,
                                             int32_t* target_argmax,
                                             int32_t* in_top16,
                                             dflash_stream_t stream) {
  using namespace dflash;
  if (!(target_logits && topi && target_argmax && in_top16))
    return DFLASH_ERR_INVALID_ARG;
  if (B < 1 || K < 1 || K > DFLASH_MAX_K || V < 1 ||
      (long long)B * K > (1 << 20))
    return DFLASH_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  const dflash_status st = current_device_info(&sms, &err);
  if (st != DFLASH_OK) return st;
  const int vec4 = (V % 4 == 0) &&
                   ((reinterpret_cast<uintptr_t>(target_logits) & 15) == 0);
  top16_recall_kernel<<<B * K, kRecallThreads, 0,
                        reinterpret_cast<cudaStream_t>(stream)>>>(
      target_logits, topi, K, V, vec4, target_argmax, in_top16, err);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
