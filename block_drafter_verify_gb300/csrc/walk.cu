// Step a4: the walk through the K x 16 candidate lattice.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): the only
// sequential step; starting from the verified token, greedy follows the best
// successor and sampling draws from the pair scores.
//
// One CTA of 128 threads per sequence.  All four warps stage the
// sequence's K x 16 x 16 scores in shared memory with 16-byte loads (at most
// eight per thread, all in flight at once), then warp 0 walks
// (walk_sequence, walk.cuh): the K dependent steps read on-chip memory only.
#include "kernels.h"
#include "walk.cuh"

namespace dflash {
namespace {

constexpr int kWalkThreads = 128;

__global__ void __launch_bounds__(kWalkThreads)
    path_walk_kernel(const float* __restrict__ scores,
                     const int* __restrict__ topi, int B, int K, float T,
                     float invT, uint64_t seed, uint64_t cycle,
                     int* __restrict__ slot, int* __restrict__ draft,
                     float* __restrict__ q, int* err) {
  extern __shared__ float4 s_scores4[];
  const float* s_scores = reinterpret_cast<const float*>(s_scores4);
  __shared__ int s_topi[DFLASH_MAX_K * kC];
  const int b = blockIdx.x;
  for (int i = threadIdx.x; i < K * kC; i += kWalkThreads)
    s_topi[i] = topi[(size_t)b * K * kC + i];
  const float4* src =
      reinterpret_cast<const float4*>(scores + (size_t)b * K * kC * kC);
  const int n4 = K * kC * kC / 4;  // <= 1024: eight per thread
  float4 st[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = threadIdx.x + u * kWalkThreads;
    if (i < n4) st[u] = src[i];
  }
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = threadIdx.x + u * kWalkThreads;
    if (i < n4) s_scores4[i] = st[u];
  }
  __syncthreads();
  if (threadIdx.x >= 32) return;
  walk_sequence(s_scores, s_topi, b, K, T, invT, seed, cycle, slot, draft, q,
                err);
}

}  // namespace

cudaError_t launch_path_walk(const float* scores, const int* topi, int B,
                             int K, float T, uint64_t seed, uint64_t cycle,
                             int* slot, int* draft, float* q, int* err,
                             cudaStream_t s) {
  const size_t smem = (size_t)K * kC * kC * sizeof(float);
  const float invT = T > 0.f ? 1.f / T : 0.f;
  path_walk_kernel<<<B, kWalkThreads, smem, s>>>(scores, topi, B, K, T, invT,
                                                 seed, cycle, slot, draft, q,
                                                 err);
  return cudaGetLastError();
}

}  // namespace dflash
