// Step a4: the walk through the K x 16 candidate lattice.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): the only
// sequential step; starting from the verified token, greedy follows the best
// successor and sampling draws from the pair scores.
//
// One CTA of 128 threads per sequence.  All four warps stage the
// sequence's K x 16 x 16 scores in shared memory with 16-byte loads (at most
// eight per thread, all in flight at once), then warp 0 walks: the K
// dependent steps read on-chip memory only.  Lane j < 16 owns candidate
// slot j; argmax, max, the exp weights' prefix sum and the draw are warp
// shuffles and one ballot.
#include "kernels.h"

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
  const int b = blockIdx.x, lane = threadIdx.x;
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
  // lane t draws position t's uniform up front (off the serial chain)
  const float u_lane = (T > 0.f && lane < K)
                           ? philox_uniform(seed, b, lane, kPurposeWalk, cycle)
                           : 0.f;

  int prev = 0;  // row 0 of position 0 is the anchor's row
  for (int t = 0; t < K; ++t) {
    const int rowbase = (b * K + t) * kC;
    const float v =
        lane < kC ? s_scores[(t * kC + prev) * kC + lane] : -INFINITY;
    int j;
    float qj;
    if (T == 0.f) {
      float bv = v;
      int bi = lane;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      j = bi;
      qj = (lane == j) ? 1.f : 0.f;
    } else {
      const float mx = warp_max(v);
      const float w = (v != -INFINITY) ? __expf((v - mx) * invT) : 0.f;
      float cum = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, cum, o);
        if (lane >= o) cum += n;
      }
      const float tot = __shfl_sync(0xffffffffu, cum, 31);
      const float u = __shfl_sync(0xffffffffu, u_lane, t);
      const float thr = u * tot;
      const unsigned above = __ballot_sync(0xffffffffu, lane < kC && cum > thr);
      const unsigned live = __ballot_sync(0xffffffffu, w > 0.f);
      if (above) j = __ffs(above) - 1;
      else j = live ? 31 - __clz(live) : 0;  // u*tot rounded up to tot
      if (mx == -INFINITY && lane == 0) raise_error(err, kErrBadIndex);
      qj = tot > 0.f ? w / tot : 0.f;
    }
    if (lane < kC) q[rowbase + lane] = qj;
    if (lane == 0) {
      const int tok = s_topi[t * kC + j];
      slot[b * K + t] = j;
      draft[b * K + t] = tok;
      if (tok < 0) raise_error(err, kErrBadIndex);
    }
    prev = j;
  }
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
