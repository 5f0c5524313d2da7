// Step a4: the walk through the K x 16 candidate lattice.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): the only
// sequential step; starting from the verified token, greedy follows the best
// successor and sampling draws from the pair scores.
//
// One warp per sequence.  The sequence's K x 16 x 16 scores are staged in
// shared memory with 16-byte loads first, so the K dependent steps read
// on-chip memory only.  Lane j < 16 owns candidate slot j; argmax, max, the
// exp weights' prefix sum and the draw are warp shuffles and one ballot.
#include "kernels.h"

namespace dflash {
namespace {

__global__ void __launch_bounds__(32)
    path_walk_kernel(const float* __restrict__ scores,
                     const int* __restrict__ topi, int B, int K, float T,
                     float invT, uint64_t seed, uint64_t cycle,
                     int* __restrict__ slot, int* __restrict__ draft,
                     float* __restrict__ q, int* err) {
  extern __shared__ float4 s_scores4[];
  const float* s_scores = reinterpret_cast<const float*>(s_scores4);
  const int b = blockIdx.x, lane = threadIdx.x;
  const float4* src =
      reinterpret_cast<const float4*>(scores + (size_t)b * K * kC * kC);
  for (int i = lane; i < K * kC * kC / 4; i += 32) s_scores4[i] = src[i];
  __syncwarp();

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
      const float u = philox_uniform(seed, b, t, kPurposeWalk, cycle);
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
      const int tok = topi[rowbase + j];
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
  path_walk_kernel<<<B, 32, smem, s>>>(scores, topi, B, K, T, invT, seed,
                                       cycle, slot, draft, q, err);
  return cudaGetLastError();
}

}  // namespace dflash
