// The walk of one sequence through its K x 16 candidate lattice, by one
// warp, from scores and candidate ids already in shared memory.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): the only
// sequential step; starting from the verified token, greedy follows the best
// successor and sampling draws from the pair scores.  Lane j < 16 owns
// candidate slot j; argmax, max, the exp weights' prefix sum and the draw
// are warp shuffles and one ballot.  Lane t draws position t's uniform
// before the walk starts, off the serial chain.
#pragma once

#include "kernels.h"

namespace dflash {

__device__ __forceinline__ void walk_sequence(
    const float* s_scores /* [K][16][16] */, const int* s_topi /* [K][16] */,
    int b, int K, float T, float invT, uint64_t seed, uint64_t cycle,
    int* __restrict__ slot, int* __restrict__ draft, float* __restrict__ q,
    int* err) {
  const int lane = threadIdx.x & 31;
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

}  // namespace dflash
