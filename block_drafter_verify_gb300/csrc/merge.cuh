// Merge of the per-strip top-16 partials of one row into its top-16 and
// logsumexp ("Sixteen candidates per position", DFlash 2: Block diffusion,
// wearing a drafter's coat): used by topk_merge_kernel and by the draft
// tail kernel.
//
// A group of kMergeWarps warps handles one row.  Warp w prefetches the lists
// of strips w, w+8, ... (all loads in flight at once) and folds each into a
// sorted top-16 held by lanes 0..15 with a bitonic merge: lanes 0..15 hold
// the current list best-first, lanes 16..31 the new list worst-first, and
// five compare-exchange steps (distance 16, 8, 4, 2, 1) sort the 32
// entries.  A list whose best entry does not beat the current 16th is
// skipped.  The group's first warp then merges the eight warp lists in warp
// order; (max, sum) pairs are folded per warp in strip order and then in
// warp order.  The result does not depend on timing.
#pragma once

#include "kernels.h"

namespace dflash {

constexpr int kMergeWarps = 8;
constexpr int kMaxPerWarp = (kMaxStrips + kMergeWarps - 1) / kMergeWarps;

// Order of the top-16: larger value first, lower id on equal values.
__device__ __forceinline__ bool ranks_ahead(float v1, int i1, float v2,
                                            int i2) {
  return v1 > v2 || (v1 == v2 && (unsigned)i1 < (unsigned)i2);
}

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

// Best-first bitonic sort of 32 (value, id) pairs, one per lane: larger
// value first, lower id first among equal values.
__device__ __forceinline__ void warp_sort32(float& v, int& i, int lane) {
#pragma unroll
  for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
    for (int d = size >> 1; d; d >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, v, d);
      const int oi = __shfl_xor_sync(0xffffffffu, i, d);
      const bool best_first = ((lane & size) == 0) || size == 32;
      const bool lower = (lane & d) == 0;
      const bool other_ahead = ranks_ahead(ov, oi, v, i);
      const bool mine_ahead = ranks_ahead(v, i, ov, oi);
      if ((lower == best_first) ? other_ahead : mine_ahead) { v = ov; i = oi; }
    }
  }
}

// Phase 1, warp gw (0..kMergeWarps-1) of the group merging row m: fold the
// strips gw, gw + 8, ... of the row.  Returns the warp's top-16 on lanes
// 0..15 (tv, ti) and its (max, sum exp) pair (rm, rs).
__device__ __forceinline__ void merge_fold_warp(const TopkPartials& P,
                                                int nstrip, int m, int gw,
                                                int lane, float& tv, int& ti,
                                                float& rm, float& rs) {
  const size_t base = (size_t)m * nstrip;
  const int k = lane < kC ? lane : 31 - lane;  // lanes 16..31: reversed
  float nv[kMaxPerWarp], pm[kMaxPerWarp], ps[kMaxPerWarp];
  int ni[kMaxPerWarp];
#pragma unroll
  for (int j = 0; j < kMaxPerWarp; ++j) {  // every load in flight at once
    const int st = gw + j * kMergeWarps;
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
  tv = -INFINITY;
  ti = -1;
  rm = -INFINITY;
  rs = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxPerWarp; ++j) {
    const int st = gw + j * kMergeWarps;
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
}

// Phase 2, the group's first warp: merge warps 1.. of the group (their
// lists and pairs staged as s_v/s_i [kMergeWarps][16], s_m/s_s
// [kMergeWarps]) into its own (tv, ti, rm, rs), in warp order.  rm/rs are
// meaningful on lane 0.
__device__ __forceinline__ void merge_combine(const float (*s_v)[kC],
                                              const int (*s_i)[kC],
                                              const float* s_m,
                                              const float* s_s, int lane,
                                              float& tv, int& ti, float& rm,
                                              float& rs) {
  const int k = lane < kC ? lane : 31 - lane;
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
}

}  // namespace dflash
