// Shared device helpers of the CUDA library: error word bits, element loads,
// warp reductions and the Philox4x32-10 generator.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dflash.h"

namespace dflash {

constexpr int kC = DFLASH_CANDIDATES;  // candidates per position
constexpr int kMaxStrips = 160;        // vocab strips per row in the partials

// Bits of the sticky device error word (see dflash_check).
enum : int {
  kErrNonfinite = 1,
  kErrBadIndex = 2,
  kErrTimeout = 4,
};

__device__ __forceinline__ void raise_error(int* err, int bit) {
  atomicOr(err, bit);
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream serialization attribute may start while the previous kernel on the
// stream is still running; pdl_wait() blocks the calling thread until that
// kernel has completed and its memory is visible, pdl_trigger() lets the
// next such kernel start.  Both are no-ops in a normal launch.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch configuration with programmatic stream serialization (plus an
// optional cluster size).
struct PdlLaunch {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  PdlLaunch(dim3 grid, dim3 block, size_t smem, cudaStream_t s,
            int cluster_x = 0) {
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int n = 1;
    if (cluster_x > 0) {
      attr[1].id = cudaLaunchAttributeClusterDimension;
      attr[1].val.clusterDim.x = cluster_x;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
  }
};

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// (max, sum of exp(x - max)) pairs combined; an empty side has max = -inf.
__device__ __forceinline__ void lse_combine(float& m, float& s, float m2,
                                            float s2, float scale) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; s = s2; return; }
  float mx = fmaxf(m, m2);
  s = s * __expf((m - mx) * scale) + s2 * __expf((m2 - mx) * scale);
  m = mx;
}

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies with the
// key bumped by the Weyl constants between rounds.
struct U32x4 { uint32_t x, y, z, w; };

__device__ __forceinline__ U32x4 philox4x32_10(U32x4 c, uint32_t k0,
                                               uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) { k0 += 0x9E3779B9u; k1 += 0xBB67AE85u; }
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = U32x4{hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0};
  }
  return c;
}

enum : uint32_t { kPurposeWalk = 0, kPurposeAccept = 1, kPurposeResample = 2 };

// 24-bit uniform integer of stream (b, t, purpose, cycle); u = value * 2^-24.
__device__ __forceinline__ uint32_t philox_u24(uint64_t seed, uint32_t b,
                                               uint32_t t, uint32_t purpose,
                                               uint64_t cycle) {
  U32x4 r = philox4x32_10(U32x4{b, t, purpose, (uint32_t)cycle},
                          (uint32_t)seed, (uint32_t)(seed >> 32));
  return r.x >> 8;
}
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint32_t b,
                                                uint32_t t, uint32_t purpose,
                                                uint64_t cycle) {
  return (float)philox_u24(seed, b, t, purpose, cycle) * 0x1p-24f;
}

// Top-16 candidate partials written per (row, vocab strip) by the LM-head
// kernels and folded by the merge kernel.  Layout [row][strip][16] and
// [row][strip]; each list sorted by (value desc, id asc), padded with
// (-inf, -1).
struct TopkPartials {
  float* v;
  int* i;
  float* m;  // running max of the strip (natural-log units)
  float* s;  // sum of exp(x - m) over the strip
};

}  // namespace dflash
