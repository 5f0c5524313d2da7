// Per-row E4M3 quantization of bf16 matrices, for the LM head with 8-bit
// operands: the weight W_lm once when it is loaded, the conv output y every
// cycle.  The pages ship quantized drafter builds ("What a block-diffusion
// drafter is", A 2B Drafter Made a 27B Model 3.4x Faster; "What Comes
// Next", DFlash 2: Keep Drafting Parallel); this library's 8-bit format is
// OCP FP8 E4M3 with one fp32 scale per row.
//
//   scale_i = max_k |x_ik| / 448   (1 for an all-zero row)
//   code_ik = e4m3(x_ik / scale_i), round to nearest even, saturated
//
// Both divisions are correctly rounded fp32 divisions, so the codes are a
// deterministic function of the input.  One CTA of four warps per row;
// rows up to 4096 wide stay in registers between the maximum and the
// conversion, wider rows are read twice (the second time from L1).
#include <cuda_fp8.h>

#include "kernels.h"

namespace dflash {
namespace {

constexpr int kQuantWarps = 4;  // warps per row (one CTA per row)
constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint2 encode8(const float (&f)[8], float s) {
  uint32_t w[2];
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[4 * h2], s), __fdiv_rn(f[4 * h2 + 1], s)),
        __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
        make_float2(__fdiv_rn(f[4 * h2 + 2], s), __fdiv_rn(f[4 * h2 + 3], s)),
        __NV_SATFINITE, __NV_E4M3);
    w[h2] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
  return make_uint2(w[0], w[1]);
}

__device__ __forceinline__ void fold8(const float (&f)[8], float& amax,
                                      bool& bad) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    bad |= !isfinite(f[k]);
    amax = fmaxf(amax, fabsf(f[k]));
  }
}

// One CTA of kQuantWarps warps per row; the row's 8-element chunks are
// dealt to the CTA's threads in turn (chunk i to thread i mod 128).
// kChunks > 0: each thread holds its kChunks chunks in registers (all
// loads in flight at once, no second read); 0: two passes over the row,
// the second from L1.  The row's max |x| is reduced over the warps
// through shared memory; max and the divisions do not depend on the order.
template <int kChunks>
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_e4m3_rows_kernel(const __nv_bfloat16* __restrict__ x, int R,
                              int H, uint8_t* __restrict__ codes,
                              float* __restrict__ scale, int* err) {
  // The next launch may start now: it waits for this grid's completion
  // before it reads the codes.
  pdl_trigger();
  pdl_wait();  // x may be written by the previous launch
  constexpr int kT = kQuantWarps * 32;
  __shared__ float s_amax[kQuantWarps];
  __shared__ int s_bad;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const long long row = blockIdx.x;
  if (row >= R) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + row * H);
  uint2* dst = reinterpret_cast<uint2*>(codes + row * H);
  const int n8 = H / 8;
  float amax = 0.f;
  bool bad = false;
  uint4 v[kChunks > 0 ? kChunks : 1];
  if constexpr (kChunks > 0) {
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      const int i = tid + kT * j;
      v[j] = i < n8 ? src[i] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      float f[8];
      unpack8(v[j], f);
      fold8(f, amax, bad);
    }
  } else {
    for (int i = tid; i < n8; i += kT) {
      float f[8];
      unpack8(src[i], f);
      fold8(f, amax, bad);
    }
  }
  if (tid == 0) s_bad = 0;
#pragma unroll
  for (int o = 16; o; o >>= 1)
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_amax[wid] = amax;
  __syncthreads();
  if (bad) s_bad = 1;
  float m = s_amax[0];
#pragma unroll
  for (int w = 1; w < kQuantWarps; ++w) m = fmaxf(m, s_amax[w]);
  const float s = m > 0.f ? __fdiv_rn(m, kE4m3Max) : 1.f;
  if constexpr (kChunks > 0) {
#pragma unroll
    for (int j = 0; j < kChunks; ++j) {
      const int i = tid + kT * j;
      if (i < n8) {
        float f[8];
        unpack8(v[j], f);
        dst[i] = encode8(f, s);
      }
    }
  } else {
    for (int i = tid; i < n8; i += kT) {
      float f[8];
      unpack8(src[i], f);
      dst[i] = encode8(f, s);
    }
  }
  __syncthreads();
  if (tid == 0) {
    scale[row] = s;
    if (s_bad) raise_error(err, kErrNonfinite);
  }
}

}  // namespace

cudaError_t launch_quantize_e4m3_rows(const __nv_bfloat16* x, int R, int H,
                                      uint8_t* codes, float* scale, int* err,
                                      cudaStream_t s) {
  if (R > 0x7fffffff) return cudaErrorInvalidValue;
  PdlLaunch L(dim3((unsigned)R), dim3(kQuantWarps * 32), 0, s);
  const int n8 = H / 8;
  constexpr int kT = kQuantWarps * 32;
  if (n8 <= kT * 2)
    return cudaLaunchKernelEx(&L.cfg, quantize_e4m3_rows_kernel<2>, x, R, H,
                              codes, scale, err);
  if (n8 <= kT * 4)
    return cudaLaunchKernelEx(&L.cfg, quantize_e4m3_rows_kernel<4>, x, R, H,
                              codes, scale, err);
  return cudaLaunchKernelEx(&L.cfg, quantize_e4m3_rows_kernel<0>, x, R, H,
                            codes, scale, err);
}

}  // namespace dflash
