// Step a1 on CUDA cores: the two-tap dynamic depthwise convolution.
//
// "Suffix-decay convolution" (DFlash 2: Block diffusion, wearing a drafter's
// coat) and "The two fixes" (A 2B Drafter Made a 27B Model 3.4x Faster):
// each position's representation is mixed with its predecessor's through
// two per-channel taps computed from the position itself,
//   y_t[c] = (W0 h_t)[c] * h_t[c] + (W1 h_t)[c] * h_{t-1}[c],  h_{-1} = 0.
//
// One warp per (row, channel): the lanes split the hidden dimension for the
// two dot products, lane 0 applies the taps and rounds y to the storage
// type.  Used for fp32 storage.
#include "kernels.h"

namespace dflash {
namespace {

constexpr int kThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kThreads)
    conv_simt_kernel(const T* __restrict__ h, const T* __restrict__ w_conv,
                     int B, int K, int H, T* __restrict__ y) {
  const long long gw = (long long)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  const long long M = (long long)B * K;
  if (gw >= M * H) return;
  const int m = (int)(gw / H), c = (int)(gw % H);
  const T* hr = h + (size_t)m * H;
  const T* w0 = w_conv + (size_t)c * H;
  const T* w1 = w_conv + (size_t)(H + c) * H;
  float a0 = 0.f, a1 = 0.f;
  for (int k = lane; k < H; k += 32) {
    const float hv = to_f32(hr[k]);
    a0 = fmaf(to_f32(w0[k]), hv, a0);
    a1 = fmaf(to_f32(w1[k]), hv, a1);
  }
  a0 = warp_sum(a0);
  a1 = warp_sum(a1);
  if (lane == 0) {
    const int t = m % K;
    const float prev = t > 0 ? to_f32(h[(size_t)(m - 1) * H + c]) : 0.f;
    y[(size_t)m * H + c] = from_f32<T>(a0 * to_f32(hr[c]) + a1 * prev);
  }
}

}  // namespace

template <typename T>
cudaError_t launch_conv_simt(const T* h, const T* w_conv, int B, int K, int H,
                             T* y, cudaStream_t s) {
  const long long warps = (long long)B * K * H;
  const long long blocks = (warps + kThreads / 32 - 1) / (kThreads / 32);
  conv_simt_kernel<T><<<(unsigned)blocks, kThreads, 0, s>>>(h, w_conv, B, K,
                                                            H, y);
  return cudaGetLastError();
}

template cudaError_t launch_conv_simt<float>(const float*, const float*, int,
                                             int, int, float*, cudaStream_t);
template cudaError_t launch_conv_simt<__nv_bfloat16>(const __nv_bfloat16*,
                                                     const __nv_bfloat16*, int,
                                                     int, int, __nv_bfloat16*,
                                                     cudaStream_t);

}  // namespace dflash
