// The step after verify in a draft-verify loop: commit each sequence's
// emitted tokens and hand the last one over as the next cycle's anchor.
//
// "What a block-diffusion drafter is" (A 2B Drafter Made a 27B Model 3.4x
// Faster. Same Exact Output.): the target verifies the whole run and the
// matching prefix is kept; "How many tokens survive": the acceptance
// length is the mean number of draft tokens kept per verification pass.
//
// One warp per sequence: lanes copy the n + 1 emitted tokens, lane 0 moves
// the anchor and the length and adds the sequence to the statistics.
#include "kernels.h"

namespace dflash {

// SM count and device error word of the current device (api.cu).
dflash_status current_device_info(int* sms, int** err);

namespace {

constexpr int kWarpsPerCta = 8;

__global__ void __launch_bounds__(kWarpsPerCta * 32)
    commit_kernel(const int* __restrict__ n_accepted,
                  const int* __restrict__ out_tok, int B, int K,
                  int* __restrict__ anchor, int* __restrict__ tokens,
                  int* __restrict__ length, int capacity,
                  unsigned long long* __restrict__ stats, int* err) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
  if (b >= B) return;
  const int n = n_accepted[b];
  if (n < 0 || n > K) {
    if (lane == 0) raise_error(err, kErrBadIndex);
    return;
  }
  const int len = length[b];
  const int* src = out_tok + (size_t)b * (K + 1);
  if (lane <= n) {
    const long long pos = (long long)len + lane;
    if (pos >= 0 && pos < capacity)
      tokens[(size_t)b * capacity + pos] = src[lane];
    else
      raise_error(err, kErrBadIndex);  // buffer full: the token is dropped
  }
  if (lane == 0) {
    anchor[b] = src[n];
    length[b] = len + n + 1;
    atomicAdd(&stats[0], (unsigned long long)n);
    atomicAdd(&stats[1], 1ull);
    atomicAdd(&stats[2], (unsigned long long)(n + 1));
    atomicAdd(&stats[3 + n], 1ull);
  }
}

}  // namespace
}  // namespace dflash

extern "C" dflash_status dflash_commit(const int32_t* n_accepted,
                                       const int32_t* out_tok, int B, int K,
                                       int32_t* anchor, int32_t* tokens,
                                       int32_t* length, int capacity,
                                       int64_t* stats,
                                       dflash_stream_t stream) {
  using namespace dflash;
  if (!(n_accepted && out_tok && anchor && tokens && length && stats))
    return DFLASH_ERR_INVALID_ARG;
  if (B < 1 || B > (1 << 20) || K < 1 || K > DFLASH_MAX_K || capacity < 1)
    return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(stats) & 7) return DFLASH_ERR_INVALID_ARG;
  int sms = 0;
  int* err = nullptr;
  const dflash_status st = current_device_info(&sms, &err);
  if (st != DFLASH_OK) return st;
  const int blocks = (B + kWarpsPerCta - 1) / kWarpsPerCta;
  commit_kernel<<<blocks, kWarpsPerCta * 32, 0,
                  reinterpret_cast<cudaStream_t>(stream)>>>(
      n_accepted, out_tok, B, K, anchor, tokens, length, capacity,
      reinterpret_cast<unsigned long long*>(stats), err);
  return cudaGetLastError() == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}
