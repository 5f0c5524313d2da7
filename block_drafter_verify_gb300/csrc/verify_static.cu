// dflash_verify_noalloc: the verify step for callers that cannot allocate
// device memory.
//
// Some callers of this library cannot call cudaMalloc (or any allocator)
// when they verify: a serving loop whose device memory is carved up and
// owned by another engine's allocator, code that runs inside a region that
// must not allocate (a latency-critical decode loop that forbids allocator
// synchronisation, or a host thread that has no handle on the caller's
// memory pool), or a plain C caller that never links an allocator at all.
// For them this entry point keeps the verify scratch in a fixed-size array
// that the library itself holds in device memory; the caller passes only
// inputs and outputs.
//
// The scratch is a file-scope __device__ array of kStaticScratchBytes
// (4 MiB): every GPU that loads this library holds it until the process
// exits.  Host code cannot use the array's name as a device address (in host
// code it is only a stand-in), so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current, checks
// the result and caches it; every later call on that device reuses it.
// That first call therefore should be made before any stream capture.
//
// Every call uses the same array and the array keeps the last call's
// contents: each call clears the part that must start at zero (the ticket
// counters) on its stream before its kernels run.  Calls whose kernels
// overlap on the GPU (different streams, or different host threads on one
// device) race on the array; serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"

namespace dflash {

// Shared with dflash_verify (api.cu): the argument checks other than the
// scratch memory, and the launch (tickets zeroed, profiling events of the
// verify stage).
bool verify_args_ok(const float* target_logits, const int32_t* draft,
                    const int32_t* topi, const float* q, int B, int K, int V,
                    float T, const int32_t* n_accepted,
                    const int32_t* out_tok);
dflash_status verify_run(const float* target_logits, const int32_t* draft,
                         const int32_t* topi, const float* q, int B, int K,
                         int V, float T, uint64_t seed, uint64_t cycle,
                         int32_t* n_accepted, int32_t* out_tok,
                         const VerifyWs& w, cudaStream_t s, bool zeroed);

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;  // 4 MiB

static __device__ __align__(256) unsigned char
    g_verify_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_verify_scratch on the current device (looked up once).
dflash_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || !p)
      return DFLASH_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DFLASH_OK;
}

}  // namespace
}  // namespace dflash

extern "C" dflash_status dflash_verify_noalloc(
    const float* target_logits, const int32_t* draft, const int32_t* topi,
    const float* q, int B, int K, int V, float T, uint64_t seed,
    uint64_t cycle, int32_t* n_accepted, int32_t* out_tok,
    dflash_stream_t stream) {
  using namespace dflash;
  if (!verify_args_ok(target_logits, draft, topi, q, B, K, V, T, n_accepted,
                      out_tok))
    return DFLASH_ERR_INVALID_ARG;
  // sizes whose scratch does not fit the fixed array are refused
  if (verify_ws_layout(B, K, V, nullptr, nullptr) > kStaticScratchBytes)
    return DFLASH_ERR_UNSUPPORTED;
  void* base = nullptr;
  const dflash_status st = scratch_address(&base);
  if (st != DFLASH_OK) return st;
  VerifyWs w;
  verify_ws_layout(B, K, V, base, &w);
  return verify_run(target_logits, draft, topi, q, B, K, V, T, seed, cycle,
                    n_accepted, out_tok, w,
                    reinterpret_cast<cudaStream_t>(stream), false);
}
