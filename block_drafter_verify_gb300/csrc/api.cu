// The C ABI declared in include/dflash.h: host-side argument checks,
// workspace carving and kernel launches.  Nothing here allocates memory.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "kernels.h"

using namespace dflash;

namespace {

__device__ int g_err_word;  // sticky device error bits (kErr*)

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int* err = nullptr;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_mu;

dflash_status device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return DFLASH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return DFLASH_ERR_CUDA;
    if (major != 10 || minor != 3) return DFLASH_ERR_UNSUPPORTED;  // sm_103a only
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return DFLASH_ERR_CUDA;
    d.err = static_cast<int*>(p);
    d.ready = true;
  }
  *out = &d;
  return DFLASH_OK;
}

// Limit of the tensor-core kernels' bounded waits for later launches
// (dflash_set_wait_limit_ns).
std::atomic<uint64_t> g_wait_ns{kWaitLimitNs};

// Caller-supplied timing events per stage (dflash_profile_stage).
enum Stage { kStConv = 0, kStLmhead, kStMerge, kStPair, kStWalk, kStVerifyRows,
             kStQuant, kNumStages };
cudaEvent_t g_prof[kNumStages][2] = {};

// Inside a stream capture the records become event-record nodes of the
// graph (cudaEventRecordExternal), so that a replay stamps the events.
inline void record_stage_event(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
      cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

struct StageTimer {
  int st;
  cudaStream_t s;
  StageTimer(int stage, cudaStream_t stream) : st(stage), s(stream) {
    if (g_prof[st][0]) record_stage_event(g_prof[st][0], s);
  }
  ~StageTimer() {
    if (g_prof[st][1]) record_stage_event(g_prof[st][1], s);
  }
};

inline bool aligned(const void* p, uintptr_t a) {
  return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}
inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

#define REQUIRE(cond)                                   \
  do {                                                  \
    if (!(cond)) return DFLASH_ERR_INVALID_ARG;         \
  } while (0)

inline dflash_status cuda_status(cudaError_t e) {
  return e == cudaSuccess ? DFLASH_OK : DFLASH_ERR_CUDA;
}

bool sizes_ok(int B, int K, int H, int V) {
  if (B < 1 || K < 1 || K > DFLASH_MAX_K || V < 1 || H < 0) return false;
  const long long M = (long long)B * K;
  return M <= (1 << 20) && (long long)V <= (1LL << 30) &&
         M * (long long)(H > 0 ? H : 1) <= (1LL << 40);
}

// Workspace of dflash_lmhead_topk: y (room for fp32), the per-strip top-16
// partials of every row, then the LM head's shared row bounds
// [B*K, kBoundSlots] fp32.
size_t lmhead_ws_layout(int B, int K, int H, int V, void* base, void** y,
                        TopkPartials* P, float** row_bound = nullptr) {
  (void)V;
  const size_t M = (size_t)B * K;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = align256(off);
    char* r = p ? p + off : nullptr;
    off += bytes;
    return r;
  };
  void* yy = take(M * H * sizeof(float));
  TopkPartials pp;
  pp.v = reinterpret_cast<float*>(take((size_t)kMaxStrips * M * kC * sizeof(float)));
  pp.i = reinterpret_cast<int*>(take((size_t)kMaxStrips * M * kC * sizeof(int)));
  pp.m = reinterpret_cast<float*>(take((size_t)kMaxStrips * M * sizeof(float)));
  pp.s = reinterpret_cast<float*>(take((size_t)kMaxStrips * M * sizeof(float)));
  float* rb = reinterpret_cast<float*>(take(M * kBoundSlots * sizeof(float)));
  if (y) *y = yy;
  if (P) *P = pp;
  if (row_bound) *row_bound = rb;
  return align256(off);
}

// Workspace of dflash_draft: the LM-head workspace, then the gate
// [B*K, DFLASH_MAX_RANK] fp32, one walk ticket per sequence, and every
// row's walk step from each predecessor slot: the chosen slot [B*K, 16]
// int32 and q [B*K, 16, 16] fp32.
size_t draft_ws_layout(int B, int K, int H, int V, void* base, float** gate,
                       unsigned** tickets = nullptr, int** walk_j = nullptr,
                       float** walk_q = nullptr) {
  const size_t M = (size_t)B * K;
  const size_t lm = align256(lmhead_ws_layout(B, K, H, V, nullptr, nullptr,
                                              nullptr));
  const size_t g = align256(M * DFLASH_MAX_RANK * sizeof(float));
  const size_t tk = align256((size_t)B * sizeof(unsigned));
  const size_t wj = align256(M * kC * sizeof(int));
  char* p = static_cast<char*>(base);
  if (gate) *gate = reinterpret_cast<float*>(p + lm);
  if (tickets) *tickets = reinterpret_cast<unsigned*>(p + lm + g);
  if (walk_j) *walk_j = reinterpret_cast<int*>(p + lm + g + tk);
  if (walk_q) *walk_q = reinterpret_cast<float*>(p + lm + g + tk + wj);
  return align256(lm + g + tk + wj + M * kC * kC * sizeof(float));
}

// Workspace of dflash_draft_e4m3: dflash_draft's, then the E4M3 codes of y
// [B*K, H] and their row scales [B*K] fp32.
size_t draft_e4m3_ws_layout(int B, int K, int H, int V, void* base,
                            uint8_t** y_codes, float** y_scale) {
  const size_t d = align256(draft_ws_layout(B, K, H, V, nullptr, nullptr));
  const size_t c = align256((size_t)B * K * H);
  char* p = static_cast<char*>(base);
  if (y_codes) *y_codes = reinterpret_cast<uint8_t*>(p + d);
  if (y_scale) *y_scale = reinterpret_cast<float*>(p + d + c);
  return align256(d + c + (size_t)B * K * sizeof(float));
}

// 8-bit LM-head operands for lmhead_tc_path: W_lm as E4M3 codes and row
// scales, and where to put y's codes and scales.
struct E4m3Head {
  const uint8_t* w_codes;
  const float* w_scale;
  uint8_t* y_codes;
  float* y_scale;
};

// bf16 storage: conv and LM head on the tensor cores (tcgen05 + TMA).  With
// w_gate (and conv_w) the conv launch also writes the pair selector's gate
// [B*K, r] fp32 to `gate`.  With q8 (and conv_w) y is quantized per row to
// E4M3 and the LM head runs on the 8-bit operands (w_lm unused).
dflash_status lmhead_tc_path(const __nv_bfloat16* h,
                            const __nv_bfloat16* conv_w,
                            const __nv_bfloat16* w_lm, int B, int K, int H,
                            int V, float* topv, int* topi, float* lse,
                            void* ws, const DeviceState& d, cudaStream_t s,
                            const __nv_bfloat16* w_gate = nullptr, int r = 0,
                            float* gate = nullptr,
                            unsigned* tickets = nullptr,
                            TopkPartials* P_out = nullptr,
                            int* strips_out = nullptr,
                            const E4m3Head* q8 = nullptr,
                            unsigned* vz = nullptr, int nvz = 0) {
  void* yv = nullptr;
  TopkPartials P;
  float* row_bound = nullptr;
  lmhead_ws_layout(B, K, H, V, ws, &yv, &P, &row_bound);
  const int M = B * K;
  const __nv_bfloat16* a = h;
  cudaError_t e;
  // the conv launch resets the LM head's shared row bounds; without a conv
  // the LM head runs without them
  if (!conv_w) row_bound = nullptr;
  if (conv_w) {
    CUtensorMap mh, mw, mg;
    if (!make_tmap_bf16_2d(&mh, h, H, M, 64, 128) ||
        !make_tmap_bf16_2d(&mw, conv_w, H, 2 * (uint64_t)H, 64,
                           conv_tc_bc(M, H)))
      return DFLASH_ERR_CUDA;
    if (w_gate &&
        !make_tmap_bf16_2d(&mg, w_gate, H, r, 64, conv_tc_bc(M, H)))
      return DFLASH_ERR_CUDA;
    __nv_bfloat16* y = static_cast<__nv_bfloat16*>(yv);
    {
      StageTimer tm(kStConv, s);
      e = launch_conv_tc(mh, mw, w_gate ? &mg : nullptr, h, B, K, H, r, y,
                         gate, tickets, row_bound, M * kBoundSlots, d.err, s,
                         g_wait_ns.load(), vz, nvz);
    }
    if (e != cudaSuccess) return DFLASH_ERR_CUDA;
    a = y;
  }
  CUtensorMap my, mw;
  const uint32_t w_box = lmhead_tc_pairs(M) ? 128 : 256;
  if (q8 && conv_w) {
    {
      StageTimer tm(kStQuant, s);
      e = launch_quantize_e4m3_rows(a, M, H, q8->y_codes, q8->y_scale, d.err,
                                    s);
    }
    if (e != cudaSuccess) return DFLASH_ERR_CUDA;
    if (!make_tmap_u8_2d(&my, q8->y_codes, H, M, 128, 128) ||
        !make_tmap_u8_2d(&mw, q8->w_codes, H, V, 128, w_box))
      return DFLASH_ERR_CUDA;
  } else if (!make_tmap_bf16_2d(&my, a, H, M, 64, 128) ||
             !make_tmap_bf16_2d(&mw, w_lm, H, V, 64, w_box)) {
    return DFLASH_ERR_CUDA;
  }
  int strips = 0;
  {
    StageTimer tm(kStLmhead, s);
    e = launch_lmhead_tc(my, mw, M, H, V, d.sms, P, d.err, &strips, s,
                         q8 && conv_w ? q8->y_scale : nullptr,
                         q8 && conv_w ? q8->w_scale : nullptr, row_bound,
                         g_wait_ns.load());
  }
  if (e != cudaSuccess) return DFLASH_ERR_CUDA;
  if (P_out) {  // the caller merges (draft tail)
    *P_out = P;
    *strips_out = strips;
    return DFLASH_OK;
  }
  StageTimer tm(kStMerge, s);
  return cuda_status(launch_topk_merge(P, strips, M, topv, topi, lse, s));
}

// fp32 storage: exact fp32 products on the CUDA cores.
template <typename T>
dflash_status lmhead_impl(const T* h, const T* conv_w, const T* w_lm, int B,
                          int K, int H, int V, float* topv, int* topi,
                          float* lse, void* ws, const DeviceState& d,
                          cudaStream_t s, TopkPartials* P_out = nullptr,
                          int* strips_out = nullptr) {
  void* yv = nullptr;
  TopkPartials P;
  lmhead_ws_layout(B, K, H, V, ws, &yv, &P);
  const int M = B * K;
  const T* a = h;
  cudaError_t e;
  if (conv_w) {
    T* y = static_cast<T*>(yv);
    {
      StageTimer tm(kStConv, s);
      e = launch_conv_simt<T>(h, conv_w, B, K, H, y, s);
    }
    if (e != cudaSuccess) return DFLASH_ERR_CUDA;
    a = y;
  }
  const int ns = lmhead_simt_strips(M, V, d.sms);
  {
    StageTimer tm(kStLmhead, s);
    e = launch_lmhead_simt<T>(a, w_lm, M, H, V, ns, P, s);
  }
  if (e != cudaSuccess) return DFLASH_ERR_CUDA;
  if (P_out) {  // the caller merges
    *P_out = P;
    *strips_out = ns;
    return DFLASH_OK;
  }
  StageTimer tm(kStMerge, s);
  return cuda_status(launch_topk_merge(P, ns, M, topv, topi, lse, s));
}

}  // namespace

namespace dflash {
// SM count and device error word of the current device, for entry points
// defined in other files.
dflash_status current_device_info(int* sms, int** err) {
  DeviceState* d = nullptr;
  const dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  *sms = d->sms;
  *err = d->err;
  return DFLASH_OK;
}

// The checks dflash_verify and dflash_verify_noalloc share (everything but
// the scratch memory): pointers, sizes, temperature, alignment.
bool verify_args_ok(const float* target_logits, const int32_t* draft,
                    const int32_t* topi, const float* q, int B, int K, int V,
                    float T, const int32_t* n_accepted,
                    const int32_t* out_tok) {
  return target_logits && draft && topi && q && n_accepted && out_tok &&
         sizes_ok(B, K, 0, V) && T >= 0.f && T < INFINITY &&
         aligned(target_logits, 16);
}

// Zero the tickets of workspace w (unless an earlier launch of the same
// call did: zeroed), then launch the verify kernel on the current device,
// inside the verify stage's profiling events.
dflash_status verify_run(const float* target_logits, const int32_t* draft,
                         const int32_t* topi, const float* q, int B, int K,
                         int V, float T, uint64_t seed, uint64_t cycle,
                         int32_t* n_accepted, int32_t* out_tok,
                         const VerifyWs& w, cudaStream_t s, bool zeroed) {
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  if (!zeroed &&
      cudaMemsetAsync(w.counters, 0, w.counter_bytes, s) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  StageTimer tm(kStVerifyRows, s);
  return cuda_status(launch_verify(target_logits, draft, topi, q, B, K, V, T,
                                   seed, cycle, n_accepted, out_tok, w, d->sms,
                                   d->err, s));
}
}  // namespace dflash

extern "C" {

size_t dflash_workspace_bytes(int which, int B, int K, int H, int V) {
  if (!sizes_ok(B, K, which == 0 ? H : 0, V)) return 0;
  if (which == 0) {
    if (H < 8) return 0;
    return lmhead_ws_layout(B, K, H, V, nullptr, nullptr, nullptr);
  }
  if (which == 1) return verify_ws_layout(B, K, V, nullptr, nullptr);
  if (which == 2) {
    if (H < 8) return 0;
    return draft_ws_layout(B, K, H, V, nullptr, nullptr);
  }
  if (which == 3) {
    if (H < 16) return 0;
    return draft_e4m3_ws_layout(B, K, H, V, nullptr, nullptr, nullptr);
  }
  return 0;
}

dflash_status dflash_quantize_e4m3_rows(const void* x, int R, int H,
                                        uint8_t* codes, float* scale,
                                        dflash_stream_t stream) {
  REQUIRE(x && codes && scale);
  REQUIRE(R >= 1 && H >= 16 && H % 16 == 0 &&
          (long long)R * H <= (1LL << 40));
  REQUIRE(aligned(x, 16) && aligned(codes, 16) && aligned(scale, 4));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  return cuda_status(launch_quantize_e4m3_rows(
      static_cast<const __nv_bfloat16*>(x), R, H, codes, scale, d->err,
      reinterpret_cast<cudaStream_t>(stream)));
}

dflash_status dflash_lmhead_topk(const void* h, const void* conv_w,
                                 const void* w_lm, int B, int K, int H, int V,
                                 dflash_dtype dt, float* topv, int32_t* topi,
                                 float* lse, void* ws, size_t ws_bytes,
                                 dflash_stream_t stream) {
  REQUIRE(h && w_lm && topv && topi && lse && ws);
  REQUIRE(sizes_ok(B, K, H, V) && H >= 8 && H % 8 == 0);
  REQUIRE(dt == DFLASH_BF16 || dt == DFLASH_FP32);
  REQUIRE(aligned(ws, 256) && aligned(h, 16) && aligned(w_lm, 16));
  REQUIRE(!conv_w || aligned(conv_w, 16));
  REQUIRE(ws_bytes >= lmhead_ws_layout(B, K, H, V, nullptr, nullptr, nullptr));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == DFLASH_FP32)
    return lmhead_impl<float>(static_cast<const float*>(h),
                              static_cast<const float*>(conv_w),
                              static_cast<const float*>(w_lm), B, K, H, V,
                              topv, topi, lse, ws, *d, s);
  return lmhead_tc_path(static_cast<const __nv_bfloat16*>(h),
                        static_cast<const __nv_bfloat16*>(conv_w),
                        static_cast<const __nv_bfloat16*>(w_lm), B, K, H, V,
                        topv, topi, lse, ws, *d, s);
}

dflash_status dflash_pair_score(const float* topv, const int32_t* topi,
                                const int32_t* anchor, const void* h,
                                const void* w_gate, const void* e_in,
                                const void* e_out, int B, int K, int H, int V,
                                int r, dflash_dtype dt, float* scores,
                                dflash_stream_t stream) {
  REQUIRE(topv && topi && anchor && h && w_gate && e_in && e_out && scores);
  REQUIRE(sizes_ok(B, K, H, V) && H >= 8 && H % 8 == 0 && r >= 1 &&
          r <= DFLASH_MAX_RANK);
  REQUIRE(dt == DFLASH_BF16 || dt == DFLASH_FP32);
  REQUIRE(aligned(h, 16) && aligned(w_gate, 16) && aligned(e_in, 16) &&
          aligned(e_out, 16));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  StageTimer tm(kStPair, s);
  if (dt == DFLASH_FP32)
    e = launch_pair_score<float>(topv, topi, anchor,
                                 static_cast<const float*>(h),
                                 static_cast<const float*>(w_gate),
                                 static_cast<const float*>(e_in),
                                 static_cast<const float*>(e_out), B, K, H, V,
                                 r, scores, d->err, s);
  else
    e = launch_pair_score<__nv_bfloat16>(
        topv, topi, anchor, static_cast<const __nv_bfloat16*>(h),
        static_cast<const __nv_bfloat16*>(w_gate),
        static_cast<const __nv_bfloat16*>(e_in),
        static_cast<const __nv_bfloat16*>(e_out), B, K, H, V, r, scores,
        d->err, s);
  return cuda_status(e);
}

dflash_status dflash_path_walk(const float* scores, const int32_t* topi,
                               int B, int K, float T, uint64_t seed,
                               uint64_t cycle, int32_t* slot, int32_t* draft,
                               float* q, dflash_stream_t stream) {
  REQUIRE(scores && topi && slot && draft && q);
  REQUIRE(B >= 1 && K >= 1 && K <= DFLASH_MAX_K && B <= (1 << 20));
  REQUIRE(T >= 0.f && T < INFINITY);
  REQUIRE(aligned(scores, 16));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StageTimer tm(kStWalk, s);
  return cuda_status(launch_path_walk(scores, topi, B, K, T, seed, cycle,
                                      slot, draft, q, d->err, s));
}

}  // extern "C"

namespace dflash {
namespace {

// Steps a1-a4 on the tensor cores (bf16 storage with a conv; q8: the
// 8-bit LM head): the gate rides along with the conv, which also zeroes the
// walk tickets (and vz, nvz words: the cycle's verify tickets); one launch
// after the LM head merges its partials, scores the pairs and walks each
// sequence.
dflash_status draft_tc(const void* h, const void* conv_w, const void* w_lm,
                       const E4m3Head* q8, const void* w_gate,
                       const void* e_in, const void* e_out,
                       const int32_t* anchor, int B, int K, int H, int V,
                       int r, float T, uint64_t seed, uint64_t cycle,
                       float* topv, int32_t* topi, float* lse, float* scores,
                       int32_t* slot, int32_t* draft, float* q, void* ws,
                       const DeviceState& d, cudaStream_t s, unsigned* vz,
                       int nvz) {
  using bf = __nv_bfloat16;
  float* gate = nullptr;
  unsigned* tickets = nullptr;
  int* walk_j = nullptr;
  float* walk_q = nullptr;
  draft_ws_layout(B, K, H, V, ws, &gate, &tickets, &walk_j, &walk_q);
  TopkPartials P;
  int strips = 0;
  const dflash_status st = lmhead_tc_path(
      static_cast<const bf*>(h), static_cast<const bf*>(conv_w),
      static_cast<const bf*>(w_lm), B, K, H, V, topv, topi, lse, ws, d, s,
      static_cast<const bf*>(w_gate), r, gate, tickets, &P, &strips, q8, vz,
      nvz);
  if (st != DFLASH_OK) return st;
  StageTimer tm(kStPair, s);
  return cuda_status(launch_draft_tail<bf>(
      P, strips, anchor, gate, static_cast<const bf*>(e_in),
      static_cast<const bf*>(e_out), B, K, V, r, T, seed, cycle, topv, topi,
      lse, scores, slot, draft, q, tickets, walk_j, walk_q, d.err, s));
}

// dflash_draft; with vz (nvz words) the tensor-core path also zeroes them
// and sets *zeroed.
dflash_status draft_call(const void* h, const void* conv_w, const void* w_lm,
                         const void* w_gate, const void* e_in,
                         const void* e_out, const int32_t* anchor, int B,
                         int K, int H, int V, int r, dflash_dtype dt, float T,
                         uint64_t seed, uint64_t cycle, float* topv,
                         int32_t* topi, float* lse, float* scores,
                         int32_t* slot, int32_t* draft, float* q, void* ws,
                         size_t ws_bytes, dflash_stream_t stream,
                         unsigned* vz, int nvz, bool* zeroed) {
  REQUIRE(h && w_lm && w_gate && e_in && e_out && anchor && topv && topi &&
          lse && scores && slot && draft && q && ws);
  REQUIRE(sizes_ok(B, K, H, V) && H >= 8 && H % 8 == 0 && r >= 1 &&
          r <= DFLASH_MAX_RANK);
  REQUIRE(dt == DFLASH_BF16 || dt == DFLASH_FP32);
  REQUIRE(T >= 0.f && T < INFINITY);
  REQUIRE(aligned(ws, 256) && aligned(h, 16) && aligned(w_lm, 16) &&
          aligned(w_gate, 16) && aligned(e_in, 16) && aligned(e_out, 16) &&
          aligned(scores, 16));
  REQUIRE(!conv_w || aligned(conv_w, 16));
  REQUIRE(ws_bytes >= draft_ws_layout(B, K, H, V, nullptr, nullptr));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dt == DFLASH_BF16 && conv_w) {
    if (zeroed) *zeroed = vz != nullptr;
    return draft_tc(h, conv_w, w_lm, nullptr, w_gate, e_in, e_out, anchor, B,
                    K, H, V, r, T, seed, cycle, topv, topi, lse, scores, slot,
                    draft, q, ws, *d, s, vz, nvz);
  }
  if (zeroed) *zeroed = false;
  st = dflash_lmhead_topk(h, conv_w, w_lm, B, K, H, V, dt, topv, topi, lse,
                          ws, ws_bytes, stream);
  if (st != DFLASH_OK) return st;
  st = dflash_pair_score(topv, topi, anchor, h, w_gate, e_in, e_out, B, K, H,
                         V, r, dt, scores, stream);
  if (st != DFLASH_OK) return st;
  return dflash_path_walk(scores, topi, B, K, T, seed, cycle, slot, draft, q,
                          stream);
}

// dflash_draft_e4m3; with vz (nvz words) the conv launch also zeroes them.
dflash_status draft_e4m3_call(
    const void* h, const void* conv_w, const uint8_t* w_lm_codes,
    const float* w_lm_scale, const void* w_gate, const void* e_in,
    const void* e_out, const int32_t* anchor, int B, int K, int H, int V,
    int r, float T, uint64_t seed, uint64_t cycle, float* topv,
    int32_t* topi, float* lse, float* scores, int32_t* slot, int32_t* draft,
    float* q, void* ws, size_t ws_bytes, dflash_stream_t stream,
    unsigned* vz, int nvz) {
  REQUIRE(h && conv_w && w_lm_codes && w_lm_scale && w_gate && e_in &&
          e_out && anchor && topv && topi && lse && scores && slot && draft &&
          q && ws);
  REQUIRE(sizes_ok(B, K, H, V) && H >= 16 && H % 16 == 0 && r >= 1 &&
          r <= DFLASH_MAX_RANK);
  REQUIRE(T >= 0.f && T < INFINITY);
  REQUIRE(aligned(ws, 256) && aligned(h, 16) && aligned(conv_w, 16) &&
          aligned(w_lm_codes, 16) && aligned(w_lm_scale, 4) &&
          aligned(w_gate, 16) && aligned(e_in, 16) && aligned(e_out, 16) &&
          aligned(scores, 16));
  REQUIRE(ws_bytes >=
          draft_e4m3_ws_layout(B, K, H, V, nullptr, nullptr, nullptr));
  DeviceState* d = nullptr;
  const dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  E4m3Head q8{w_lm_codes, w_lm_scale, nullptr, nullptr};
  draft_e4m3_ws_layout(B, K, H, V, ws, &q8.y_codes, &q8.y_scale);
  return draft_tc(h, conv_w, nullptr, &q8, w_gate, e_in, e_out, anchor, B, K,
                  H, V, r, T, seed, cycle, topv, topi, lse, scores, slot,
                  draft, q, ws, *d, reinterpret_cast<cudaStream_t>(stream),
                  vz, nvz);
}

}  // namespace
}  // namespace dflash

extern "C" {

dflash_status dflash_draft(const void* h, const void* conv_w, const void* w_lm,
                           const void* w_gate, const void* e_in,
                           const void* e_out, const int32_t* anchor, int B,
                           int K, int H, int V, int r, dflash_dtype dt,
                           float T, uint64_t seed, uint64_t cycle, float* topv,
                           int32_t* topi, float* lse, float* scores,
                           int32_t* slot, int32_t* draft, float* q, void* ws,
                           size_t ws_bytes, dflash_stream_t stream) {
  return draft_call(h, conv_w, w_lm, w_gate, e_in, e_out, anchor, B, K, H, V,
                    r, dt, T, seed, cycle, topv, topi, lse, scores, slot,
                    draft, q, ws, ws_bytes, stream, nullptr, 0, nullptr);
}

dflash_status dflash_draft_e4m3(
    const void* h, const void* conv_w, const uint8_t* w_lm_codes,
    const float* w_lm_scale, const void* w_gate, const void* e_in,
    const void* e_out, const int32_t* anchor, int B, int K, int H, int V,
    int r, float T, uint64_t seed, uint64_t cycle, float* topv,
    int32_t* topi, float* lse, float* scores, int32_t* slot, int32_t* draft,
    float* q, void* ws, size_t ws_bytes, dflash_stream_t stream) {
  return draft_e4m3_call(h, conv_w, w_lm_codes, w_lm_scale, w_gate, e_in,
                         e_out, anchor, B, K, H, V, r, T, seed, cycle, topv,
                         topi, lse, scores, slot, draft, q, ws, ws_bytes,
                         stream, nullptr, 0);
}

dflash_status dflash_cycle(
    const void* h, const void* conv_w, const void* w_lm,
    const float* w_lm_scale, const void* w_gate, const void* e_in,
    const void* e_out, const int32_t* anchor, const float* target_logits,
    int B, int K, int H, int V, int r, dflash_dtype dt, float T,
    uint64_t seed, uint64_t cycle, float* topv, int32_t* topi, float* lse,
    float* scores, int32_t* slot, int32_t* draft, float* q,
    int32_t* n_accepted, int32_t* out_tok, void* ws_draft,
    size_t ws_draft_bytes, void* ws_verify, size_t ws_verify_bytes,
    dflash_stream_t stream) {
  REQUIRE(verify_args_ok(target_logits, draft, topi, q, B, K, V, T,
                         n_accepted, out_tok));
  REQUIRE(ws_verify && aligned(ws_verify, 256));
  REQUIRE(ws_verify_bytes >= verify_ws_layout(B, K, V, nullptr, nullptr));
  REQUIRE(!w_lm_scale || dt == DFLASH_BF16);
  VerifyWs w;
  verify_ws_layout(B, K, V, ws_verify, &w);
  const int nvz = (int)(w.counter_bytes / sizeof(unsigned));
  bool zeroed = true;
  dflash_status st =
      w_lm_scale
          ? draft_e4m3_call(h, conv_w, static_cast<const uint8_t*>(w_lm),
                            w_lm_scale, w_gate, e_in, e_out, anchor, B, K, H,
                            V, r, T, seed, cycle, topv, topi, lse, scores,
                            slot, draft, q, ws_draft, ws_draft_bytes, stream,
                            w.counters, nvz)
          : draft_call(h, conv_w, w_lm, w_gate, e_in, e_out, anchor, B, K, H,
                       V, r, dt, T, seed, cycle, topv, topi, lse, scores,
                       slot, draft, q, ws_draft, ws_draft_bytes, stream,
                       w.counters, nvz, &zeroed);
  if (st != DFLASH_OK) return st;
  return verify_run(target_logits, draft, topi, q, B, K, V, T, seed, cycle,
                    n_accepted, out_tok, w,
                    reinterpret_cast<cudaStream_t>(stream), zeroed);
}

dflash_status dflash_verify(const float* target_logits, const int32_t* draft,
                            const int32_t* topi, const float* q, int B, int K,
                            int V, float T, uint64_t seed, uint64_t cycle,
                            int32_t* n_accepted, int32_t* out_tok, void* ws,
                            size_t ws_bytes, dflash_stream_t stream) {
  REQUIRE(verify_args_ok(target_logits, draft, topi, q, B, K, V, T,
                         n_accepted, out_tok));
  REQUIRE(ws && aligned(ws, 256));
  REQUIRE(ws_bytes >= verify_ws_layout(B, K, V, nullptr, nullptr));
  VerifyWs w;
  verify_ws_layout(B, K, V, ws, &w);
  return verify_run(target_logits, draft, topi, q, B, K, V, T, seed, cycle,
                    n_accepted, out_tok, w,
                    reinterpret_cast<cudaStream_t>(stream), false);
}

dflash_status dflash_lmhead_topk_shard(const void* h, const void* conv_w,
                                       const void* w_lm_shard, int B, int K,
                                       int H, int V_shard, int v0,
                                       dflash_dtype dt, float* part_v,
                                       int32_t* part_i, float* part_m,
                                       float* part_s, void* ws,
                                       size_t ws_bytes,
                                       dflash_stream_t stream) {
  REQUIRE(h && w_lm_shard && part_v && part_i && part_m && part_s && ws);
  REQUIRE(sizes_ok(B, K, H, V_shard) && H >= 8 && H % 8 == 0);
  REQUIRE(v0 >= 0 && (long long)v0 + V_shard <= (1LL << 30));
  REQUIRE(dt == DFLASH_BF16 || dt == DFLASH_FP32);
  REQUIRE(aligned(ws, 256) && aligned(h, 16) && aligned(w_lm_shard, 16));
  REQUIRE(!conv_w || aligned(conv_w, 16));
  REQUIRE(ws_bytes >=
          lmhead_ws_layout(B, K, H, V_shard, nullptr, nullptr, nullptr));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TopkPartials P;
  int strips = 0;
  if (dt == DFLASH_FP32)
    st = lmhead_impl<float>(static_cast<const float*>(h),
                            static_cast<const float*>(conv_w),
                            static_cast<const float*>(w_lm_shard), B, K, H,
                            V_shard, nullptr, nullptr, nullptr, ws, *d, s, &P,
                            &strips);
  else
    st = lmhead_tc_path(static_cast<const __nv_bfloat16*>(h),
                        static_cast<const __nv_bfloat16*>(conv_w),
                        static_cast<const __nv_bfloat16*>(w_lm_shard), B, K,
                        H, V_shard, nullptr, nullptr, nullptr, ws, *d, s,
                        nullptr, 0, nullptr, nullptr, &P, &strips);
  if (st != DFLASH_OK) return st;
  StageTimer tm(kStMerge, s);
  return cuda_status(launch_topk_merge(P, strips, B * K, part_v, part_i,
                                       nullptr, s, v0, part_m, part_s));
}

dflash_status dflash_topk_merge_shards(const float* part_v,
                                       const int32_t* part_i,
                                       const float* part_m,
                                       const float* part_s, int S, int M,
                                       float* topv, int32_t* topi, float* lse,
                                       dflash_stream_t stream) {
  REQUIRE(part_v && part_i && part_m && part_s && topv && topi && lse);
  REQUIRE(S >= 1 && S <= DFLASH_MAX_SHARDS && M >= 1 && M <= (1 << 20));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  StageTimer tm(kStMerge, s);
  return cuda_status(launch_shard_merge(part_v, part_i, part_m, part_s, S, M,
                                        topv, topi, lse, s));
}

dflash_status dflash_verify_shard_stats(const float* target_shard,
                                        const int32_t* draft,
                                        const int32_t* topi, int B, int K,
                                        int V_shard, int v0, int V, float T,
                                        float* stats, void* ws,
                                        size_t ws_bytes,
                                        dflash_stream_t stream) {
  REQUIRE(target_shard && draft && topi && stats && ws);
  REQUIRE(sizes_ok(B, K, 0, V_shard) && sizes_ok(B, K, 0, V));
  REQUIRE(v0 >= 0 && (long long)v0 + V_shard <= V);
  REQUIRE(T >= 0.f && T < INFINITY);
  REQUIRE(aligned(ws, 256) && aligned(target_shard, 16) && aligned(stats, 4));
  REQUIRE(ws_bytes >= verify_ws_layout(B, K, V_shard, nullptr, nullptr));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  VerifyWs w;
  verify_ws_layout(B, K, V_shard, ws, &w);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(w.counters, 0, w.counter_bytes, s) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  StageTimer tm(kStVerifyRows, s);
  return cuda_status(launch_verify(target_shard, draft, topi, nullptr, B, K,
                                   V_shard, T, 0, 0, nullptr, nullptr, w,
                                   d->sms, d->err, s, v0, stats));
}

dflash_status dflash_verify_shard_decide(
    const float* stats, int S, const int32_t* draft, const int32_t* topi,
    const float* q, int B, int K, int V, float T, uint64_t seed,
    uint64_t cycle, int32_t* n_accepted, int32_t* out_tok, float* plan,
    dflash_stream_t stream) {
  REQUIRE(stats && draft && topi && q && n_accepted && out_tok && plan);
  REQUIRE(S >= 1 && S <= DFLASH_MAX_SHARDS && sizes_ok(B, K, 0, V));
  REQUIRE(T >= 0.f && T < INFINITY);
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  return cuda_status(launch_verify_shard_decide(
      stats, S, draft, topi, q, B, K, V, T, seed, cycle, n_accepted, out_tok,
      plan, d->err, reinterpret_cast<cudaStream_t>(stream)));
}

dflash_status dflash_verify_shard_draw(const float* target_shard,
                                       const float* plan,
                                       const int32_t* topi, const float* q,
                                       int shard, int B, int K, int V_shard,
                                       int v0, float T, int32_t* out_tok,
                                       void* ws, size_t ws_bytes,
                                       dflash_stream_t stream) {
  REQUIRE(target_shard && plan && topi && q && out_tok && ws);
  REQUIRE(shard >= 0 && shard < DFLASH_MAX_SHARDS);
  REQUIRE(sizes_ok(B, K, 0, V_shard) && v0 >= 0 &&
          (long long)v0 + V_shard <= (1LL << 30));
  REQUIRE(T >= 0.f && T < INFINITY);
  REQUIRE(aligned(ws, 256) && aligned(target_shard, 16));
  REQUIRE(ws_bytes >= verify_ws_layout(B, K, V_shard, nullptr, nullptr));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  VerifyWs w;
  verify_ws_layout(B, K, V_shard, ws, &w);
  return cuda_status(launch_verify_shard_draw(
      target_shard, plan, topi, q, shard, B, K, V_shard, v0, T, out_tok, w,
      d->err, reinterpret_cast<cudaStream_t>(stream)));
}

dflash_status dflash_philox4x32(const uint32_t* ctr, uint64_t seed,
                                uint32_t* out, int64_t n,
                                dflash_stream_t stream) {
  REQUIRE(n >= 0 && (n == 0 || (ctr && out)));
  REQUIRE(aligned(ctr, 16) && aligned(out, 16));
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  return cuda_status(launch_philox(ctr, seed, out, n,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

dflash_status dflash_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns ? ns : kWaitLimitNs);
  return DFLASH_OK;
}

dflash_status dflash_profile_stage(int stage, void* begin, void* end) {
  REQUIRE(stage >= 0 && stage < kNumStages);
  REQUIRE((begin == nullptr) == (end == nullptr));
  g_prof[stage][0] = static_cast<cudaEvent_t>(begin);
  g_prof[stage][1] = static_cast<cudaEvent_t>(end);
  return DFLASH_OK;
}

dflash_status dflash_check(dflash_stream_t stream) {
  DeviceState* d = nullptr;
  dflash_status st = device_state(&d);
  if (st != DFLASH_OK) return st;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, d->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  if (word) {
    const int zero = 0;
    if (cudaMemcpy(d->err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  if (word & kErrTimeout) return DFLASH_ERR_DEVICE_TIMEOUT;
  if (word & kErrNonfinite) return DFLASH_ERR_NONFINITE;
  if (word & kErrBadIndex) return DFLASH_ERR_BAD_INDEX;
  return DFLASH_OK;
}

const char* dflash_status_string(dflash_status st) {
  switch (st) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported";
    case DFLASH_ERR_CUDA: return "CUDA runtime error";
    case DFLASH_ERR_NONFINITE: return "non-finite target logit";
    case DFLASH_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case DFLASH_ERR_BAD_INDEX: return "token index out of range";
  }
  return "unknown status";
}

}  // extern "C"
