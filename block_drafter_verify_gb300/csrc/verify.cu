// Steps a5 + a6: rejection-sampling verify with residual / bonus draw.
//
// "Lossless, with conditions I did not used to state" (DFlash 2: Block
// diffusion, wearing a drafter's coat): accept a draft token with
// probability min(1, p/q) and resample from the residual on rejection.
//
// Two launches:
//   verify_rows      grid (B*(K+1), chunks): every target row is split into
//                    chunks; a CTA reduces its chunk to (max, sum exp) at
//                    T > 0 or (max, first argmax) at T = 0.  The last CTA of
//                    a row folds the chunk partials in a fixed order; the
//                    last row of a sequence runs the accept tests of all K
//                    positions in parallel (one lane each) and keeps the
//                    prefix before the first rejection.
//   verify_resample  (T > 0 only) grid (B, chunks of whole 4096-token
//                    slabs): every CTA sums the fixed-point residual weights
//                    of one chunk of row n_b; the last CTA of the sequence
//                    finds the chunk that holds the draw with a block scan
//                    and scans it slab by slab, 16 tokens per thread held in
//                    registers.
// Residual weights are integers (units of 2^-40 of the row maximum's
// weight), so their sums are exact and the draw does not depend on the
// grid.  "Last CTA" is found with an atomic ticket: nothing ever waits.
// Every loop keeps several independent loads in flight.
#include <algorithm>

#include "kernels.h"

namespace dflash {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kSeg = 16;                // tokens per thread per slab
constexpr int kSlab = kThreads * kSeg;  // 4096 tokens

__device__ __forceinline__ bool arg_better(float v1, int i1, float v2,
                                           int i2) {
  return v1 > v2 || (v1 == v2 && (unsigned)i1 < (unsigned)i2);
}

// exp((x - m) / T): the one formula every weight in this file uses.
__device__ __forceinline__ float rel_weight(float x, float m, float invT) {
  return __expf((x - m) * invT);
}

// Fixed-point weight of e in [0, 1]: floor(e * 2^40).
__device__ __forceinline__ unsigned long long quant(float e) {
  return __float2ull_rz(e * 1099511627776.0f);
}

__device__ __forceinline__ unsigned long long warp_sum_u64(
    unsigned long long v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Online (max, sum exp) update with one element.
__device__ __forceinline__ void online_lse(float x, float& m, float& s,
                                           float invT) {
  if (x > m) {
    s = s * __expf((m - x) * invT) + 1.f;
    m = x;
  } else if (x != -INFINITY) {
    s += __expf((x - m) * invT);
  }
}

// Fold a second (max, sum) or (max, argmax) partial into the first.
__device__ __forceinline__ void fold(bool greedy, float& a, float& s, int& i,
                                     float a2, float s2, int i2, float invT) {
  if (greedy) {
    if (arg_better(a2, i2, a, i)) { a = a2; i = i2; }
  } else {
    lse_combine(a, s, a2, s2, invT);
  }
}

// Inclusive block scan of one uint64 per thread; also returns the block
// total.  `s_red` holds kWarps values.
__device__ __forceinline__ unsigned long long block_incl_scan(
    unsigned long long v, unsigned long long* s_red,
    unsigned long long* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  __syncthreads();
  if (lane == 31) s_red[wid] = v;
  __syncthreads();
  unsigned long long pre = 0, tot = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < wid) pre += s_red[w];
    tot += s_red[w];
  }
  *total = tot;
  return v + pre;
}

__global__ void __launch_bounds__(kThreads)
    verify_rows_kernel(const float* __restrict__ L,
                       const int* __restrict__ draft,
                       const int* __restrict__ topi,
                       const float* __restrict__ q, int B, int K, int V,
                       int nchunk, int chunk, float T, float invT,
                       uint64_t seed, uint64_t cycle,
                       int* __restrict__ n_accepted, int* __restrict__ out_tok,
                       VerifyWs ws, int* err, int vec4) {
  const int row = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int K1 = K + 1, rows = B * K1;
  const int b = row / K1;
  const float* x = L + (size_t)row * V;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  bool bad = false;
  float a = -INFINITY, sacc = 0.f;  // (m, s) or (max value, -)
  int ai = 0x7fffffff;              // first argmax (T == 0)
  const bool greedy = (T == 0.f);

  auto take = [&](float xv, int v) {
    bad |= !(xv < INFINITY);
    if (greedy) {
      if (xv > a) { a = xv; ai = v; }
    } else {
      online_lse(xv, a, sacc, invT);
    }
  };
  if (vec4) {
    const float4* x4 = reinterpret_cast<const float4*>(x);
    int v = v0 + tid * 4;
    for (; v + 3 * kThreads * 4 < v1; v += 4 * kThreads * 4) {
      float4 f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) f[u] = x4[(v + u * kThreads * 4) >> 2];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int vv = v + u * kThreads * 4;
        take(f[u].x, vv); take(f[u].y, vv + 1);
        take(f[u].z, vv + 2); take(f[u].w, vv + 3);
      }
    }
    for (; v < v1; v += kThreads * 4) {
      const float4 f = x4[v >> 2];
      take(f.x, v); take(f.y, v + 1); take(f.z, v + 2); take(f.w, v + 3);
    }
  } else {
    int v = v0 + tid;
    for (; v + 3 * kThreads < v1; v += 4 * kThreads) {
      float f[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) f[u] = x[v + u * kThreads];
#pragma unroll
      for (int u = 0; u < 4; ++u) take(f[u], v + u * kThreads);
    }
    for (; v < v1; v += kThreads) take(x[v], v);
  }
  if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0)
    raise_error(err, kErrNonfinite);

  // block reduction in a fixed tree: lanes, then warps in order
  __shared__ float s_a[kWarps], s_s[kWarps];
  __shared__ int s_i[kWarps];
  __shared__ int s_last;
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float oa = __shfl_xor_sync(0xffffffffu, a, o);
    const float os = __shfl_xor_sync(0xffffffffu, sacc, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ai, o);
    fold(greedy, a, sacc, ai, oa, os, oi, invT);
  }
  if ((tid & 31) == 0) {
    s_a[tid >> 5] = a;
    s_s[tid >> 5] = sacc;
    s_i[tid >> 5] = ai;
  }
  __syncthreads();
  if (tid == 0) {
    float ra = s_a[0], rs = s_s[0];
    int ri = s_i[0];
    for (int w = 1; w < kWarps; ++w)
      fold(greedy, ra, rs, ri, s_a[w], s_s[w], s_i[w], invT);
    ws.chunk_part[(size_t)row * nchunk + c] =
        make_float2(ra, greedy ? __int_as_float(ri) : rs);
    __threadfence();
    s_last = (atomicAdd(&ws.counters[row], 1u) == (unsigned)(nchunk - 1));
  }
  __syncthreads();
  if (!s_last || tid >= 32) return;

  // ---- last CTA of this row (warp 0): fold the chunks in a fixed tree ---
  __threadfence();
  const int lane = tid;
  float ra = -INFINITY, rs = 0.f;
  int ri = 0x7fffffff;
  for (int cc = lane; cc < nchunk; cc += 32) {  // nchunk <= 64
    const float2 p = __ldcg(&ws.chunk_part[(size_t)row * nchunk + cc]);
    fold(greedy, ra, rs, ri, p.x, p.y, __float_as_int(p.y), invT);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float oa = __shfl_xor_sync(0xffffffffu, ra, o);
    const float os = __shfl_xor_sync(0xffffffffu, rs, o);
    const int oi = __shfl_xor_sync(0xffffffffu, ri, o);
    fold(greedy, ra, rs, ri, oa, os, oi, invT);
  }
  int last_row = 0;
  if (lane == 0) {
    if (ra == -INFINITY) {  // every logit of the row is -inf: no distribution
      raise_error(err, kErrNonfinite);
      ri = 0; ra = 0.f; rs = 1.f;
    }
    ws.row_m[row] = ra;
    ws.row_z[row] = rs;
    ws.row_arg[row] = ri;
    __threadfence();
    last_row = (atomicAdd(&ws.counters[rows + b], 1u) == (unsigned)K);
  }
  if (!__shfl_sync(0xffffffffu, last_row, 0)) return;

  // ---- last row of sequence b: the K accept tests, one lane each --------
  __threadfence();
  bool ok = true;
  if (lane < K) {
    const int t = lane;
    const int d = draft[b * K + t];
    const int rr = b * K1 + t;
    if (d < 0 || d >= V) {
      raise_error(err, kErrBadIndex);
      ok = false;
    } else if (greedy) {
      ok = (d == __ldcg(&ws.row_arg[rr]));
    } else {
      float qd = 0.f;
      bool found = false;
#pragma unroll
      for (int j = 0; j < kC; ++j) {
        const int cj = topi[(b * K + t) * kC + j];
        const float qj = q[(b * K + t) * kC + j];
        if (!found && cj == d) { qd = qj; found = true; }
      }
      if (!found) raise_error(err, kErrBadIndex);
      const float pd = rel_weight(L[(size_t)rr * V + d],
                                  __ldcg(&ws.row_m[rr]), invT) /
                       __ldcg(&ws.row_z[rr]);
      const float u = philox_uniform(seed, b, t, kPurposeAccept, cycle);
      ok = u * qd < pd;
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < K && !ok);
  const int n = rej ? __ffs(rej) - 1 : K;
  if (lane == 0) {
    n_accepted[b] = n;
    ws.n_row[b] = n;
  }
  if (lane <= K) {
    int tok = lane < n ? draft[b * K + lane] : -1;
    if (greedy && lane == n) tok = __ldcg(&ws.row_arg[b * K1 + n]);
    out_tok[b * K1 + lane] = tok;  // at T > 0 slot n is drawn next launch
  }
}

// Fixed-point weight of token v: the residual max(0, e - q Z) for a
// candidate of the rejected row, e itself otherwise (and for every token
// when drawing from p).
__device__ __forceinline__ unsigned long long token_weight(
    float xv, int v, float m, float invT, bool use_raw, const int* s_ci,
    const float* s_qz) {
  const float e = rel_weight(xv, m, invT);
  float w = e;
  if (!use_raw) {
#pragma unroll
    for (int j = 0; j < kC; ++j)
      if (s_ci[j] == v) w = fmaxf(e - s_qz[j], 0.f);
  }
  return quant(w);
}

// Load kSeg consecutive logits starting at v (-inf past v1).
__device__ __forceinline__ void load_seg(const float* x, int v, int v1,
                                         int vec4, float (&f)[kSeg]) {
  if (vec4 && v + kSeg <= v1) {
    const float4* p = reinterpret_cast<const float4*>(x + v);
#pragma unroll
    for (int u = 0; u < kSeg / 4; ++u) {
      const float4 t = p[u];
      f[4 * u] = t.x;
      f[4 * u + 1] = t.y;
      f[4 * u + 2] = t.z;
      f[4 * u + 3] = t.w;
    }
  } else {
#pragma unroll
    for (int u = 0; u < kSeg; ++u) f[u] = (v + u < v1) ? x[v + u] : -INFINITY;
  }
}

__global__ void __launch_bounds__(kThreads)
    verify_resample_kernel(const float* __restrict__ L,
                           const int* __restrict__ topi,
                           const float* __restrict__ q, int B, int K, int V,
                           int nchunk2, int chunk2, float invT, uint64_t seed,
                           uint64_t cycle, int* __restrict__ out_tok,
                           VerifyWs ws, int* err, int vec4) {
  const int b = blockIdx.x, c = blockIdx.y, tid = threadIdx.x;
  const int K1 = K + 1, rows = B * K1;
  const int n = ws.n_row[b];
  const int rr = b * K1 + n;
  const float m = ws.row_m[rr], Z = ws.row_z[rr];
  const float* x = L + (size_t)rr * V;
  __shared__ int s_ci[kC];
  __shared__ float s_qz[kC];
  __shared__ unsigned long long s_red[kWarps], s_red2[kWarps];
  __shared__ int s_last, s_use_raw, s_cstar;
  __shared__ unsigned long long s_theta, s_cum;
  if (tid < kC) {
    if (n < K) {
      s_ci[tid] = topi[(b * K + n) * kC + tid];
      s_qz[tid] = q[(b * K + n) * kC + tid] * Z;
    } else {
      s_ci[tid] = -1;
      s_qz[tid] = 0.f;
    }
  }
  __syncthreads();

  // ---- chunk sums: raw weights quant(e), residual = raw + corrections ----
  const int v0 = c * chunk2, v1 = min(V, v0 + chunk2);
  unsigned long long raw = 0;
  for (int s0 = v0; s0 < v1; s0 += kSlab) {
    float f[kSeg];
    load_seg(x, s0 + tid * kSeg, v1, vec4, f);
#pragma unroll
    for (int u = 0; u < kSeg; ++u) raw += quant(rel_weight(f[u], m, invT));
  }
  long long corr = 0;
  if (tid < kC) {
    const int ci = s_ci[tid];
    if (ci >= v0 && ci < v1) {
      const float e = rel_weight(x[ci], m, invT);
      corr = (long long)quant(fmaxf(e - s_qz[tid], 0.f)) - (long long)quant(e);
    }
  }
  raw = warp_sum_u64(raw);
  corr = (long long)warp_sum_u64((unsigned long long)corr);
  if ((tid & 31) == 0) s_red[tid >> 5] = raw;
  __syncthreads();
  if (tid == 0) {
    unsigned long long tr = 0;
    for (int w = 0; w < kWarps; ++w) tr += s_red[w];
    const unsigned long long tres = tr + (unsigned long long)corr;
    ws.res_part[((size_t)b * nchunk2 + c) * 2 + 0] = tr;
    ws.res_part[((size_t)b * nchunk2 + c) * 2 + 1] = tres;
    __threadfence();
    s_last = (atomicAdd(&ws.counters[rows + B + b], 1u) ==
              (unsigned)(nchunk2 - 1));
  }
  __syncthreads();
  if (!s_last) return;

  // ---- last CTA of the sequence: locate the chunk of the draw ------------
  __threadfence();
  unsigned long long p_res = 0, p_raw = 0;
  if (tid < nchunk2) {  // nchunk2 <= kThreads
    p_raw = __ldcg(&ws.res_part[((size_t)b * nchunk2 + tid) * 2 + 0]);
    p_res = __ldcg(&ws.res_part[((size_t)b * nchunk2 + tid) * 2 + 1]);
  }
  const unsigned long long wres = warp_sum_u64(p_res);
  const unsigned long long wraw = warp_sum_u64(p_raw);
  if ((tid & 31) == 0) {
    s_red[tid >> 5] = wres;
    s_red2[tid >> 5] = wraw;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long R = 0, R0 = 0;
    for (int w = 0; w < kWarps; ++w) {
      R += s_red[w];
      R0 += s_red2[w];
    }
    const int use_raw = (R == 0);  // degenerate residual: draw from p
    if (use_raw) R = R0;
    const unsigned long long u24 =
        philox_u24(seed, b, K, kPurposeResample, cycle);
    // theta = floor(u24 * R / 2^24); the product needs up to 82 bits
    const unsigned long long hi = __umul64hi(R, u24), lo = R * u24;
    s_theta = (hi << 40) | (lo >> 24);
    s_use_raw = use_raw;
    s_cstar = -1;
  }
  __syncthreads();
  const bool use_raw = s_use_raw;
  const unsigned long long theta = s_theta;
  {
    const unsigned long long p = use_raw ? p_raw : p_res;
    unsigned long long tot;
    const unsigned long long incl = block_incl_scan(p, s_red, &tot);
    if (tid < nchunk2 && incl - p <= theta && theta < incl) {
      s_cstar = tid;
      s_cum = incl - p;
    }
  }
  __syncthreads();
  if (s_cstar < 0) {  // cannot happen: theta is below the total
    if (tid == 0) raise_error(err, kErrBadIndex);
    return;
  }
  // ---- scan chunk c* slab by slab, 16 tokens per thread in registers -----
  const int w0 = s_cstar * chunk2, w1 = min(V, w0 + chunk2);
  unsigned long long base = s_cum;
  for (int s0 = w0; s0 < w1; s0 += kSlab) {
    float f[kSeg];
    const int v = s0 + tid * kSeg;
    load_seg(x, v, w1, vec4, f);
    unsigned long long wts[kSeg], tsum = 0;
#pragma unroll
    for (int u = 0; u < kSeg; ++u) {
      wts[u] = (v + u < w1)
                   ? token_weight(f[u], v + u, m, invT, use_raw, s_ci, s_qz)
                   : 0ull;
      tsum += wts[u];
    }
    unsigned long long tot;
    const unsigned long long incl = block_incl_scan(tsum, s_red, &tot);
    const unsigned long long lo_b = base + incl - tsum;
    if (tsum > 0 && lo_b <= theta && theta < lo_b + tsum) {
      unsigned long long acc = lo_b;
      int pick = -1;
#pragma unroll
      for (int u = 0; u < kSeg; ++u) {
        acc += wts[u];
        if (pick < 0 && acc > theta) pick = v + u;
      }
      out_tok[b * K1 + n] = pick;
    }
    if (theta < base + tot) break;  // uniform across the block
    base += tot;
  }
}

__global__ void philox_kernel(const uint32_t* __restrict__ ctr, uint64_t seed,
                              uint32_t* __restrict__ out, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const uint4 c = reinterpret_cast<const uint4*>(ctr)[i];
  const U32x4 r = philox4x32_10(U32x4{c.x, c.y, c.z, c.w}, (uint32_t)seed,
                                (uint32_t)(seed >> 32));
  reinterpret_cast<uint4*>(out)[i] = make_uint4(r.x, r.y, r.z, r.w);
}

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

int verify_chunks(int parts, int V, int target_ctas, int* chunk) {
  const int max_chunks =
      std::min(kVerifyMaxChunks, std::max(1, (V + 1023) / 1024));
  int n = std::min(max_chunks, std::max(1, (target_ctas + parts - 1) / parts));
  *chunk = (((V + n - 1) / n) + 3) & ~3;
  return (V + *chunk - 1) / *chunk;
}

}  // namespace

size_t verify_ws_layout(int B, int K, int V, void* base, VerifyWs* o) {
  (void)V;
  const size_t rows = (size_t)B * (K + 1);
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    off = align256(off);
    char* r = p ? p + off : nullptr;
    off += bytes;
    return r;
  };
  VerifyWs w{};
  w.chunk_part =
      reinterpret_cast<float2*>(take(rows * kVerifyMaxChunks * sizeof(float2)));
  w.row_m = reinterpret_cast<float*>(take(rows * sizeof(float)));
  w.row_z = reinterpret_cast<float*>(take(rows * sizeof(float)));
  w.row_arg = reinterpret_cast<int*>(take(rows * sizeof(int)));
  w.n_row = reinterpret_cast<int*>(take((size_t)B * sizeof(int)));
  w.res_part = reinterpret_cast<unsigned long long*>(take(
      (size_t)B * kResampleMaxChunks * 2 * sizeof(unsigned long long)));
  w.counter_bytes = (rows + 2 * (size_t)B) * sizeof(unsigned);
  w.counters = reinterpret_cast<unsigned*>(take(w.counter_bytes));
  if (o) *o = w;
  return align256(off);
}

// The caller zeroes ws.counters on the stream before this launch.
cudaError_t launch_verify_rows(const float* L, const int* draft,
                               const int* topi, const float* q, int B, int K,
                               int V, float T, uint64_t seed, uint64_t cycle,
                               int* n_accepted, int* out_tok,
                               const VerifyWs& ws, int num_sms, int* err,
                               cudaStream_t s) {
  const int rows = B * (K + 1);
  int chunk = 0;
  const int nchunk = verify_chunks(rows, V, 4 * num_sms, &chunk);
  const int vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(L) & 15) == 0);
  const float invT = T > 0.f ? 1.f / T : 0.f;
  verify_rows_kernel<<<dim3(rows, nchunk), kThreads, 0, s>>>(
      L, draft, topi, q, B, K, V, nchunk, chunk, T, invT, seed, cycle,
      n_accepted, out_tok, ws, err, vec4);
  return cudaGetLastError();
}

cudaError_t launch_verify_resample(const float* L, const int* topi,
                                   const float* q, int B, int K, int V,
                                   float T, uint64_t seed, uint64_t cycle,
                                   int* out_tok, const VerifyWs& ws,
                                   int num_sms, int* err, cudaStream_t s) {
  (void)num_sms;
  // chunks are whole slabs of 4096 tokens, at most kResampleMaxChunks
  const int slabs = (V + kSlab - 1) / kSlab;
  const int per = (slabs + kResampleMaxChunks - 1) / kResampleMaxChunks;
  const int chunk2 = per * kSlab;
  const int nchunk2 = (V + chunk2 - 1) / chunk2;
  const int vec4 = (V % 4 == 0) && ((reinterpret_cast<uintptr_t>(L) & 15) == 0);
  const float invT = 1.f / T;
  verify_resample_kernel<<<dim3(B, nchunk2), kThreads, 0, s>>>(
      L, topi, q, B, K, V, nchunk2, chunk2, invT, seed, cycle, out_tok, ws,
      err, vec4);
  return cudaGetLastError();
}

cudaError_t launch_philox(const uint32_t* ctr, uint64_t seed, uint32_t* out,
                          int64_t n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (n + threads - 1) / threads;
  philox_kernel<<<(unsigned)blocks, threads, 0, s>>>(ctr, seed, out, n);
  return cudaGetLastError();
}

}  // namespace dflash
