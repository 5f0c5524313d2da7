// Step a3: context gate and low-rank bilinear pair scores.
//
// "A Lightweight Path Selector" (DFlash 2: Keep Drafting Parallel): every
// adjacent pair (predecessor a, candidate b) is scored at once as the
// drafter's own logit of b plus a 256-dim embedding match under a context
// gate of h_t — no backbone or LM-head pass.
//
// One launch, no scratch memory: a cluster of 8 CTAs owns 16 rows (b, t).
//   1. gate pre-activations z = W_g h of the 16 rows over this CTA's eighth
//      of the hidden dimension.  bf16 storage: the h rows and W_g rows are
//      staged unconverted with cp.async (zero-filled past the slice) and
//      contracted on the tensor cores (mma.sync m16n8k16, bf16 x bf16 ->
//      fp32; warp w owns gate columns 32w .. 32w+31).  fp32 storage: exact
//      fp32 products on the CUDA cores, W_g staged in 64-column panels;
//   2. the partial sums are added over the cluster through distributed
//      shared memory, in cluster-rank order, and CTA k keeps the gates
//      g = sigmoid(z) of rows 2k and 2k+1;
//   3. CTA k writes the 16 x 16 scores of each of its two rows from the 16
//      predecessor rows of E_in and the 16 candidate rows of E_out (scaled
//      by g).  Those 64 embedding rows are fetched with cp.async while step
//      1 runs: right after the first W_g panel's copies are issued, the CTA
//      reads its rows' candidate lists and starts the gathers.
#include <cooperative_groups.h>

#include <algorithm>
#include <type_traits>

#include "kernels.h"
#include "merge.cuh"

namespace cg = cooperative_groups;

namespace dflash {
namespace {

constexpr int kCluster = 8;     // CTAs per cluster (split of the hidden dim)
constexpr int kRows = 16;       // rows (b, t) per cluster
constexpr int kRowsPerCta = kRows / kCluster;
constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPanel = 64;           // fp32 path: W_g columns per panel
constexpr int kPanelStride = kPanel + 4;  // 16-byte rows, no bank conflicts
constexpr int kKP = 128;             // bf16 path: hidden columns per panel
constexpr int kLdsB = kKP + 8;       // padded bf16 row: conflict-free reads

// Shared memory of phase 1, in floats (phase 3 reuses the same region).
__host__ __device__ constexpr size_t work_floats(int hs, bool bf16) {
  return bf16 ? (size_t)(kRows + 256) * kLdsB / 2
              : (size_t)kRows * hs + (size_t)256 * kPanelStride;
}

// 16-byte vector of storage elements converted to fp32.
template <typename T>
struct Vec16 {
  __device__ __forceinline__ static void to_f32(const uint4& u, float* f);
};
template <>
__device__ __forceinline__ void Vec16<float>::to_f32(const uint4& u,
                                                     float* f) {
  f[0] = __uint_as_float(u.x); f[1] = __uint_as_float(u.y);
  f[2] = __uint_as_float(u.z); f[3] = __uint_as_float(u.w);
}
template <>
__device__ __forceinline__ void Vec16<__nv_bfloat16>::to_f32(const uint4& u,
                                                             float* f) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
__device__ __forceinline__ void cp_async16(void* dst, const void* src,
                                           int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src), "r"(src_bytes)
               : "memory");
}
// 4-byte asynchronous copy global -> shared.
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// D += A B for one 16 x 8 x 16 tile, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0,
                                          uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0,
                                          uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t ld_b32(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint32_t*>(p);
}

// Phase 1, bf16 storage: part[row][n] = sum over this CTA's slice of
// h[m0 + row][k] * W_g[n][k], on the tensor cores.  The slice length is a
// multiple of 8 (H is), so every 16-byte copy is either whole or skipped.
template <typename Prologue>
__device__ __forceinline__ void gate_partial_mma(
    const __nv_bfloat16* __restrict__ h, const __nv_bfloat16* __restrict__ w,
    int M, int H, int r, int m0, int k0, int klen, float* part, float* work,
    Prologue&& after_first_issue) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  __nv_bfloat16* hs_ = reinterpret_cast<__nv_bfloat16*>(work);  // [16][kLdsB]
  __nv_bfloat16* ws_ = hs_ + kRows * kLdsB;                      // [256][kLdsB]
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
  constexpr int kChunks = kKP / 8;  // 16-byte chunks per staged row
  for (int p0 = 0; p0 < klen; p0 += kKP) {
    const int pw = min(kKP, klen - p0);
    __syncthreads();  // the previous panel is consumed
    for (int i = tid; i < kRows * kChunks; i += kThreads) {
      const int row = i / kChunks, ch = i % kChunks;
      const bool ok = m0 + row < M && ch * 8 < pw;
      cp_async16(hs_ + row * kLdsB + ch * 8,
                 ok ? h + (size_t)(m0 + row) * H + k0 + p0 + ch * 8 : h,
                 ok ? 16 : 0);
    }
    for (int i = tid; i < 256 * kChunks; i += kThreads) {
      const int n = i / kChunks, ch = i % kChunks;
      const bool ok = n < r && ch * 8 < pw;
      cp_async16(ws_ + n * kLdsB + ch * 8,
                 ok ? w + (size_t)n * H + k0 + p0 + ch * 8 : w, ok ? 16 : 0);
    }
    if (p0 == 0) after_first_issue();
    cp_async_wait_all();
    __syncthreads();
    const int ksteps = (pw + 15) / 16;  // columns past pw are zeros
    for (int kk = 0; kk < ksteps; ++kk) {
      const int kc = kk * 16 + 2 * c;
      const uint32_t a0 = ld_b32(hs_ + g * kLdsB + kc);
      const uint32_t a1 = ld_b32(hs_ + (g + 8) * kLdsB + kc);
      const uint32_t a2 = ld_b32(hs_ + g * kLdsB + kc + 8);
      const uint32_t a3 = ld_b32(hs_ + (g + 8) * kLdsB + kc + 8);
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) {
        const __nv_bfloat16* wr = ws_ + ((warp * 4 + nt) * 8 + g) * kLdsB + kc;
        mma_16816(acc[nt], a0, a1, a2, a3, ld_b32(wr), ld_b32(wr + 8));
      }
    }
  }
  if (klen <= 0) after_first_issue();
  __syncthreads();  // part aliases the staged tiles
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    const int n = (warp * 4 + nt) * 8 + 2 * c;
    part[g * 256 + n] = acc[nt][0];
    part[g * 256 + n + 1] = acc[nt][1];
    part[(g + 8) * 256 + n] = acc[nt][2];
    part[(g + 8) * 256 + n + 1] = acc[nt][3];
  }
}

// Phase 1, fp32 storage: exact fp32 products on the CUDA cores.
__device__ __forceinline__ void gate_partial_simt(
    const float* __restrict__ h, const float* __restrict__ w_gate, int M,
    int H, int r, int m0, int k0, int klen, int hs, float* part,
    float* work) {
  using T = float;
  constexpr int EPV = 4;               // elements per 16-byte vector
  constexpr int VPR = kPanel / EPV;    // vectors per panel row
  const int tid = threadIdx.x;
  float* hsl = work;                   // kRows * hs
  float* panel = hsl + kRows * hs;     // 256 * kPanelStride
  {  // h slice of the 16 rows: 16-byte loads, a batch issued before use
    const int vrow = hs / EPV;                 // vectors per row slice
    constexpr int kBatch = 8;                  // loads in flight per thread
    for (int i0 = 0; i0 < kRows * vrow; i0 += kBatch * kThreads) {
      uint4 hv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + tid + u * kThreads;
        const int rr = i / vrow, cv = i % vrow;
        const int m = m0 + rr;
        hv[u] = (rr < kRows && m < M && cv * EPV < klen)
                    ? *reinterpret_cast<const uint4*>(h + (size_t)m * H + k0 +
                                                      cv * EPV)
                    : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + tid + u * kThreads;
        const int rr = i / vrow, cv = i % vrow;
        if (rr < kRows) {
          float f[EPV];
          Vec16<T>::to_f32(hv[u], f);
#pragma unroll
          for (int e = 0; e < EPV; ++e) hsl[rr * hs + cv * EPV + e] = f[e];
        }
      }
    }
  }
  float acc[kRows];
#pragma unroll
  for (int rr = 0; rr < kRows; ++rr) acc[rr] = 0.f;
  constexpr int kLoads = 256 * VPR / kThreads;  // 16-byte loads per thread
  for (int p0 = 0; p0 < klen; p0 += kPanel) {
    const int pw = min(kPanel, klen - p0);
    uint4 buf[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = tid + u * kThreads;
      const int g = i / VPR, cv = i % VPR;
      buf[u] = (g < r && cv * EPV < pw)
                   ? *reinterpret_cast<const uint4*>(
                         w_gate + (size_t)g * H + k0 + p0 + cv * EPV)
                   : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();  // previous panel fully consumed
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
      const int i = tid + u * kThreads;
      const int g = i / VPR, cv = i % VPR;
      float f[EPV];
      Vec16<T>::to_f32(buf[u], f);
      float4* dst = reinterpret_cast<float4*>(panel + g * kPanelStride + cv * EPV);
#pragma unroll
      for (int e = 0; e < EPV / 4; ++e)
        dst[e] = make_float4(f[4 * e], f[4 * e + 1], f[4 * e + 2], f[4 * e + 3]);
    }
    __syncthreads();
    if (tid < r) {
      // four columns per step: one 16-byte load of W_g, one per row of h
      const float4* wrow = reinterpret_cast<const float4*>(panel + tid * kPanelStride);
      for (int c4 = 0; c4 < pw / 4; ++c4) {
        const float4 w = wrow[c4];
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) {
          const float4 hv =
              *reinterpret_cast<const float4*>(hsl + rr * hs + p0 + 4 * c4);
          acc[rr] = fmaf(w.x, hv.x, acc[rr]);
          acc[rr] = fmaf(w.y, hv.y, acc[rr]);
          acc[rr] = fmaf(w.z, hv.z, acc[rr]);
          acc[rr] = fmaf(w.w, hv.w, acc[rr]);
        }
      }
    }
  }
  __syncthreads();  // part aliases the staged slice and panel
  if (tid < r) {
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) part[rr * 256 + tid] = acc[rr];
  }
}

// The 16 x 16 scores of one row (b, t), whole CTA:
//   S[i][j] = topv[j] + sum_k E_in[pred_i, k] g[k] E_out[cand_j, k]
// (-inf where pred_i or cand_j is padding).  The embedding rows are staged
// raw in st ([table][16][r], 0 = E_in) when `vec`, else read from the
// tables here.  work holds two fp32 tiles of 16 rows; thread tid < 128
// writes S[tid / 16][tid % 16] and S[tid / 16 + 8][tid % 16].
template <int NT, typename T>
__device__ __forceinline__ void score_row(
    const T* st, bool vec, const int* pred, const int* cand,
    const float* g_row, const T* __restrict__ e_in,
    const T* __restrict__ e_out, int r, float* work,
    const float* __restrict__ topv_row, float* __restrict__ out,
    float* s_out = nullptr) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // fp32 tiles with 16-byte aligned rows when r allows (float4 reads)
  const bool r4 = (r % 4) == 0;
  const int rs = r4 ? r + 4 : r + 1;
  float* ein_s = work;              // [16][rs]
  float* eout_s = work + kC * rs;   // [16][rs], scaled by the gate
  if (vec) {
    // warp w converts staged rows w, w + 8, ...; lane l its 16-byte chunks
    constexpr int epc = 16 / sizeof(T);  // elements per chunk
    const int cpr = r / epc;
    for (int rowi = warp; rowi < 2 * kC; rowi += NT / 32) {
      const bool outt = rowi >= kC;
      float* dst = (outt ? eout_s : ein_s) + (rowi % kC) * rs;
      const T* srow = st + (size_t)rowi * r;
      for (int ch = lane; ch < cpr; ch += 32) {
        float f[epc > 4 ? 8 : 4];
        Vec16<T>::to_f32(*reinterpret_cast<const uint4*>(srow + ch * epc), f);
        if (r4) {  // 16-byte stores (rows are 16-byte aligned)
#pragma unroll
          for (int e = 0; e < epc; e += 4) {
            float4 o = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
            if (outt) {
              const float4 g4 =
                  *reinterpret_cast<const float4*>(g_row + ch * epc + e);
              o.x *= g4.x; o.y *= g4.y; o.z *= g4.z; o.w *= g4.w;
            }
            *reinterpret_cast<float4*>(dst + ch * epc + e) = o;
          }
        } else {
#pragma unroll
          for (int e = 0; e < epc; ++e)
            dst[ch * epc + e] = outt ? f[e] * g_row[ch * epc + e] : f[e];
        }
      }
    }
  } else {
    for (int i = tid; i < kC * r; i += NT) {
      const int row = i / r, k = i % r;
      const int a = pred[row], c = cand[row];
      ein_s[row * rs + k] = a >= 0 ? to_f32(e_in[(size_t)a * r + k]) : 0.f;
      eout_s[row * rs + k] =
          c >= 0 ? to_f32(e_out[(size_t)c * r + k]) * g_row[k] : 0.f;
    }
  }
  __syncthreads();
  // thread tid < 128: outputs (i, jj) and (i + 8, jj), sharing eb's loads
  if (tid >= kC * kC / 2) return;
  const int i = tid / kC, jj = tid % kC;
  const float* ea = ein_s + i * rs;
  const float* ea8 = ein_s + (i + 8) * rs;
  const float* eb = eout_s + jj * rs;
  float sc = 0.f, sd = 0.f;
  int k = 0;
  if (r4) {  // four partial sums (k mod 4) per output, added at the end
    float s1 = 0.f, s2 = 0.f, s3 = 0.f, d1 = 0.f, d2 = 0.f, d3 = 0.f;
#pragma unroll 4
    for (; k < r; k += 4) {
      const float4 b4 = *reinterpret_cast<const float4*>(eb + k);
      const float4 a4 = *reinterpret_cast<const float4*>(ea + k);
      const float4 c4 = *reinterpret_cast<const float4*>(ea8 + k);
      sc = fmaf(a4.x, b4.x, sc);
      s1 = fmaf(a4.y, b4.y, s1);
      s2 = fmaf(a4.z, b4.z, s2);
      s3 = fmaf(a4.w, b4.w, s3);
      sd = fmaf(c4.x, b4.x, sd);
      d1 = fmaf(c4.y, b4.y, d1);
      d2 = fmaf(c4.z, b4.z, d2);
      d3 = fmaf(c4.w, b4.w, d3);
    }
    sc = (sc + s1) + (s2 + s3);
    sd = (sd + d1) + (d2 + d3);
  }
  for (; k < r; ++k) {
    sc = fmaf(ea[k], eb[k], sc);
    sd = fmaf(ea8[k], eb[k], sd);
  }
  const float tj = topv_row[jj];
  const bool cj = cand[jj] >= 0;
  const float o0 = (pred[i] >= 0 && cj) ? tj + sc : -INFINITY;
  const float o1 = (pred[i + 8] >= 0 && cj) ? tj + sd : -INFINITY;
  out[i * kC + jj] = o0;
  out[(i + 8) * kC + jj] = o1;
  if (s_out) {
    s_out[i * kC + jj] = o0;
    s_out[(i + 8) * kC + jj] = o1;
  }
}

// Token of (table, slot i) for row m: candidates topi[m, i] (table 1) or
// their predecessors, the anchor at t = 0 else topi[m - 1, i] (table 0);
// -1 for padding, and out-of-range ids are flagged and treated as padding.
__device__ __forceinline__ int row_token(const int* __restrict__ topi,
                                         const int* __restrict__ anchor, int m,
                                         int K, int V, int tab, int i,
                                         int* err) {
  const int b = m / K, t = m % K;
  int tok = tab == 1 ? topi[(size_t)m * kC + i]
                     : (t == 0 ? anchor[b] : topi[(size_t)(m - 1) * kC + i]);
  if (tok < -1 || tok >= V) {
    raise_error(err, kErrBadIndex);
    tok = -1;
  }
  return tok;
}

// Gathers of the 2 x 16 embedding rows of tokens tok[tab][i] into st
// ([table][16][r]) by 16-byte asynchronous copies; padding rows are zeros.
template <typename T, int NT = kThreads>
__device__ __forceinline__ void gather_rows(T* st, const int (*tok)[kC],
                                            const T* __restrict__ e_in,
                                            const T* __restrict__ e_out,
                                            int r) {
  const int cpr = r * (int)sizeof(T) / 16;  // 16-byte chunks per row
  for (int idx = threadIdx.x; idx < 2 * kC * cpr; idx += NT) {
    const int rowi = idx / cpr, ch = idx % cpr;  // rowi = tab * 16 + i
    const int tab = rowi / kC;
    const int t = tok[tab][rowi % kC];
    const T* src = (tab == 0 ? e_in : e_out) + (size_t)max(t, 0) * r;
    cp_async16(st + (size_t)rowi * r + ch * (16 / sizeof(T)),
               reinterpret_cast<const char*>(src) + ch * 16, t >= 0 ? 16 : 0);
  }
}

// Row stride (bf16 elements) of the staged embedding rows of the
// tensor-core scores: r rounded up to whole k-steps of 16, plus 8 so that
// the fragment loads of 8 rows x 4 columns hit 32 distinct banks.
__host__ __device__ constexpr int mma_ld(int r) { return (r + 15) / 16 * 16 + 8; }

// As gather_rows, into rows of stride ld, with the elements [r, ld - 8)
// zeroed (r % 8 == 0).
__device__ __forceinline__ void gather_rows_ld(__nv_bfloat16* st, int ld,
                                               const int (*tok)[kC],
                                               const __nv_bfloat16* e_in,
                                               const __nv_bfloat16* e_out,
                                               int r) {
  const int cpr = r / 8;                    // 16-byte chunks per row
  const int cpad = (ld - 8) / 8;            // chunks up to the k-step
  for (int idx = threadIdx.x; idx < 2 * kC * cpad; idx += kThreads) {
    const int rowi = idx / cpad, ch = idx % cpad;
    __nv_bfloat16* dst = st + (size_t)rowi * ld + ch * 8;
    if (ch >= cpr) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
      continue;
    }
    const int tab = rowi / kC;
    const int t = tok[tab][rowi % kC];
    const __nv_bfloat16* src = (tab == 0 ? e_in : e_out) + (size_t)max(t, 0) * r;
    cp_async16(dst, src + ch * 8, t >= 0 ? 16 : 0);
  }
}

// bf16 splitting of an fp32 value x = hi + mid + lo + e, |e| <= 2^-24 |x|
// (each step keeps the next 8 significant bits; the differences are exact
// in fp32).
__device__ __forceinline__ void split3_bf16(float x, __nv_bfloat16& hi,
                                            __nv_bfloat16& mid,
                                            __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  const float r1 = x - __bfloat162float(hi);
  mid = __float2bfloat16_rn(r1);
  lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
}

// The 16 x 16 scores of one row (b, t) on the tensor cores, whole CTA
// (256 threads), from the staged raw rows st ([table][16][ld], 0 = E_in,
// padded with zeros to the k-step):
//   S[i][j] = topv[j] + sum_k E_in[pred_i, k] X[j, k],
//   X[j, k] = g[k] E_out[cand_j, k]  (fp32),
// with X split into three bf16 parts so that every product of the
// mma.sync m16n8k16 (bf16 x bf16 -> fp32) is exact and the sum matches
// fp32 evaluation: E_in is bf16 already, X = X_hi + X_mid + X_lo to 2^-24.
// Warp w takes column block w & 1 (8 candidates) and every fourth k-step
// from w >> 1; the four partial tiles are added in a fixed order.
// work: >= 3 * 16 * ld bf16 + 4 * 256 fp32.
__device__ __forceinline__ void score_row_mma(
    const __nv_bfloat16* st, int ld, const int* pred, const int* cand,
    const float* g_row, int r, float* work, const float* topv_row,
    float* __restrict__ out, float* s_out) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kp = ld - 8;                        // padded k extent
  __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(work);  // [3][16][ld]
  float* part = work + (3 * kC * ld + 1) / 2;   // [4][16][16]
  const __nv_bfloat16* eo = st + (size_t)kC * ld;
  const int cpr = kp / 8;
  for (int idx = tid; idx < kC * cpr; idx += kThreads) {
    const int j = idx / cpr, ch = idx % cpr;
    float f[8];
    Vec16<__nv_bfloat16>::to_f32(
        *reinterpret_cast<const uint4*>(eo + (size_t)j * ld + ch * 8), f);
    __align__(16) __nv_bfloat16 h8[8], m8[8], l8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int k = ch * 8 + e;
      const float x = k < r ? f[e] * g_row[k] : 0.f;
      split3_bf16(x, h8[e], m8[e], l8[e]);
    }
    const size_t o = (size_t)j * ld + ch * 8;
    *reinterpret_cast<uint4*>(xs + o) = *reinterpret_cast<const uint4*>(h8);
    *reinterpret_cast<uint4*>(xs + kC * ld + o) =
        *reinterpret_cast<const uint4*>(m8);
    *reinterpret_cast<uint4*>(xs + 2 * kC * ld + o) =
        *reinterpret_cast<const uint4*>(l8);
  }
  __syncthreads();
  {
    const int g = lane >> 2, c = lane & 3;
    const int nt = warp & 1, kq = warp >> 1;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    const __nv_bfloat16* ea = st + g * ld + 2 * c;
    const __nv_bfloat16* xb = xs + (nt * 8 + g) * ld + 2 * c;
    for (int k0 = kq * 16; k0 < kp; k0 += 64) {
      const uint32_t a0 = ld_b32(ea + k0);
      const uint32_t a1 = ld_b32(ea + 8 * ld + k0);
      const uint32_t a2 = ld_b32(ea + k0 + 8);
      const uint32_t a3 = ld_b32(ea + 8 * ld + k0 + 8);
#pragma unroll
      for (int pp = 0; pp < 3; ++pp) {
        const __nv_bfloat16* xr = xb + pp * kC * ld + k0;
        mma_16816(acc, a0, a1, a2, a3, ld_b32(xr), ld_b32(xr + 8));
      }
    }
    float* pq = part + kq * kC * kC;
    const int col = nt * 8 + 2 * c;
    pq[g * kC + col] = acc[0];
    pq[g * kC + col + 1] = acc[1];
    pq[(g + 8) * kC + col] = acc[2];
    pq[(g + 8) * kC + col + 1] = acc[3];
  }
  __syncthreads();
  const int i = tid / kC, j = tid % kC;  // kThreads == 256 == 16 x 16
  const float v = ((part[tid] + part[256 + tid]) + part[512 + tid]) +
                  part[768 + tid];
  const float o = (pred[i] >= 0 && cand[j] >= 0) ? topv_row[j] + v : -INFINITY;
  out[tid] = o;
  s_out[tid] = o;
}

template <typename T>
__global__ void __cluster_dims__(kCluster, 1, 1) __launch_bounds__(kThreads)
    pair_score_kernel(const float* __restrict__ topv,
                      const int* __restrict__ topi,
                      const int* __restrict__ anchor, const T* __restrict__ h,
                      const T* __restrict__ w_gate, const T* __restrict__ e_in,
                      const T* __restrict__ e_out, int B, int K, int H, int V,
                      int r, int hs, int work_len, float* __restrict__ scores,
                      int* err) {
  extern __shared__ float4 smem4[];
  float* smem = reinterpret_cast<float*>(smem4);
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int tid = threadIdx.x;
  const int M = B * K;
  const int m0 = (blockIdx.x / kCluster) * kRows;
  const int k0 = crank * hs, k1 = min(H, k0 + hs);
  const int klen = max(0, k1 - k0);

  float* gate = smem;                           // kRowsPerCta * 256
  float* work = gate + kRowsPerCta * 256;       // phase 1, then phase 3
  float* part = work;  // [kRows][256]: written once phase 1's tiles are done
  // raw embedding rows [row j][table (0 = E_in, 1 = E_out)][16][r]
  T* estage = reinterpret_cast<T*>(work + work_len);
  __shared__ int s_tok[kRowsPerCta][2][kC];
  // the embedding rows come in by 16-byte copies when rows are whole
  // 16-byte vectors (the tables are 16-byte aligned)
  const bool vec = (r * (int)sizeof(T)) % 16 == 0;

  // Indices of this CTA's rows (b, t): candidates topi[b,t,:] and their
  // predecessors (the anchor at t = 0, else topi[b,t-1,:]); then the
  // gathers of their embedding rows, in flight during phase 1.
  auto fetch_rows = [&]() {
    if (tid < kRowsPerCta * 2 * kC) {
      const int j = tid / (2 * kC), tab = (tid / kC) & 1, i = tid % kC;
      const int m = m0 + crank * kRowsPerCta + j;
      s_tok[j][tab][i] = m < M ? row_token(topi, anchor, m, K, V, tab, i, err)
                               : -1;
    }
    __syncthreads();
    if (vec)
      for (int j = 0; j < kRowsPerCta; ++j)
        gather_rows(estage + (size_t)j * 2 * kC * r, s_tok[j], e_in, e_out, r);
  };

  // ---- phase 1: partial z[row][k] over this CTA's hidden slice ----------
  if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    gate_partial_mma(h, w_gate, M, H, r, m0, k0, klen, part, work, fetch_rows);
  } else {
    fetch_rows();
    gate_partial_simt(h, w_gate, M, H, r, m0, k0, klen, hs, part, work);
  }
  cluster.sync();

  // ---- phase 2: add the 8 slices (rank order) for this CTA's two rows ---
  if (tid < r) {
#pragma unroll
    for (int j = 0; j < kRowsPerCta; ++j) {
      const int rr = crank * kRowsPerCta + j;
      float z = 0.f;
      for (int c = 0; c < kCluster; ++c) {
        const float* peer = cluster.map_shared_rank(part, c);
        z += peer[rr * 256 + tid];
      }
      gate[j * 256 + tid] = 1.f / (1.f + __expf(-z));
    }
  }
  cp_async_wait_all();  // the embedding rows (normally long since landed)
  cluster.sync();       // peers are done reading this CTA's partials

  // ---- phase 3: 16 x 16 scores of each row --------------------------------
  for (int j = 0; j < kRowsPerCta; ++j) {
    const int m = m0 + crank * kRowsPerCta + j;
    if (m >= M) break;
    if (j > 0) __syncthreads();  // the previous row's tiles are consumed
    score_row<kThreads>(estage + (size_t)j * 2 * kC * r, vec, s_tok[j][0], s_tok[j][1],
              gate + j * 256, e_in, e_out, r, work, topv + (size_t)m * kC,
              scores + (size_t)m * kC * kC);
  }
}

// Pair scores of one row (b, t) per CTA from a precomputed gate: the
// candidate and predecessor ids, the gate row and the 32 embedding rows
// come in by asynchronous copies, then score_row.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    pair_score_gated_kernel(const float* __restrict__ topv,
                            const int* __restrict__ topi,
                            const int* __restrict__ anchor,
                            const float* __restrict__ gate,
                            const T* __restrict__ e_in,
                            const T* __restrict__ e_out, int K, int V, int r,
                            float* __restrict__ scores, int* err) {
  extern __shared__ float4 smem4[];
  float* g_row = reinterpret_cast<float*>(smem4);        // [256]
  float* work = g_row + DFLASH_MAX_RANK;                  // two 16-row tiles
  T* st = reinterpret_cast<T*>(work + 2 * kC * (DFLASH_MAX_RANK + 4));
  __shared__ int s_tok[2][kC];
  const int m = blockIdx.x, tid = threadIdx.x;
  const bool vec = (r * (int)sizeof(T)) % 16 == 0;
  const float* grow = gate + (size_t)m * r;
  if (r % 4 == 0) {
    for (int c = tid; c < r / 4; c += kThreads)
      cp_async16(g_row + 4 * c, grow + 4 * c, 16);
  } else {
    for (int k = tid; k < r; k += kThreads) g_row[k] = grow[k];
  }
  if (tid < 2 * kC)
    s_tok[tid / kC][tid % kC] =
        row_token(topi, anchor, m, K, V, tid / kC, tid % kC, err);
  __syncthreads();
  if (vec) gather_rows(st, s_tok, e_in, e_out, r);
  cp_async_wait_all();
  __syncthreads();
  score_row<kThreads>(st, vec, s_tok[0], s_tok[1], g_row, e_in, e_out, r,
                      work, topv + (size_t)m * kC,
                      scores + (size_t)m * kC * kC);
}

// Merge of one row's nstrip strip lists staged in shared memory (sv/si
// [nstrip][16], best first; sm/ss [nstrip] pairs) by a group of warps:
// warp gw of ngw takes the lists gw, gw + ngw, ...: it sorts their best
// entries (a warp bitonic sort) and folds the lists in that order with
// bitonic merges, stopping at the first list whose best entry cannot enter
// the top-16 (so at most 16 merges); then the group's first warp merges the
// group's lists in warp order.  Same top-16 as topk_merge_kernel; lse may
// differ in the last bits (another summation order).
// (max, sum exp) pairs of the strips gw, gw + ngw, ... of one row, folded
// by a warp: each lane its strips in order, then the lanes in a fixed tree.
__device__ __forceinline__ void fold_pairs_smem(const float* sm,
                                                const float* ss, int nstrip,
                                                int gw, int ngw, float& rm,
                                                float& rs) {
  const int lane = threadIdx.x & 31;
  const int nl = gw < nstrip ? (nstrip - gw + ngw - 1) / ngw : 0;  // lists
  rm = -INFINITY;
  rs = 0.f;
  for (int j = lane; j < nl; j += 32) {
    const int st = gw + ngw * j;
    lse_combine(rm, rs, sm[st], ss[st], 1.f);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float om = __shfl_down_sync(0xffffffffu, rm, o);
    const float os = __shfl_down_sync(0xffffffffu, rs, o);
    if (lane + o < 32) lse_combine(rm, rs, om, os, 1.f);
  }
  rm = __shfl_sync(0xffffffffu, rm, 0);
  rs = __shfl_sync(0xffffffffu, rs, 0);
}

__device__ __forceinline__ void fold_lists_smem(const float* sv,
                                                const int* si,
                                                const float* sm,
                                                const float* ss, int nstrip,
                                                int gw, int ngw, float& tv,
                                                int& ti, float& rm,
                                                float& rs) {
  const int lane = threadIdx.x & 31;
  const int k = lane < kC ? lane : 31 - lane;  // lanes 16..31: reversed
  const int nl = gw < nstrip ? (nstrip - gw + ngw - 1) / ngw : 0;  // lists
  tv = -INFINITY;
  ti = -1;
  fold_pairs_smem(sm, ss, nstrip, gw, ngw, rm, rs);
  // top-16: 32 lists at a time, taken in the order of their best entries;
  // once a list's best cannot enter the top-16, no later one can
  for (int j0 = 0; j0 < nl; j0 += 32) {
    const int j = j0 + lane;
    float hv = -INFINITY;
    int hi = -1, hs = -1;
    if (j < nl) {
      hs = gw + ngw * j;
      hv = sv[hs * kC];
      hi = si[hs * kC];
    }
    // bitonic sort of the 32 heads, best first
#pragma unroll
    for (int size = 2; size <= 32; size <<= 1) {
#pragma unroll
      for (int d = size >> 1; d; d >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, hv, d);
        const int oi = __shfl_xor_sync(0xffffffffu, hi, d);
        const int os = __shfl_xor_sync(0xffffffffu, hs, d);
        const bool best_first = ((lane & size) == 0) || size == 32;
        const bool lower = (lane & d) == 0;
        const bool other_ahead = ranks_ahead(ov, oi, hv, hi);
        const bool mine_ahead = ranks_ahead(hv, hi, ov, oi);
        if ((lower == best_first) ? other_ahead : mine_ahead) {
          hv = ov; hi = oi; hs = os;
        }
      }
    }
    for (int p = 0; p < 32; ++p) {
      const float bv = __shfl_sync(0xffffffffu, hv, p);
      const int bi = __shfl_sync(0xffffffffu, hi, p);
      const int bs = __shfl_sync(0xffffffffu, hs, p);
      if (bs < 0 ||
          !ranks_ahead(bv, bi, __shfl_sync(0xffffffffu, tv, kC - 1),
                       __shfl_sync(0xffffffffu, ti, kC - 1)))
        break;
      float v = lane < kC ? tv : sv[bs * kC + k];
      int i = lane < kC ? ti : si[bs * kC + k];
      bitonic_merge32(v, i, lane);
      tv = v;
      ti = i;
    }
  }
}

// The drafting steps after the LM head, for bf16 storage with the gate
// precomputed by the conv launch: one CTA per row m = (b, t).
//   1. one round of asynchronous copies: the gate row and the strip lists
//      of rows m and m - 1 (the predecessors of row m are row m - 1's
//      candidates; the anchor at t = 0);
//   2. warps 0-3 merge row m (and write topv/topi/lse), warps 4-7 row m - 1;
//   3. the 32 embedding rows by asynchronous copies; the 16 x 16 scores;
//   4. the sequence's last row to finish (atomic ticket, zeroed by the conv
//      launch) walks it: all K x 16 rows' step quantities are computed in
//      parallel first, so the K serial steps are lookups.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    draft_tail_kernel(TopkPartials P, int nstrip,
                      const int* __restrict__ anchor,
                      const float* __restrict__ gate,
                      const T* __restrict__ e_in, const T* __restrict__ e_out,
                      int K, int V, int r, float Tt, float invT, uint64_t seed,
                      uint64_t cycle, float* __restrict__ topv,
                      int* __restrict__ topi, float* __restrict__ lse,
                      float* __restrict__ scores, int* __restrict__ slot,
                      int* __restrict__ draft, float* __restrict__ q,
                      unsigned* __restrict__ tickets,
                      int* __restrict__ walk_j, float* __restrict__ walk_q,
                      int* err) {
  extern __shared__ float4 smem4[];
  float* g_row = reinterpret_cast<float*>(smem4);    // [256]
  float* work = g_row + DFLASH_MAX_RANK;              // score tiles / walk
  T* st = reinterpret_cast<T*>(work + 2 * kC * (DFLASH_MAX_RANK + 4));
  float* lists = reinterpret_cast<float*>(st + 2 * kC * mma_ld(r));
  // words of one row's lists, rounded to 16 bytes for the copies
  const int lw = (nstrip * (2 * kC + 2) + 3) & ~3;
  __shared__ int s_tok[2][kC];
  __shared__ float s_topv[kC];
  __shared__ int s_ids[DFLASH_MAX_K * kC];
  __shared__ int s_arg[DFLASH_MAX_K * kC];
  __shared__ float s_S[kC * kC];
  __shared__ int s_prev[DFLASH_MAX_K], s_pick[DFLASH_MAX_K];
  __shared__ float s_mv[2][kWarps / 2][kC], s_mm[2][kWarps / 2],
      s_ms[2][kWarps / 2];
  __shared__ int s_mi[2][kWarps / 2][kC];
  __shared__ float s_th[2], s_sv[2][64], s_lm[2][32], s_bv[2][kC];
  __shared__ int s_wt[2][kWarps / 2], s_si[2][64], s_bi[2][kC];
  __shared__ int s_flag;
  const int m = blockIdx.x, b = m / K, t = m % K;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool vec = (r * (int)sizeof(T)) % 16 == 0;
  pdl_wait();  // the LM head's partials (and, before it, the gate)
  if (tid == 0) pdl_trigger();

  // ---- 1. gate row and strip lists ---------------------------------------
  const float* grow = gate + (size_t)m * r;
  if (r % 4 == 0) {
    for (int c = tid; c < r / 4; c += kThreads)
      cp_async16(g_row + 4 * c, grow + 4 * c, 16);
  } else {
    for (int k = tid; k < r; k += kThreads) g_row[k] = grow[k];
  }
  for (int j = 0; j < (t > 0 ? 2 : 1); ++j) {
    const size_t base = (size_t)(m - j) * nstrip;
    float* L = lists + j * lw;
    for (int c = tid; c < nstrip * kC / 4; c += kThreads) {
      cp_async16(L + 4 * c, P.v + base * kC + 4 * c, 16);
      cp_async16(L + nstrip * kC + 4 * c, P.i + base * kC + 4 * c, 16);
    }
    for (int c = tid; c < nstrip; c += kThreads) {
      cp_async4(L + 2 * nstrip * kC + c, P.m + base + c);
      cp_async4(L + 2 * nstrip * kC + nstrip + c, P.s + base + c);
    }
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- 2. merges: warps 0-3 row m, warps 4-7 row m - 1 ------------------
  // The row's top 16 come from few of its strip lists.  A bound th, the
  // 16th largest of 32 lane maxima of the lists' best entries (each lane
  // owns distinct strips, so at least 16 values of distinct columns reach
  // th), is at most the row's 16th value: no entry below it can make the
  // top 16.  The entries >= th of every list (a prefix of each sorted
  // list; usually a few dozen in all) are gathered and sorted once.  When
  // more than kCap survive (many equal values), the lists are folded
  // whole by bitonic merges instead.
  {
    constexpr int kG = kWarps / 2;  // warps per row
    constexpr int kGT = kG * 32;    // threads per row
    constexpr int kCap = 64;
    const int g = warp / kG, gw = warp % kG, lt = tid % kGT;
    const bool act = g == 0 || t > 0;  // row m - 1 exists
    const float* L = lists + g * lw;
    const float* sv = L;
    const int* si = reinterpret_cast<const int*>(L + nstrip * kC);
    const float* sm = L + 2 * nstrip * kC;
    const float* ss = sm + nstrip;
    float rm = -INFINITY, rs = 0.f;
    if (gw == 0) {
      // th: the lane maximum ranked 16th (values descending, lanes
      // ascending on equal values), by counting the maxima ranked ahead
      float mx = -INFINITY;
      if (act)
        for (int q = lane; q < nstrip; q += 32) mx = fmaxf(mx, sv[q * kC]);
      s_lm[g][lane] = mx;
      __syncwarp();
      int ahead = 0;
#pragma unroll 8
      for (int k = 0; k < 32; ++k) {
        const float o = s_lm[g][k];
        ahead += (o > mx || (o == mx && k < lane)) ? 1 : 0;
      }
      if (ahead == kC - 1) s_th[g] = mx;
    }
    if (act) fold_pairs_smem(sm, ss, nstrip, gw, kG, rm, rs);
    if (lane == 0) { s_mm[g][gw] = rm; s_ms[g][gw] = rs; }
    __syncthreads();
    // survivors of lists lt, lt + kGT, ... (nstrip <= 160 < 2 kGT)
    const float th = s_th[g];
    int c0 = 0, c1 = 0;
    if (act) {
      if (lt < nstrip)
        while (c0 < kC && sv[lt * kC + c0] >= th) ++c0;
      if (lt + kGT < nstrip)
        while (c1 < kC && sv[(lt + kGT) * kC + c1] >= th) ++c1;
    }
    const int cnt = c0 + c1;
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    if (lane == 31) s_wt[g][gw] = incl;
    __syncthreads();
    int pos = incl - cnt, total = 0;
#pragma unroll
    for (int w2 = 0; w2 < kG; ++w2) {
      const int x = s_wt[g][w2];
      if (w2 < gw) pos += x;
      total += x;
    }
    const bool direct = total <= kCap;
    if (act && direct) {
      for (int k = 0; k < c0; ++k, ++pos) {
        s_sv[g][pos] = sv[lt * kC + k];
        s_si[g][pos] = si[lt * kC + k];
      }
      for (int k = 0; k < c1; ++k, ++pos) {
        s_sv[g][pos] = sv[(lt + kGT) * kC + k];
        s_si[g][pos] = si[(lt + kGT) * kC + k];
      }
      for (int p2 = total + lt; p2 < kCap; p2 += kGT) {
        s_sv[g][p2] = -INFINITY;
        s_si[g][p2] = -1;
      }
    }
    float tv = -INFINITY;
    int ti = -1;
    if (act && !direct) {
      float rm2, rs2;  // the pairs are folded above
      fold_lists_smem(sv, si, sm, ss, nstrip, gw, kG, tv, ti, rm2, rs2);
    }
    if (lane < kC) { s_mv[g][gw][lane] = tv; s_mi[g][gw][lane] = ti; }
    __syncthreads();
    // the survivors' top 16: survivor lt goes to its rank (the number of
    // survivors ranked ahead of it, so every rank below 16 is taken once)
    if (act && direct) {
      if (lt < total) {
        const float v = s_sv[g][lt];
        const int i = s_si[g][lt];
        int ahead = 0;  // equal entries (padding: -inf, -1) in list order
        for (int k = 0; k < total; ++k) {
          const float ov = s_sv[g][k];
          const int oi = s_si[g][k];
          ahead += (ranks_ahead(ov, oi, v, i) ||
                    (ov == v && oi == i && k < lt)) ? 1 : 0;
        }
        if (ahead < kC) { s_bv[g][ahead] = v; s_bi[g][ahead] = i; }
      }
      if (total + lt < kC) {  // fewer than 16 survivors: padding
        s_bv[g][total + lt] = -INFINITY;
        s_bi[g][total + lt] = -1;
      }
    }
    __syncthreads();
    if (gw == 0) {
      if (act) {
        for (int w2 = 1; w2 < kG; ++w2)
          lse_combine(rm, rs, s_mm[g][w2], s_ms[g][w2], 1.f);
        if (direct) {  // placed by rank below
          tv = s_bv[g][lane & (kC - 1)];
          ti = s_bi[g][lane & (kC - 1)];
        } else {
          const int k = lane < kC ? lane : 31 - lane;
          for (int w2 = 1; w2 < kG; ++w2) {
            float v = lane < kC ? tv : s_mv[g][w2][k];
            int i = lane < kC ? ti : s_mi[g][w2][k];
            bitonic_merge32(v, i, lane);
            tv = v;
            ti = i;
          }
        }
      } else {  // t = 0: every predecessor is the anchor
        ti = anchor[b];
        if (ti < -1 || ti >= V) {
          if (lane == 0) raise_error(err, kErrBadIndex);
          ti = -1;
        }
      }
      // the lists come from the LM head; after a failed launch they may
      // hold anything, and the ids index the embedding tables below
      if (act && lane < kC && (ti < -1 || ti >= V)) {
        raise_error(err, kErrBadIndex);
        ti = -1;
        tv = -INFINITY;
      }
      if (g == 0) {
        if (lane < kC) {
          topv[(size_t)m * kC + lane] = tv;
          topi[(size_t)m * kC + lane] = ti;
          s_topv[lane] = tv;
          s_tok[1][lane] = ti;
        }
        if (lane == 0) lse[m] = rm + logf(rs);
      } else if (lane < kC) {
        s_tok[0][lane] = ti;
      }
    }
  }
  __syncthreads();

  // ---- 3. embedding rows and scores --------------------------------------
  // bf16 rows of whole 16-byte chunks: tensor-core scores; otherwise the
  // fp32 dot products
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  const bool tc_scores = kBf16 && r % 8 == 0;
  if (tc_scores) {
    if constexpr (kBf16)
      gather_rows_ld(st, mma_ld(r), s_tok, e_in, e_out, r);
  } else if (vec) {
    gather_rows(st, s_tok, e_in, e_out, r);
  }
  cp_async_wait_all();
  __syncthreads();
  if (tc_scores) {
    if constexpr (kBf16)
      score_row_mma(st, mma_ld(r), s_tok[0], s_tok[1], g_row, r, work,
                    s_topv, scores + (size_t)m * kC * kC, s_S);
  } else {
    score_row<kThreads>(st, vec, s_tok[0], s_tok[1], g_row, e_in, e_out, r,
                        work, s_topv, scores + (size_t)m * kC * kC, s_S);
  }
  __syncthreads();

  // ---- 3b. the walk's step from every predecessor slot of this row ------
  // Half-warp i takes predecessor slot i (the 16 scores S[i][.]): the
  // argmax at T = 0 (lowest slot on ties), else the weights
  // w = exp((S - max) / T), their running sums and total, and the slot the
  // walk's uniform of position t selects (the first running sum above
  // u * total; the last slot of positive weight if rounding leaves none;
  // -1 if no slot has weight), and q = w / total.  The uniform depends on
  // (b, t) only, so every predecessor's step is known here and the walk
  // itself only follows the chosen slots.
  {
    const int i = tid / kC, jj = tid % kC;
    const float v = s_S[tid];
    int jstar;
    float qv;
    if (Tt == 0.f) {
      float bv = v;
      int bi = jj;
#pragma unroll
      for (int o = 8; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o, 16);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o, 16);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      jstar = bi;
      qv = jj == bi ? 1.f : 0.f;
    } else {
      float mx = v;
#pragma unroll
      for (int o = 8; o; o >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o, 16));
      const float wv = (v != -INFINITY) ? __expf((v - mx) * invT) : 0.f;
      float cum = wv;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        const float n = __shfl_up_sync(0xffffffffu, cum, o, 16);
        if (jj >= o) cum += n;
      }
      const float tot = __shfl_sync(0xffffffffu, cum, 15, 16);
      const float u = philox_uniform(seed, b, t, kPurposeWalk, cycle);
      const int sh = lane & 16;  // this half-warp's lanes in the ballots
      const unsigned above =
          (__ballot_sync(0xffffffffu, cum > u * tot) >> sh) & 0xFFFFu;
      const unsigned live =
          (__ballot_sync(0xffffffffu, wv > 0.f) >> sh) & 0xFFFFu;
      jstar = above ? __ffs(above) - 1 : (live ? 31 - __clz(live) : -1);
      qv = tot > 0.f ? wv / tot : 0.f;
    }
    walk_q[(size_t)m * kC * kC + tid] = qv;
    if (jj == 0) walk_j[(size_t)m * kC + i] = jstar;
  }

  // ---- 4. the last row of sequence b walks it -----------------------------
  // (the barrier orders the CTA's score and walk-step stores before thread
  // 0's fence, which makes them visible before its ticket)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_flag = (atomicAdd(&tickets[b], 1u) == (unsigned)(K - 1));
  }
  __syncthreads();
  if (!s_flag) return;
  __threadfence();
  // every row's steps are known: follow the chosen slots from the anchor's
  // row (slot 0 of position 0), then write each position's q, slot, draft
  for (int i2 = tid; i2 < K * kC; i2 += kThreads) {
    s_arg[i2] = __ldcg(walk_j + (size_t)b * K * kC + i2);
    s_ids[i2] = __ldcg(topi + (size_t)b * K * kC + i2);
  }
  __syncthreads();
  if (tid == 0) {
    int prev = 0;
    for (int tt = 0; tt < K; ++tt) {
      int j = s_arg[tt * kC + prev];
      if (j < 0) {  // the walk reached a slot with no weight
        raise_error(err, kErrBadIndex);
        j = 0;
      }
      s_prev[tt] = prev;
      s_pick[tt] = j;
      prev = j;
    }
  }
  __syncthreads();
  for (int i2 = tid; i2 < K * kC; i2 += kThreads) {
    const int tt = i2 / kC, jj = i2 % kC;
    const size_t rr = (size_t)b * K + tt;
    q[rr * kC + jj] = __ldcg(walk_q + (rr * kC + s_prev[tt]) * kC + jj);
  }
  if (tid < K) {
    const int j = s_pick[tid];
    const int tok = s_ids[tid * kC + j];
    slot[b * K + tid] = j;
    draft[b * K + tid] = tok;
    if (tok < 0) raise_error(err, kErrBadIndex);
  }
}

}  // namespace

template <typename T>
cudaError_t launch_pair_score(const float* topv, const int* topi,
                              const int* anchor, const T* h, const T* w_gate,
                              const T* e_in, const T* e_out, int B, int K,
                              int H, int V, int r, float* scores, int* err,
                              cudaStream_t s) {
  const int M = B * K;
  // hidden slice per cluster rank, a multiple of 8 so 16-byte loads align
  const int hs = ((H + kCluster - 1) / kCluster + 7) & ~7;
  const size_t work = std::max(
      {work_floats(hs, std::is_same<T, __nv_bfloat16>::value),
       (size_t)kRows * 256, (size_t)2 * kC * (r + 4)});
  const size_t estage = (size_t)kRowsPerCta * 2 * kC * r * sizeof(T);
  const size_t smem =
      ((size_t)kRowsPerCta * 256 + work) * sizeof(float) + estage;
  cudaError_t e = cudaFuncSetAttribute(
      pair_score_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const int clusters = (M + kRows - 1) / kRows;
  pair_score_kernel<T><<<clusters * kCluster, kThreads, smem, s>>>(
      topv, topi, anchor, h, w_gate, e_in, e_out, B, K, H, V, r, hs,
      (int)work, scores, err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pair_score_gated(const float* topv, const int* topi,
                                    const int* anchor, const float* gate,
                                    const T* e_in, const T* e_out, int B,
                                    int K, int V, int r, float* scores,
                                    int* err, cudaStream_t s) {
  const size_t smem = (size_t)(DFLASH_MAX_RANK + 2 * kC * (DFLASH_MAX_RANK + 4)) *
                          sizeof(float) +
                      (size_t)2 * kC * r * sizeof(T);
  cudaError_t e = cudaFuncSetAttribute(
      pair_score_gated_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  pair_score_gated_kernel<T><<<B * K, kThreads, smem, s>>>(
      topv, topi, anchor, gate, e_in, e_out, K, V, r, scores, err);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_draft_tail(TopkPartials P, int nstrip, const int* anchor,
                              const float* gate, const T* e_in,
                              const T* e_out, int B, int K, int V, int r,
                              float T_, uint64_t seed, uint64_t cycle,
                              float* topv, int* topi, float* lse,
                              float* scores, int* slot, int* draft, float* q,
                              unsigned* tickets, int* walk_j, float* walk_q,
                              int* err, cudaStream_t s) {
  const size_t smem =
      (size_t)(DFLASH_MAX_RANK + 2 * kC * (DFLASH_MAX_RANK + 4)) *
          sizeof(float) +
      (size_t)2 * kC * mma_ld(r) * sizeof(T) +
      (size_t)2 * ((nstrip * (2 * kC + 2) + 3) & ~3) * sizeof(float);
  cudaError_t e = cudaFuncSetAttribute(
      draft_tail_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  const float invT = T_ > 0.f ? 1.f / T_ : 0.f;
  PdlLaunch L(dim3(B * K), dim3(kThreads), smem, s);
  return cudaLaunchKernelEx(&L.cfg, draft_tail_kernel<T>, P, nstrip, anchor,
                            gate, e_in, e_out, K, V, r, T_, invT, seed, cycle,
                            topv, topi, lse, scores, slot, draft, q, tickets,
                            walk_j, walk_q, err);
}

template cudaError_t launch_draft_tail<__nv_bfloat16>(
    TopkPartials, int, const int*, const float*, const __nv_bfloat16*,
    const __nv_bfloat16*, int, int, int, int, float, uint64_t, uint64_t,
    float*, int*, float*, float*, int*, int*, float*, unsigned*, int*,
    float*, int*, cudaStream_t);

template cudaError_t launch_pair_score_gated<float>(
    const float*, const int*, const int*, const float*, const float*,
    const float*, int, int, int, int, float*, int*, cudaStream_t);
template cudaError_t launch_pair_score_gated<__nv_bfloat16>(
    const float*, const int*, const int*, const float*, const __nv_bfloat16*,
    const __nv_bfloat16*, int, int, int, int, float*, int*, cudaStream_t);

template cudaError_t launch_pair_score<float>(const float*, const int*,
                                              const int*, const float*,
                                              const float*, const float*,
                                              const float*, int, int, int,
                                              int, int, float*, int*,
                                              cudaStream_t);
template cudaError_t launch_pair_score<__nv_bfloat16>(
    const float*, const int*, const int*, const __nv_bfloat16*,
    const __nv_bfloat16*, const __nv_bfloat16*, const __nv_bfloat16*, int,
    int, int, int, int, float*, int*, cudaStream_t);

}  // namespace dflash
