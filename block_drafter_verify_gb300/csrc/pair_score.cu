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
// tables here.  work holds two fp32 tiles of 16 rows; thread tid writes
// S[tid / 16][tid % 16].
template <typename T>
__device__ __forceinline__ void score_row(
    const T* st, bool vec, const int* pred, const int* cand,
    const float* g_row, const T* __restrict__ e_in,
    const T* __restrict__ e_out, int r, float* work,
    const float* __restrict__ topv_row, float* __restrict__ out) {
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
    for (int rowi = warp; rowi < 2 * kC; rowi += kWarps) {
      const bool outt = rowi >= kC;
      float* dst = (outt ? eout_s : ein_s) + (rowi % kC) * rs;
      const T* srow = st + (size_t)rowi * r;
      for (int ch = lane; ch < cpr; ch += 32) {
        float f[epc > 4 ? 8 : 4];
        Vec16<T>::to_f32(*reinterpret_cast<const uint4*>(srow + ch * epc), f);
#pragma unroll
        for (int e = 0; e < epc; ++e)
          dst[ch * epc + e] = outt ? f[e] * g_row[ch * epc + e] : f[e];
      }
    }
  } else {
    for (int i = tid; i < kC * r; i += kThreads) {
      const int row = i / r, k = i % r;
      const int a = pred[row], c = cand[row];
      ein_s[row * rs + k] = a >= 0 ? to_f32(e_in[(size_t)a * r + k]) : 0.f;
      eout_s[row * rs + k] =
          c >= 0 ? to_f32(e_out[(size_t)c * r + k]) * g_row[k] : 0.f;
    }
  }
  __syncthreads();
  const int i = tid / kC, jj = tid % kC;
  float sc = 0.f;
  const float* ea = ein_s + i * rs;
  const float* eb = eout_s + jj * rs;
  int k = 0;
  if (r4) {
    for (; k < r; k += 4) {
      const float4 a4 = *reinterpret_cast<const float4*>(ea + k);
      const float4 b4 = *reinterpret_cast<const float4*>(eb + k);
      sc = fmaf(a4.x, b4.x, sc);
      sc = fmaf(a4.y, b4.y, sc);
      sc = fmaf(a4.z, b4.z, sc);
      sc = fmaf(a4.w, b4.w, sc);
    }
  }
  for (; k < r; ++k) sc = fmaf(ea[k], eb[k], sc);
  const bool valid = pred[i] >= 0 && cand[jj] >= 0;
  out[tid] = valid ? topv_row[jj] + sc : -INFINITY;
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
template <typename T>
__device__ __forceinline__ void gather_rows(T* st, const int (*tok)[kC],
                                            const T* __restrict__ e_in,
                                            const T* __restrict__ e_out,
                                            int r) {
  const int cpr = r * (int)sizeof(T) / 16;  // 16-byte chunks per row
  for (int idx = threadIdx.x; idx < 2 * kC * cpr; idx += kThreads) {
    const int rowi = idx / cpr, ch = idx % cpr;  // rowi = tab * 16 + i
    const int tab = rowi / kC;
    const int t = tok[tab][rowi % kC];
    const T* src = (tab == 0 ? e_in : e_out) + (size_t)max(t, 0) * r;
    cp_async16(st + (size_t)rowi * r + ch * (16 / sizeof(T)),
               reinterpret_cast<const char*>(src) + ch * 16, t >= 0 ? 16 : 0);
  }
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
    score_row(estage + (size_t)j * 2 * kC * r, vec, s_tok[j][0], s_tok[j][1],
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
  score_row(st, vec, s_tok[0], s_tok[1], g_row, e_in, e_out, r, work,
            topv + (size_t)m * kC, scores + (size_t)m * kC * kC);
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
