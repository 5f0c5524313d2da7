// Step a1 on the 5th-generation tensor cores: the two-tap dynamic depthwise
// convolution for bf16 storage, fused into the GEMM that computes its taps.
//
// "Suffix-decay convolution" (DFlash 2: Block diffusion, wearing a drafter's
// coat): each position is mixed with its predecessor through per-channel
// taps computed from the position, y_t = (W0 h_t) * h_t + (W1 h_t) * h_{t-1}
// with h_{-1} = 0.
//
// One CTA per (128-row tile, BC-channel tile), 192 threads.  The B operand
// of each stage stacks W0 rows [c0, c0+BC) over W1 rows [c0, c0+BC), so one
// tcgen05.mma M=128 N=2BC yields both taps of BC channels (TMEM columns
// 0..BC-1 = W0 h, BC..2BC-1 = W1 h).  The epilogue (warps 2-5, thread = row)
// reads both halves, loads h_t and h_{t-1} for the channels, applies the
// taps in fp32 and writes y rounded to bf16 — the A operand of the LM head.
//
// What bounds the launch is what each SM takes in (about 48 bytes per SM
// cycle): the whole h tile per channel tile.  So for 129 to 1023 rows the
// tiles are 64 channels wide and K is split over the two CTAs of a
// cluster (KS = 2): each takes in half of h and of W (512 KB per CTA at
// H = 2048 against 768 KB for 32-channel tiles over all of K, with the same
// number of CTAs), then each writes the partial sums of the other's half
// of the columns into the other's shared memory, arrives on its barrier,
// and adds what it received to its own half: CTA kh finishes channels
// [c0 + 32 kh, c0 + 32 kh + 32) (gate tiles: columns [64 kh, 64 kh + 64)).
//
// Optionally the same launch also computes the pair selector's context gate
// g_t = sigmoid(W_g h_t) ("A Lightweight Path Selector", DFlash 2: Keep
// Drafting Parallel), which reads the same h tiles: extra tiles after the
// channel tiles take 2BC gate rows each as their B operand (W_g rows
// [g0, g0+2BC) in two BC-row boxes) and write g in fp32.
#include "kernels.h"
#include "tc_ptx.cuh"

namespace dflash {
namespace {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int THREADS = 192;
// Limit of the drain waits after a give-up (copies and MMAs in flight
// complete in microseconds); the other waits take the launch's wait_ns.
constexpr uint64_t WAIT_NS = 2000000000ull;

// BC channels per CTA: the B operand is BC rows of W0 over BC rows of W1
// (MMA N = 2 BC).  32 for few rows (more CTAs), 128 when there are many
// rows (M >= 1024), where the N = 64 tiles leave the tensor cores idle.
template <int BC, int KS>
struct ConvCfg {
  static constexpr int STAGES = BC == 32 ? 8 : (BC == 64 ? 5 : 4);
  static constexpr int B_BYTES = 2 * BC * BK * 2;  // W0 part, then W1 part
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BC;
  // K split: the 64 partial sums per row received from the other CTA, as
  // 16 columns of 128 rows of float4 (one warp's remote store, and later
  // its load, of a column covers 512 contiguous bytes: a scattered layout,
  // a row's 64 sums together, made each remote store 32 separate pieces
  // and the send took 4k SM cycles)
  static constexpr int XBUF_BYTES = KS == 2 ? BM * 64 * 4 : 0;
};

template <int STAGES>
struct Bars {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull;
  uint64_t drain;
  uint64_t xbar;  // K split: the other CTA's 128 epilogue threads arrived
  uint32_t tmem_base;
  int abort;
};
template <int BC, int KS>
constexpr size_t conv_bars_bytes() {
  return (sizeof(Bars<ConvCfg<BC, KS>::STAGES>) + 15) & ~size_t(15);
}
template <int BC, int KS>
constexpr size_t conv_smem_bytes() {
  return 1024 +
         (size_t)ConvCfg<BC, KS>::STAGES * ConvCfg<BC, KS>::STAGE_BYTES +
         conv_bars_bytes<BC, KS>() + ConvCfg<BC, KS>::XBUF_BYTES;
}

__device__ __forceinline__ bool wait_timeout(uint64_t* bar, uint32_t parity) {
  int never = 0;
  return tc::mbar_wait_bounded(bar, parity, &never, WAIT_NS);
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(p[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

template <int BC, int KS>
__global__ void __launch_bounds__(THREADS, 1)
    conv_tc_kernel(const __grid_constant__ CUtensorMap map_h,
                   const __grid_constant__ CUtensorMap map_wc,
                   const __grid_constant__ CUtensorMap map_wg,
                   const __nv_bfloat16* __restrict__ h, int M, int K, int H,
                   int r, __nv_bfloat16* __restrict__ y,
                   float* __restrict__ gate, unsigned* __restrict__ tickets,
                   int ntickets, float* __restrict__ row_bound, int nbound,
                   int* err, uint64_t wait_ns, unsigned* __restrict__ tickets2,
                   int ntickets2) {
  using Cf = ConvCfg<BC, KS>;
  constexpr int STAGES = Cf::STAGES;
  constexpr int B_BYTES = Cf::B_BYTES;
  constexpr int STAGE_BYTES = Cf::STAGE_BYTES;
  constexpr uint32_t TMEM_COLS = Cf::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars<STAGES>* bars =
      reinterpret_cast<Bars<STAGES>*>(smem + STAGES * STAGE_BYTES);
  float* xbuf = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES +
                                         conv_bars_bytes<BC, KS>());
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // tiles [0, H/BC): conv channel tiles; after them: 2BC-row gate tiles.
  // K split: the two CTAs of a cluster (kh = 0, 1) share one tile.
  const int kh = KS == 2 ? (int)(blockIdx.x & 1) : 0;
  const int tile = KS == 2 ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int conv_tiles = (H + BC - 1) / BC;
  const bool is_gate = tile >= conv_tiles;
  const int c0 = is_gate ? (tile - conv_tiles) * 2 * BC : tile * BC;
  const int mtile = blockIdx.y;
  const int kblocks = (H + BK - 1) / BK;
  const int kbh = KS == 2 ? (kblocks + 1) / 2 : kblocks;
  const int kb_lo = kh == 0 ? 0 : kbh, kb_hi = kh == 0 ? kbh : kblocks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    tc::mbar_init(&bars->tfull, 1);
    tc::mbar_init(&bars->drain, 1);
    tc::mbar_init(&bars->xbar, 4 * 32);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  if constexpr (KS == 2)
    tc::cluster_sync();  // both CTAs' barriers exist before any arrival
  else
    __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;
  // everything above is on-chip set-up; h may come from the previous launch
  pdl_wait();
  if (threadIdx.x == 0) pdl_trigger();
  if (tickets && blockIdx.x == 0 && blockIdx.y == 0)
    for (int i = threadIdx.x; i < ntickets; i += THREADS) tickets[i] = 0u;
  if (tickets2) {  // a later launch's tickets (the cycle's verify)
    const int lin = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = lin * THREADS + threadIdx.x; i < ntickets2;
         i += gridDim.x * gridDim.y * THREADS)
      tickets2[i] = 0u;
  }
  if (row_bound) {  // the next launch's shared row bounds start unset
    const int lin = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = lin * THREADS + threadIdx.x; i < nbound;
         i += gridDim.x * gridDim.y * THREADS)
      row_bound[i] = -INFINITY;
  }

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!tc::mbar_wait_bounded(&bars->empty[stage], phase ^ 1, abort,
                                   wait_ns))
          break;
        tc::mbar_arrive_expect_tx(&bars->full[stage], STAGE_BYTES);
        uint8_t* b = sb + stage * B_BYTES;
        tc::tma_load_2d(sa + stage * A_BYTES, &map_h, &bars->full[stage],
                        kb * BK, mtile * BM);
        if (is_gate) {
          tc::tma_load_2d(b, &map_wg, &bars->full[stage], kb * BK, c0);
          tc::tma_load_2d(b + BC * BK * 2, &map_wg, &bars->full[stage],
                          kb * BK, c0 + BC);
        } else {
          tc::tma_load_2d(b, &map_wc, &bars->full[stage], kb * BK, c0);
          tc::tma_load_2d(b + BC * BK * 2, &map_wc, &bars->full[stage],
                          kb * BK, H + c0);
        }
        issued |= 1u << stage;
        last_par = (last_par & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      for (int s = 0; s < STAGES; ++s)
        if ((issued >> s) & 1)
          wait_timeout(&bars->full[s], (last_par >> s) & 1);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(BM, 2 * BC);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int kb = kb_lo; kb < kb_hi; ++kb) {
        if (!tc::mbar_wait_bounded(&bars->full[stage], phase, abort,
                                   wait_ns)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a0 = tc::smem_u32(sa + stage * A_BYTES);
        const uint32_t b0 = tc::smem_u32(sb + stage * B_BYTES);
#pragma unroll
        for (int k = 0; k < BK / 16; ++k)
          tc::mma_bf16(tmem, tc::sdesc_k_sw128(a0 + k * 32),
                       tc::sdesc_k_sw128(b0 + k * 32), idesc,
                       (kb != kb_lo) || (k != 0));
        tc::mma_commit(&bars->empty[stage]);
        if (++stage == STAGES) { stage = 0; phase ^= 1; }
      }
      if (ok) tc::mma_commit(&bars->tfull);
      tc::mma_commit(&bars->drain);
      wait_timeout(&bars->drain, 0);
    }
  } else {
    const int q = warp & 3;
    const int row = q * 32 + lane;  // within the tile (TMEM lane)
    const int m = mtile * BM + row;
    const bool has_prev = (m % K) != 0;
    // conv tiles: the channels this CTA writes (all BC, or its 32 of the
    // K-split tile's 64)
    const int cme = KS == 2 ? c0 + 32 * kh : c0;
    // h_t and h_{t-1} of its first 32 channels, loaded while the MMAs run
    uint4 hc0[4], hp0[4];
    const bool pre = !is_gate && m < M;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      hc0[g] = make_uint4(0u, 0u, 0u, 0u);
      hp0[g] = hc0[g];
      if (pre && cme + g * 8 < H) {
        const __nv_bfloat16* hr = h + (size_t)m * H + cme + g * 8;
        hc0[g] = *reinterpret_cast<const uint4*>(hr);
        if (has_prev) hp0[g] = *reinterpret_cast<const uint4*>(hr - H);
      }
    }
    // gate rows [g0, g0 + 32) of this row from 32 pre-activations.  The
    // fast reciprocal divide (within 2 ulp; 0 for divisors past 2^126, the
    // sigmoid's limit there): the correctly rounded divide's per-value
    // latency chain, 64 values per thread in a warp per scheduler, made the
    // gate tiles' epilogue 9k SM cycles and them the launch's last CTAs
    auto write_gate = [&](int g0, const float (&z)[32]) {
      float* gr = gate + (size_t)m * r + g0;
      float g[32];
#pragma unroll
      for (int j = 0; j < 32; ++j)
        g[j] = __fdividef(1.f, 1.f + __expf(-z[j]));
      if (r % 4 == 0 && g0 + 32 <= r) {
#pragma unroll
        for (int j = 0; j < 32; j += 4)
          *reinterpret_cast<float4*>(gr + j) =
              make_float4(g[j], g[j + 1], g[j + 2], g[j + 3]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (g0 + j < r) gr[j] = g[j];
      }
    };
    // y of channels [cc, cc + 32) of this row from their two taps
    auto write_conv = [&](int cc, const float (&w0)[32],
                          const float (&w1)[32], bool first) {
      const __nv_bfloat16* hr = h + (size_t)m * H + cc;
      __nv_bfloat16* yr = y + (size_t)m * H + cc;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        if (cc + g * 8 >= H) break;
        float hc[8], hp[8];
        bf16x8_to_f32(first ? hc0[g]
                            : *reinterpret_cast<const uint4*>(hr + g * 8),
                      hc);
        if (has_prev)
          bf16x8_to_f32(
              first ? hp0[g]
                    : *reinterpret_cast<const uint4*>(hr - H + g * 8),
              hp);
        uint4 out;
        __nv_bfloat162* o = reinterpret_cast<__nv_bfloat162*>(&out);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int j = g * 8 + 2 * i;
          const float y0 =
              w0[j] * hc[2 * i] + (has_prev ? w1[j] * hp[2 * i] : 0.f);
          const float y1 = w0[j + 1] * hc[2 * i + 1] +
                           (has_prev ? w1[j + 1] * hp[2 * i + 1] : 0.f);
          o[i] = __floats2bfloat162_rn(y0, y1);
        }
        *reinterpret_cast<uint4*>(yr + g * 8) = out;
      }
    };
    const bool got = tc::mbar_wait_bounded(&bars->tfull, 0, abort, wait_ns);
    if (__all_sync(0xffffffffu, got)) {
      tc::fence_after_sync();
      const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16);
      if constexpr (KS == 2) {
        // columns of the other CTA's half (first and second 32) and of
        // this CTA's half
        const int o0 = is_gate ? 64 * (1 - kh) : 32 * (1 - kh);
        const int o1 = is_gate ? o0 + 32 : o0 + 64;
        const int m0 = is_gate ? 64 * kh : 32 * kh;
        const int m1 = is_gate ? m0 + 32 : m0 + 64;
        float w0[32], w1[32];
        tc::tmem_ld_x32(tb + o0, w0);
        tc::tmem_ld_x32(tb + o1, w1);
        const uint32_t peer = (uint32_t)(kh ^ 1);
        const uint32_t xr =
            tc::mapa_shared(tc::smem_u32(xbuf) + row * 16, peer);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          tc::st_cluster_v4(xr + j * (BM * 16), w0[4 * j], w0[4 * j + 1],
                            w0[4 * j + 2], w0[4 * j + 3]);
          tc::st_cluster_v4(xr + (8 + j) * (BM * 16), w1[4 * j],
                            w1[4 * j + 1], w1[4 * j + 2], w1[4 * j + 3]);
        }
        tc::mbar_arrive_cluster(
            tc::mapa_shared(tc::smem_u32(&bars->xbar), peer));
        tc::tmem_ld_x32(tb + m0, w0);
        tc::tmem_ld_x32(tb + m1, w1);
        const bool xok =
            tc::mbar_wait_cluster_bounded(&bars->xbar, 0, abort, wait_ns);
        if (__all_sync(0xffffffffu, xok)) {
          const float4* xs = reinterpret_cast<const float4*>(xbuf) + row;
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float4 a = xs[j * BM], b = xs[(8 + j) * BM];
            w0[4 * j] += a.x;
            w0[4 * j + 1] += a.y;
            w0[4 * j + 2] += a.z;
            w0[4 * j + 3] += a.w;
            w1[4 * j] += b.x;
            w1[4 * j + 1] += b.y;
            w1[4 * j + 2] += b.z;
            w1[4 * j + 3] += b.w;
          }
          if (m < M) {
            if (is_gate) {
              write_gate(c0 + m0, w0);
              write_gate(c0 + m0 + 32, w1);
            } else {
              write_conv(cme, w0, w1, true);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int cg = 0; cg < BC / 32; ++cg) {
          float w0[32], w1[32];
          tc::tmem_ld_x32(tb + cg * 32, w0);
          tc::tmem_ld_x32(tb + BC + cg * 32, w1);
          if (m >= M) continue;
          if (is_gate) {
            // columns [0, BC) are z of gate rows c0 .., [BC, 2 BC) of
            // c0 + BC ..
            write_gate(c0 + cg * 32, w0);
            write_gate(c0 + BC + cg * 32, w1);
          } else {
            write_conv(c0 + cg * 32, w0, w1, cg == 0);
          }
        }
      }
    } else {
      *abort = 1;
    }
  }

  tc::fence_before_sync();
  // K split: neither CTA leaves while the other may still write into its
  // shared memory or arrive on its barrier
  if constexpr (KS == 2)
    tc::cluster_sync();
  else
    __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars->abort) raise_error(err, kErrTimeout);
}

}  // namespace

// Channels per tile: 128 for many rows (M >= 1024, where narrower tiles
// leave the tensor cores idle); 64 with K split over a cluster of two CTAs
// for more than one row tile (at one tile, mostly rows past M, the
// exchange costs more than the halved intake saves) when K has at least
// two 64-wide blocks; else 32.
int conv_tc_bc(int M, int H) {
  return M >= 1024 ? 128 : (M > BM && H >= 2 * BK ? 64 : 32);
}

namespace {
template <int BC, int KS>
cudaError_t launch_conv_bc(const CUtensorMap& map_h, const CUtensorMap& map_wc,
                           const CUtensorMap* map_wg, const __nv_bfloat16* h,
                           int B, int K, int H, int r, __nv_bfloat16* y,
                           float* gate, unsigned* tickets, float* row_bound,
                           int nbound, int* err, cudaStream_t s,
                           uint64_t wait_ns, unsigned* tickets2,
                           int ntickets2) {
  const int M = B * K;
  cudaError_t e = cudaFuncSetAttribute(
      conv_tc_kernel<BC, KS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)conv_smem_bytes<BC, KS>());
  if (e != cudaSuccess) return e;
  const int gate_tiles = map_wg ? (r + 2 * BC - 1) / (2 * BC) : 0;
  const dim3 grid(((H + BC - 1) / BC + gate_tiles) * KS, (M + BM - 1) / BM);
  PdlLaunch L(grid, dim3(THREADS), conv_smem_bytes<BC, KS>(), s,
              KS == 2 ? 2 : 0);
  return cudaLaunchKernelEx(&L.cfg, conv_tc_kernel<BC, KS>, map_h, map_wc,
                            map_wg ? *map_wg : map_wc, h, M, K, H, r, y, gate,
                            tickets, B, row_bound, nbound, err, wait_ns,
                            tickets2, ntickets2);
}
}  // namespace

cudaError_t launch_conv_tc(const CUtensorMap& map_h, const CUtensorMap& map_wc,
                           const CUtensorMap* map_wg, const __nv_bfloat16* h,
                           int B, int K, int H, int r, __nv_bfloat16* y,
                           float* gate, unsigned* tickets, float* row_bound,
                           int nbound, int* err, cudaStream_t s,
                           uint64_t wait_ns, unsigned* tickets2,
                           int ntickets2) {
  switch (conv_tc_bc(B * K, H)) {
    case 128:
      return launch_conv_bc<128, 1>(map_h, map_wc, map_wg, h, B, K, H, r, y,
                                    gate, tickets, row_bound, nbound, err, s,
                                    wait_ns, tickets2, ntickets2);
    case 64:
      return launch_conv_bc<64, 2>(map_h, map_wc, map_wg, h, B, K, H, r, y,
                                   gate, tickets, row_bound, nbound, err, s,
                                   wait_ns, tickets2, ntickets2);
    default:
      return launch_conv_bc<32, 1>(map_h, map_wc, map_wg, h, B, K, H, r, y,
                                   gate, tickets, row_bound, nbound, err, s,
                                   wait_ns, tickets2, ntickets2);
  }
}

}  // namespace dflash
