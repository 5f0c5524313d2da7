// Step a2 on the 5th-generation tensor cores: drafter LM head
// U = y W_lm^T (bf16 x bf16 -> fp32) with an epilogue that keeps, per row,
// an online logsumexp and the 16 largest logits, so U never reaches HBM.
// The same kernel also runs with 8-bit operands: E4M3 codes of y and W_lm
// with one fp32 scale per row each (kind::f8f6f4; a stage then holds 128
// codes of every row instead of 64 bf16, the same bytes); the epilogue
// multiplies each logit by its column's scale and applies the row's scale
// in the exponent and to the outputs.
//
// "Sixteen candidates per position" (DFlash 2: Block diffusion, wearing a
// drafter's coat) and "A Lightweight Path Selector" (DFlash 2: Keep Drafting
// Parallel): U_t is the drafter's own logit; 16 candidates are kept per slot.
//
// Persistent kernel, one CTA per SM, 64 + 32 * EPI_WARPS threads:
//   warp 0      TMA producer: y tile [128 rows x 128 bytes] and W tile per
//               stage, 128-byte swizzle;
//   warp 1      MMA issuer (one thread): tcgen05.mma N=256 into one of two
//               TMEM accumulators (2 x 256 fp32 columns);
//   warps 2..   epilogue: thread = one row (TMEM lane), reads 32 columns at
//               a time with tcgen05.ld, folds them into (max, sum exp) and a
//               register-resident sorted top-16, while the MMA fills the
//               other accumulator.  Four warps, or eight for the 8-bit pair
//               variant (two per lane quarter, half of the columns each,
//               their lists merged at the end).
// Two variants:
//   single  (one row tile, M <= 128): W tile [256 rows] per stage, 4
//           stages, M=128 MMAs (cta_group::1);
//   pair    (two or more row tiles): a cluster of two CTAs computes the rows
//           of two row tiles against one W tile with M=256 MMAs
//           (cta_group::2).  Each CTA loads its own y tile and one half
//           [128 rows] of the W tile, so W crosses L2 -> SM once per pair
//           instead of once per row tile and a stage is 32 KB: 6 stages
//           (5 for the 8-bit variant, whose epilogue needs more room).
//           The even CTA issues the MMAs; its full barriers count both
//           CTAs' copies, and its commits arrive on both CTAs' barriers.
// Unit u (a CTA, or a pair) owns row group (u mod row_groups) and the vocab
// tiles strip, strip + strips, ... (strip = u / row_groups), so the units
// that share a vocab tile run it at the same time and W_lm is read from HBM
// about once.  Each CTA writes one top-16 / (max, sum) partial per row;
// topk_merge (or the draft tail) folds them.
// Candidate insertions dominate the epilogue.  They are pruned twice: in a
// unit's first tile, where the list is empty, by the 16th largest of 32
// column-group maxima (at least 16 of the tile's values reach it), and in
// every tile by the running maxima that 16 (32 for at most 8 rows) units
// of the row group publish in the workspace (values of distinct columns,
// so a value below 16 of them cannot make the row's top 16).
// Every wait is time-bounded; on a timeout the CTA stops issuing, drains
// its copies and MMAs, frees TMEM, flags the error word and exits.
#include <algorithm>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace dflash {
namespace {

constexpr int BM = 128, BN = 256;
constexpr int ROW_BYTES = 128;  // bytes of each operand row per stage
constexpr int A_BYTES = BM * ROW_BYTES;  // 16 KB
constexpr uint32_t TMEM_COLS = 2 * BN;
// 2 s: far beyond any real wait.  The limit of the drain waits after a
// give-up, and of every wait of the CTA-pair variant; the single-CTA
// variant's other waits take the launch's wait_ns.
constexpr uint64_t WAIT_NS = 2000000000ull;
constexpr float LOG2E = 1.4426950408889634f;

// EPI_WARPS epilogue warps: 4 (thread = row, all BN columns of a tile),
// or 8 for CTA pairs with 8-bit operands, whose W tiles arrive twice as
// fast: then two warps share each TMEM lane quarter and take half of the
// tile's columns each, and the two halves' lists are merged at the end.
template <bool kPair, bool kFp8>
struct Cfg {
  static constexpr int EPI_WARPS = kPair && kFp8 ? 8 : 4;
  static constexpr int HALVES = EPI_WARPS / 4;
  static constexpr int THREADS = 64 + 32 * EPI_WARPS;
  static constexpr int STAGES = !kPair ? 4 : (EPI_WARPS == 8 ? 5 : 6);
  static constexpr int B_ROWS = kPair ? BN / 2 : BN;  // W rows per CTA
  static constexpr int B_BYTES = B_ROWS * ROW_BYTES;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int CTAS = kPair ? 2 : 1;
};
// Elements of K per stage and per MMA: 64 and 16 for bf16, 128 and 32 for
// E4M3; either way each MMA step advances 32 bytes along the row.
template <bool kFp8>
struct Elem {
  static constexpr int BK = kFp8 ? 128 : 64;
  static constexpr int MMA_K = kFp8 ? 32 : 16;
};

template <int STAGES>
struct Bars {
  uint64_t full[STAGES];   // pair: only the even CTA's are used
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];      // pair: only the even CTA's are used
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr int XS_STRIDE = 33;  // padded row of the per-thread chunk stage
// Shared memory after the stages and barriers: the per-thread chunk
// stage, (8-bit operands) each epilogue warp's copy of its columns'
// scales for the current tile, and (two halves) the second half's lists
// for the final merge (16 values, 16 ids, max, sum per row).
template <bool kPair, bool kFp8>
struct Smem {
  using C = Cfg<kPair, kFp8>;
  static constexpr size_t XS = (size_t)C::EPI_WARPS * 32 * XS_STRIDE * 4;
  static constexpr size_t WS = kFp8 ? (size_t)4 * BN * 4 : 0;
  static constexpr size_t MERGE = C::HALVES == 2 ? (size_t)BM * 34 * 4 : 0;
  static constexpr size_t BARS = (sizeof(Bars<C::STAGES>) + 15) & ~size_t(15);
  static constexpr size_t TOTAL =
      1024 + (size_t)C::STAGES * C::STAGE_BYTES + BARS + XS + WS + MERGE;
};
template <bool kPair, bool kFp8>
constexpr size_t smem_bytes() {
  return Smem<kPair, kFp8>::TOTAL;
}

__device__ __forceinline__ bool wait_timeout(uint64_t* bar, uint32_t parity) {
  int never = 0;
  return tc::mbar_wait_bounded(bar, parity, &never, WAIT_NS);
}

// Insert xv (> tv[15], id larger than every held id) into the sorted list:
// entry p becomes max(tv[p], min(xv, tv[p-1])), and the ids follow the
// comparisons of xv with the old entries (an equal value keeps its place).
__device__ __forceinline__ void topk_insert(float (&tv)[kC], int (&ti)[kC],
                                            float xv, int xi) {
  bool c[kC];
#pragma unroll
  for (int p = 0; p < kC; ++p) c[p] = xv > tv[p];
#pragma unroll
  for (int p = kC - 1; p >= 1; --p) {
    ti[p] = c[p - 1] ? ti[p - 1] : (c[p] ? xi : ti[p]);
    tv[p] = fmaxf(tv[p], fminf(xv, tv[p - 1]));
  }
  ti[0] = c[0] ? xi : ti[0];
  tv[0] = fmaxf(tv[0], xv);
}

// Order of the lists: value descending, then id ascending (for merging
// lists whose ids interleave).
__device__ __forceinline__ bool topk_before(float xv, int xi, float tv,
                                            int ti) {
  return xv > tv || (xv == tv && xi < ti);
}

// The 16th largest of 32 values: both halves sorted descending by bitonic
// networks of min/max steps, then max(a[i], b[15-i]) is the top 16 of the
// union (in some order), whose minimum is returned.
__device__ __forceinline__ float kth16_of_32(float (&g)[32]) {
#pragma unroll
  for (int h = 0; h < 32; h += 16)
#pragma unroll
    for (int k = 2; k <= 16; k <<= 1)
#pragma unroll
      for (int j = k >> 1; j > 0; j >>= 1)
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int l = i ^ j;
          if (l > i) {
            const float a = g[h + i], b = g[h + l];
            const bool desc = (i & k) == 0;
            g[h + i] = desc ? fmaxf(a, b) : fminf(a, b);
            g[h + l] = desc ? fminf(a, b) : fmaxf(a, b);
          }
        }
  float lo = INFINITY;
#pragma unroll
  for (int i = 0; i < 16; ++i) lo = fminf(lo, fmaxf(g[i], g[31 - i]));
  return lo;
}

// Columns at or beyond V take no part in the row.
__device__ __forceinline__ void mask_tail(float (&x)[32], int col0, int V) {
  if (col0 + 32 > V) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (col0 + i >= V) x[i] = -INFINITY;
  }
}

// Fold 32 logits of this thread's row into its running (max, sum exp), the
// exponent taken as 2^(l2e * x) (l2e = log2 e times the row's positive
// scale).  Returns the chunk maximum.
// With gmax, also the maxima of the chunk's kG column groups (kG = 8:
// columns {i, i+8, .., i+24}; kG = 4: {i, i+4, .., i+28}).
template <int kG = 0>
__device__ __forceinline__ float fold_chunk(const float (&x)[32], float l2e,
                                            float& run_m, float& run_s,
                                            float* gmax = nullptr) {
  float t[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) t[i] = fmaxf(x[i], x[i + 16]);
#pragma unroll
  for (int w = 8; w >= 1; w >>= 1) {
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
    if (kG == w) {
#pragma unroll
      for (int i = 0; i < w; ++i) gmax[i] = t[i];
    }
  }
  const float cm = t[0];
  if (cm > run_m) {
    run_s *= tc::ex2_approx((run_m - cm) * l2e);
    run_m = cm;
  }
  // a warp whose columns so far are all beyond V (the second half of a
  // last tile) still has run_m = -inf: its terms are exactly 0, not
  // 2^(-inf + inf)
  const float nb = run_m == -INFINITY ? 0.f : -run_m * l2e;
  float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int i = 0; i < 32; ++i) s[i & 3] += tc::ex2_approx(fmaf(x[i], l2e, nb));
  run_s += (s[0] + s[1]) + (s[2] + s[3]);
  return cm;
}

// Bitmask of the columns that beat the row's current 16th value thr and
// reach lo (their values are staged in xs); cm is the chunk maximum.
__device__ __forceinline__ unsigned chunk_candidates(const float (&x)[32],
                                                     float cm, float thr,
                                                     float lo, float* xs) {
  unsigned mask = 0;
  if (cm > thr && cm >= lo) {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      mask |= (x[i] > thr && x[i] >= lo ? 1u : 0u) << i;
      xs[i] = x[i];
    }
  }
  return mask;
}

template <bool kPair, bool kFp8>
__global__ void __launch_bounds__(Cfg<kPair, kFp8>::THREADS, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap map_y,
                     const __grid_constant__ CUtensorMap map_w, int M, int H,
                     int V, int row_groups, int strips, TopkPartials P,
                     const float* __restrict__ y_scale,
                     const float* __restrict__ w_scale,
                     float* __restrict__ row_bound, int* err,
                     uint64_t wait_ns) {
  using C = Cfg<kPair, kFp8>;
  // the launch's limit for the work waits; CTA pairs keep the long one (an
  // early give-up there could leave one CTA's last copy in flight, counted
  // on the other CTA's barrier, when the pair exits)
  const uint64_t lim = kPair ? WAIT_NS : wait_ns;
  using SM = Smem<kPair, kFp8>;
  constexpr int STAGES = C::STAGES;
  constexpr int BK = Elem<kFp8>::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sa = smem;
  uint8_t* sb = smem + STAGES * A_BYTES;
  Bars<STAGES>* bars =
      reinterpret_cast<Bars<STAGES>*>(smem + STAGES * C::STAGE_BYTES);
  float* xs_all =
      reinterpret_cast<float*>(smem + STAGES * C::STAGE_BYTES + SM::BARS);
  float* ws_all = xs_all + SM::XS / 4;     // 8-bit operands only
  float* mg_all = ws_all + SM::WS / 4;     // two halves only
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a pair is a cluster of two consecutive blocks; rank 0 leads
  const int rank = kPair ? (int)(blockIdx.x & 1) : 0;
  const bool leader = rank == 0;
  const int unit = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int group = unit % row_groups, strip = unit / row_groups;
  const int mtile = kPair ? 2 * group + rank : group;
  const int vtiles = (V + BN - 1) / BN;
  const int kblocks = (H + BK - 1) / BK;
  const int my_tiles =
      strip < vtiles ? (vtiles - strip + strips - 1) / strips : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&bars->full[s], 1);
      tc::mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars->tfull[b], 1);
      tc::mbar_init(&bars->tempty[b], C::EPI_WARPS * C::CTAS);
    }
    tc::mbar_init(&bars->drain, 1);
    bars->abort = 0;
    tc::fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tc::tmem_alloc_pair(&bars->tmem_base, TMEM_COLS);
      tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(&bars->tmem_base, TMEM_COLS);
      tc::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_map(&map_y);
    tc::tma_prefetch_map(&map_w);
  }
  tc::fence_before_sync();
  if constexpr (kPair)
    tc::cluster_sync();  // both CTAs' barriers exist before any copy lands
  else
    __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort = &bars->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // full barriers of the MMA-issuing CTA, as cluster addresses
      const uint32_t full0 =
          kPair ? tc::mapa_shared(tc::smem_u32(&bars->full[0]), 0)
                : tc::smem_u32(&bars->full[0]);
      int stage = 0;
      uint32_t phase = 0, issued = 0, last_par = 0;
      bool ok = true;
      // The W tiles of the first stages go out before waiting for the
      // launch that writes y (W_lm is an input no launch writes); each
      // stage's full barrier already expects both of its tiles.
      const int pre = min(STAGES, my_tiles * kblocks);
      auto load_w = [&](int j, int s) {
        const int vt = strip + (j / kblocks) * strips, kb = j % kblocks;
        uint8_t* b_dst = sb + s * C::B_BYTES;
        if constexpr (kPair) {
          if (leader)
            tc::mbar_arrive_expect_tx(&bars->full[s], 2 * C::STAGE_BYTES);
          tc::tma_load_2d_pair(b_dst, &map_w, full0 + s * 8, kb * BK,
                               vt * BN + rank * C::B_ROWS);
        } else {
          tc::mbar_arrive_expect_tx(&bars->full[s], C::STAGE_BYTES);
          tc::tma_load_2d(b_dst, &map_w, &bars->full[s], kb * BK, vt * BN);
        }
      };
      for (int j = 0; j < pre; ++j) load_w(j, j);
      pdl_wait();
      pdl_trigger();
      int j = 0;
      for (int it = 0; it < my_tiles && ok; ++it) {
        for (int kb = 0; kb < kblocks; ++kb, ++j) {
          if (!tc::mbar_wait_bounded(&bars->empty[stage], phase ^ 1, abort,
                                     lim)) {
            ok = false;
            break;
          }
          uint8_t* a_dst = sa + stage * A_BYTES;
          if (j >= pre) load_w(j, stage);
          if constexpr (kPair) {
            tc::tma_load_2d_pair(a_dst, &map_y, full0 + stage * 8, kb * BK,
                                 mtile * BM);
          } else {
            tc::tma_load_2d(a_dst, &map_y, &bars->full[stage], kb * BK,
                            mtile * BM);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
      }
      // leave no copy in flight (a pair's full barriers count both CTAs'
      // copies; the closing cluster barrier keeps the odd CTA until then)
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if ((issued >> s) & 1)
            wait_timeout(&bars->full[s], (last_par >> s) & 1);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA
    if (lane == 0 && leader) {
      constexpr uint32_t idesc =
          kFp8 ? tc::idesc_e4m3_f32(BM * C::CTAS, BN)
               : tc::idesc_bf16_f32(BM * C::CTAS, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; it < my_tiles && ok; ++it) {
        const int b = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!tc::mbar_wait_bounded(&bars->tempty[b], aph ^ 1, abort, lim)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t d = tmem + b * BN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!tc::mbar_wait_bounded(&bars->full[stage], phase, abort,
                                     lim)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a0 = tc::smem_u32(sa + stage * A_BYTES);
          const uint32_t b0 = tc::smem_u32(sb + stage * C::B_BYTES);
#pragma unroll
          for (int k = 0; k < BK / Elem<kFp8>::MMA_K; ++k) {
            const uint64_t ad = tc::sdesc_k_sw128(a0 + k * 32);
            const uint64_t bd = tc::sdesc_k_sw128(b0 + k * 32);
            if constexpr (kPair && kFp8)
              tc::mma_e4m3_pair(d, ad, bd, idesc, (kb | k) != 0);
            else if constexpr (kPair)
              tc::mma_bf16_pair(d, ad, bd, idesc, (kb | k) != 0);
            else if constexpr (kFp8)
              tc::mma_e4m3(d, ad, bd, idesc, (kb | k) != 0);
            else
              tc::mma_bf16(d, ad, bd, idesc, (kb | k) != 0);
          }
          if constexpr (kPair)
            tc::mma_commit_pair_mc(&bars->empty[stage], 3);
          else
            tc::mma_commit(&bars->empty[stage]);
          if (++stage == STAGES) { stage = 0; phase ^= 1; }
        }
        if (ok) {
          if constexpr (kPair)
            tc::mma_commit_pair_mc(&bars->tfull[b], 3);
          else
            tc::mma_commit(&bars->tfull[b]);
        }
      }
      // every MMA issued completes before TMEM is released
      if constexpr (kPair)
        tc::mma_commit_pair_mc(&bars->drain, 1);
      else
        tc::mma_commit(&bars->drain);
      wait_timeout(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int CH = BN / 32 / C::HALVES;  // 32-column chunks per warp
    const int ew = warp - 2;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int half = ew >> 2;  // which part of each tile's columns
    const int m = mtile * BM + q * 32 + lane;
    float* xs = xs_all + (ew * 32 + lane) * XS_STRIDE;
    float* wsc = ws_all + ew * (BN / C::HALVES);  // this warp's col scales
    // y's row scales come from the previous launch, which also reset the
    // shared row bounds: wait for it here too (the producer waits anyway)
    if (kFp8 || row_bound) pdl_wait();
    // 8-bit operands: logit = srow * (acc * w_scale); the row factor is
    // positive, so candidates are ranked on acc * w_scale and srow enters
    // the exponent's scale and the final values only
    const float srow = kFp8 && m < M ? y_scale[m] : 1.f;
    const float l2e = kFp8 ? srow * LOG2E : LOG2E;
    // accumulator-free barriers of the MMA-issuing CTA
    const uint32_t tempty0 =
        kPair ? tc::mapa_shared(tc::smem_u32(&bars->tempty[0]), 0)
              : tc::smem_u32(&bars->tempty[0]);
    float tv[kC];
    int ti[kC];
#pragma unroll
    for (int k = 0; k < kC; ++k) { tv[k] = -INFINITY; ti[k] = -1; }
    float run_m = -INFINITY, run_s = 0.f;
    bool ok = true;
    // Shared row bounds: the lists of nslots units (strips 0.. of the row
    // group, each half of a tile's columns its own slot) publish their
    // running maxima; these are values of distinct columns, so a value
    // below 16 of them cannot make the row's top 16 and no unit needs to
    // insert it.  Usually the bound is the smallest of 16 slots; for at
    // most 8 rows (single CTAs, so only a few threads per CTA read it) the
    // 16th largest of 32, a tighter bound that costs 32 loads and a
    // sorting network per tile.  Unset slots hold -inf; reads may be
    // stale, which only weakens the bound.
    const bool wide = !kPair && M <= 8;
    const int nslots = wide ? 32 : 16;
    const int bslot = strip * C::HALVES + half;
    // rows nslots floats apart, so many rows stay packed
    float* rb = row_bound && m < M ? row_bound + (size_t)m * nslots
                                   : nullptr;
    auto publish = [&]() {
      if (rb && bslot < nslots) rb[bslot] = run_m;
    };
    auto read_bound = [&]() {
      float bd = -INFINITY;
      if (rb) {
        const float4* r4 = reinterpret_cast<const float4*>(rb);
        if (!wide) {
          bd = INFINITY;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float4 f = __ldcg(r4 + k);
            bd = fminf(bd, fminf(fminf(f.x, f.y), fminf(f.z, f.w)));
          }
        } else {
          float g[32];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 f = __ldcg(r4 + k);
            g[4 * k] = f.x;
            g[4 * k + 1] = f.y;
            g[4 * k + 2] = f.z;
            g[4 * k + 3] = f.w;
          }
          bd = kth16_of_32(g);
        }
      }
      return bd;
    };
    for (int it = 0; it < my_tiles; ++it) {
      const int vt = strip + it * strips;
      const int b = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      float wreg[CH];
      if constexpr (kFp8) {  // loads in flight during the wait
#pragma unroll
        for (int j = 0; j < CH; ++j) {
          const int v = vt * BN + (half * CH + j) * 32 + lane;
          wreg[j] = v < V ? __ldg(w_scale + v) : 0.f;
        }
      }
      const bool got = tc::mbar_wait_bounded(&bars->tfull[b], aph, abort,
                                             lim);
      if (!__all_sync(0xffffffffu, got)) {
        *abort = 1;
        ok = false;
        break;
      }
      if constexpr (kFp8) {
        __syncwarp();  // the previous tile's reads of wsc are done
#pragma unroll
        for (int j = 0; j < CH; ++j) wsc[j * 32 + lane] = wreg[j];
        __syncwarp();
      }
      tc::fence_after_sync();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(b * BN);
      // chunk c of this warp's columns: TMEM -> registers, scaled, tail
      auto load_chunk = [&](int c, float (&x)[32]) {
        const int cc = half * CH + c;
        tc::tmem_ld_x32(tbase + cc * 32, x);
        if constexpr (kFp8) {
          const float4* w4 = reinterpret_cast<const float4*>(wsc + c * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 f = w4[i];
            x[4 * i] *= f.x;
            x[4 * i + 1] *= f.y;
            x[4 * i + 2] *= f.z;
            x[4 * i + 3] *= f.w;
          }
        }
        mask_tail(x, vt * BN + cc * 32, V);
      };
      // insert the chunk's candidates, every lane its own row in step
      auto insert = [&](unsigned mask, int col0) {
        while (__any_sync(0xffffffffu, mask != 0)) {
          // straight-line for every lane: a lane without a candidate
          // inserts -inf, which changes nothing
          const int i = max(__ffs(mask) - 1, 0);
          const float xv = mask ? xs[i] : -INFINITY;
          mask &= mask - 1;
          topk_insert(tv, ti, xv, col0 + i);
        }
      };
      float lo = -INFINITY;
      if (it == 0) {
        // First tile: the list is empty, so most columns would be inserted
        // one by one.  A first pass folds (max, sum) and keeps the maxima
        // of 32 column groups; lo, the 16th largest of them, is reached by
        // at least 16 of the tile's values, so no value below lo can make
        // the top 16, and the second pass inserts only values >= lo.
#pragma unroll 1
        for (int c = 0; c < CH; ++c) {
          __syncwarp();
          float x[32];
          load_chunk(c, x);
          fold_chunk<32 / CH>(x, l2e, run_m, run_s, xs + c * (32 / CH));
        }
        float gm[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) gm[i] = xs[i];
        lo = kth16_of_32(gm);
        publish();
      }
      lo = fmaxf(lo, read_bound());
#pragma unroll 1
      for (int c = 0; c < CH; ++c) {
        __syncwarp();
        float x[32];
        load_chunk(c, x);
        float cm;
        if (it == 0) {  // folded above
          cm = x[0];
#pragma unroll
          for (int i = 1; i < 32; ++i) cm = fmaxf(cm, x[i]);
        } else {
          cm = fold_chunk(x, l2e, run_m, run_s);
          // the tile's running maximum is final: publish it now, so the
          // store is done before the accumulator is handed back (that
          // arrive's release would wait for it)
          if (c == CH - 1) publish();
        }
        insert(chunk_candidates(x, cm, tv[kC - 1], lo, xs),
               vt * BN + (half * CH + c) * 32);
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if constexpr (kPair)
          tc::mbar_arrive_cluster(tempty0 + b * 8);
        else
          tc::mbar_arrive(&bars->tempty[b]);
      }
    }
    if constexpr (C::HALVES == 2) {
      // the second half's warps hand their lists to the first half's; every
      // epilogue thread reaches both barriers once (also after a timeout)
      float* mg = mg_all + (q * 32 + lane) * 34;
      if (half == 1) {
#pragma unroll
        for (int k = 0; k < kC; ++k) {
          mg[k] = tv[k];
          mg[kC + k] = __int_as_float(ti[k]);
        }
        mg[32] = run_m;
        mg[33] = run_s;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::EPI_WARPS * 32) : "memory");
      if (half == 0) {
        // Merge of two sorted lists: the better of entry k and the other
        // list's entry 15 - k are the top 16 of both, in bitonic order,
        // which four rounds of compare-exchanges (distance 8, 4, 2, 1)
        // sort best first.
#pragma unroll
        for (int k = 0; k < kC; ++k) {
          const float bv = mg[kC - 1 - k];
          const int bi = __float_as_int(mg[2 * kC - 1 - k]);
          if (topk_before(bv, bi, tv[k], ti[k])) {
            tv[k] = bv;
            ti[k] = bi;
          }
        }
#pragma unroll
        for (int dd = kC / 2; dd; dd >>= 1) {
#pragma unroll
          for (int k = 0; k < kC; ++k) {
            const int l = k ^ dd;
            if (l > k && topk_before(tv[l], ti[l], tv[k], ti[k])) {
              const float fv = tv[k];
              const int fi = ti[k];
              tv[k] = tv[l];
              ti[k] = ti[l];
              tv[l] = fv;
              ti[l] = fi;
            }
          }
        }
        const float m1 = mg[32], s1 = mg[33];
        const float mm = fmaxf(run_m, m1);
        if (mm != -INFINITY)
          run_s = run_s * tc::ex2_approx((run_m - mm) * l2e) +
                  s1 * tc::ex2_approx((m1 - mm) * l2e);
        run_m = mm;
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::EPI_WARPS * 32) : "memory");
    }
    if (ok && half == 0 && !*abort && m < M) {
      if constexpr (kFp8) {
#pragma unroll
        for (int k = 0; k < kC; ++k) tv[k] *= srow;
        run_m *= srow;
      }
      const size_t pr = (size_t)m * strips + strip;
      float4* pv = reinterpret_cast<float4*>(P.v + pr * kC);
      int4* pi = reinterpret_cast<int4*>(P.i + pr * kC);
#pragma unroll
      for (int k = 0; k < kC / 4; ++k) {
        pv[k] = make_float4(tv[4 * k], tv[4 * k + 1], tv[4 * k + 2],
                            tv[4 * k + 3]);
        pi[k] = make_int4(ti[4 * k], ti[4 * k + 1], ti[4 * k + 2],
                          ti[4 * k + 3]);
      }
      P.m[pr] = run_m;
      P.s[pr] = run_s;
    }
  }

  tc::fence_before_sync();
  if constexpr (kPair)
    tc::cluster_sync();  // the pair's MMAs and copies are done in both CTAs
  else
    __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    if constexpr (kPair)
      tc::tmem_dealloc_pair(tmem, TMEM_COLS);
    else
      tc::tmem_dealloc(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && bars->abort) raise_error(err, kErrTimeout);
}

}  // namespace

bool lmhead_tc_pairs(int M) { return (M + BM - 1) / BM >= 2; }

namespace {
// Pairs the device can hold at once (a pair needs two SMs of one TPC).
template <bool kFp8>
int max_resident_pairs(int num_sms) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return num_sms / 2;
  if (cached[dev] > 0) return cached[dev];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms);
  cfg.blockDim = dim3(Cfg<true, kFp8>::THREADS);
  cfg.dynamicSmemBytes = smem_bytes<true, kFp8>();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaFuncSetAttribute(lmhead_tc_kernel<true, kFp8>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes<true, kFp8>()) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, lmhead_tc_kernel<true, kFp8>,
                                     &cfg) != cudaSuccess ||
      n < 1) {
    (void)cudaGetLastError();
    n = num_sms / 2;
  }
  cached[dev] = n;
  return n;
}
}  // namespace

int lmhead_tc_grid(int M, int V, int num_sms, int* row_groups, int* strips,
                   bool fp8) {
  const bool pairs = lmhead_tc_pairs(M);
  const int ctas = pairs ? 2 : 1;
  const int rt = (M + BM - 1) / BM;
  const int rg = (rt + ctas - 1) / ctas;  // units per vocab strip
  const int vt = (V + BN - 1) / BN;
  const int units = !pairs ? num_sms
                    : fp8  ? max_resident_pairs<true>(num_sms)
                           : max_resident_pairs<false>(num_sms);
  int st = std::max(1, units / rg);
  st = std::min(std::min(st, vt), kMaxStrips);
  *row_groups = rg;
  *strips = st;
  return rg * st * ctas;
}

namespace {
template <bool kFp8>
cudaError_t launch_variant(const CUtensorMap& map_y, const CUtensorMap& map_w,
                           int M, int H, int V, int num_sms, TopkPartials P,
                           int* err, int* strips_out, cudaStream_t s,
                           const float* y_scale, const float* w_scale,
                           float* row_bound, uint64_t wait_ns) {
  int rg = 0, st = 0;
  const int grid = lmhead_tc_grid(M, V, num_sms, &rg, &st, kFp8);
  *strips_out = st;
  if (!lmhead_tc_pairs(M)) {
    cudaError_t e = cudaFuncSetAttribute(
        lmhead_tc_kernel<false, kFp8>,
        cudaFuncAttributeMaxDynamicSharedMemorySize,
        (int)smem_bytes<false, kFp8>());
    if (e != cudaSuccess) return e;
    PdlLaunch L(dim3(grid), dim3(Cfg<false, kFp8>::THREADS),
                smem_bytes<false, kFp8>(), s);
    return cudaLaunchKernelEx(&L.cfg, lmhead_tc_kernel<false, kFp8>, map_y,
                              map_w, M, H, V, rg, st, P, y_scale, w_scale,
                              row_bound, err, wait_ns);
  }
  cudaError_t e = cudaFuncSetAttribute(
      lmhead_tc_kernel<true, kFp8>,
      cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem_bytes<true, kFp8>());
  if (e != cudaSuccess) return e;
  PdlLaunch L(dim3(grid), dim3(Cfg<true, kFp8>::THREADS),
              smem_bytes<true, kFp8>(), s, 2);
  return cudaLaunchKernelEx(&L.cfg, lmhead_tc_kernel<true, kFp8>, map_y,
                            map_w, M, H, V, rg, st, P, y_scale, w_scale,
                            row_bound, err, wait_ns);
}
}  // namespace

cudaError_t launch_lmhead_tc(const CUtensorMap& map_y, const CUtensorMap& map_w,
                             int M, int H, int V, int num_sms, TopkPartials P,
                             int* err, int* strips_out, cudaStream_t s,
                             const float* y_scale, const float* w_scale,
                             float* row_bound, uint64_t wait_ns) {
  if (y_scale && w_scale)
    return launch_variant<true>(map_y, map_w, M, H, V, num_sms, P, err,
                                strips_out, s, y_scale, w_scale, row_bound,
                                wait_ns);
  return launch_variant<false>(map_y, map_w, M, H, V, num_sms, P, err,
                               strips_out, s, nullptr, nullptr, row_bound,
                               wait_ns);
}

}  // namespace dflash
