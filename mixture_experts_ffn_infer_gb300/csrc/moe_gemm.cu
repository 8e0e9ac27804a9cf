// Grouped GEMMs of the routed experts on the fifth-generation tensor core.
//
// "SwiGLU output" page, MLP class: expert(x) = down(silu(gate x) * up x);
// "Element-wise product" page: h = silu(gate x) (.) (up x);
// "Mixture of experts" page, moe_infer: each expert runs on the contiguous
// slice of sorted rows routed to it, outputs go back to their positions and
// are weighted by topk_weight;
// "Input features" page, quantisation config: weights are e4m3 with one fp32
// scale per 128 x 128 block.
//
// One persistent CTA per SM walks a list of work units.  A unit is one tile of
// at most NTOK sorted rows of one expert times two blocks of 128 weight rows:
// gate and up of the same 128 output features (gate/up pass), or down row
// blocks 2j and 2j + 1 (down pass; the units of a last round that would leave
// most SMs idle are cut into single row blocks).  The weights are the MMA's M side (128
// rows) and the tokens its N side ("swap AB").  The e4m3 weight tiles go from
// global memory to shared memory by bulk copy (tiled layout: both blocks of
// KPS consecutive K blocks in one copy) or TMA (row-major layout) and
// straight into tcgen05.mma kind::f8f6f4 - no conversion.  The activations
// arrive in the e4m3 split format (split3.cuh), rows interleaved with three
// term slots; the N side of each MMA holds the TT live terms of NTOK tokens
// (N = TT NTOK): two for the bf16 features of gate/up, three for h in down,
// one for either under the dynamic FP8 scheme.  Per 128-wide K block:
//
//   warp 0      weight producer: stages of KPS K blocks x both weight blocks
//               into a ring.
//   warp 2      activation producer: a 3-D box of NTOK rows x TT terms x 128 bytes
//               into its own ring, so neither ring throttles the other.
//   warp 1      MMA issuer (one thread, elected): 4 x tcgen05.mma (M=128,
//               N=TT NTOK, K=32) per weight block into a fresh fp32 partial
//               in tensor memory.
//   warps 4-7   epilogue: per token, sum its TT term columns, multiply by
//               the weight block's fp32 scale and the activation block's factor
//               (2^-s, or the FP8 scale) and add to fp32 accumulators in
//               registers - the exact block-scaled product of the dequantised
//               operands.
//
// After the last K block the epilogue writes, per valid token column,
//   gate/up pass : h = silu(g) * u in the split format (one block scale per
//                  row and 128 features, found with a max over the 4 warps),
//                  or as one dynamic-FP8 term (scale amax / 448) with the
//                  other two terms zero
//   down pass    : f16(topk_weight * o) -> rows[flat position][feature], both blocks
//
// Both passes are dependent launches (gate/up behind the row gather, down
// behind gate/up): the weight producer starts at once, the activation producer
// and the epilogue wait for the previous grid first.  Every wait is bounded; a
// wait that gives up raises the CTA's abort flag and the device error word, the
// roles drain their in-flight copies and MMAs and the kernel returns normally.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "split3.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarpProducer = 0;     // weight loads
constexpr int kWarpMma = 1;
constexpr int kWarpActProducer = 2;  // activation loads
constexpr int kWarpEpi0 = 4;         // epilogue: warps 4..7 -> tensor-memory lane quarters 0..3

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NTOK, int TT, int KPS, int WST, int BST, int DST>
struct Cfg {
  static_assert(NTOK <= 32, "one token per lane for the activation exponents");
  static_assert(TT >= 1 && TT <= 3, "one to three e4m3 terms per token");
  static constexpr int kNB = TT * NTOK;                  // MMA N: the live e4m3 terms of every token
  static constexpr int kWTile = 128 * 128;               // e4m3 weight tile bytes
  static constexpr int kWKb = 2 * kWTile;                // both weight blocks of one K block
  static constexpr int kWStage = KPS * kWKb;             // one weight stage: [K block][block][tile]
  static constexpr int kBStage = kNB * 128;              // one K block of split activations
  static constexpr int kDCols = 2 * kNB;                 // tensor-memory columns of one partial buffer
  static constexpr int kTmemCols = pow2_at_least(DST * kDCols);
  static constexpr int kNumBars = 2 * WST + 2 * BST + 2 * DST + 2 + 1;
  static constexpr int kBOffset = WST * kWStage;
  static constexpr int kBarOffset = kBOffset + BST * kBStage;
  static constexpr int kRedOffset = kBarOffset + kNumBars * 8 + 16;
  static constexpr int kSmem = 1024 + kRedOffset + 2 * 4 * NTOK * 4;
  static_assert(kBStage % 1024 == 0, "activation stages must stay 1024-byte aligned");
  static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
  static_assert(kNB % 16 == 0 && kNB <= 256, "MMA N for M = 128");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

struct GemmArgs {
  const uint8_t* w_tiled;   // non-null: weights in the tiled layout, streamed with bulk copies
  const float* s0;          // scales of block 0 / block 1 [E][n_nb][num_kb]
  const float* s1;
  const TileDesc* tiles;
  const int32_t* n_tiles;
  int32_t n_nb;
  int32_t num_kb;
  int32_t pair;             // 1: unit = row blocks 2j, 2j + 1 of w0 (down); 0: row block j of w0 and w1
  const float* act_inv;     // [num_kb][act_rows]: 2^-s of each activation block
  int32_t act_rows;
  void* out;                // gate/up: h terms [3 act_rows][n_nb*128] e4m3; down: rows [.][n_nb*128] f16
  float* out_inv;           // gate/up: [n_nb][act_rows] factor of each h block
  int32_t fp8;              // gate/up: h as one dynamic-FP8 term (scale amax / 448) instead of three
  const int32_t* sorted_pos;
  const float* topk_weight;
  uint32_t* err;
};

// The unit list.  Units [0, n_pair) are token tile u / upt times its unit row
// u % upt (two weight blocks).  Down pass: when the last, partial round of units
// would keep at most half of the CTAs busy, its units are cut into their two
// row blocks (units n_pair + 2i and n_pair + 2i + 1 are the blocks of unit
// n_pair + i), so twice as many SMs stream the tail, each half as long.  Only
// with an even number of row blocks, where every pair is complete.
struct UnitList {
  int n_pair;
  int total;
};

__device__ __forceinline__ UnitList unit_list(const GemmArgs& a, int upt) {
  const int U = *a.n_tiles * upt, G = static_cast<int>(gridDim.x);
  const int q = U / G, r = U - q * G;
  if (!a.pair || (a.n_nb & 1) || r == 0 || 2 * r > G) return UnitList{U, U};
  return UnitList{q * G, q * G + 2 * r};
}

struct Unit16 {
  int tile, ru, nb0, nb1;
  int half;  // -1: both blocks of the unit row; 0 or 1: that block of the down pair alone
  bool has1;
};

__device__ __forceinline__ Unit16 unit16(const GemmArgs& a, int u, int upt, const UnitList& L) {
  Unit16 x;
  int v = u;
  x.half = -1;
  if (u >= L.n_pair) {
    v = L.n_pair + ((u - L.n_pair) >> 1);
    x.half = (u - L.n_pair) & 1;
  }
  x.tile = v / upt;
  x.ru = v % upt;
  if (x.half >= 0) {
    x.nb0 = x.nb1 = 2 * x.ru + x.half;
    x.has1 = false;
  } else {
    x.nb0 = a.pair ? 2 * x.ru : x.ru;
    x.nb1 = a.pair ? 2 * x.ru + 1 : x.ru;
    x.has1 = x.nb1 < a.n_nb;
  }
  return x;
}

// Bounded wait used while winding down: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return;
}

__device__ __forceinline__ void mma_f8_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <bool GATEUP, int NTOK, int TT, int KPS, int WST, int BST, int DST>
__global__ void __launch_bounds__(kThreads, 1)
moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                const __grid_constant__ CUtensorMap tm_act, const GemmArgs a) {
  using C = Cfg<NTOK, TT, KPS, WST, BST, DST>;
  constexpr int NB = C::kNB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOffset;
  // weight ring, activation ring, partial-accumulator buffers
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto empty_w = [&](int i) { return bar0 + 8u * (WST + i); };
  auto full_b = [&](int i) { return bar0 + 8u * (2 * WST + i); };
  auto empty_b = [&](int i) { return bar0 + 8u * (2 * WST + BST + i); };
  auto dfull = [&](int i) { return bar0 + 8u * (2 * WST + 2 * BST + i); };
  auto dempty = [&](int i) { return bar0 + 8u * (2 * WST + 2 * BST + DST + i); };
  auto redbar = [&](int i) { return bar0 + 8u * (2 * WST + 2 * BST + 2 * DST + i); };  // epilogue exchange
  const uint32_t drain_bar = bar0 + 8u * (C::kNumBars - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOffset + C::kNumBars * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  float* red = reinterpret_cast<float*>(smem + C::kRedOffset);  // [2][4 warps][NTOK] block maxima

  // The dependent launch behind this grid (down behind gate/up, the combine behind down)
  // may be placed now: this grid was placed only after every kernel before its own
  // predecessor had ended, so a dependent that reads weights without waiting reads
  // finished ones; it waits for this grid to end before it reads this grid's results.
  pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < WST; ++i) {
      mbar_init(full_w(i), 1);
      mbar_init(empty_w(i), 1);  // one MMA commit
    }
    for (int i = 0; i < BST; ++i) {
      mbar_init(full_b(i), 1);
      mbar_init(empty_b(i), 1);
    }
    for (int i = 0; i < DST; ++i) {
      mbar_init(dfull(i), 1);
      mbar_init(dempty(i), 4);  // the four epilogue warps
    }
    mbar_init(redbar(0), 4);
    mbar_init(redbar(1), 4);
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    if (!a.w_tiled) {
      prefetch_tmap(&tm_w0);
      prefetch_tmap(&tm_w1);
    }
    prefetch_tmap(&tm_act);
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_nb = a.n_nb, num_kb = a.num_kb;
  const int upt = a.pair ? (n_nb + 1) / 2 : n_nb;  // units per tile
  const UnitList L = unit_list(a, upt);
  const int total_units = L.total;
  // tiled layout: K block kb of unit row ru of expert e, both blocks (32 KB)
  auto unit_off = [&](int e, int ru, int kb) {
    return ((static_cast<int64_t>(e) * upt + ru) * num_kb + kb) * C::kWKb;
  };

  if (warp == kWarpProducer) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      // No L2 prefetch ahead of the stages: with six 32-64 KB stages per SM in
      // flight the stream already saturates HBM, and extra prefetch requests
      // measured 5-7 % slower.
      uint32_t w_issued = 0;  // weight stages issued
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit16 un = unit16(a, u, upt, L);
        const int e = a.tiles[un.tile].expert;
        for (int kb = 0; kb < num_kb; kb += KPS) {
          const uint32_t it = w_issued;
          const int sw = it % WST;
          const int nk = min(KPS, num_kb - kb);
          if (!wait_bounded(empty_w(sw), ((it / WST) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t wst = sbase + sw * C::kWStage;
          if (a.w_tiled && un.half < 0) {
            // the stage's K blocks, both weight blocks each, are one contiguous
            // region already in the swizzled image: one bulk copy
            mbar_arrive_expect_tx(full_w(sw), nk * C::kWKb);
            bulk_load(wst, a.w_tiled + unit_off(e, un.ru, kb), nk * C::kWKb, full_w(sw), pol_w);
          } else if (a.w_tiled) {
            // one block of the pair: its 16 KB tile of each K block, to the stage's first slot
            mbar_arrive_expect_tx(full_w(sw), nk * C::kWTile);
            for (int j = 0; j < nk; ++j)
              bulk_load(wst + j * C::kWKb, a.w_tiled + unit_off(e, un.ru, kb + j) + un.half * C::kWTile, C::kWTile,
                        full_w(sw), pol_w);
          } else {
            mbar_arrive_expect_tx(full_w(sw), nk * (un.has1 ? 2 : 1) * C::kWTile);
            for (int j = 0; j < nk; ++j) {
              tma_load_3d(wst + j * C::kWKb, &tm_w0, full_w(sw), (kb + j) * 128, un.nb0 * 128, e, pol_w);
              if (un.has1)
                tma_load_3d(wst + j * C::kWKb + C::kWTile, &tm_w1, full_w(sw), (kb + j) * 128, un.nb1 * 128, e,
                            pol_w);
            }
          }
          ++w_issued;
        }
      }
      if (!ok)  // wait for the copies already in flight before the CTA exits
        for (uint32_t i = w_issued > WST ? w_issued - WST : 0; i < w_issued; ++i)
          wait_drain(full_w(i % WST), (i / WST) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpActProducer) {
    pdl_wait();  // the activations are the previous kernel's output
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      uint32_t b_issued = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const int row0 = a.tiles[unit16(a, u, upt, L).tile].row_start;
        for (int kb = 0; kb < num_kb; ++kb) {
          const uint32_t it = b_issued;
          const int sb = it % BST;
          if (!wait_bounded(empty_b(sb), ((it / BST) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t bst = sbase + C::kBOffset + sb * C::kBStage;
          mbar_arrive_expect_tx(full_b(sb), C::kBStage);
          tma_load_3d(bst, &tm_act, full_b(sb), kb * 128, 0, row0, pol_a);  // [NTOK rows][TT terms][128 B]
          ++b_issued;
        }
      }
      if (!ok)
        for (uint32_t i = b_issued > BST ? b_issued - BST : 0; i < b_issued; ++i)
          wait_drain(full_b(i % BST), (i / BST) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // One elected thread runs the whole loop: its waits, MMAs and commits.
    if (elect_one()) {
      constexpr uint32_t idesc = idesc_f16_f32(128, NB);  // kind::f8f6f4: E4M3 has format code 0, as f16
      uint32_t it = 0, wt = 0;  // K blocks and weight stages consumed
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const bool has1 = unit16(a, u, upt, L).has1;
        for (int kb0 = 0; ok && kb0 < num_kb; kb0 += KPS, ++wt) {
          const int sw = wt % WST;
          const int nk = min(KPS, num_kb - kb0);
          if (!wait_bounded(full_w(sw), (wt / WST) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t wst = sbase + sw * C::kWStage;
          const uint64_t wdesc = desc_kmajor_sw128(wst);
          for (int j = 0; j < nk; ++j, ++it) {
            const int sb = it % BST, sd = it % DST;
            if (!wait_bounded(full_b(sb), (it / BST) & 1, abort_flag, a.err) ||
                !wait_bounded(dempty(sd), ((it / DST) & 1) ^ 1, abort_flag, a.err)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t bdesc = desc_kmajor_sw128(sbase + C::kBOffset + sb * C::kBStage);
            const uint64_t wj = desc_advance(wdesc, j * C::kWKb);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              if (m == 1 && !has1) break;
              const uint32_t d_addr = tmem + (sd * 2 + m) * NB;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_f8_ss(d_addr, desc_advance(wj, m * C::kWTile + kk * 32), desc_advance(bdesc, kk * 32), idesc,
                          kk > 0 ? 1u : 0u);
            }
            tc_commit(empty_b(sb));
            tc_commit(dfull(sd));
          }
          if (ok) tc_commit(empty_w(sw));  // the stage's weights are free once its MMAs complete
        }
      }
      tc_commit(drain_bar);  // every MMA issued above has completed once this arrives
      wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    pdl_wait();  // activation exponents come from the previous kernel
    const int q = warp - kWarpEpi0;
    const int r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ui) {
      const Unit16 un = unit16(a, u, upt, L);
      const TileDesc td = a.tiles[un.tile];
      const float* sc0 = a.s0 + (static_cast<int64_t>(td.expert) * n_nb + un.nb0) * num_kb;
      const float* sc1 = a.s1 + (static_cast<int64_t>(td.expert) * n_nb + (un.has1 ? un.nb1 : un.nb0)) * num_kb;
      float acc[2][NTOK];
#pragma unroll
      for (int m = 0; m < 2; ++m)
#pragma unroll
        for (int j = 0; j < NTOK; ++j) acc[m][j] = 0.f;
      // Down pass: destination rows and router weights of the tile, loaded now so their
      // latency hides behind the K loop instead of stalling the end of the unit.
      int dest[GATEUP ? 1 : NTOK];
      float wgt[GATEUP ? 1 : NTOK];
      if (!GATEUP) {
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          const int row = td.row_start + j;
          dest[j] = j < td.n_valid ? (a.sorted_pos ? __ldg(a.sorted_pos + row) : row) : 0;
        }
#pragma unroll
        for (int j = 0; j < NTOK; ++j)
          wgt[j] = (j < td.n_valid && a.topk_weight) ? __ldg(a.topk_weight + dest[j]) : 1.0f;
      }
      // Per K block: the two blocks' weight scales and, in lane j, the 2^-s of token j's
      // activation block ([kb][row]); each iteration loads the next block's, so the
      // latency hides behind the wait, and the lanes' values reach all lanes by shuffle.
      const float* inv0 = a.act_inv + td.row_start;
      const bool tok_lane = lane < NTOK && lane < td.n_valid;
      float s0n = __ldg(sc0), s1n = __ldg(sc1);
      float sxn = tok_lane ? __ldg(inv0 + lane) : 0.f;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int sd = it % DST;
        const float s0v = s0n, s1v = s1n, sx_lane = sxn;
        if (kb + 1 < num_kb) {
          s0n = __ldg(sc0 + kb + 1);
          s1n = __ldg(sc1 + kb + 1);
          sxn = tok_lane ? __ldg(inv0 + static_cast<int64_t>(kb + 1) * a.act_rows + lane) : 0.f;
        }
        ok = __all_sync(0xffffffffu, wait_bounded(dfull(sd), (it / DST) & 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < NTOK / 16; ++c) {  // 16 tokens (16 TT tensor-memory columns) at a time
          float sx[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) sx[j] = __shfl_sync(0xffffffffu, sx_lane, 16 * c + j);
#pragma unroll
          for (int m = 0; m < 2; ++m) {
            if (m == 1 && !un.has1) break;
            const float sv = m == 0 ? s0v : s1v;
            uint32_t p[16 * TT];
#pragma unroll
            for (int c0 = 0; c0 < 16 * TT; c0 += 16)
              tmem_ld16(tmem + lane_base + (sd * 2 + m) * NB + 16 * TT * c + c0,
                        *reinterpret_cast<uint32_t(*)[16]>(&p[c0]));
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float part = __uint_as_float(p[TT * j]);  // the token's terms, first to last
#pragma unroll
              for (int t = 1; t < TT; ++t) part += __uint_as_float(p[TT * j + t]);
              acc[m][16 * c + j] = fmaf(sv * sx[j], part, acc[m][16 * c + j]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty(sd));
      }
      if (!ok) break;
      bool overflow = false;
      if (GATEUP) {
        // h = silu(g) * u, then the split format with one exponent per (row, 128 features):
        // the block maximum is taken over the 128 threads (4 warps x 32 lanes).
        // The exchange goes through red[ui & 1] and an mbarrier of four arrivals, so a
        // warp can be one unit ahead of the others and every wait stays bounded.
        float* rb = red + (ui & 1) * 4 * NTOK;
        float* hv = acc[0];  // h overwrites the gate accumulators
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          const float g = acc[0][j];
          hv[j] = g / (1.0f + expf(-g)) * acc[1][j];
          overflow |= (j < td.n_valid) && !isfinite(hv[j]);
          const float m = warp_max(fabsf(hv[j]));
          if (lane == 0) rb[q * NTOK + j] = m;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(redbar(ui & 1));
        ok = __all_sync(0xffffffffu, wait_bounded(redbar(ui & 1), (ui >> 1) & 1, abort_flag, a.err));
        if (!ok) break;
        uint8_t* hterm = static_cast<uint8_t*>(a.out);
        const int64_t ld = static_cast<int64_t>(n_nb) * 128;
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          if (j < td.n_valid) {
            const float m = fmaxf(fmaxf(rb[j], rb[NTOK + j]), fmaxf(rb[2 * NTOK + j], rb[3 * NTOK + j]));
            uint8_t t1, t2 = 0, t3 = 0;
            float factor;
            if (a.fp8) {  // dynamic FP8: one term, scale amax / 448
              factor = fp8_block_scale(m);
              t1 = float_to_e4m3(__fdiv_rn(hv[j], factor));
            } else {
              const int sexp = split_exponent(m);
              split3(ldexpf(hv[j], sexp), t1, t2, t3);
              factor = ldexpf(1.0f, -sexp);
            }
            const int64_t row = td.row_start + j;
            uint8_t* dst = hterm + (3 * row) * ld + un.nb0 * 128 + r;
            dst[0] = t1;
            dst[ld] = t2;
            dst[2 * ld] = t3;
            if (r == 0) a.out_inv[static_cast<int64_t>(un.nb0) * a.act_rows + row] = factor;
          }
        }
      } else {
        uint16_t* rows = static_cast<uint16_t*>(a.out);
        const int64_t ld = static_cast<int64_t>(n_nb) * 128;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m == 1 && !un.has1) break;
          const int nb = m == 0 ? un.nb0 : un.nb1;
#pragma unroll
          for (int j = 0; j < NTOK; ++j) {
            if (j < td.n_valid) {
              const __half hh = __float2half_rn(acc[m][j] * wgt[GATEUP ? 0 : j]);
              overflow |= __hisinf(hh) != 0 || __hisnan(hh);
              rows[static_cast<int64_t>(dest[GATEUP ? 0 : j]) * ld + nb * 128 + r] = __half_as_ushort(hh);
            }
          }
        }
      }
      if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(a.err, DEV_ERR_RANGE);
    }
  }
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

template <bool GATEUP, int NTOK, int TT, int KPS, int WST, int BST, int DST>
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s) {
  using C = Cfg<NTOK, TT, KPS, WST, BST, DST>;
  auto kern = moe_gemm_kernel<GATEUP, NTOK, TT, KPS, WST, BST, DST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  GemmArgs a;
  a.w_tiled = g.w_tiled;
  a.s0 = g.s0;
  a.s1 = g.s1;
  a.tiles = g.tiles;
  a.n_tiles = g.n_tiles;
  a.n_nb = g.n_nb;
  a.num_kb = g.num_kb;
  a.pair = GATEUP ? 0 : 1;
  a.act_inv = g.act_inv;
  a.act_rows = g.act_rows;
  a.out = g.out;
  a.out_inv = g.out_inv;
  a.fp8 = g.fp8 ? 1 : 0;
  a.sorted_pos = g.sorted_pos;
  a.topk_weight = g.topk_weight;
  a.err = g.err;
  // dependent launches: gate/up after the row gather (its CTAs fit beside the gather's,
  // so they start streaming weights at once) and down after gate/up (each CTA starts
  // streaming down weights as soon as its SM's gate/up CTA exits); both wait for
  // their predecessor before they read activations
  return launch_maybe_overlapped(kern, g.num_sms, kThreads, C::kSmem, s, !GATEUP || g.overlap, *g.w0, *g.w1,
                                 *g.act, a);
}

}  // namespace

// Each weight stage is one bulk copy of 32 KB: on GB300 an SM completes bulk
// copies at a roughly fixed rate (about 3.5 million per second) up to 32 KB, so
// the bytes per copy and the copies in flight set the bandwidth (a probe
// streaming from HBM into shared memory: 8 KB copies cap at 29 GB/s per SM;
// 32 KB copies reach 47-48 GB/s per SM, 7.4 TB/s in total, with two or more
// in flight).
// Decode-sized tiles (16 tokens; MMA N = 16 per live term: 32 for the two terms
// of gate/up's bf16 features, 48 for h's three in down, 16 under dynamic FP8):
//   gate/up: 6 stages of 1 K block x (gate, up) = 32 KB, 4 activation stages of
//            2 KB per term, 4 partial buffers
//   down:    5 stages of 1 K block x 2 row blocks = 32 KB, 4 activation stages,
//            4 partial buffers (five 32 KB stages measured 2.7 % faster than
//            three of 64 KB)
// Wide tiles (up to 128 tokens) go to moe_gemm_wide.cu.
cudaError_t launch_gateup(const GemmLaunch& g, cudaStream_t s) {
  if (g.ntok == kNTokWide) return g.fp8 ? launch_gateup_wide(g, s) : launch_gateup_f16(g, s);
  if (g.ntok != kNTokSmall) return cudaErrorInvalidValue;
  if (g.terms == 2) return launch_gemm<true, kNTokSmall, 2, 1, 6, 4, 4>(g, s);
  if (g.terms == 1) return launch_gemm<true, kNTokSmall, 1, 1, 6, 4, 4>(g, s);
  return cudaErrorInvalidValue;
}
cudaError_t launch_down(const GemmLaunch& g, cudaStream_t s) {
  if (g.ntok == kNTokWide) return g.fp8 ? launch_down_wide(g, s) : launch_down_f16(g, s);
  if (g.ntok != kNTokSmall) return cudaErrorInvalidValue;
  if (g.terms == 3) return launch_gemm<false, kNTokSmall, 3, 1, 5, 4, 4>(g, s);
  if (g.terms == 1) return launch_gemm<false, kNTokSmall, 1, 1, 5, 4, 4>(g, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
