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
// at most kNTok sorted rows of one expert times one block of 128 weight rows
// (128 output features).  The weights are the MMA's M side (128 rows) and the
// tokens its N side ("swap AB"), so a decode tile of 1-3 tokens still fills
// the instruction.  Per 128-wide K block:
//
//   warp 0      TMA producer: e4m3 weight tile(s) 128 x 128 and the f16
//               activation tile kNTok x 128 into a ring of shared-memory stages.
//   warps 4-7   converters: thread r owns weight row r; it reads its 128 bytes
//               (128-byte swizzle), converts e4m3 -> f16 exactly and stores
//               the row into tensor memory as the MMA's A operand.
//   warp 1      MMA issuer: 8 x tcgen05.mma kind::f16 (M=128, N=kNTok, K=16),
//               A from tensor memory, B from shared memory, into a fresh fp32
//               partial accumulator in tensor memory.
//   warps 8-11  epilogue: load the partial, multiply it by the block's fp32
//               scale and add it to fp32 accumulators in registers.  That is
//               the exact block-scaled product (the scale is constant over the
//               128 x 128 block), without rounding weight * scale.
//
// After the last K block the epilogue writes, per valid token column,
//   gate/up pass : h = f16(silu(g) * u)            -> h[row][feature]
//   down pass    : f16(topk_weight * o)            -> rows[flat position][feature]
// Converted weights never touch shared memory, so shared-memory bandwidth is
// spent only on the TMA writes, the converters' reads and the small B tiles.
//
// Every wait is bounded; a wait that gives up raises the CTA's abort flag and
// the device error word, the roles drain their in-flight copies and MMAs and
// the kernel returns normally.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 384;
constexpr int kWarpProducer = 0;
constexpr int kWarpMma = 1;
constexpr int kWarpConv0 = 4;  // warps 4..7 -> tensor-memory lane quarters 0..3
constexpr int kWarpEpi0 = 8;   // warps 8..11 -> lane quarters 0..3

constexpr int pow2_at_least(int v) {
  int p = 32;
  while (p < v) p <<= 1;
  return p;
}

template <int NMAT, int NTOK, int STAGES>
struct Cfg {
  static constexpr int kWTile = 128 * 128;               // e4m3 weight tile bytes
  static constexpr int kBBox = NTOK * 128;               // one 64-column f16 activation box
  static constexpr int kStage = NMAT * kWTile + 2 * kBBox;
  static constexpr int kACols = 64;                      // tensor-memory columns of a converted tile
  static constexpr int kATotal = 2 * NMAT * kACols;      // two A stages
  static constexpr int kDTotal = 2 * NMAT * NTOK;        // two partial-accumulator buffers
  static constexpr int kTmemCols = pow2_at_least(kATotal + kDTotal);
  static constexpr int kNumBars = 2 * STAGES + 9;
  static constexpr int kBarBytes = kNumBars * 8 + 16;
  static constexpr int kSmem = 1024 + STAGES * kStage + kBarBytes;
  static_assert(kBBox % 1024 == 0, "activation boxes must stay 1024-byte aligned");
  static_assert(kTmemCols <= 512, "tensor memory holds 512 columns");
  static_assert(NTOK % 16 == 0 && NTOK >= 16 && NTOK <= 256, "MMA N for M = 128");
};

struct GemmArgs {
  const float* s0;
  const float* s1;
  const TileDesc* tiles;
  const int32_t* n_tiles;
  int32_t n_nb;
  int32_t num_kb;
  void* out;
  const int32_t* sorted_pos;
  const float* topk_weight;
  uint32_t* err;
};

// Bounded wait used while winding down: ignores the abort flag.
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return;
}

// 16 e4m3 bytes -> 8 words of two f16 each (lower K index in the low half).
__device__ __forceinline__ void cvt_e4m3x16_f16(const uint4 v, uint32_t* o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), __NV_E4M3);
    o[2 * q] = static_cast<uint32_t>(lo.x) | (static_cast<uint32_t>(lo.y) << 16);
    o[2 * q + 1] = static_cast<uint32_t>(hi.x) | (static_cast<uint32_t>(hi.y) << 16);
  }
}

template <int NMAT, int NTOK, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                const __grid_constant__ CUtensorMap tm_act, const GemmArgs a) {
  using C = Cfg<NMAT, NTOK, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + STAGES * C::kStage;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto afull = [&](int i) { return bar0 + 8u * (2 * STAGES + i); };
  auto aempty = [&](int i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  auto dfull = [&](int i) { return bar0 + 8u * (2 * STAGES + 4 + i); };
  auto dempty = [&](int i) { return bar0 + 8u * (2 * STAGES + 6 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + STAGES * C::kStage + C::kNumBars * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 4 + 1);  // four converter warps + one MMA commit
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(afull(i), 4);
      mbar_init(aempty(i), 1);
      mbar_init(dfull(i), 1);
      mbar_init(dempty(i), 4);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpProducer && lane == 0) {
    prefetch_tmap(&tm_w0);
    if (NMAT == 2) prefetch_tmap(&tm_w1);
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
  const int total_units = *a.n_tiles * n_nb;

  if (warp == kWarpProducer) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const TileDesc td = a.tiles[u / n_nb];
        const int nb = u % n_nb;
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          if (!wait_bounded(empty(s), ((it / STAGES) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * C::kStage;
          mbar_arrive_expect_tx(full(s), C::kStage);
          tma_load_3d(st, &tm_w0, full(s), kb * 128, nb * 128, td.expert, pol_w);
          if (NMAT == 2) tma_load_3d(st + C::kWTile, &tm_w1, full(s), kb * 128, nb * 128, td.expert, pol_w);
          tma_load_2d(st + NMAT * C::kWTile, &tm_act, full(s), kb * 128, td.row_start, pol_a);
          tma_load_2d(st + NMAT * C::kWTile + C::kBBox, &tm_act, full(s), kb * 128 + 64, td.row_start, pol_a);
        }
      }
      if (!ok)  // wait for the copies already in flight before the CTA exits
        for (uint32_t i = it > STAGES ? it - STAGES : 0; i < it; ++i) wait_drain(full(i % STAGES), (i / STAGES) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(128, NTOK);
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % STAGES;
          const int sa = it & 1;
          const uint32_t pa = (it >> 1) & 1;
          if (!wait_bounded(full(s), (it / STAGES) & 1, abort_flag, a.err) ||
              !wait_bounded(afull(sa), pa, abort_flag, a.err) ||
              !wait_bounded(dempty(sa), pa ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t bst = sbase + s * C::kStage + NMAT * C::kWTile;
#pragma unroll
          for (int m = 0; m < NMAT; ++m) {
            const uint32_t d_addr = tmem + C::kATotal + (sa * NMAT + m) * NTOK;
            const uint32_t a_addr = tmem + (sa * NMAT + m) * C::kACols;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint32_t baddr = bst + (kk >> 2) * C::kBBox + (kk & 3) * 32;
              mma_f16_ts(d_addr, a_addr + kk * 8, desc_kmajor_sw128(baddr), idesc, kk > 0 ? 1u : 0u);
            }
          }
          tc_commit(aempty(sa));
          tc_commit(empty(s));
          tc_commit(dfull(sa));
        }
      }
      tc_commit(drain_bar);  // every MMA issued above has completed once this arrives
      wait_drain(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpConv0 && warp < kWarpConv0 + 4) {
    const int q = warp - kWarpConv0;
    const int r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % STAGES;
        const int sa = it & 1;
        // Every lane waits (each gets the barrier's acquire); the vote keeps the
        // warp converged for the .sync.aligned tensor-memory stores.
        ok = __all_sync(0xffffffffu, wait_bounded(full(s), (it / STAGES) & 1, abort_flag, a.err) &&
                                         wait_bounded(aempty(sa), ((it >> 1) & 1) ^ 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint32_t row = sbase + s * C::kStage + m * C::kWTile + r * 128;
          uint32_t v[64];
#pragma unroll
          for (int c = 0; c < 8; ++c) cvt_e4m3x16_f16(lds128(row + ((c ^ (r & 7)) << 4)), v + 8 * c);
          const uint32_t taddr = tmem + lane_base + (sa * NMAT + m) * C::kACols;
#pragma unroll
          for (int j = 0; j < 4; ++j) tmem_st16(taddr + 16 * j, v + 16 * j);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull(sa));
          mbar_arrive(empty(s));
        }
      }
    }
  } else if (warp >= kWarpEpi0 && warp < kWarpEpi0 + 4) {
    const int q = warp - kWarpEpi0;
    const int r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const TileDesc td = a.tiles[u / n_nb];
      const int nb = u % n_nb;
      const float* sc0 = a.s0 + (static_cast<int64_t>(td.expert) * n_nb + nb) * num_kb;
      const float* sc1 = NMAT == 2 ? a.s1 + (static_cast<int64_t>(td.expert) * n_nb + nb) * num_kb : sc0;
      float acc[NMAT][NTOK];
#pragma unroll
      for (int m = 0; m < NMAT; ++m)
#pragma unroll
        for (int j = 0; j < NTOK; ++j) acc[m][j] = 0.f;
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int sd = it & 1;
        const float s0v = __ldg(sc0 + kb);
        const float s1v = NMAT == 2 ? __ldg(sc1 + kb) : 0.f;
        ok = __all_sync(0xffffffffu, wait_bounded(dfull(sd), (it >> 1) & 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        uint32_t p[NMAT][NTOK];
#pragma unroll
        for (int m = 0; m < NMAT; ++m)
#pragma unroll
          for (int j0 = 0; j0 < NTOK; j0 += 16)
            tmem_ld16(tmem + lane_base + C::kATotal + (sd * NMAT + m) * NTOK + j0,
                      *reinterpret_cast<uint32_t(*)[16]>(&p[m][j0]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty(sd));
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          acc[0][j] = fmaf(s0v, __uint_as_float(p[0][j]), acc[0][j]);
          if (NMAT == 2) acc[NMAT - 1][j] = fmaf(s1v, __uint_as_float(p[NMAT - 1][j]), acc[NMAT - 1][j]);
        }
      }
      if (!ok) break;
      bool overflow = false;
      if (NMAT == 2) {
        uint16_t* h = static_cast<uint16_t*>(a.out);
        const int64_t ld = static_cast<int64_t>(n_nb) * 128;
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          if (j < td.n_valid) {
            const float g = acc[0][j], uu = acc[NMAT - 1][j];
            const float hv = g / (1.0f + expf(-g)) * uu;
            const __half hh = __float2half_rn(hv);
            overflow |= __hisinf(hh) != 0 || __hisnan(hh);
            h[static_cast<int64_t>(td.row_start + j) * ld + nb * 128 + r] = __half_as_ushort(hh);
          }
        }
      } else {
        uint16_t* rows = static_cast<uint16_t*>(a.out);
        const int64_t ld = static_cast<int64_t>(n_nb) * 128;
#pragma unroll
        for (int j = 0; j < NTOK; ++j) {
          if (j < td.n_valid) {
            const int row = td.row_start + j;
            const int dest = a.sorted_pos ? a.sorted_pos[row] : row;
            const float w = a.topk_weight ? a.topk_weight[dest] : 1.0f;
            const __half hh = __float2half_rn(acc[0][j] * w);
            overflow |= __hisinf(hh) != 0 || __hisnan(hh);
            rows[static_cast<int64_t>(dest) * ld + nb * 128 + r] = __half_as_ushort(hh);
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

template <int NMAT, int NTOK, int STAGES>
cudaError_t launch_gemm(const GemmLaunch& g, cudaStream_t s) {
  using C = Cfg<NMAT, NTOK, STAGES>;
  auto kern = moe_gemm_kernel<NMAT, NTOK, STAGES>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  GemmArgs a;
  a.s0 = g.s0;
  a.s1 = g.s1;
  a.tiles = g.tiles;
  a.n_tiles = g.n_tiles;
  a.n_nb = g.n_nb;
  a.num_kb = g.num_kb;
  a.out = g.out;
  a.sorted_pos = g.sorted_pos;
  a.topk_weight = g.topk_weight;
  a.err = g.err;
  kern<<<g.num_sms, kThreads, C::kSmem, s>>>(*g.w0, NMAT == 2 ? *g.w1 : *g.w0, *g.act, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gateup(const GemmLaunch& g, cudaStream_t s) { return launch_gemm<2, kNTok, 6>(g, s); }
cudaError_t launch_down(const GemmLaunch& g, cudaStream_t s) { return launch_gemm<1, kNTok, 10>(g, s); }

}  // namespace moe
