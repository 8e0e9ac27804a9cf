// Grouped GEMMs of the routed experts for batches with more than a few rows
// per expert, on f16 operands with the weight block scale folded in on chip.
//
// "SwiGLU output" page, MLP class: expert(x) = down(silu(gate x) * up x);
// "Element-wise product" page: h = silu(gate x) (.) (up x);
// "Mixture of experts" page, moe_infer: each expert runs on its contiguous
// slice of sorted rows, outputs return to their positions weighted by
// topk_weight; "Input features" page, quantisation config: e4m3 weights with
// one fp32 scale per 128 x 128 block.
//
// The weights are the MMA's M side (128 rows per weight block = the 128
// tensor-memory lanes) and the tokens its N side (up to 128, rounded up to a
// multiple of 16 per tile).  A unit is one token tile times two 128-row weight
// blocks: gate and up of the same output features (gate/up pass) or two
// consecutive row blocks of down (down pass).
//
//  * Converter warps read each K block's e4m3 weight tile from shared memory
//    (landed by a bulk copy of the tiled layout, or by TMA from the row-major
//    one), turn every code into f16 exactly and multiply it by the block's
//    scale times 2^cw (one f16 product, rounded to nearest), and store the
//    rows into tensor memory as the MMA's A operand.  cw is a power of two per
//    (expert, weight block), chosen from the largest scale of the block's row
//    so that 448 * scale * 2^cw stays inside [2^14, 2^15): every product is a
//    normal f16 and the rounding costs at most 2^-11 of it.
//  * Tokens arrive as f16 rows: x (or the normalised row) times a power of two
//    per token, exact for a bf16 value (gather / RMSNorm kernels); h as the
//    plain f16 of silu(g) * u.
//  * The MMAs (tcgen05.mma kind::f16, A from tensor memory, B from shared
//    memory) accumulate the whole K extent into one fp32 accumulator per
//    weight block in tensor memory.  No per-K-block partials leave the tensor
//    core: the block scales are already inside the operands.
//  * At the end of a unit the epilogue reads the accumulators once, multiplies
//    by 2^-cw (and the token's power of two), and writes
//      gate/up: h = f16(silu(g) * u)        -> h[row][feature]
//      down:    f16(topk_weight * o)        -> rows[flat position][feature]
//
// Tensor memory (512 columns): accumulators of the two weight blocks in
// columns 0-127 and 128-255 (one column per token), two A stages of 128
// columns (64 per weight block: 128 f16 of K per lane) in 256-511.
//
// Warps (512 threads = 4 warpgroups, one CTA per SM, persistent over the unit
// list; warpgroups 0 and 1 hand registers to the epilogue warpgroups):
//   0      weight producer: one 32 KB copy per K block (both tiles) into the
//          weight ring (3 stages, or 2 when the tile list marks its weights as
//          shared by the experts' several tiles)
//   1      MMA issuer (one thread, elected)
//   2      token producer: one TMA box [2 panels][rows][64 f16] per K block, the
//          tile's rows rounded up to 32, into the token ring (4 or 5 stages)
//   3      idle
//   4..7   converters: warp 4 + q owns tensor-memory lanes 32q..32q+31, i.e.
//          weight row 32q + lane of both blocks
//   8..15  epilogue: warp w reads lanes 32 (w % 4).. (output features) and
//          tokens 64 ((w - 8) / 4) .. +63 of both accumulators with one wait,
//          releases them (the next unit's MMAs start) and forms and writes its
//          outputs (straight from registers, a 64-byte store per token) while
//          the next unit's K blocks are converted and multiplied.
//
// Every wait is bounded; a wait that gives up raises the abort flag and the
// device error word, and every role drains what it has in flight before the
// kernel returns.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreadsF = 512;
constexpr int kWarpW = 0;
constexpr int kWarpMmaF = 1;
constexpr int kWarpTok = 2;
constexpr int kWarpConv = 4;   // warps 4..7: converters
constexpr int kWarpEpi = 8;    // warps 8..15: epilogue
constexpr int kTokMax = kNTokWide;
constexpr int kWTileF = 128 * 128;             // e4m3 bytes of one 128 x 128 weight tile
constexpr int kWStageF = 2 * kWTileF;          // both weight blocks of one K block
constexpr int kTPanel = kTokMax * 128;         // one 64-column panel of 128 token rows (f16)
constexpr int kTStage = 2 * kTPanel;           // a K block of 128 tokens: two panels, one TMA box
constexpr uint32_t kTmemColsF = 512;
constexpr uint32_t kAccCols = 128;             // accumulator columns per weight block
constexpr uint32_t kAOff = 256;                // first A stage column
constexpr uint32_t kAStageCols = 128;          // both blocks' A of one K block
constexpr int kAStages = 2;

// Registers per thread after the split: warpgroup 0 (copies, MMA) and the
// converters (warpgroup 1) give up registers, the two epilogue warpgroups take
// them.  Each warpgroup executes exactly one setmaxnreg.  The pool is the
// launch's threads x the kernel's register count (128 at 512 threads); the
// launcher checks that the split fits it before every launch, since an increase
// that cannot be met never returns.
constexpr int kRegsLow = 56;
constexpr int kRegsConv = 96;
constexpr int kRegsEpi = 176;
constexpr int kRegsAtLaunch = 128;  // 65536 / 512
static_assert(128 * kRegsLow + 128 * kRegsConv + 256 * kRegsEpi <= kThreadsF * kRegsAtLaunch, "register split");

// Seven 32 KB operand stages, split between the weight ring and the token ring
// at run time: 3 + 4 when weights stream from DRAM, 2 + 5 when nearly every
// tile's weights are shared with the expert's other tiles (they come from L2
// after the first tile, and the token stream needs the deeper ring).
struct F16Cfg {
  static constexpr int kStages = 7;
  static constexpr int kWMax = 3;   // weight stages at most
  static constexpr int kTMax = 5;   // token stages at most
  static constexpr int kBarOff = kStages * kWStageF;
  // full / empty of each ring at its largest, A stages, accumulators full / empty, drain
  static constexpr int kNumBars = 2 * kWMax + 2 * kTMax + 2 * kAStages + 2 + 1;
  static constexpr int kSmem = 1024 + kBarOff + kNumBars * 8 + 16;
  static_assert(kWStageF == kTStage && kTStage % 1024 == 0, "operand stages stay 1024-byte aligned");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

// Stage and phase parity of the i-th use of a ring of A (is_a) or B stages;
// both sizes are compile-time constants, so no division at run time.
template <int A, int B>
__device__ __forceinline__ int ring_stage(uint32_t i, bool is_a, uint32_t& parity) {
  const uint32_t q = is_a ? i / A : i / B;
  parity = q & 1u;
  return static_cast<int>(i - q * (is_a ? A : B));
}

struct F16Args {
  const uint8_t* w_tiled;   // non-null: tiled layout (both blocks of a K block in 32 KB), bulk copies
  const float* s0;          // [E][n_nb][num_kb]
  const float* s1;
  const TileDesc* tiles;
  const int32_t* n_tiles;
  int32_t n_nb;             // 128-row blocks of the weight matrix
  int32_t num_kb;           // K / 128
  int32_t pair;             // 1: unit = row blocks 2j, 2j+1 of w0 (down); 0: row block j of w0 and w1
  const float* tok_scale;   // [act_rows] power of two the token's f16 row was divided by (NULL = 1)
  int32_t act_rows;         // rows of the token matrix (and of h)
  void* out;                // gate/up: h in panels [n_nb*2][act_rows][64] f16; down: rows [.][n_nb*128] f16
  const int32_t* sorted_pos;
  const float* topk_weight;
  uint32_t* err;
};

struct UnitF {
  int e, row0, nv, ru, nb0, nb1;
  int reuse;  // tiles of the unit's chunk: units that read the same weights side by side
  bool has1;
};

// Unit u: within each chunk of an expert's tiles the units run weight-row
// block first (the tile list's chunk field), as in the e4m3 wide kernel, so
// the tiles reading the same weights run side by side and share them in L2.
__device__ __forceinline__ UnitF unit_f(const F16Args& a, int u, int upt) {
  const int code = a.tiles[u / upt].chunk;
  const int first = u / upt - (code & 0xff), n = code >> 8;
  const int l = u - first * upt;
  const TileDesc td = a.tiles[first + l % n];
  const int j = l / n;
  UnitF x;
  x.e = td.expert;
  x.row0 = td.row_start;
  x.nv = td.n_valid;
  x.ru = j;
  x.nb0 = a.pair ? 2 * j : j;
  x.nb1 = a.pair ? 2 * j + 1 : j;
  x.has1 = x.nb1 < a.n_nb;
  x.reuse = n;
  return x;
}

// Rows of the token box that brings a tile of nv rows: nv rounded up to 32 (the
// maps hold boxes of 32, 64, 96 and 128 rows).  The box's second panel starts
// right after its rows, at rows * 128 bytes (a multiple of 4 KB).
__device__ __forceinline__ int box_rows_of(int nv) { return min(kTokMax, (max(nv, 1) + 31) & ~31); }

__device__ __forceinline__ void wait_drain_f(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return;
}

// The power of two cw of one weight block: 448 * max_kb scale[kb] * 2^cw lies in
// [2^14, 2^15), so every code * scale * 2^cw is a normal f16 below 2^15.  All 32
// lanes of the calling warp take part; every lane returns the same value.
// Limited to [-100, 100] (scales outside about 2^-110..2^90 are not in use).
__device__ __forceinline__ int pow2_of_max(float m) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float v = m * 448.0f;
  if (!(v > 0.f) || !(v < 3.0e38f)) return 0;
  int ex;
  frexpf(v, &ex);  // v = f * 2^ex, f in [0.5, 1)
  return max(-100, min(100, 15 - ex));
}
// A weight block's scales held by a warp, lane l keeping K blocks l and l + 32
// (the rest, for K above 64 blocks, is read when used).
struct BlockScales {
  const float* sc;
  float lo, hi;
  int cw;
  __device__ __forceinline__ void load(const float* p, int num_kb, int lane) {
    sc = p;
    lo = lane < num_kb ? __ldg(p + lane) : 0.f;
    hi = lane + 32 < num_kb ? __ldg(p + lane + 32) : 0.f;
    float m = fmaxf(lo, hi);
    for (int kb = lane + 64; kb < num_kb; kb += 32) m = fmaxf(m, __ldg(p + kb));
    cw = pow2_of_max(m);
  }
  // scale of K block kb (warp-uniform kb; every lane takes part)
  __device__ __forceinline__ float at(int kb) const {
    const float v = __shfl_sync(0xffffffffu, kb < 32 ? lo : hi, kb & 31);
    return kb < 64 ? v : __ldg(sc + kb);
  }
};

// 16 e4m3 codes (16 consecutive K of one weight row) -> 8 words of two f16,
// each code * s2 rounded to nearest (lower K in the low half).
__device__ __forceinline__ void cvt16_scaled(const uint4 v, __half2 s2, uint32_t* o) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] & 0xffffu), __NV_E4M3);
    const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w[q] >> 16), __NV_E4M3);
    const __half2 a = __hmul2(__half2(lo), s2), b = __hmul2(__half2(hi), s2);
    o[2 * q] = *reinterpret_cast<const uint32_t*>(&a);
    o[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&b);
  }
}

__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// End of a unit for one epilogue warp (lanes 32q.. = output features 32q..,
// tokens 64 half .. + 63): read the warp's 64 columns of both accumulators
// with one wait and release them; then, token by token, form the outputs and
// write them straight from registers: the 32 lanes hold 32 consecutive
// features of the token, one 64-byte store per token and weight block.
template <bool GATEUP>
__device__ __forceinline__ bool unit_epilogue(const F16Args& a, const UnitF un, const int cw0, const int cw1,
                                              const uint32_t ui, const uint32_t tmem, const int q, const int half,
                                              const uint32_t dfull, const uint32_t dempty,
                                              volatile uint32_t* abort_flag) {
  const int lane = threadIdx.x & 31;
  const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
  const float f0 = ldexpf(1.0f, -cw0), f1 = ldexpf(1.0f, -cw1);
  const int t0 = half * 64;
  const int nt = min(64, un.nv - t0);  // valid tokens of this warp (may be <= 0)
  const bool has1 = GATEUP || un.has1;
  // per-token values, lane l holding tokens t0 + l and t0 + 32 + l
  float tf[2];
  int dstv[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = t0 + lane + 32 * i;
    const int64_t row = un.row0 + t;
    tf[i] = 1.0f;
    dstv[i] = static_cast<int>(row);
    if (t < un.nv) {
      if (GATEUP) {
        if (a.tok_scale) tf[i] = __ldg(a.tok_scale + row);
      } else {
        dstv[i] = a.sorted_pos ? __ldg(a.sorted_pos + row) : static_cast<int>(row);
        tf[i] = a.topk_weight ? __ldg(a.topk_weight + dstv[i]) : 1.0f;
      }
    }
  }
  if (!__all_sync(0xffffffffu, wait_bounded(dfull, ui & 1, abort_flag, a.err))) return false;
  tc_fence_after();
  uint32_t p0[64], p1[64];
  if (nt > 0) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      tmem_ld16(tmem + lane_base + t0 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&p0[16 * c]));
      if (has1) tmem_ld16(tmem + lane_base + kAccCols + t0 + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&p1[16 * c]));
    }
    tmem_ld_wait();
  }
  // the accumulators are in registers: the next unit's MMAs may overwrite them
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(dempty);
  bool overflow = false;
  const int f = q * 32 + lane;  // this lane's feature within the 128-row block
#pragma unroll
  for (int jj = 0; jj < 64; ++jj) {
    if (jj >= nt) break;
    const float tfj = __shfl_sync(0xffffffffu, tf[jj >> 5], jj & 31);
    const int dst = __shfl_sync(0xffffffffu, dstv[jj >> 5], jj & 31);
    if (GATEUP) {
      const float gg = __uint_as_float(p0[jj]) * (f0 * tfj), uu = __uint_as_float(p1[jj]) * (f1 * tfj);
      const float v0 = silu_f(gg) * uu;
      overflow |= !(fabsf(v0) < 65520.f);  // f16 rounds these to inf
      // h panels of 64 features: panel 2 nb0 + f / 64, row dst (the sorted row)
      const int64_t panel = 2 * un.nb0 + (f >> 6);
      *reinterpret_cast<__half*>(static_cast<uint8_t*>(a.out) + panel * a.act_rows * 128 +
                                 static_cast<int64_t>(dst) * 128 + (f & 63) * 2) = __float2half_rn(v0);
    } else {
      __half* orow = static_cast<__half*>(a.out) + static_cast<int64_t>(dst) * a.n_nb * 128;
      const float v0 = __uint_as_float(p0[jj]) * (f0 * tfj);
      overflow |= !(fabsf(v0) < 65520.f);
      orow[un.nb0 * 128 + f] = __float2half_rn(v0);
      if (has1) {
        const float v1 = __uint_as_float(p1[jj]) * (f1 * tfj);
        overflow |= !(fabsf(v1) < 65520.f);
        orow[un.nb1 * 128 + f] = __float2half_rn(v1);
      }
    }
  }
  if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(a.err, DEV_ERR_RANGE);
  return true;
}

__device__ __forceinline__ void regs_dec_low() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsLow));
}
__device__ __forceinline__ void regs_dec_conv() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsConv));
}
__device__ __forceinline__ void regs_inc_epi() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
}

template <bool GATEUP>
__global__ void __launch_bounds__(kThreadsF, 1)
moe_gemm_f16_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                    const __grid_constant__ CUtensorMap tm_tok, const __grid_constant__ CUtensorMap tm_tok32,
                    const __grid_constant__ CUtensorMap tm_tok64, const __grid_constant__ CUtensorMap tm_tok96,
                    const F16Args a) {
  using C = F16Cfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  constexpr int WM = C::kWMax, TM = C::kTMax;
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto empty_w = [&](int i) { return bar0 + 8u * (WM + i); };
  auto full_t = [&](int i) { return bar0 + 8u * (2 * WM + i); };
  auto empty_t = [&](int i) { return bar0 + 8u * (2 * WM + TM + i); };
  auto afull = [&](int i) { return bar0 + 8u * (2 * WM + 2 * TM + i); };
  auto aempty = [&](int i) { return bar0 + 8u * (2 * WM + 2 * TM + kAStages + i); };
  const uint32_t dfull = bar0 + 8u * (2 * WM + 2 * TM + 2 * kAStages);
  const uint32_t dempty = dfull + 8u;
  const uint32_t drain_bar = bar0 + 8u * (C::kNumBars - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < WM; ++i) {
      mbar_init(full_w(i), 1);
      mbar_init(empty_w(i), 4);  // the four converter warps
    }
    for (int i = 0; i < TM; ++i) {
      mbar_init(full_t(i), 1);
      mbar_init(empty_t(i), 1);  // one MMA commit
    }
    for (int i = 0; i < kAStages; ++i) {
      mbar_init(afull(i), 4);    // the four converter warps
      mbar_init(aempty(i), 1);   // one MMA commit
    }
    mbar_init(dfull, 1);
    mbar_init(dempty, 8);        // the eight epilogue warps
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpW && lane == 0) {
    if (!a.w_tiled) {
      prefetch_tmap(&tm_w0);
      prefetch_tmap(&tm_w1);
    }
    prefetch_tmap(&tm_tok);
    prefetch_tmap(&tm_tok32);
    prefetch_tmap(&tm_tok64);
    prefetch_tmap(&tm_tok96);
  }
  if (warp == kWarpMmaF) {
    tmem_alloc(smem_u32(tmem_slot), kTmemColsF);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_nb = a.n_nb, num_kb = a.num_kb;
  const int upt = a.pair ? (n_nb + 1) / 2 : n_nb;  // units per tile
  const int total_units = a.n_tiles[0] * upt;
  // the stage split (set with the tile list): weight stages 3 (w3) or 2, token stages the rest
  const bool w3 = a.n_tiles[2] == 0;
  const uint32_t tbase = sbase + (w3 ? 3 : 2) * kWStageF;
  // tiled layout: K block kb of unit row ru of expert e, both blocks (32 KB)
  auto unit_off = [&](int e, int ru, int kb) {
    return ((static_cast<int64_t>(e) * upt + ru) * num_kb + kb) * kWStageF;
  };

  if (warp < kWarpConv) regs_dec_low();  // warpgroup 0: copies, MMA
  if (warp == kWarpW) {
    if (lane == 0) {
      // weights read by one tile leave L2 first; weights that the chunk's other tiles
      // read next to it stay at normal priority
      const uint64_t pol_once = policy_evict_first(), pol_shared = policy_evict_normal();
      uint32_t wi = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const UnitF un = unit_f(a, u, upt);
        const uint64_t pol_w = un.reuse > 1 ? pol_shared : pol_once;
        for (int kb = 0; kb < num_kb; ++kb) {
          uint32_t pw;
          const int sw = ring_stage<3, 2>(wi, w3, pw);
          if (!wait_bounded(empty_w(sw), pw ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + sw * kWStageF;
          if (a.w_tiled) {
            mbar_arrive_expect_tx(full_w(sw), kWStageF);
            bulk_load(dst, a.w_tiled + unit_off(un.e, un.ru, kb), kWStageF, full_w(sw), pol_w);
          } else {
            mbar_arrive_expect_tx(full_w(sw), (un.has1 ? 2 : 1) * kWTileF);
            tma_load_3d(dst, &tm_w0, full_w(sw), kb * 128, un.nb0 * 128, un.e, pol_w);
            if (un.has1) tma_load_3d(dst + kWTileF, &tm_w1, full_w(sw), kb * 128, un.nb1 * 128, un.e, pol_w);
          }
          ++wi;
        }
      }
      if (!ok) {
        const uint32_t nw = w3 ? 3u : 2u;  // copies possibly in flight: the ring's last uses
        for (uint32_t i = wi > nw ? wi - nw : 0; i < wi; ++i) {
          uint32_t pw;
          const int sw = ring_stage<3, 2>(i, w3, pw);
          wait_drain_f(full_w(sw), pw);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpTok) {
    pdl_wait();  // the token rows are the previous kernel's output
    // Everything before this kernel in the stream has completed: the dependent launch
    // behind it may be placed and stream its weights.
    pdl_launch_dependents();
    if (lane == 0) {
      const uint64_t pol_t = policy_evict_last();
      uint32_t ti = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const UnitF un = unit_f(a, u, upt);
        // the tile's rows rounded up to 32: the box that brings them (panel 1 follows its rows)
        const int rb = box_rows_of(un.nv);
        const CUtensorMap* tm = rb == 32 ? &tm_tok32 : rb == 64 ? &tm_tok64 : rb == 96 ? &tm_tok96 : &tm_tok;
        for (int kb = 0; kb < num_kb; ++kb) {
          uint32_t pt;
          const int st = ring_stage<4, 5>(ti, w3, pt);
          if (!wait_bounded(empty_t(st), pt ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = tbase + st * kTStage;
          mbar_arrive_expect_tx(full_t(st), rb * 256);
          tma_load_3d(dst, tm, full_t(st), 0, un.row0, 2 * kb, pol_t);  // panels 2 kb and 2 kb + 1
          ++ti;
        }
      }
      if (!ok) {
        const uint32_t nt = w3 ? 4u : 5u;
        for (uint32_t i = ti > nt ? ti - nt : 0; i < ti; ++i) {
          uint32_t pt;
          const int st = ring_stage<4, 5>(i, w3, pt);
          wait_drain_f(full_t(st), pt);
        }
      }
    }
    __syncwarp();
  } else if (warp == kWarpMmaF) {
    // One elected thread runs the whole loop: its waits, MMAs and commits.
    if (elect_one()) {
      uint32_t it = 0, ui = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ui) {
        const UnitF un = unit_f(a, u, upt);
        const int n_mma = (max(un.nv, 1) + 15) & ~15;  // N: the tile's rows, a multiple of 16
        const uint32_t idesc = idesc_f16_f32(128, n_mma);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          uint32_t pt;
          const int st = ring_stage<4, 5>(it, w3, pt), sa = it % kAStages;
          // the first K block overwrites the accumulators: they must have been read out
          if ((kb == 0 && !wait_bounded(dempty, (ui & 1) ^ 1, abort_flag, a.err)) ||
              !wait_bounded(full_t(st), pt, abort_flag, a.err) ||
              !wait_bounded(afull(sa), (it / kAStages) & 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t tb = tbase + st * kTStage;
          const uint64_t bdesc0 = desc_kmajor_sw128(tb), bdesc1 = desc_kmajor_sw128(tb + box_rows_of(un.nv) * 128);
#pragma unroll
          // K step outer, weight block inner: the two MMAs of a K step read the same token slice
          // back to back (measured 7.5 % faster on gate/up of the full block than block outer)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = desc_advance(kk < 4 ? bdesc0 : bdesc1, (kk & 3) * 32);
#pragma unroll
            for (int m = 0; m < 2; ++m) {
              if (m == 1 && !un.has1) break;
              mma_f16_ts(tmem + m * kAccCols, tmem + kAOff + sa * kAStageCols + m * 64 + kk * 8, bd, idesc,
                         (kb > 0 || kk > 0) ? 1u : 0u);
            }
          }
          tc_commit(empty_t(st));
          tc_commit(aempty(sa));
          if (kb == num_kb - 1) tc_commit(dfull);
        }
      }
      tc_commit(drain_bar);  // every MMA issued above has completed once this arrives
      wait_drain_f(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpConv && warp < kWarpEpi) {
    // converters: weight row r of both blocks, K block by K block, into the A stages
    regs_dec_conv();
    const int q = warp - kWarpConv;
    const int r = q * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
      const UnitF un = unit_f(a, u, upt);
      BlockScales b0, b1;
      b0.load(a.s0 + (static_cast<int64_t>(un.e) * n_nb + un.nb0) * num_kb, num_kb, lane);
      b1.load(a.s1 + (static_cast<int64_t>(un.e) * n_nb + (un.has1 ? un.nb1 : un.nb0)) * num_kb, num_kb, lane);
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        uint32_t pw;
        const int sw = ring_stage<3, 2>(it, w3, pw), sa = it % kAStages;
        const float s0v = b0.at(kb), s1v = b1.at(kb);
        // Every lane waits (each gets the barrier's acquire); the vote keeps the warp
        // converged for the .sync.aligned tensor-memory stores.
        ok = __all_sync(0xffffffffu, wait_bounded(full_w(sw), pw, abort_flag, a.err) &&
                                         wait_bounded(aempty(sa), ((it / kAStages) & 1) ^ 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m == 1 && !un.has1) break;
          const __half2 s2 = __half2half2(__float2half_rn(m == 0 ? ldexpf(s0v, b0.cw) : ldexpf(s1v, b1.cw)));
          const uint32_t row = sbase + sw * kWStageF + m * kWTileF + r * 128;
#pragma unroll
          for (int hv = 0; hv < 2; ++hv) {  // half a row (64 codes) at a time
            uint32_t v[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) cvt16_scaled(lds128(row + (((4 * hv + c) ^ (r & 7)) << 4)), s2, v + 8 * c);
            const uint32_t taddr = tmem + lane_base + kAOff + sa * kAStageCols + m * 64 + hv * 32;
            tmem_st16(taddr, v);
            tmem_st16(taddr + 16, v + 16);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(afull(sa));
          mbar_arrive(empty_w(sw));
        }
      }
    }
  } else if (warp >= kWarpEpi) {
    // epilogue: the accumulators of each unit, read once at its end
    regs_inc_epi();
    pdl_wait();  // token scales, positions and router weights come from earlier kernels
    const int q = warp & 3;
    const int half = (warp - kWarpEpi) >> 2;
    uint32_t ui = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x, ++ui) {
      const UnitF un = unit_f(a, u, upt);
      const float* sc0 = a.s0 + (static_cast<int64_t>(un.e) * n_nb + un.nb0) * num_kb;
      const float* sc1 = a.s1 + (static_cast<int64_t>(un.e) * n_nb + (un.has1 ? un.nb1 : un.nb0)) * num_kb;
      float m0 = 0.f, m1 = 0.f;
      for (int kb = lane; kb < num_kb; kb += 32) {
        m0 = fmaxf(m0, __ldg(sc0 + kb));
        m1 = fmaxf(m1, __ldg(sc1 + kb));
      }
      const int cw0 = pow2_of_max(m0), cw1 = pow2_of_max(m1);
      if (!unit_epilogue<GATEUP>(a, un, cw0, cw1, ui, tmem, q, half, dfull, dempty, abort_flag)) break;
    }
  }
  __syncthreads();
  if (warp == kWarpMmaF) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsF);
  }
}

template <bool GATEUP>
cudaError_t launch_f16(const GemmLaunch& g, cudaStream_t s) {
  using C = F16Cfg;
  auto kern = moe_gemm_f16_kernel<GATEUP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (!g.act_box || !g.act_box_rows[0] || !g.act_box_rows[1] || !g.act_box_rows[2]) return cudaErrorInvalidValue;
  // The register split waits until the pool covers it: launch only if it does.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kThreadsF < 128 * kRegsLow + 128 * kRegsConv + 256 * kRegsEpi) return cudaErrorInvalidConfiguration;
  F16Args a;
  a.w_tiled = g.w_tiled;
  a.s0 = g.s0;
  a.s1 = g.s1;
  a.tiles = g.tiles;
  a.n_tiles = g.n_tiles;
  a.n_nb = g.n_nb;
  a.num_kb = g.num_kb;
  a.pair = GATEUP ? 0 : 1;
  a.tok_scale = g.act_inv;
  a.act_rows = g.act_rows;
  a.out = g.out;
  a.sorted_pos = g.sorted_pos;
  a.topk_weight = g.topk_weight;
  a.err = g.err;
  // gate/up behind the row gather, down behind gate/up: dependent launches that stream
  // weights while their predecessor drains (both wait for its rows before reading them)
  return launch_maybe_overlapped(kern, g.num_sms, kThreadsF, C::kSmem, s, GATEUP ? g.overlap : true, *g.w0, *g.w1,
                                 *g.act_box, *g.act_box_rows[0], *g.act_box_rows[1], *g.act_box_rows[2], a);
}

}  // namespace

// Stages: seven 32 KB operand stages (F16Cfg), three for weights (both blocks of
// one K block; released as soon as they are converted) and four for tokens (128
// rows x 128 f16, one TMA box each), or two and five when the tile list marks its
// weights as shared; 225 KB of shared memory.  What bounds the K-block period
// (timestamps, copy probes, timing-only knock-outs): with one tile per expert
// the weight stream from DRAM (the gate/up pass reaches the copy bandwidth);
// with several tiles per expert the tensor pipe and the token stream, whose
// boxes queue behind the SM's weight copies (~3,000 cycles from issue to use).
cudaError_t launch_gateup_f16(const GemmLaunch& g, cudaStream_t s) { return launch_f16<true>(g, s); }
cudaError_t launch_down_f16(const GemmLaunch& g, cudaStream_t s) { return launch_f16<false>(g, s); }

}  // namespace moe
