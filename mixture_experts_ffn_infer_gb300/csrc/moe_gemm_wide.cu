// Grouped GEMMs of the routed experts for batches with more than a few rows
// per expert, under dynamic FP8 activations.
//
// "SwiGLU output" page, MLP class: expert(x) = down(silu(gate x) * up x);
// "Mixture of experts" page, moe_infer: each expert runs on its contiguous
// slice of sorted rows, outputs return to their positions weighted by
// topk_weight; "Input features" page, quantisation config: e4m3 weights with
// one fp32 scale per 128 x 128 block, activation_scheme "dynamic" (e4m3
// activations with one scale amax / 448 per 128 features).
//
// Weights and activations are both e4m3 codes, straight into tcgen05.mma
// kind::f8f6f4; each K block (128) of the product gets its own fp32 partial,
// multiplied by the weight block's scale and the activation group's scale in
// the epilogue.  The arrangement is for tiles of up to 128 tokens:
//
//  * Tokens are the MMA's M side (128 rows = the 128 tensor-memory lanes) and
//    two 128-row weight blocks its N side (N = 256): gate and up of the same
//    output features (gate/up pass) or two consecutive row blocks of down
//    (down pass).  The two 16 KB weight tiles of a K block sit back to back in
//    shared memory and form one 256-row operand.
//  * Two partial buffers of 256 columns fill tensor memory's 512 columns.
//  * An epilogue thread owns one token (its tensor-memory lane) and 64 output
//    features of each weight block.  Per K block it adds
//    s_weight * s_act * partial to fp32 registers; at the end of a unit it
//    writes its token's features with 32-byte stores.
//
// Warps (384 threads = 3 warpgroups, one CTA per SM, persistent over the unit
// list; warpgroup 0 hands registers to the epilogue warpgroups):
//   0      weight producer: the K block's two 16 KB tiles (one 32 KB bulk copy
//          of the tiled layout, or 3-D TMA of the row-major layout), and an L2
//          prefetch ahead when several token tiles share an expert's weights
//   1      MMA issuer (one thread, elected)
//   2      activation producer: one TMA box [128 rows][128 bytes] per K block
//   3      idle
//   4..11  epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31 (the
//          tile's tokens) and features 64 ((w - 4) / 4) .. +63 of each block
//
// At the end of a unit the gate/up epilogue forms h = silu(g) * u, takes each
// token's maximum over the 128 features of the unit (its 64 and the other
// half's, exchanged as floats through shared memory and an eight-arrival
// mbarrier) and writes the codes of h / s, s = amax / 448; the down epilogue
// writes f16(topk_weight * o) to the row's flat position.  Every wait is
// bounded; a wait that gives up raises the abort flag and the device error
// word, and every role drains what it has in flight before the kernel returns.
#include <cuda_fp16.h>

#include "common.cuh"
#include "split3.cuh"

namespace moe {
namespace {

constexpr int kThreadsW = 384;
constexpr int kWarpWeights = 0;
constexpr int kWarpIssue = 1;
constexpr int kWarpAct = 2;
constexpr int kWarpEpi = 4;  // warps 4..11 (warpgroups 1 and 2)
constexpr int kTileMax = kNTokWide;
constexpr int kHalfF = 64;   // output features of each block per epilogue thread
constexpr uint32_t kTmemColsW = 512;
constexpr int kWTileBytes = 128 * 128;

template <int WST, int AST>
struct WideCfg {
  static constexpr int kWStage = 2 * kWTileBytes;          // both weight blocks of one K block
  static constexpr int kAStage = kTileMax * 128;           // the activation box: 128 rows of codes
  static constexpr int kAOff = WST * kWStage;
  // h block maxima [parity][half][128 tokens]
  static constexpr int kRedOff = kAOff + AST * kAStage;
  static constexpr int kRedBytes = 2 * 2 * kTileMax * 4;
  static constexpr int kBarOff = kRedOff + kRedBytes;
  static constexpr int kNumBars = 2 * WST + 2 * AST + 2 * 2 + 2 + 1;
  static constexpr int kSmem = 1024 + kBarOff + kNumBars * 8 + 16;
  static constexpr int kPrefetch = (128 * 1024) / kWStage;  // L2 prefetch distance in K blocks
  static_assert(kAStage % 1024 == 0 && kAOff % 1024 == 0, "operand stages stay 1024-byte aligned");
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

struct WideArgs {
  const uint8_t* w_tiled;   // non-null: tiled layout (both blocks of a K block in 32 KB), bulk copies
  const float* s0;          // [E][n_nb][num_kb]
  const float* s1;
  const TileDesc* tiles;
  const int32_t* n_tiles;
  int32_t n_nb;             // 128-row blocks of the weight matrix
  int32_t num_kb;           // K / 128
  int32_t pair;             // 1: unit = row blocks 2j, 2j+1 of w0 (down); 0: row block j of w0 and w1
  int32_t l2_prefetch;      // prefetch weights into L2 ahead of their copies
  const float* act_inv;     // [num_kb][act_rows]
  int32_t act_rows;
  void* out;                // gate/up: h term planes [3][act_rows][n_nb*128]; down: rows [.][n_nb*128] f16
  float* out_inv;           // gate/up: [n_nb][act_rows]
  const int32_t* sorted_pos;
  const float* topk_weight;
  uint32_t* err;
};

struct Unit {
  int e, row0, nv, ru, nb0, nb1;
  bool has1;
};

// Unit u.  Within each chunk of an expert's tiles the units run weight-row
// block first: the chunk's n tiles take units first*upt .. (first+n)*upt - 1,
// unit row j of tile first + i being unit first*upt + j*n + i, so the tiles
// that read the same weights are neighbours in the unit list and run at the
// same time (their weights are read from DRAM once and from L2 after that).
__device__ __forceinline__ Unit unit_of(const WideArgs& a, int u, int upt) {
  const int code = a.tiles[u / upt].chunk;  // a tile of the same chunk
  const int first = u / upt - (code & 0xff), n = code >> 8;
  const int l = u - first * upt;
  const TileDesc td = a.tiles[first + l % n];
  const int j = l / n;
  Unit x;
  x.e = td.expert;
  x.row0 = td.row_start;
  x.nv = td.n_valid;
  x.ru = j;
  x.nb0 = a.pair ? 2 * j : j;
  x.nb1 = a.pair ? 2 * j + 1 : j;
  x.has1 = x.nb1 < a.n_nb;
  return x;
}

__device__ __forceinline__ void wait_drain_w(uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitLimitCycles) return;
}

// Registers per thread after the split: warpgroup 0 (copies, MMA) gives up
// registers, the two epilogue warpgroups take them.  The pool is the launch's
// threads x the kernel's register count; the launcher checks that the split
// fits it before every launch, since an increase that cannot be met never returns.
constexpr int kRegsProducer = 56;
constexpr int kRegsEpilogue = 224;
constexpr int kRegsAtLaunch = 168;  // 65536 / 384, rounded down to a multiple of 8
static_assert(128 * kRegsProducer + 256 * kRegsEpilogue <= kThreadsW * kRegsAtLaunch, "register split");

__device__ __forceinline__ void regs_dec_producer() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsProducer));
}
__device__ __forceinline__ void regs_inc_epilogue() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpilogue));
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                       uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&p)[64]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld16(taddr + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&p[16 * c]));
}

// silu(g) = g / (1 + e^-g) with the fast exponential and division; for
// g < -87 the denominator overflows and the result is 0 (the exact value is
// below 1e-36).
__device__ __forceinline__ float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

template <bool GATEUP, int WST, int AST>
__global__ void __launch_bounds__(kThreadsW, 1)
moe_gemm_wide_kernel(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
                     const __grid_constant__ CUtensorMap tm_act, const WideArgs a) {
  using C = WideCfg<WST, AST>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + C::kBarOff;
  auto full_w = [&](int i) { return bar0 + 8u * i; };
  auto empty_w = [&](int i) { return bar0 + 8u * (WST + i); };
  auto full_a = [&](int i) { return bar0 + 8u * (2 * WST + i); };
  auto empty_a = [&](int i) { return bar0 + 8u * (2 * WST + AST + i); };
  auto dfull = [&](int i) { return bar0 + 8u * (2 * WST + 2 * AST + i); };
  auto dempty = [&](int i) { return bar0 + 8u * (2 * WST + 2 * AST + 2 + i); };
  auto redbar = [&](int par) { return bar0 + 8u * (2 * WST + 2 * AST + 4 + par); };
  const uint32_t drain_bar = bar0 + 8u * (C::kNumBars - 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kBarOff + C::kNumBars * 8);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  uint8_t* red = smem + C::kRedOff;

  // the down pass's dependent (the combine) may be placed now; it waits for this grid to end
  if (!GATEUP) pdl_launch_dependents();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < WST; ++i) {
      mbar_init(full_w(i), 1);
      mbar_init(empty_w(i), 1);
    }
    for (int i = 0; i < AST; ++i) {
      mbar_init(full_a(i), 1);
      mbar_init(empty_a(i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(dfull(i), 1);
      mbar_init(dempty(i), 8);  // the eight epilogue warps
      mbar_init(redbar(i), 8);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == kWarpWeights && lane == 0) {
    if (!a.w_tiled) {
      prefetch_tmap(&tm_w0);
      prefetch_tmap(&tm_w1);
    }
    prefetch_tmap(&tm_act);
  }
  if (warp == kWarpIssue) {
    tmem_alloc(smem_u32(tmem_slot), kTmemColsW);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int n_nb = a.n_nb, num_kb = a.num_kb;
  const int upt = a.pair ? (n_nb + 1) / 2 : n_nb;  // units per tile
  const int total_units = *a.n_tiles * upt;
  // tiled layout: K block kb of unit row ru of expert e, both blocks (32 KB)
  auto unit_off = [&](int e, int ru, int kb) {
    return ((static_cast<int64_t>(e) * upt + ru) * num_kb + kb) * (2 * kWTileBytes);
  };

  if (warp < kWarpEpi) regs_dec_producer();
  if (warp == kWarpWeights) {
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int pf_u = blockIdx.x, pf_kb = 0;
      Unit pf{};
      auto prefetch_one = [&]() {
        if (!a.l2_prefetch || pf_u >= total_units) return;
        if (pf_kb == 0) pf = unit_of(a, pf_u, upt);
        if (a.w_tiled) {
          bulk_prefetch_l2(a.w_tiled + unit_off(pf.e, pf.ru, pf_kb), 2 * kWTileBytes);
        } else {
          tma_prefetch_3d(&tm_w0, pf_kb * 128, pf.nb0 * 128, pf.e);
          if (pf.has1) tma_prefetch_3d(&tm_w1, pf_kb * 128, pf.nb1 * 128, pf.e);
        }
        if (++pf_kb == num_kb) {
          pf_kb = 0;
          pf_u += gridDim.x;
        }
      };
      for (int i = 0; i < C::kPrefetch; ++i) prefetch_one();
      uint32_t wi = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit un = unit_of(a, u, upt);
        for (int kb = 0; kb < num_kb; ++kb) {
          const int sw = wi % WST;
          if (!wait_bounded(empty_w(sw), ((wi / WST) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          const uint32_t dst = sbase + sw * C::kWStage;
          if (a.w_tiled) {
            // both weight blocks of the K block are one contiguous 32 KB image
            mbar_arrive_expect_tx(full_w(sw), 2 * kWTileBytes);
            bulk_load(dst, a.w_tiled + unit_off(un.e, un.ru, kb), 2 * kWTileBytes, full_w(sw), pol_w);
          } else {
            mbar_arrive_expect_tx(full_w(sw), (un.has1 ? 2 : 1) * kWTileBytes);
            tma_load_3d(dst, &tm_w0, full_w(sw), kb * 128, un.nb0 * 128, un.e, pol_w);
            if (un.has1) tma_load_3d(dst + kWTileBytes, &tm_w1, full_w(sw), kb * 128, un.nb1 * 128, un.e, pol_w);
          }
          ++wi;
          prefetch_one();
        }
      }
      if (!ok)
        for (uint32_t i = wi > WST ? wi - WST : 0; i < wi; ++i) wait_drain_w(full_w(i % WST), (i / WST) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpAct) {
    pdl_wait();  // the activations are the previous kernel's output
    if (lane == 0) {
      const uint64_t pol_a = policy_evict_last();
      uint32_t ai = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const int row0 = unit_of(a, u, upt).row0;
        for (int kb = 0; kb < num_kb; ++kb) {
          const int sa = ai % AST;
          if (!wait_bounded(empty_a(sa), ((ai / AST) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_a(sa), C::kAStage);
          tma_load_3d(sbase + C::kAOff + sa * C::kAStage, &tm_act, full_a(sa), kb * 128, row0, 0, pol_a);
          ++ai;
        }
      }
      if (!ok)
        for (uint32_t i = ai > AST ? ai - AST : 0; i < ai; ++i) wait_drain_w(full_a(i % AST), (i / AST) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpIssue) {
    // One elected thread runs the whole loop: its waits, MMAs and commits.
    if (elect_one()) {
      uint32_t it = 0;
      bool ok = true;
      for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x) {
        const Unit un = unit_of(a, u, upt);
        // kind::f8f6f4 with E4M3 operands: format code 0, the same bits as f16
        const uint32_t idesc = idesc_f16_f32(128, un.has1 ? 256 : 128);
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int sw = it % WST, sa = it % AST, sd = it & 1;
          if (!wait_bounded(full_w(sw), (it / WST) & 1, abort_flag, a.err) ||
              !wait_bounded(full_a(sa), (it / AST) & 1, abort_flag, a.err) ||
              !wait_bounded(dempty(sd), ((it >> 1) & 1) ^ 1, abort_flag, a.err)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t wdesc = desc_kmajor_sw128(sbase + sw * C::kWStage);
          const uint64_t adesc = desc_kmajor_sw128(sbase + C::kAOff + sa * C::kAStage);
          const uint32_t d = tmem + static_cast<uint32_t>(sd) * 256;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_f8(d, desc_advance(adesc, kk * 32), desc_advance(wdesc, kk * 32), idesc, kk > 0 ? 1u : 0u);
          tc_commit(empty_w(sw));
          tc_commit(empty_a(sa));
          tc_commit(dfull(sd));
        }
      }
      tc_commit(drain_bar);  // every MMA issued above has completed once this arrives
      wait_drain_w(drain_bar, 0);
    }
    __syncwarp();
  } else if (warp >= kWarpEpi) {
    regs_inc_epilogue();
    pdl_wait();  // activation exponents come from the previous kernel
    const int q = warp & 3;                  // tensor-memory lane quarter: tokens 32q..32q+31
    const int hf = (warp - kWarpEpi) >> 2;   // feature half of each weight block
    const int tok = q * 32 + lane;           // this thread's token within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    uint32_t it = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; ok && u < total_units; u += gridDim.x, ++ui) {
      const Unit un = unit_of(a, u, upt);
      const bool valid = tok < un.nv;
      const int64_t row = un.row0 + tok;
      const float* sc0 = a.s0 + (static_cast<int64_t>(un.e) * n_nb + un.nb0) * num_kb;
      const float* sc1 = a.s1 + (static_cast<int64_t>(un.e) * n_nb + (un.has1 ? un.nb1 : un.nb0)) * num_kb;
      const float* inv = a.act_inv + row;
      // down pass: destination row and router weight, loaded now so their
      // latency hides behind the K loop
      int dst = 0;
      float wg = 1.f;
      if (!GATEUP && valid) {
        dst = a.sorted_pos ? __ldg(a.sorted_pos + row) : static_cast<int>(row);
        wg = a.topk_weight ? __ldg(a.topk_weight + dst) : 1.f;
      }
      float acc0[kHalfF], acc1[kHalfF];
#pragma unroll
      for (int j = 0; j < kHalfF; ++j) acc0[j] = acc1[j] = 0.f;
      // this K block's factors; each iteration loads the next block's
      float sx = valid ? __ldg(inv) : 0.f;
      float s0v = __ldg(sc0), s1v = __ldg(sc1);
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        float nsx = 0.f, ns0 = 0.f, ns1 = 0.f;
        if (kb + 1 < num_kb) {
          nsx = valid ? __ldg(inv + static_cast<int64_t>(kb + 1) * a.act_rows) : 0.f;
          ns0 = __ldg(sc0 + kb + 1);
          ns1 = __ldg(sc1 + kb + 1);
        }
        const int sd = it & 1;
        ok = __all_sync(0xffffffffu, wait_bounded(dfull(sd), (it >> 1) & 1, abort_flag, a.err));
        if (!ok) break;
        tc_fence_after();
        const uint32_t tcol = tmem + lane_base + static_cast<uint32_t>(sd) * 256 + hf * kHalfF;
        uint32_t p[kHalfF];
        tmem_ld64(tcol, p);
        tmem_ld_wait();
        if (un.has1) {
          const float c0 = s0v * sx;
#pragma unroll
          for (int j = 0; j < kHalfF; ++j) acc0[j] = fmaf(c0, __uint_as_float(p[j]), acc0[j]);
          tmem_ld64(tcol + 128, p);
          tmem_ld_wait();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(dempty(sd));  // the partials are in registers now
        if (un.has1) {
          const float c1 = s1v * sx;
#pragma unroll
          for (int j = 0; j < kHalfF; ++j) acc1[j] = fmaf(c1, __uint_as_float(p[j]), acc1[j]);
        } else {
          const float c0 = s0v * sx;
#pragma unroll
          for (int j = 0; j < kHalfF; ++j) acc0[j] = fmaf(c0, __uint_as_float(p[j]), acc0[j]);
        }
        sx = nsx;
        s0v = ns0;
        s1v = ns1;
      }
      if (!ok) break;
      bool overflow = false;
      if (GATEUP) {
        // h = silu(g) * u; one scale per (token, 128 features) from the maximum of
        // this thread's 64 features and the other half's, exchanged through
        // red[ui & 1] and an eight-arrival mbarrier.
        float m = 0.f;
#pragma unroll
        for (int j = 0; j < kHalfF; ++j) {
          acc0[j] = silu_fast(acc0[j]) * acc1[j];
          m = fmaxf(m, fabsf(acc0[j]));
          overflow |= !(fabsf(acc0[j]) <= 3.0e38f);
        }
        overflow &= valid;
        const int64_t ld = static_cast<int64_t>(n_nb) * 128;
        uint8_t* hp = static_cast<uint8_t*>(a.out) + row * ld + un.nb0 * 128 + hf * kHalfF;
        float* rf = reinterpret_cast<float*>(red) + (ui & 1) * 2 * kTileMax;
        rf[hf * kTileMax + tok] = m;
        __syncwarp();
        if (lane == 0) mbar_arrive(redbar(ui & 1));
        ok = __all_sync(0xffffffffu, wait_bounded(redbar(ui & 1), (ui >> 1) & 1, abort_flag, a.err));
        if (!ok) break;
        if (valid) {
          const float sc = fp8_block_scale(fmaxf(m, rf[(hf ^ 1) * kTileMax + tok]));
#pragma unroll
          for (int v = 0; v < kHalfF / 32; ++v) {
            uint32_t t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float* x4 = acc0 + 32 * v + 4 * i;
              const uint32_t lo = __nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(x4[0], sc), __fdiv_rn(x4[1], sc)), __NV_SATFINITE, __NV_E4M3);
              const uint32_t hi = __nv_cvt_float2_to_fp8x2(
                  make_float2(__fdiv_rn(x4[2], sc), __fdiv_rn(x4[3], sc)), __NV_SATFINITE, __NV_E4M3);
              t[i] = lo | (hi << 16);
            }
            stg256(hp + 32 * v, t);
          }
          if (hf == 0) a.out_inv[static_cast<int64_t>(un.nb0) * a.act_rows + row] = sc;
        }
      } else if (valid) {
        uint16_t* o = static_cast<uint16_t*>(a.out) + static_cast<int64_t>(dst) * n_nb * 128 + hf * kHalfF;
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          if (m == 1 && !un.has1) break;
          const float* src = m == 0 ? acc0 : acc1;
#pragma unroll
          for (int v = 0; v < kHalfF / 16; ++v) {
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float x0 = src[16 * v + 2 * i] * wg, x1 = src[16 * v + 2 * i + 1] * wg;
              overflow |= !(fabsf(x0) < 65520.f) || !(fabsf(x1) < 65520.f);  // f16 rounds these to inf
              const __half2 h2 = __floats2half2_rn(x0, x1);
              w[i] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            stg256(o + (m == 0 ? un.nb0 : un.nb1) * 128 + 16 * v, w);
          }
        }
      }
      if (__any_sync(0xffffffffu, overflow) && lane == 0) atomicOr(a.err, DEV_ERR_RANGE);
    }
  }
  __syncthreads();
  if (warp == kWarpIssue) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemColsW);
  }
}

template <bool GATEUP, int WST, int AST>
cudaError_t launch_wide(const GemmLaunch& g, cudaStream_t s) {
  using C = WideCfg<WST, AST>;
  auto kern = moe_gemm_wide_kernel<GATEUP, WST, AST>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  if (!g.act_box) return cudaErrorInvalidValue;
  // The register split waits until the pool covers it: launch only if it does.
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kThreadsW < 128 * kRegsProducer + 256 * kRegsEpilogue) return cudaErrorInvalidConfiguration;
  WideArgs a;
  a.w_tiled = g.w_tiled;
  a.s0 = g.s0;
  a.s1 = g.s1;
  a.tiles = g.tiles;
  a.n_tiles = g.n_tiles;
  a.n_nb = g.n_nb;
  a.num_kb = g.num_kb;
  a.pair = GATEUP ? 0 : 1;
  a.l2_prefetch = g.l2_prefetch ? 1 : 0;
  a.act_inv = g.act_inv;
  a.act_rows = g.act_rows;
  a.out = g.out;
  a.out_inv = g.out_inv;
  a.sorted_pos = g.sorted_pos;
  a.topk_weight = g.topk_weight;
  a.err = g.err;
  // gate/up behind the row gather starts streaming weights on any SM with room
  return launch_maybe_overlapped(kern, g.num_sms, kThreadsW, C::kSmem, s, GATEUP && g.overlap, *g.w0, *g.w1,
                                 *g.act_box, a);
}

}  // namespace

// Stages (dynamic FP8, one term): four 32 KB weight stages (both blocks of one
// K block) and four 16 KB activation stages; about 195 KB of shared memory.
cudaError_t launch_gateup_wide(const GemmLaunch& g, cudaStream_t s) {
  if (g.terms == 1 && g.fp8) return launch_wide<true, 4, 4>(g, s);
  return cudaErrorInvalidValue;
}
cudaError_t launch_down_wide(const GemmLaunch& g, cudaStream_t s) {
  if (g.terms == 1 && g.fp8) return launch_wide<false, 4, 4>(g, s);
  return cudaErrorInvalidValue;
}

}  // namespace moe
