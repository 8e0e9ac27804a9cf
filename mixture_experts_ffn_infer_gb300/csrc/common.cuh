// Shared definitions of the CUDA library: device error bits, the bounded
// mbarrier wait, tile descriptors and the launchers each .cu file exports.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace moe {

// Bits of the device error word (first 4 bytes of the workspace).
enum : uint32_t {
  DEV_ERR_ROUTING = 1u << 0,
  DEV_ERR_TIMEOUT = 1u << 1,
  DEV_ERR_RANGE = 1u << 2,
};

// A pipeline wait gives up after this many SM clocks (about one second at
// the GB300's maximum clock); it then flags DEV_ERR_TIMEOUT and the kernel
// winds down instead of hanging the GPU.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Waits until phase `parity` of the mbarrier has completed.  Returns false
// (and stops waiting) when another role of the CTA has aborted or when the
// bound is exceeded, in which case it raises the abort flag itself.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                             uint32_t* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *abort_flag = 1u;
      atomicOr(err, DEV_ERR_TIMEOUT);
      return false;
    }
  }
}

// One GEMM tile of the grouped GEMMs: `n_valid` consecutive rows of the
// sorted activation matrix starting at `row_start`, all routed to `expert`.
// The tiles of one expert's slice are grouped into chunks of at most
// kTileChunk consecutive tiles; `chunk` holds the tile's index within its chunk
// (bits 0-7) and the chunk's tile count (bits 8-15).
struct TileDesc {
  int32_t expert;
  int32_t row_start;
  int32_t n_valid;
  int32_t chunk;
};

// Written beside a tile count (n_tiles[2], the count in n_tiles[0]): 1 when at
// least 90 % of the tiles belong to experts cut into two or more tiles, whose
// weights are then read by several tiles and mostly from L2 after the first;
// the f16 GEMM then gives its token ring the deeper share of its stages.
__host__ __device__ inline int32_t tiles_share_weights(int multi_tiles, int tiles) {
  return tiles > 0 && 10LL * multi_tiles >= 9LL * tiles ? 1 : 0;
}

constexpr int kTileChunk = 8;
__host__ __device__ inline int32_t tile_chunk_code(int idx_in_slice, int tiles_in_slice) {
  const int c = idx_in_slice / kTileChunk;
  const int left = tiles_in_slice - c * kTileChunk;
  return (idx_in_slice % kTileChunk) | ((left < kTileChunk ? left : kTileChunk) << 8);
}

// Token tile widths of the grouped GEMMs.  Decode-like batches (a few rows per
// expert) use 16-token tiles whose live activation terms sit side by side on
// the MMA's N axis (N = 16 x terms: 32 for x, 48 for h, 16 under dynamic FP8);
// from 24 rows per expert on, tiles of up to 128 tokens on the MMA's M side
// with the terms stacked along K.
constexpr int kNTokSmall = 16;
constexpr int kNTokWide = 128;
__host__ __device__ constexpr int tile_tokens(int64_t rows, int64_t experts) {
  return rows >= 24 * experts ? kNTokWide : kNTokSmall;
}

// Where the sorted activation rows live and in which format.
//   16-token tiles: e4m3 split-format codes (split3.cuh), rows interleaved
//                   with three term slots, [rows][3][K] (row_stride 3K,
//                   term_stride K; the live terms first)
//   wide tiles:     f16 values in panels of 64 columns, [K/64][rows][64]
//                   (row_stride 128 bytes within a panel, term_stride =
//                   rows * 128 bytes between panels), so that one TMA box
//                   brings a K block of 128 columns of a tile as two 16 KB
//                   panels; each row is divided by a power of two of its own
//                   (kept in the factor array, one per row), so a bf16 value
//                   is held exactly
//   fp8 != 0:       the dynamic FP8 scheme, one e4m3 term per value with the
//                   scale amax / 448 per 128 columns (the first slot of the
//                   16-token layout, or one plane [rows][K] for wide tiles)
// The factor array holds, per (128 columns, row), 2^-s of the split format or
// the FP8 scale ([K/128][rows]); for f16 rows, per row, the power of two to
// multiply the row by ([rows]).
struct SplitLayout {
  int64_t row_stride;
  int64_t term_stride;
  int32_t terms;
  int32_t fp8;
  int32_t f16;
};
inline SplitLayout split_layout(bool wide, int64_t rows, int64_t K, int terms, bool fp8) {
  if (wide && !fp8) return SplitLayout{128, rows * 128, 1, 0, 1};
  const int32_t t = fp8 ? 1 : terms, f = fp8 ? 1 : 0;
  return wide ? SplitLayout{K, rows * K, t, f, 0} : SplitLayout{3 * K, K, t, f, 0};
}

// Launch with programmatic stream serialization when `overlap`: the kernel may
// start while the previous kernel in the stream finishes (it calls pdl_wait
// before it reads that kernel's results).
template <typename... P, typename... A>
cudaError_t launch_maybe_overlapped(void (*kern)(P...), int grid, int block, size_t smem, cudaStream_t s,
                                    bool overlap, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = overlap ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A&&>(args)...);
}

// ---------------------------------------------------------------- launchers
// routing.cu
// scratch: route_scratch_ints(n k, E) ints (none for small batches, which one CTA plans).
// tiles / n_tiles non-null: also cut the GEMM tile plan of ntok-row tiles from the offsets.
int64_t route_scratch_ints(int64_t R, int32_t E);
cudaError_t launch_route_permute(const int32_t* ids, int32_t n, int32_t k, int32_t E, int32_t* counts,
                                 int32_t* offsets, int32_t* sorted_pos, int32_t* inv_pos, int32_t validate,
                                 int32_t* scratch, uint32_t* err, int32_t ntok, TileDesc* tiles, int32_t* n_tiles,
                                 cudaStream_t s);
cudaError_t launch_build_tiles(const int32_t* offsets, int32_t E, int32_t ntok, TileDesc* tiles,
                               int32_t* n_tiles, cudaStream_t s);
cudaError_t launch_bounded_wait_selftest(uint32_t* err, cudaStream_t s);
cudaError_t launch_identity_tiles(int32_t rows, int32_t ntok, TileDesc* tiles, int32_t* n_tiles, cudaStream_t s);

// elementwise.cu
// Sorted activation rows in the split format from the bf16 tokens: inv_pos [n k]
// gives each routed slot's sorted position (-1: none; a null inv_pos keeps the
// slots' own order, position t k + j).
cudaError_t launch_gather_rows(const uint16_t* x_bf16, const int32_t* inv_pos, int32_t n, int32_t k, int32_t d,
                               uint8_t* xs, SplitLayout lay, float* xs_inv, cudaStream_t s);
// inv_pos from sorted_pos (entries that no sorted row names become -1).
cudaError_t launch_invert_positions(const int32_t* sorted_pos, int32_t R, int32_t* inv, cudaStream_t s);
cudaError_t launch_rmsnorm_scatter(const uint16_t* h_bf16, const uint16_t* gain_bf16, float eps, int32_t n,
                                   int32_t d, int32_t k, const int32_t* inv_pos, uint8_t* xs, SplitLayout lay,
                                   float* xs_inv, uint8_t* xs_shared, SplitLayout lay_shared, float* xs_shared_inv,
                                   cudaStream_t s);
// Tiled layout (moe_pack_weights): paired = 0 interleaves src0 and src1 (gate, up)
// per row block; paired = 1 interleaves row blocks 2u, 2u + 1 of src0 (down).
int64_t pack_tile_count(int32_t num_experts, int32_t rows, int32_t cols, int32_t paired);
cudaError_t launch_pack_tiles(const uint8_t* src0, const uint8_t* src1, uint8_t* dst, int32_t num_experts,
                              int32_t rows, int32_t cols, int32_t paired, cudaStream_t s);
cudaError_t launch_combine(const uint16_t* rows_f16, const uint16_t* shared_f16, const uint16_t* resid_bf16,
                           int32_t n, int32_t k, int32_t d, void* out, int32_t out_fp32, cudaStream_t s);

// ep.cu (expert parallelism: the steps on either side of the exchanges)
cudaError_t launch_ep_send_plan(const int32_t* ids, int32_t R, int32_t E, int32_t ep, const int32_t* offsets,
                                const int32_t* inv_pos, int64_t capacity, int32_t* send_counts, int32_t* tok_slot,
                                uint32_t* err, cudaStream_t s);
cudaError_t launch_ep_gather(const uint16_t* x, const int32_t* tok_slot, int32_t n, int32_t k, int32_t d,
                             int64_t n_slots, uint16_t* send, cudaStream_t s);
int64_t ep_regroup_scratch_ints(int32_t epr, int32_t ep);
cudaError_t launch_ep_regroup(const int32_t* cnt, int32_t epr, int32_t ep, int64_t capacity, int64_t n_slots,
                              int32_t* local_counts, int32_t* local_offsets, int32_t* row_pos, int32_t* pos_row,
                              int32_t* scratch, uint32_t* err, cudaStream_t s);
cudaError_t launch_ep_combine(const uint16_t* back, const int32_t* tok_slot, const float* topk_weight, int32_t n,
                              int32_t k, int32_t d, int64_t n_slots, void* out, int32_t out_fp32, cudaStream_t s);

// moe_gemm.cu
struct GemmLaunch {
  // weights: 3-D maps over [E][rows][K] e4m3, box 128 x 128 x 1, 128-byte swizzle
  const CUtensorMap* w0;        // gate (gate/up pass) or down (down pass)
  const CUtensorMap* w1;        // up (gate/up pass only)
  const CUtensorMap* act;       // 16-token tiles: 3-D map over [rows][3][K] e4m3, box 128 x terms x 16
  const CUtensorMap* act_box_rows[3];  // wide tiles, exact scheme: boxes of 32, 64 and 96 token rows
  const CUtensorMap* act_box;   // wide tiles: f16 panels [K/64][rows][64], box 64 x 128 rows x 2 panels
                                //   (exact scheme; act_box_rows[i] the same with boxes of 32 (i + 1) rows), or
                                //   3-D map over [terms][rows][K], box 128 x 128 rows x terms (FP8)
  int32_t ntok;                 // token tile width (kNTokSmall or kNTokWide)
  int32_t terms;                // live activation terms per row (1 to 3)
  bool fp8;                     // dynamic FP8 activations: gate/up writes h as one e4m3 term, scale amax / 448
  // Tiled layout (moe_pack_weights): both weight blocks of a unit per K block, 32 KB,
  // consecutive K blocks contiguous; used instead of w0 / w1 when non-null.
  const uint8_t* w_tiled;
  const float* s0;              // scales [E][n_nb][num_kb]
  const float* s1;
  const TileDesc* tiles;
  const int32_t* n_tiles;       // [0] tile count, [2] tiles_share_weights of the list
  int32_t n_nb;                 // weight-row blocks of 128 (output features / 128)
  // A unit is one token tile times two weight blocks: gate/up pass = row block j
  // of w0 and of w1; down pass = row blocks 2j and 2j + 1 of w0.
  int32_t num_kb;               // K / 128
  const float* act_inv;         // [num_kb][act_rows] factor of each activation block (2^-s, or the FP8 scale);
                                //   f16 rows: [act_rows] power of two of each row (NULL = 1)
  int32_t act_rows;             // rows of the sorted activation matrix
  void* out;                    // gate/up: h (layout of the next pass); down: rows [.][n_nb*128] f16
  float* out_inv;               // gate/up: [n_nb][act_rows] factor of each h block
  const int32_t* sorted_pos;    // down: flat position of each sorted row (NULL = identity)
  const float* topk_weight;     // down: flat router weights (NULL = 1)
  uint32_t* err;
  int num_sms;
  bool overlap;                 // gate/up: launched behind the row gather (dependent launch)
  bool l2_prefetch;             // wide tiles: prefetch weights into L2 ahead of their copies
};
cudaError_t launch_gateup(const GemmLaunch& g, cudaStream_t s);
cudaError_t launch_down(const GemmLaunch& g, cudaStream_t s);
// moe_gemm_f16.cu (the two above forward wide tiles of the exact scheme here):
// f16 token rows, weights converted to f16 with their block scale on chip
cudaError_t launch_gateup_f16(const GemmLaunch& g, cudaStream_t s);
cudaError_t launch_down_f16(const GemmLaunch& g, cudaStream_t s);
// moe_gemm_wide.cu (wide tiles of the dynamic FP8 scheme)
cudaError_t launch_gateup_wide(const GemmLaunch& g, cudaStream_t s);
cudaError_t launch_down_wide(const GemmLaunch& g, cudaStream_t s);

}  // namespace moe
