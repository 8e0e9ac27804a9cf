// Routing plan of the routed-expert forward ("Mixture of experts" page,
// moe_infer: per-expert token counts and the sort of the flattened expert ids).
//
// route_permute_kernel: one CTA of 1024 threads replaces the page's one-hot
// scatter + column sum + argsort with a counting sort that is stable by
// construction.  Each warp owns a contiguous chunk of the flattened ids and
// walks it 32 entries at a time; __match_any_sync groups the lanes that carry
// the same expert so one lane updates the warp's private count (no atomics),
// and the rank of a lane among its peers is a popcount of the lower peers.
// Pass 1 builds per-warp histograms in shared memory, a block scan turns them
// into per-(warp, expert) starting positions, pass 2 repeats the walk and
// writes sorted_pos / inv_pos.  Order = (expert, warp, round, lane) = (expert,
// flat index): identical to a stable argsort.
//
// Large batches use the same walk spread over many CTAs: route_count_kernel
// counts per (CTA chunk, expert), route_scan_kernel turns the counts into
// tokens_per_expert, expert_offsets and each chunk's starting position per
// expert, route_scatter_kernel repeats the walk and writes the positions.  The
// order is (expert, chunk, warp, round, lane) = (expert, flat index) again.
//
// build_tiles_kernel: cuts every expert's contiguous slice into tiles of at
// most `ntok` rows for the grouped GEMMs, on the device, so nothing is copied
// back to the host (the page's loop reads the counts on the host instead).
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
// Up to this many flattened entries one CTA builds the plan; above it, chunks of
// kChunkEntries entries per CTA.
constexpr int64_t kSingleCtaEntries = 8192;
constexpr int kChunkEntries = 2048;

// Exclusive scan of one int per thread over the whole CTA; `*total` gets the sum.
__device__ int block_exclusive_scan(int v, int* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    warp_sums[lane] = w;  // inclusive
  }
  __syncthreads();
  const int before = warp > 0 ? warp_sums[warp - 1] : 0;
  *total = warp_sums[kWarps - 1];
  __syncthreads();
  return before + x - v;
}

// Tiles of at most ntok rows over every expert's slice [offsets[e], offsets[e+1]),
// in expert order; the whole CTA (kThreads threads) takes part.  n_tiles[0] gets
// the tile count, n_tiles[2] the weight-sharing flag (tiles_share_weights).
__device__ void cta_build_tiles(const int32_t* __restrict__ offsets, int E, int ntok, TileDesc* __restrict__ tiles,
                                int32_t* __restrict__ n_tiles, int* warp_sums) {
  const int tid = threadIdx.x;
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int local = 0, local_multi = 0;
  for (int e = e0; e < e1; ++e) {
    const int nt_e = (offsets[e + 1] - offsets[e] + ntok - 1) / ntok;
    local += nt_e;
    if (nt_e >= 2) local_multi += nt_e;
  }
  int total, multi;
  int t = block_exclusive_scan(local, warp_sums, &total);
  block_exclusive_scan(local_multi, warp_sums, &multi);
  for (int e = e0; e < e1; ++e) {
    const int beg = offsets[e], end = offsets[e + 1];
    const int nt_e = (end - beg + ntok - 1) / ntok;
    for (int i = 0; i < nt_e; ++i) {
      const int r = beg + i * ntok;
      tiles[t++] = TileDesc{e, r, min(ntok, end - r), tile_chunk_code(i, nt_e)};
    }
  }
  if (tid == 0) {
    n_tiles[0] = total;
    n_tiles[2] = tiles_share_weights(multi, total);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
route_permute_kernel(const int32_t* __restrict__ ids, int32_t n, int32_t k, int32_t E, int32_t* __restrict__ counts,
                     int32_t* __restrict__ offsets, int32_t* __restrict__ sorted_pos, int32_t* __restrict__ inv_pos,
                     int32_t validate, int32_t reset_err, uint32_t* err, int32_t ntok, TileDesc* __restrict__ tiles,
                     int32_t* __restrict__ n_tiles) {
  extern __shared__ int32_t smem[];
  int32_t* wcnt = smem;                  // [kWarps][E]: counts, then running positions
  int32_t* warp_sums = smem + kWarps * E;  // [32]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = n * k;
  pdl_wait();  // launched behind the previous kernel in the stream: nothing is touched before it ends
  pdl_launch_dependents();  // the row gather may be placed now; it waits for this plan

  if (reset_err && tid == 0) *err = 0u;  // a new routing plan starts a new error record
  for (int i = tid; i < kWarps * E; i += kThreads) wcnt[i] = 0;
  __syncthreads();

  // Contiguous chunk of the flattened ids per warp, a multiple of 32 entries.
  const int chunk = (((R + kWarps - 1) / kWarps) + 31) & ~31;
  const int beg = min(warp * chunk, R), end = min(beg + chunk, R);
  int32_t* mine = wcnt + warp * E;

  bool bad = false;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids[i] : -1;
    const bool valid = i < end && e >= 0 && e < E;
    bad |= (i < end) && !valid;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  if (bad) atomicOr(err, DEV_ERR_ROUTING);
  if (validate) {
    for (int t = tid; t < n; t += kThreads) {
      const int32_t* row = ids + static_cast<int64_t>(t) * k;
      bool dup = false;
      for (int a = 1; a < k; ++a)
        for (int b = 0; b < a; ++b) dup |= row[a] == row[b];
      if (dup) atomicOr(err, DEV_ERR_ROUTING);
    }
  }
  __syncthreads();

  // counts[e], offsets[e] and the starting position of each (warp, expert).
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int local = 0;
  for (int e = e0; e < e1; ++e) {
    int c = 0;
    for (int w = 0; w < kWarps; ++w) c += wcnt[w * E + e];
    counts[e] = c;
    local += c;
  }
  int total;
  int run = block_exclusive_scan(local, warp_sums, &total);
  for (int e = e0; e < e1; ++e) {
    offsets[e] = run;
    for (int w = 0; w < kWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  if (tid == 0) offsets[E] = total;
  __syncthreads();

  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids[i] : -1;
    const bool valid = i < end && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid) {
      const int pos = mine[e] + __popc(peers & ((1u << lane) - 1u));
      sorted_pos[pos] = i;
      if (inv_pos) inv_pos[i] = pos;
    } else if (i < end && inv_pos) {
      inv_pos[i] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  for (int i = total + tid; i < R; i += kThreads) sorted_pos[i] = -1;
  if (tiles) {  // the GEMMs' tile plan from the offsets this CTA wrote
    __syncthreads();
    cta_build_tiles(offsets, E, ntok, tiles, n_tiles, warp_sums);
  }
}

// ------------------------------------------------------------ many CTAs
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kWarpEntries = kChunkEntries / kChunkWarps;  // a multiple of 32

// Walk of one warp over [beg, end): per-expert counts of the warp into mine[].
__device__ __forceinline__ bool warp_count(const int32_t* __restrict__ ids, int beg, int end, int E, int lane,
                                           int32_t* mine) {
  bool bad = false;
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids[i] : -1;
    const bool valid = i < end && e >= 0 && e < E;
    bad |= (i < end) && !valid;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  return bad;
}

__global__ void __launch_bounds__(kChunkThreads) route_count_kernel(const int32_t* __restrict__ ids, int32_t n,
                                                                    int32_t k, int32_t E, int32_t validate,
                                                                    int32_t* __restrict__ chunk_counts, uint32_t* err) {
  extern __shared__ int32_t wcnt[];  // [kChunkWarps][E]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = n * k;
  for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) wcnt[i] = 0;
  __syncthreads();
  const int beg = min(static_cast<int>(blockIdx.x) * kChunkEntries + warp * kWarpEntries, R);
  const int end = min(beg + kWarpEntries, min((static_cast<int>(blockIdx.x) + 1) * kChunkEntries, R));
  if (warp_count(ids, beg, end, E, lane, wcnt + warp * E)) atomicOr(err, DEV_ERR_ROUTING);
  if (validate) {
    for (int t = blockIdx.x * kChunkThreads + tid; t < n; t += gridDim.x * kChunkThreads) {
      const int32_t* row = ids + static_cast<int64_t>(t) * k;
      bool dup = false;
      for (int a = 1; a < k; ++a)
        for (int b = 0; b < a; ++b) dup |= row[a] == row[b];
      if (dup) atomicOr(err, DEV_ERR_ROUTING);
    }
  }
  __syncthreads();
  for (int e = tid; e < E; e += kChunkThreads) {
    int c = 0;
    for (int w = 0; w < kChunkWarps; ++w) c += wcnt[w * E + e];
    chunk_counts[static_cast<int64_t>(blockIdx.x) * E + e] = c;
  }
}

// One CTA: totals per expert, the exclusive scan over experts, and each chunk's
// starting position per expert (written over its count).
__global__ void __launch_bounds__(kThreads, 1) route_scan_kernel(int32_t* __restrict__ chunk_counts, int32_t chunks,
                                                                 int32_t E, int32_t* __restrict__ counts,
                                                                 int32_t* __restrict__ offsets, int32_t ntok,
                                                                 TileDesc* __restrict__ tiles,
                                                                 int32_t* __restrict__ n_tiles) {
  __shared__ int warp_sums[32];
  const int tid = threadIdx.x;
  const int per = (E + kThreads - 1) / kThreads;
  const int e0 = min(tid * per, E), e1 = min(e0 + per, E);
  int local = 0;
  for (int e = e0; e < e1; ++e) {
    int c = 0;
    for (int ch = 0; ch < chunks; ++ch) c += chunk_counts[static_cast<int64_t>(ch) * E + e];
    counts[e] = c;
    local += c;
  }
  int total;
  int run = block_exclusive_scan(local, warp_sums, &total);
  for (int e = e0; e < e1; ++e) {
    offsets[e] = run;
    for (int ch = 0; ch < chunks; ++ch) {
      int32_t* v = chunk_counts + static_cast<int64_t>(ch) * E + e;
      const int c = *v;
      *v = run;
      run += c;
    }
  }
  if (tid == 0) offsets[E] = total;
  if (tiles) {
    __syncthreads();
    cta_build_tiles(offsets, E, ntok, tiles, n_tiles, warp_sums);
  }
}

__global__ void __launch_bounds__(kChunkThreads) route_scatter_kernel(const int32_t* __restrict__ ids, int32_t n,
                                                                      int32_t k, int32_t E,
                                                                      const int32_t* __restrict__ chunk_base,
                                                                      const int32_t* __restrict__ offsets,
                                                                      int32_t* __restrict__ sorted_pos,
                                                                      int32_t* __restrict__ inv_pos) {
  extern __shared__ int32_t wcnt[];  // [kChunkWarps][E]: counts, then running positions
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int R = n * k;
  for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) wcnt[i] = 0;
  __syncthreads();
  const int cbeg = static_cast<int>(blockIdx.x) * kChunkEntries, cend = min(cbeg + kChunkEntries, R);
  const int beg = min(cbeg + warp * kWarpEntries, cend), end = min(beg + kWarpEntries, cend);
  int32_t* mine = wcnt + warp * E;
  warp_count(ids, beg, end, E, lane, mine);
  __syncthreads();
  for (int e = tid; e < E; e += kChunkThreads) {
    int run = chunk_base[static_cast<int64_t>(blockIdx.x) * E + e];
    for (int w = 0; w < kChunkWarps; ++w) {
      const int c = wcnt[w * E + e];
      wcnt[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = beg; base < end; base += 32) {
    const int i = base + lane;
    const int e = i < end ? ids[i] : -1;
    const bool valid = i < end && e >= 0 && e < E;
    const unsigned peers = __match_any_sync(0xffffffffu, valid ? e : -1);
    if (valid) {
      const int pos = mine[e] + __popc(peers & ((1u << lane) - 1u));
      sorted_pos[pos] = i;
      if (inv_pos) inv_pos[i] = pos;
    } else if (i < end && inv_pos) {
      inv_pos[i] = -1;
    }
    __syncwarp();
    if (valid && lane == __ffs(peers) - 1) mine[e] += __popc(peers);
    __syncwarp();
  }
  // positions past the valid entries name nothing
  const int total = offsets[E];
  for (int i = max(cbeg, total) + tid; i < cend; i += kChunkThreads) sorted_pos[i] = -1;
}

__global__ void __launch_bounds__(kThreads, 1)
build_tiles_kernel(const int32_t* __restrict__ offsets, int32_t E, int32_t ntok, TileDesc* __restrict__ tiles,
                   int32_t* __restrict__ n_tiles) {
  __shared__ int warp_sums[32];
  cta_build_tiles(offsets, E, ntok, tiles, n_tiles, warp_sums);
}

__global__ void identity_tiles_kernel(int32_t rows, int32_t ntok, TileDesc* tiles, int32_t* n_tiles) {
  const int nt = (rows + ntok - 1) / ntok;
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < nt; t += gridDim.x * blockDim.x)
    tiles[t] = TileDesc{0, t * ntok, min(ntok, rows - t * ntok), tile_chunk_code(t, nt)};
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    n_tiles[0] = nt;
    n_tiles[2] = tiles_share_weights(nt >= 2 ? nt : 0, nt);  // one expert: every tile shares its weights
  }
}

// One thread waits on a barrier that nothing completes, through the same bounded
// wait the GEMM pipelines use; after the bound it raises DEV_ERR_TIMEOUT and exits.
__global__ void bounded_wait_selftest_kernel(uint32_t* err) {
  __shared__ uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0u;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  wait_bounded(smem_u32(&bar), 0, &abort_flag, err);
}

}  // namespace

cudaError_t launch_bounded_wait_selftest(uint32_t* err, cudaStream_t s) {
  bounded_wait_selftest_kernel<<<1, 32, 0, s>>>(err);
  return cudaGetLastError();
}

int64_t route_scratch_ints(int64_t R, int32_t E) {
  return R > kSingleCtaEntries ? ((R + kChunkEntries - 1) / kChunkEntries) * E : 0;
}

cudaError_t launch_route_permute(const int32_t* ids, int32_t n, int32_t k, int32_t E, int32_t* counts,
                                 int32_t* offsets, int32_t* sorted_pos, int32_t* inv_pos, int32_t validate,
                                 int32_t* scratch, uint32_t* err, int32_t ntok, TileDesc* tiles, int32_t* n_tiles,
                                 cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t R = static_cast<int64_t>(n) * k;
  if (R <= kSingleCtaEntries) {
    const size_t smem = sizeof(int32_t) * (static_cast<size_t>(kWarps) * E + 32);
    cudaError_t e = cudaFuncSetAttribute(route_permute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    // dependent launch: placed while the previous kernel in the stream drains; it waits for it
    return launch_maybe_overlapped(route_permute_kernel, 1, kThreads, smem, s, true, ids, n, k, E, counts, offsets,
                                   sorted_pos, inv_pos, validate, 1, err, ntok, tiles, n_tiles);
  }
  if (!scratch) return cudaErrorInvalidValue;
  const int chunks = static_cast<int>((R + kChunkEntries - 1) / kChunkEntries);
  const size_t smem = sizeof(int32_t) * static_cast<size_t>(kChunkWarps) * E;
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(uint32_t), s);  // a new routing plan starts a new error record
  if (e != cudaSuccess) return e;
  route_count_kernel<<<chunks, kChunkThreads, smem, s>>>(ids, n, k, E, validate, scratch, err);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  route_scan_kernel<<<1, kThreads, 0, s>>>(scratch, chunks, E, counts, offsets, ntok, tiles, n_tiles);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  route_scatter_kernel<<<chunks, kChunkThreads, smem, s>>>(ids, n, k, E, scratch, offsets, sorted_pos, inv_pos);
  return cudaGetLastError();
}

cudaError_t launch_build_tiles(const int32_t* offsets, int32_t E, int32_t ntok, TileDesc* tiles, int32_t* n_tiles,
                               cudaStream_t s) {
  build_tiles_kernel<<<1, kThreads, 0, s>>>(offsets, E, ntok, tiles, n_tiles);
  return cudaGetLastError();
}

cudaError_t launch_identity_tiles(int32_t rows, int32_t ntok, TileDesc* tiles, int32_t* n_tiles, cudaStream_t s) {
  const int nt = (rows + ntok - 1) / ntok;
  const int blocks = nt > 0 ? min((nt + 255) / 256, 1024) : 1;
  identity_tiles_kernel<<<blocks, 256, 0, s>>>(rows, ntok, tiles, n_tiles);
  return cudaGetLastError();
}

}  // namespace moe
