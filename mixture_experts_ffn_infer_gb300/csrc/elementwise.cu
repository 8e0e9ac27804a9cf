// Bandwidth-bound steps around the grouped GEMMs.
//
// gather_rows_kernel    - "Mixture of experts" page, moe_infer: sorted_tokens
//                         = x[idxs // k]; each token's row is split once into
//                         the e4m3 split format the 16-token GEMMs read
//                         (split3.cuh), or quantised to dynamic FP8, and written
//                         to all of its sorted positions.
// gather_rows_f16_kernel- the same gather for the wide f16 GEMMs: the row is
//                         divided by a power of two of its own (its largest
//                         magnitude lands in [2^14, 2^15)) and stored as f16,
//                         which holds every bf16 value of the row exactly
//                         unless it lies more than 2^28 below the maximum.
// rmsnorm_scatter_kernel- "Input features" page, RMSNorm: fp32 mean of squares,
//                         h / sqrt(mean + eps) cast to bf16, times the bf16 gain
//                         in bf16; the normalised row is split once (two terms
//                         hold a bf16 value) or stored as scaled f16 (as the f16
//                         gather), and written per routed slot straight to its
//                         sorted position (inv_pos) and to the shared expert's
//                         rows.
// pack_tiles_kernel     - storage layout only: copies each 128 x 128 tile of
//                         e4m3 codes into one contiguous 16 KB block, laid out
//                         exactly as a 128-byte-swizzled TMA box lands in
//                         shared memory, the two weight blocks of a GEMM unit
//                         side by side per K block, so one bulk copy moves both.
// combine_kernel        - "Mixture of experts" page, moe_infer: sum of the
//                         token's k weighted rows (fp32, ascending slot), plus
//                         the shared expert ("forward") and the residual
//                         ("Input features" page, decoder block); 16-byte
//                         vector loads and stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "split3.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

constexpr int kRowThreads = 256;  // eight warps per row, one 128-column block per warp at a time

// The power of two s of an f16 row whose largest magnitude is m: m * 2^-s lies
// in [2^14, 2^15), inside f16's range with 28 binades of normal numbers below
// it.  0 for an all-zero or non-finite row; limited to [-126, 113] so that 2^s
// and 2^-s stay normal floats.
__device__ __forceinline__ int f16_row_exponent(float m) {
  if (!(m > 0.f) || !(m < 3.0e38f)) return 0;
  int e;
  frexpf(m, &e);  // m = f * 2^e, f in [0.5, 1)
  return max(-126, min(113, e - 15));
}

// Largest value over the CTA (kRowThreads threads; every thread gets it).
__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __syncthreads();  // red may still be read from an earlier use
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

// Four values times 2^-s as f16 (exact for bf16 inputs in range), packed in two words.
__device__ __forceinline__ uint2 f16x4_scaled(const float (&v)[4], int s) {
  const __half2 a = __floats2half2_rn(ldexpf(v[0], -s), ldexpf(v[1], -s));
  const __half2 b = __floats2half2_rn(ldexpf(v[2], -s), ldexpf(v[3], -s));
  return make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
}

// One CTA per token and column group (blockIdx.y of gridDim.y, a batch with
// fewer tokens than SMs spreads each row over several CTAs): the token's row is
// read once, each 128-column block is split once and written to every sorted
// position of the token (inv_pos).  Each warp keeps four blocks' loads in
// flight before it converts them.
__global__ void __launch_bounds__(kRowThreads) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                                  const int32_t* __restrict__ inv_pos, int32_t n,
                                                                  int32_t k, int32_t d, uint8_t* __restrict__ xs,
                                                                  SplitLayout lay, float* __restrict__ xs_inv) {
  pdl_wait();  // launched behind the routing plan, whose inv_pos it reads
  // Everything before this kernel in the stream is complete now, so the gate/up GEMM
  // may be placed and stream its weights (it waits for these rows, not for the weights).
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t R = static_cast<int64_t>(n) * k;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t dst_rows[32];
  int ndst = 0;
  for (int j = 0; j < k; ++j) {
    const int p = inv_pos ? inv_pos[t * k + j] : static_cast<int>(t * k + j);  // null: identity order
    if (p >= 0 && p < R) dst_rows[ndst++] = p;
  }
  if (ndst == 0) return;
  const uint2* src = reinterpret_cast<const uint2*>(x + t * d);
  const int nkb = d / 128;
  constexpr int kWarps = kRowThreads / 32, kBatch = 4;
  const int step = kWarps * static_cast<int>(gridDim.y);  // column blocks apart of one warp's consecutive blocks
  for (int kb0 = static_cast<int>(blockIdx.y) * kWarps + warp; kb0 < nkb; kb0 += step * kBatch) {
    uint2 w[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int kb = kb0 + step * i;
      w[i] = kb < nkb ? src[kb * 32 + lane] : make_uint2(0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int kb = kb0 + step * i;
      if (kb >= nkb) break;
      const float v[4] = {bf16_lo(w[i].x), bf16_hi(w[i].x), bf16_lo(w[i].y), bf16_hi(w[i].y)};
      uint32_t t1, t2, t3;
      const float inv = lay.fp8 ? warp_fp8_block(v, t1, t2, t3) : warp_split_block(v, t1, t2, t3);
      for (int q = 0; q < ndst; ++q) warp_store_block(xs, lay, xs_inv, R, dst_rows[q], kb, t1, t2, t3, inv, lane);
    }
  }
}

// One CTA per token: the row's largest magnitude, then the row as f16 times
// 2^-s to every sorted position of the token, and 2^s to the factor array.
// Each thread moves 8 columns at a time (16-byte loads and stores) and keeps
// its first kHeld groups in registers between the two passes.
__global__ void __launch_bounds__(kRowThreads) gather_rows_f16_kernel(const uint16_t* __restrict__ x,
                                                                      const int32_t* __restrict__ inv_pos,
                                                                      int32_t n, int32_t k, int32_t d,
                                                                      uint8_t* __restrict__ xs, SplitLayout lay,
                                                                      float* __restrict__ xs_scale) {
  constexpr int kHeld = 4;  // rows up to 8 * kRowThreads * kHeld = 8192 columns are read once
  __shared__ float red[kRowThreads / 32];
  pdl_wait();  // launched behind the routing plan, whose inv_pos it reads
  pdl_launch_dependents();
  const int64_t t = blockIdx.x;
  const int64_t R = static_cast<int64_t>(n) * k;
  int32_t dst_rows[32];
  int ndst = 0;
  for (int j = 0; j < k; ++j) {
    const int p = inv_pos ? inv_pos[t * k + j] : static_cast<int>(t * k + j);  // null: identity order
    if (p >= 0 && p < R) dst_rows[ndst++] = p;
  }
  if (ndst == 0) return;  // the whole CTA leaves together (ndst is the same for every thread)
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);  // eight bf16 per uint4
  const int n8 = d / 8;
  auto max8 = [](const uint4& w) {
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(bf16_lo(q[i])), fabsf(bf16_hi(q[i]))));
    return m;
  };
  uint4 held[kHeld];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < kHeld; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    held[i] = c < n8 ? src[c] : make_uint4(0u, 0u, 0u, 0u);
    m = fmaxf(m, max8(held[i]));
  }
  for (int c = threadIdx.x + kHeld * kRowThreads; c < n8; c += kRowThreads) m = fmaxf(m, max8(src[c]));
  const int s = f16_row_exponent(block_max(m, red));
  // columns 8c..8c+7: panel c / 8, bytes (c % 8) * 16 of the row's 128 in it
  auto store8 = [&](int c, const uint4& w) {
    const float v0[4] = {bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y)};
    const float v1[4] = {bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w)};
    const uint2 a = f16x4_scaled(v0, s), b = f16x4_scaled(v1, s);
    const uint4 o = make_uint4(a.x, a.y, b.x, b.y);
    uint8_t* panel = xs + static_cast<int64_t>(c >> 3) * lay.term_stride + (c & 7) * 16;
    for (int q = 0; q < ndst; ++q)
      *reinterpret_cast<uint4*>(panel + static_cast<int64_t>(dst_rows[q]) * lay.row_stride) = o;
  };
#pragma unroll
  for (int i = 0; i < kHeld; ++i) {
    const int c = threadIdx.x + i * kRowThreads;
    if (c < n8) store8(c, held[i]);
  }
  for (int c = threadIdx.x + kHeld * kRowThreads; c < n8; c += kRowThreads) store8(c, src[c]);
  if (threadIdx.x < ndst) xs_scale[dst_rows[threadIdx.x]] = ldexpf(1.0f, s);
}

// inv[sorted_pos[i]] = i for every valid entry; the rest stay -1 (set before).
__global__ void invert_positions_kernel(const int32_t* __restrict__ sorted_pos, int32_t R, int32_t* __restrict__ inv) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < R; i += gridDim.x * blockDim.x) {
    const int p = sorted_pos[i];
    if (p >= 0 && p < R) inv[p] = i;
  }
}

__global__ void __launch_bounds__(kRowThreads) rmsnorm_scatter_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ gain, float eps, int32_t n, int32_t d, int32_t k,
    const int32_t* __restrict__ inv_pos, uint8_t* __restrict__ xs, SplitLayout lay, float* __restrict__ xs_inv,
    uint8_t* __restrict__ xs_shared, SplitLayout lay_shared, float* __restrict__ xs_shared_inv) {
  __shared__ float red[kRowThreads / 32];
  __shared__ float s_inv;
  const int64_t t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint4* row = reinterpret_cast<const uint4*>(h + t * d);
  const int nv = d / 8;
  float ss = 0.f;
  for (int c = threadIdx.x; c < nv; c += kRowThreads) {
    const uint4 v = row[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float a = bf16_lo(w[q]), b = bf16_hi(w[q]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[warp] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kRowThreads / 32; ++w) tot += red[w];
    s_inv = 1.0f / sqrtf(tot / static_cast<float>(d) + eps);
  }
  __syncthreads();
  const float inv_rms = s_inv;

  int32_t dst_rows[32];
  int ndst = 0;
  for (int j = 0; j < k; ++j) {
    const int p = inv_pos[t * k + j];
    if (p >= 0) dst_rows[ndst++] = p;
  }
  const int64_t R = static_cast<int64_t>(n) * k;
  // the normalised row is cast to bf16, then multiplied by the bf16 gain in bf16
  auto normalised = [&](int kb, float (&v)[4]) {
    const uint2 w = reinterpret_cast<const uint2*>(h + t * d + kb * 128)[lane];
    const uint2 g = reinterpret_cast<const uint2*>(gain + kb * 128)[lane];
    v[0] = bf16_round(bf16_lo(g.x) * bf16_round(bf16_lo(w.x) * inv_rms));
    v[1] = bf16_round(bf16_hi(g.x) * bf16_round(bf16_hi(w.x) * inv_rms));
    v[2] = bf16_round(bf16_lo(g.y) * bf16_round(bf16_lo(w.y) * inv_rms));
    v[3] = bf16_round(bf16_hi(g.y) * bf16_round(bf16_hi(w.y) * inv_rms));
  };
  // f16 rows (wide tiles) need the normalised row's largest magnitude first
  int s = 0;
  if (lay.f16 || (xs_shared && lay_shared.f16)) {
    float m = 0.f;
    for (int kb = warp; kb < d / 128; kb += kRowThreads / 32) {
      float v[4];
      normalised(kb, v);
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3]))));
    }
    s = f16_row_exponent(block_max(m, red));
  }
  for (int kb = warp; kb < d / 128; kb += kRowThreads / 32) {
    float v[4];
    normalised(kb, v);
    uint2 f16v = make_uint2(0u, 0u);
    if (lay.f16 || (xs_shared && lay_shared.f16)) f16v = f16x4_scaled(v, s);
    uint32_t t1 = 0, t2 = 0, t3 = 0;
    float inv = 0.f;
    if (!lay.f16 || (xs_shared && !lay_shared.f16))
      inv = lay.fp8 || lay_shared.fp8 ? warp_fp8_block(v, t1, t2, t3) : warp_split_block(v, t1, t2, t3);
    for (int q = 0; q < ndst; ++q) {
      if (lay.f16)  // columns 4 lane.. of block kb: panel 2 kb + lane / 16
        *reinterpret_cast<uint2*>(xs + static_cast<int64_t>(2 * kb + (lane >> 4)) * lay.term_stride +
                                  static_cast<int64_t>(dst_rows[q]) * lay.row_stride + (lane & 15) * 8) = f16v;
      else
        warp_store_block(xs, lay, xs_inv, R, dst_rows[q], kb, t1, t2, t3, inv, lane);
    }
    if (xs_shared) {
      if (lay_shared.f16)
        *reinterpret_cast<uint2*>(xs_shared + static_cast<int64_t>(2 * kb + (lane >> 4)) * lay_shared.term_stride +
                                  t * lay_shared.row_stride + (lane & 15) * 8) = f16v;
      else
        warp_store_block(xs_shared, lay_shared, xs_shared_inv, n, t, kb, t1, t2, t3, inv, lane);
    }
  }
  if (lay.f16 && threadIdx.x < ndst) xs_inv[dst_rows[threadIdx.x]] = ldexpf(1.0f, s);
  if (xs_shared && lay_shared.f16 && threadIdx.x == 0) xs_shared_inv[t] = ldexpf(1.0f, s);
}

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const uint16_t* __restrict__ shared,
                                                      const uint16_t* __restrict__ resid, int32_t n, int32_t k,
                                                      int32_t d, void* __restrict__ out, int32_t out_fp32) {
  pdl_wait();  // launched behind the down GEMM: its rows are complete past this point
  const int nv = d / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(n) * nv) return;
  const int64_t t = idx / nv;
  const int c = static_cast<int>(idx - t * nv);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  for (int j = 0; j < k; ++j) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(rows + (t * k + j) * d) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = unpack_f16x2(w[q]);
      acc[2 * q] += f.x;
      acc[2 * q + 1] += f.y;
    }
  }
  if (shared) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(shared + t * d) + c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = unpack_f16x2(w[q]);
      acc[2 * q] += f.x;
      acc[2 * q + 1] += f.y;
    }
  }
  if (resid) {
    const uint4 v = reinterpret_cast<const uint4*>(resid + t * d)[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      acc[2 * q] += bf16_lo(w[q]);
      acc[2 * q + 1] += bf16_hi(w[q]);
    }
  }
  if (out_fp32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + t * d) + 2 * c;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + t * d) + c;
    *o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                    pack_bf16x2(acc[6], acc[7]));
  }
}

// One CTA per 16 KB output tile; tiles enumerated (((e * unit_rows + u) * cols/128 + c) * 2 + m).
// Source row block of tile (u, m): gate/up (paired = 0): block u of src_m;
// down (paired = 1): block 2u + m of src0, zeros past the last block.
__global__ void __launch_bounds__(256) pack_tiles_kernel(const uint8_t* __restrict__ src0,
                                                         const uint8_t* __restrict__ src1, uint8_t* __restrict__ dst,
                                                         int32_t rows, int32_t cols, int32_t paired) {
  const int64_t t = blockIdx.x;
  const int nrb = rows / 128, ncb = cols / 128;
  const int unit_rows = paired ? (nrb + 1) / 2 : nrb;
  const int m = static_cast<int>(t & 1);
  const int64_t q = t >> 1;  // (e * unit_rows + u) * ncb + c
  const int c = static_cast<int>(q % ncb);
  const int64_t eu = q / ncb;
  const int u = static_cast<int>(eu % unit_rows);
  const int64_t e = eu / unit_rows;
  const int b = paired ? 2 * u + m : u;
  const uint8_t* src = paired ? src0 : (m ? src1 : src0);
  uint8_t* d = dst + t * 16384;
  for (int i = threadIdx.x; i < 1024; i += 256) {
    const int r = i >> 3, j = i & 7;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (b < nrb)
      v = *reinterpret_cast<const uint4*>(src + (e * rows + static_cast<int64_t>(b) * 128 + r) * cols +
                                          static_cast<int64_t>(c) * 128 + j * 16);
    *reinterpret_cast<uint4*>(d + r * 128 + ((j ^ (r & 7)) << 4)) = v;
  }
}

}  // namespace

int64_t pack_tile_count(int32_t num_experts, int32_t rows, int32_t cols, int32_t paired) {
  const int64_t nrb = rows / 128;
  return static_cast<int64_t>(num_experts) * (paired ? (nrb + 1) / 2 : nrb) * (cols / 128) * 2;
}

cudaError_t launch_pack_tiles(const uint8_t* src0, const uint8_t* src1, uint8_t* dst, int32_t num_experts,
                              int32_t rows, int32_t cols, int32_t paired, cudaStream_t s) {
  const int64_t tiles = pack_tile_count(num_experts, rows, cols, paired);
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  pack_tiles_kernel<<<static_cast<unsigned>(tiles), 256, 0, s>>>(src0, src1, dst, rows, cols, paired);
  return cudaGetLastError();
}

cudaError_t launch_gather_rows(const uint16_t* x_bf16, const int32_t* inv_pos, int32_t n, int32_t k, int32_t d,
                               uint8_t* xs, SplitLayout lay, float* xs_inv, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  if (lay.f16) {
    // one CTA per token (its row's maximum is needed before any value is stored)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(n);
    cfg.blockDim = dim3(kRowThreads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gather_rows_f16_kernel, x_bf16, inv_pos, n, k, d, xs, lay, xs_inv);
  }
  // a batch smaller than the GPU spreads each row's column blocks over several CTAs
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess)
    sms = 1;
  const int nkb = d / 128;
  const int max_groups = (nkb + kRowThreads / 32 - 1) / (kRowThreads / 32);
  const int groups = n >= sms ? 1 : max(1, min(max_groups, sms / n));
  // dependent launch: placed while the routing plan finishes, waiting for it
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n, groups);
  cfg.blockDim = dim3(kRowThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, x_bf16, inv_pos, n, k, d, xs, lay, xs_inv);
}

cudaError_t launch_invert_positions(const int32_t* sorted_pos, int32_t R, int32_t* inv, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(inv, 0xff, sizeof(int32_t) * static_cast<size_t>(R), s);
  if (e != cudaSuccess) return e;
  const int blocks = min((R + 255) / 256, 4096);
  invert_positions_kernel<<<blocks, 256, 0, s>>>(sorted_pos, R, inv);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_scatter(const uint16_t* h_bf16, const uint16_t* gain_bf16, float eps, int32_t n, int32_t d,
                                   int32_t k, const int32_t* inv_pos, uint8_t* xs, SplitLayout lay, float* xs_inv,
                                   uint8_t* xs_shared, SplitLayout lay_shared, float* xs_shared_inv, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  rmsnorm_scatter_kernel<<<n, kRowThreads, 0, s>>>(h_bf16, gain_bf16, eps, n, d, k, inv_pos, xs, lay, xs_inv,
                                                   xs_shared, lay_shared, xs_shared_inv);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* rows_f16, const uint16_t* shared_f16, const uint16_t* resid_bf16,
                           int32_t n, int32_t k, int32_t d, void* out, int32_t out_fp32, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nv = static_cast<int64_t>(n) * (d / 8);
  const int blocks = static_cast<int>((nv + 255) / 256);
  // dependent launch: the CTAs are placed while the previous kernel drains and wait for it
  return launch_maybe_overlapped(combine_kernel, blocks, 256, 0, s, true, rows_f16, shared_f16, resid_bf16, n, k, d,
                                 out, out_fp32);
}

}  // namespace moe
