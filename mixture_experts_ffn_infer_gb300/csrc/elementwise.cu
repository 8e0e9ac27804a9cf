// Bandwidth-bound steps around the grouped GEMMs.
//
// gather_rows_kernel    - "Mixture of experts" page, moe_infer: sorted_tokens
//                         = x[idxs // k]; rows are converted bf16 -> f16 (exact
//                         for |x| < 65504) for the f16 tensor-core GEMMs.
// rmsnorm_scatter_kernel- "Input features" page, RMSNorm: fp32 mean of squares,
//                         rsqrt(mean + eps), times gain; the normalised row is
//                         written once per routed slot straight to its sorted
//                         position (inv_pos) and to the shared expert's rows.
// combine_kernel        - "Mixture of experts" page, moe_infer: sum of the
//                         token's k weighted rows (fp32, ascending slot), plus
//                         the shared expert ("forward") and the residual
//                         ("Input features" page, decoder block); 16-byte
//                         vector loads and stores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ float2 unpack_f16x2(uint32_t w) {
  return __half22float2(*reinterpret_cast<const __half2*>(&w));
}

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) { return pack_f16x2(bf16_lo(w), bf16_hi(w)); }

__global__ void __launch_bounds__(128) gather_rows_kernel(const uint16_t* __restrict__ x,
                                                          const int32_t* __restrict__ sorted_pos, int32_t k,
                                                          int32_t d, uint16_t* __restrict__ xs) {
  const int64_t i = blockIdx.x;
  const int p = sorted_pos[i];
  uint4* dst = reinterpret_cast<uint4*>(xs + i * d);
  const int nv = d / 8;
  if (p < 0) {
    for (int c = threadIdx.x; c < nv; c += blockDim.x) dst[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<int64_t>(p / k) * d);
  for (int c = threadIdx.x; c < nv; c += blockDim.x) {
    const uint4 v = src[c];
    dst[c] = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
  }
}

constexpr int kNormThreads = 256;

__global__ void __launch_bounds__(kNormThreads) rmsnorm_scatter_kernel(
    const uint16_t* __restrict__ h, const uint16_t* __restrict__ gain, float eps, int32_t d, int32_t k,
    const int32_t* __restrict__ inv_pos, uint16_t* __restrict__ xs, uint16_t* __restrict__ xs_shared) {
  __shared__ float red[kNormThreads / 32];
  __shared__ float s_inv;
  const int64_t t = blockIdx.x;
  const uint4* row = reinterpret_cast<const uint4*>(h + t * d);
  const uint4* g4 = reinterpret_cast<const uint4*>(gain);
  const int nv = d / 8;
  float ss = 0.f;
  for (int c = threadIdx.x; c < nv; c += kNormThreads) {
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
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
    for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
    s_inv = rsqrtf(tot / static_cast<float>(d) + eps);
  }
  __syncthreads();
  const float inv = s_inv;

  int32_t dst_rows[32];
  int ndst = 0;
  for (int j = 0; j < k; ++j) {
    const int p = inv_pos[t * k + j];
    if (p >= 0) dst_rows[ndst++] = p;
  }
  for (int c = threadIdx.x; c < nv; c += kNormThreads) {
    const uint4 v = row[c], g = g4[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      o[q] = pack_f16x2(bf16_lo(gw[q]) * (bf16_lo(w[q]) * inv), bf16_hi(gw[q]) * (bf16_hi(w[q]) * inv));
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    for (int q = 0; q < ndst; ++q) reinterpret_cast<uint4*>(xs + static_cast<int64_t>(dst_rows[q]) * d)[c] = ov;
    if (xs_shared) reinterpret_cast<uint4*>(xs_shared + t * d)[c] = ov;
  }
}

__global__ void __launch_bounds__(256) combine_kernel(const uint16_t* __restrict__ rows,
                                                      const uint16_t* __restrict__ shared,
                                                      const uint16_t* __restrict__ resid, int32_t n, int32_t k,
                                                      int32_t d, void* __restrict__ out, int32_t out_fp32) {
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

}  // namespace

cudaError_t launch_gather_rows(const uint16_t* x_bf16, const int32_t* sorted_pos, int32_t R, int32_t k, int32_t d,
                               uint16_t* xs_f16, cudaStream_t s) {
  if (R <= 0) return cudaSuccess;
  gather_rows_kernel<<<R, 128, 0, s>>>(x_bf16, sorted_pos, k, d, xs_f16);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_scatter(const uint16_t* h_bf16, const uint16_t* gain_bf16, float eps, int32_t n, int32_t d,
                                   int32_t k, const int32_t* inv_pos, uint16_t* xs_f16, uint16_t* xs_shared_f16,
                                   cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  rmsnorm_scatter_kernel<<<n, kNormThreads, 0, s>>>(h_bf16, gain_bf16, eps, d, k, inv_pos, xs_f16, xs_shared_f16);
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t* rows_f16, const uint16_t* shared_f16, const uint16_t* resid_bf16,
                           int32_t n, int32_t k, int32_t d, void* out, int32_t out_fp32, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nv = static_cast<int64_t>(n) * (d / 8);
  const int blocks = static_cast<int>((nv + 255) / 256);
  combine_kernel<<<blocks, 256, 0, s>>>(rows_f16, shared_f16, resid_bf16, n, k, d, out, out_fp32);
  return cudaGetLastError();
}

}  // namespace moe
