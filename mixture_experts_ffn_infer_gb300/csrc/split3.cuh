// Activations as two or three e4m3 terms with a power-of-two scale per 128-column block.
//
// The expert GEMMs run on the tensor core's e4m3 x e4m3 path so the FP8
// weights feed the MMA unconverted.  An activation value v of a 128-element
// block with largest magnitude m is written as
//     v * 2^s = a1 + a2 + a3,   s = 8 - frexp_exponent(m)   (so |v| * 2^s < 256),
// a1 = e4m3(v * 2^s), a2 = e4m3(remainder), a3 = e4m3(next remainder), each
// rounded to nearest.  Each term carries 4 significant bits, so a bf16 value
// (8 bits) is reproduced exactly by the first two terms whenever the block's
// range stays inside e4m3's (so bf16 rows are stored as two terms); the third
// term carries an fp32 intermediate (h) to about 12 bits.  The GEMMs sum the
// terms' partial products - in the epilogue for 16-token tiles, in the tensor
// core's accumulator for wide tiles - and multiply by 2^-s in fp32.  The
// dynamic FP8 scheme below uses the same storage with a single term.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cstdint>

#include "common.cuh"

namespace moe {

__device__ __forceinline__ float e4m3_to_float(uint8_t v) {
  return __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(v), __NV_E4M3)));
}

__device__ __forceinline__ uint8_t float_to_e4m3(float v) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}

// Block exponent s for a block whose largest magnitude is `amax` (0 for an all-zero block).
__device__ __forceinline__ int split_exponent(float amax) {
  if (!(amax > 0.f) || !(amax < 3.0e38f)) return 0;
  int e;
  frexpf(amax, &e);
  return 8 - e;
}

// v * 2^s -> three e4m3 codes (the scaled value must be below 448 in magnitude).
__device__ __forceinline__ void split3(float scaled, uint8_t& a1, uint8_t& a2, uint8_t& a3) {
  a1 = float_to_e4m3(scaled);
  const float r1 = scaled - e4m3_to_float(a1);
  a2 = float_to_e4m3(r1);
  const float r2 = r1 - e4m3_to_float(a2);
  a3 = float_to_e4m3(r2);
}

// Four consecutive values of one lane -> three packed words (one per term).
__device__ __forceinline__ void split3x4(const float (&v)[4], int s, uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  t1 = t2 = t3 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint8_t a, b, c;
    split3(ldexpf(v[i], s), a, b, c);
    t1 |= static_cast<uint32_t>(a) << (8 * i);
    t2 |= static_cast<uint32_t>(b) << (8 * i);
    t3 |= static_cast<uint32_t>(c) << (8 * i);
  }
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One warp converts one 128-column block of one row to the split format: lane
// l holds columns 4l..4l+3 in v; on return t1..t3 hold the lane's four codes of
// each term and the return value is 2^-s.
__device__ __forceinline__ float warp_split_block(const float (&v)[4], uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  m = warp_max(m);
  const int s = split_exponent(m);
  split3x4(v, s, t1, t2, t3);
  return ldexpf(1.0f, -s);
}

// Dynamic FP8 activations ("Input features" page, quantisation config:
// activation_scheme "dynamic", fmt e4m3): one e4m3 term per value, with the
// scale s = amax / 448 of its 128-column block (1 for an all-zero block),
// code = nearest e4m3 of v / s with ties to even and saturation at 448.  The
// divisions are IEEE round-to-nearest, so a bf16 input's codes are exactly
// reproducible.
__device__ __forceinline__ float fp8_block_scale(float amax) {
  const float s = __fdiv_rn(amax, 448.0f);
  return s > 0.f ? s : 1.0f;
}

// One warp, one 128-column block, lane l holding columns 4l..4l+3: t1 gets the
// lane's four codes, t2 and t3 zero; returns the block scale.
__device__ __forceinline__ float warp_fp8_block(const float (&v)[4], uint32_t& t1, uint32_t& t2, uint32_t& t3) {
  float m = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  const float s = fp8_block_scale(warp_max(m));
  t1 = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) t1 |= static_cast<uint32_t>(float_to_e4m3(__fdiv_rn(v[i], s))) << (8 * i);
  t2 = t3 = 0;
  return s;
}

// Store a block converted by warp_split_block or warp_fp8_block for sorted
// row `row` at column block kb: the codes go where `lay` puts them (as many
// terms as the layout keeps), the block's factor to inv[kb * n_rows + row].
__device__ __forceinline__ void warp_store_block(uint8_t* codes, SplitLayout lay, float* inv, int64_t n_rows,
                                                 int64_t row, int kb, uint32_t t1, uint32_t t2, uint32_t t3,
                                                 float inv_s, int lane) {
  uint8_t* base = codes + row * lay.row_stride + static_cast<int64_t>(kb) * 128;
  reinterpret_cast<uint32_t*>(base)[lane] = t1;
  if (lay.terms > 1) reinterpret_cast<uint32_t*>(base + lay.term_stride)[lane] = t2;
  if (lay.terms > 2) reinterpret_cast<uint32_t*>(base + 2 * lay.term_stride)[lane] = t3;
  if (lane == 0) inv[static_cast<int64_t>(kb) * n_rows + row] = inv_s;
}

}  // namespace moe
