// Expert parallelism: the device-side steps around the two exchanges of the
// multi-rank routed-expert forward.
//
// "Input features" page, expert construction: with ep ranks, rank r holds
// experts [r * epr, (r + 1) * epr), epr = E / ep.  "Mixture of experts" page,
// moe_infer, ep_size > 1 branch: each rank sends the rows it routes to rank
// r's experts to rank r (tokens_per_ep_rank of them, in its sorted order), a
// rank regroups what it receives by local expert (gatherd_idxs), runs its
// experts, puts the outputs back in received order, sends them back, and the
// source sums each token's k rows weighted by topk_weight.
//
// The exchanges themselves are the caller's (an all-to-all of the counts and
// of the rows); everything on either side of them is here, with no host
// synchronisation.  Rows travel in a send buffer of "slots": with capacity 0
// the rows for rank d follow the rows for ranks < d without gaps (the pages'
// packed layout, whose split sizes the caller reads back); with capacity C the
// rows for rank d sit at slots d * C .. (fixed split sizes, nothing to read
// back, unused slots carry nothing).
//
// ep_send_plan_kernel   per rank: send_counts[d] (rows for rank d) and, for
//                       each (token, slot) entry, its slot in the send buffer
//                       (its sorted position, or d * C + its place among the
//                       rows for d); -1 for an id outside [0, E).
// ep_gather_kernel      send[slot(t, j)] = x[t]: one CTA per token, the row read
//                       once and written to each of its slots.
// ep_regroup_*          receiver: the received slots grouped by local expert,
//                       ties in received order (a stable sort of the labels of
//                       the pages' regroup): per-expert counts and offsets, and
//                       the position of each received slot in that order
//                       (row_pos, -1 for an unused slot) and its inverse.
// ep_combine_kernel     out[t] = sum_j topk_weight[t][j] * back[slot(t, j)] in
//                       fp32, j ascending, where back holds the expert outputs
//                       returned to their send slots.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace moe {
namespace {

__global__ void ep_send_plan_kernel(const int32_t* __restrict__ ids, int32_t R, int32_t E, int32_t ep,
                                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ inv_pos,
                                    int64_t capacity, int32_t* __restrict__ send_counts,
                                    int32_t* __restrict__ tok_slot, uint32_t* err) {
  const int epr = E / ep;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (blockIdx.x == 0 && threadIdx.x < ep)
    send_counts[threadIdx.x] = offsets[(threadIdx.x + 1) * epr] - offsets[threadIdx.x * epr];
  if (i >= R) return;
  const int e = ids[i];
  const int p = inv_pos[i];
  if (e < 0 || e >= E || p < 0) {
    tok_slot[i] = -1;
    return;
  }
  const int d = e / epr;
  if (capacity == 0) {
    tok_slot[i] = p;
  } else {
    const int64_t within = p - offsets[d * epr];
    if (within >= capacity) {  // more rows for rank d than its block of slots holds
      tok_slot[i] = -1;
      atomicOr(err, DEV_ERR_ROUTING);
    } else {
      tok_slot[i] = static_cast<int32_t>(d * capacity + within);
    }
  }
}

constexpr int kGatherThreads = 256;

__global__ void __launch_bounds__(kGatherThreads) ep_gather_kernel(const uint16_t* __restrict__ x,
                                                                   const int32_t* __restrict__ tok_slot, int32_t k,
                                                                   int32_t d, int64_t n_slots,
                                                                   uint16_t* __restrict__ send) {
  const int64_t t = blockIdx.x;
  int32_t slots[32];
  int ns = 0;
  for (int j = 0; j < k; ++j) {
    const int s = tok_slot[t * k + j];
    if (s >= 0 && s < n_slots) slots[ns++] = s;
  }
  const uint4* src = reinterpret_cast<const uint4*>(x + t * d);
  for (int c = threadIdx.x; c < d / 8; c += kGatherThreads) {
    const uint4 v = src[c];
    for (int q = 0; q < ns; ++q) reinterpret_cast<uint4*>(send + static_cast<int64_t>(slots[q]) * d)[c] = v;
  }
}

// One thread: counts [ep][epr] (source-major, as the count exchange delivers
// them) -> the counts that fit the received slots (each source's rows must fit
// its block of `capacity` slots, all rows must fit the n_slots slots; anything
// beyond is dropped and raises MOE_ERR_ROUTING), local_counts, local_offsets,
// and per (source r, expert e) chunk its first received slot and its first
// position in expert order.  ep * epr is small: one entry per exchanged count.
__global__ void ep_regroup_prep_kernel(const int32_t* __restrict__ cnt, int32_t epr, int32_t ep, int64_t capacity,
                                       int64_t n_slots, int32_t* __restrict__ local_counts,
                                       int32_t* __restrict__ local_offsets, int32_t* __restrict__ eff,
                                       int32_t* __restrict__ recv_start, int32_t* __restrict__ exp_start,
                                       uint32_t* err) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  int64_t s = 0;
  bool clipped = false;
  for (int r = 0; r < ep; ++r) {
    if (capacity > 0) s = r * capacity;
    const int64_t end = capacity > 0 ? min(static_cast<int64_t>(r + 1) * capacity, n_slots) : n_slots;
    for (int e = 0; e < epr; ++e) {
      const int64_t c = max(0, cnt[r * epr + e]);
      const int64_t fit = max(static_cast<int64_t>(0), min(c, end - s));
      clipped |= fit < c || cnt[r * epr + e] < 0;
      eff[r * epr + e] = static_cast<int32_t>(fit);
      recv_start[r * epr + e] = static_cast<int32_t>(s);
      s += fit;
    }
  }
  recv_start[ep * epr] = static_cast<int32_t>(s);
  int32_t off = 0;
  for (int e = 0; e < epr; ++e) {
    int32_t c = 0;
    for (int r = 0; r < ep; ++r) c += eff[r * epr + e];
    local_counts[e] = c;
    local_offsets[e] = off;
    int32_t p = off;
    for (int r = 0; r < ep; ++r) {  // within an expert: sources in order
      exp_start[r * epr + e] = p;
      p += eff[r * epr + e];
    }
    off += c;
  }
  local_offsets[epr] = off;
  if (clipped) atomicOr(err, DEV_ERR_ROUTING);
}

__global__ void ep_regroup_kernel(const int32_t* __restrict__ eff, int32_t chunks, int64_t n_slots,
                                  const int32_t* __restrict__ recv_start, const int32_t* __restrict__ exp_start,
                                  int32_t* __restrict__ row_pos, int32_t* __restrict__ pos_row) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= n_slots) return;
  // last chunk whose first slot is <= i (recv_start is nondecreasing)
  int lo = 0, hi = chunks - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (recv_start[mid] <= i) lo = mid;
    else hi = mid - 1;
  }
  const int64_t j = i - recv_start[lo];
  if (j < 0 || j >= eff[lo]) {  // an unused slot (a gap after a source's rows, or past the end)
    row_pos[i] = -1;
    return;
  }
  const int p = static_cast<int>(exp_start[lo] + j);  // < local_offsets[epr] <= n_slots
  row_pos[i] = p;
  pos_row[p] = static_cast<int32_t>(i);
}

__device__ __forceinline__ float2 f16x2_to_f2(uint32_t w) { return __half22float2(*reinterpret_cast<const __half2*>(&w)); }

__device__ __forceinline__ uint32_t pack_bf16x2_ep(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__global__ void __launch_bounds__(256) ep_combine_kernel(const uint16_t* __restrict__ back,
                                                         const int32_t* __restrict__ tok_slot,
                                                         const float* __restrict__ topk_weight, int32_t n, int32_t k,
                                                         int32_t d, int64_t n_slots, void* __restrict__ out,
                                                         int32_t out_fp32) {
  const int nv = d / 8;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(n) * nv) return;
  const int64_t t = idx / nv;
  const int c = static_cast<int>(idx - t * nv);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  for (int j = 0; j < k; ++j) {
    const int s = tok_slot[t * k + j];
    if (s < 0 || s >= n_slots) continue;
    const float w = topk_weight[t * k + j];
    const uint4 v = reinterpret_cast<const uint4*>(back + static_cast<int64_t>(s) * d)[c];
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = f16x2_to_f2(wv[q]);
      acc[2 * q] = fmaf(w, f.x, acc[2 * q]);
      acc[2 * q + 1] = fmaf(w, f.y, acc[2 * q + 1]);
    }
  }
  if (out_fp32) {
    float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) + t * d) + 2 * c;
    o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  } else {
    uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + t * d) + c;
    *o = make_uint4(pack_bf16x2_ep(acc[0], acc[1]), pack_bf16x2_ep(acc[2], acc[3]), pack_bf16x2_ep(acc[4], acc[5]),
                    pack_bf16x2_ep(acc[6], acc[7]));
  }
}

}  // namespace

cudaError_t launch_ep_send_plan(const int32_t* ids, int32_t R, int32_t E, int32_t ep, const int32_t* offsets,
                                const int32_t* inv_pos, int64_t capacity, int32_t* send_counts, int32_t* tok_slot,
                                uint32_t* err, cudaStream_t s) {
  const int blocks = max(1, (R + 255) / 256);
  ep_send_plan_kernel<<<blocks, 256, 0, s>>>(ids, R, E, ep, offsets, inv_pos, capacity, send_counts, tok_slot, err);
  return cudaGetLastError();
}

cudaError_t launch_ep_gather(const uint16_t* x, const int32_t* tok_slot, int32_t n, int32_t k, int32_t d,
                             int64_t n_slots, uint16_t* send, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  ep_gather_kernel<<<n, kGatherThreads, 0, s>>>(x, tok_slot, k, d, n_slots, send);
  return cudaGetLastError();
}

int64_t ep_regroup_scratch_ints(int32_t epr, int32_t ep) { return 3 * static_cast<int64_t>(epr) * ep + 1; }

cudaError_t launch_ep_regroup(const int32_t* cnt, int32_t epr, int32_t ep, int64_t capacity, int64_t n_slots,
                              int32_t* local_counts, int32_t* local_offsets, int32_t* row_pos, int32_t* pos_row,
                              int32_t* scratch, uint32_t* err, cudaStream_t s) {
  const int chunks = epr * ep;
  int32_t* eff = scratch;                        // chunks
  int32_t* recv_start = scratch + chunks;        // chunks + 1
  int32_t* exp_start = scratch + 2 * chunks + 1; // chunks
  ep_regroup_prep_kernel<<<1, 32, 0, s>>>(cnt, epr, ep, capacity, n_slots, local_counts, local_offsets, eff,
                                          recv_start, exp_start, err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || n_slots <= 0) return e;
  const int64_t blocks = (n_slots + 255) / 256;
  ep_regroup_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(eff, chunks, n_slots, recv_start, exp_start,
                                                                  row_pos, pos_row);
  return cudaGetLastError();
}

cudaError_t launch_ep_combine(const uint16_t* back, const int32_t* tok_slot, const float* topk_weight, int32_t n,
                              int32_t k, int32_t d, int64_t n_slots, void* out, int32_t out_fp32, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t nv = static_cast<int64_t>(n) * (d / 8);
  ep_combine_kernel<<<static_cast<unsigned>((nv + 255) / 256), 256, 0, s>>>(back, tok_slot, topk_weight, n, k, d,
                                                                            n_slots, out, out_fp32);
  return cudaGetLastError();
}

}  // namespace moe
