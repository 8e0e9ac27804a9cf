// C ABI of the routed-expert forward: argument checks, workspace layout,
// tensor-map encoding and the launch sequence of each entry point.  All
// launches go to the caller's stream; nothing here synchronises except
// moe_get_error.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "moe_ffn.h"

namespace moe {
namespace {

constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kMaxEpRanks = 256;  // ranks of an expert-parallel group

// ---------------------------------------------------------------- workspace
// Sorted activations and h are kept in the split format (split3.cuh): e4m3
// codes (rows interleaved with their three terms for 16-token tiles, one plane
// per term for wide tiles; SplitLayout) plus one fp32 exponent factor per
// (128 columns, row).
struct Layout {
  size_t err = 0, n_tiles = 64, route = 256, route_end = 256;
  size_t tiles = 0, tiles_sh = 0, counts = 0, offsets = 0, sorted_pos = 0, inv_pos = 0;
  size_t xs = 0, xs_inv = 0, h = 0, h_inv = 0, xs_sh = 0, xs_sh_inv = 0, h_sh = 0, h_sh_inv = 0, sh_out = 0;
  size_t rows = 0, total = 0;
};

size_t align_up(size_t v) { return (v + 1023) & ~size_t(1023); }

bool dims_ok(const moe_dims* d) {
  return d && d->d > 0 && d->d_ff > 0 && d->d % 128 == 0 && d->d_ff % 128 == 0 && d->num_experts >= 1 &&
         d->num_experts <= kMaxExperts && d->top_k >= 1 && d->top_k <= kMaxTopK &&
         (d->act_scheme == MOE_ACT_EXACT || d->act_scheme == MOE_ACT_FP8_DYNAMIC);
}

bool fp8_act(const moe_dims* d) { return d->act_scheme == MOE_ACT_FP8_DYNAMIC; }

// Activation terms the GEMMs read: bf16 rows (x, the normalised row) and h.
int x_terms_of(bool fp8) { return fp8 ? 1 : 2; }
int h_terms_of(bool fp8) { return fp8 ? 1 : 3; }

bool make_layout(const moe_dims* d, int64_t n, int32_t dff_sh, Layout* L) {
  if (!dims_ok(d) || n < 0 || dff_sh < 0 || dff_sh % 128 != 0) return false;
  const int64_t R = n * d->top_k;
  if (R >= (int64_t(1) << 31) - 4096) return false;
  const int64_t max_tiles = R / kNTokSmall + d->num_experts + 1;  // bound for either tile width
  const int64_t max_tiles_sh = n / kNTokSmall + 2;
  size_t off = 256;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes);
    return at;
  };
  // the routing plan's scratch comes first, so moe_permute needs only a short prefix
  L->route = take(4 * size_t(route_scratch_ints(R, d->num_experts)));
  L->route_end = off;
  L->tiles = take(sizeof(TileDesc) * max_tiles);
  L->tiles_sh = take(sizeof(TileDesc) * max_tiles_sh);
  L->counts = take(4 * size_t(d->num_experts));
  L->offsets = take(4 * size_t(d->num_experts + 1));
  L->sorted_pos = take(4 * size_t(R));
  L->inv_pos = take(4 * size_t(R));
  L->xs = take(3 * size_t(R) * d->d);
  L->xs_inv = take(4 * size_t(R) * (d->d / 128));
  L->h = take(3 * size_t(R) * d->d_ff);
  L->h_inv = take(4 * size_t(R) * (d->d_ff / 128));
  L->rows = take(2 * size_t(R) * d->d);
  if (dff_sh > 0) {
    L->xs_sh = take(3 * size_t(n) * d->d);
    L->xs_sh_inv = take(4 * size_t(n) * (d->d / 128));
    L->h_sh = take(3 * size_t(n) * dff_sh);
    L->h_sh_inv = take(4 * size_t(n) * (dff_sh / 128));
    L->sh_out = take(2 * size_t(n) * d->d);
  }
  L->total = off;
  return true;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

// ---------------------------------------------------------------- tensor maps
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
  });
  return fn;
}

// [E][rows][K] e4m3, box 128 (K) x 128 (rows) x 1, 128-byte swizzle.
bool map_weights(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, uint64_t E) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {K, rows, E};
  const cuuint64_t strides[2] = {K, K * rows};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Split-format codes of `rows` sorted rows, rows interleaved with their three
// term slots: [rows][3][K] e4m3.  Box 128 (K) x `terms` slots x ntok rows, so
// only the live terms are loaded (smem order [row][term][128 B]), 128-byte
// swizzle; rows past the end read as zero.
bool map_act(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, int terms, int ntok) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {K, 3, rows};
  const cuuint64_t strides[2] = {K, 3 * K};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(terms), static_cast<cuuint32_t>(ntok)};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Wide tiles: split-format codes as term planes [terms][rows][K] e4m3, box 128 (K)
// x box_rows x terms, 128-byte swizzle; rows past the end read as zero.
bool map_act_planar(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, int terms, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {K, rows, static_cast<cuuint64_t>(terms)};
  const cuuint64_t strides[2] = {K, K * rows};
  const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(terms)};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Wide tiles of the exact scheme: f16 values in panels of 64 columns,
// [K/64][rows][64]; box 64 (128 bytes) x box_rows x 2 panels, 128-byte
// swizzle, so one copy brings a K block of 128 columns; rows past the end read
// as zero.
bool map_rows_f16(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows, int box_rows) {
  EncodeFn enc = encode_fn();
  if (!enc) return false;
  const cuuint64_t dims[3] = {64, rows, K / 64};
  const cuuint64_t strides[2] = {128, 128 * rows};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 2};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split layout of `rows` sorted rows of width K, as the tile width chosen for
// `rows` rows over `experts` experts reads it.
SplitLayout rows_layout(int64_t rows, int64_t experts, int64_t K, int terms, bool fp8) {
  return split_layout(tile_tokens(rows, experts) == kNTokWide, rows, K, terms, fp8);
}

int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Kernels the routing plan launches for R flattened entries (one CTA, or count + scan + scatter).
int route_kernels(int64_t R) { return route_scratch_ints(R, 1) > 0 ? 3 : 1; }

bool weights_ok(const moe_weights* w) {
  if (!w || !w->w_gate || !w->w_down || !w->s_gate || !w->s_up || !w->s_down || !aligned(w->w_gate, 16) ||
      !aligned(w->w_down, 16))
    return false;
  if (w->layout == MOE_LAYOUT_TILED) return true;  // w_up is part of w_gate
  return w->layout == MOE_LAYOUT_ROW_MAJOR && w->w_up && aligned(w->w_up, 16);
}

// Weight maps of a bank (row-major only; the tiled layout is read with bulk copies).
bool map_bank(const moe_weights* w, int64_t d, int64_t dff, int64_t E, CUtensorMap* g, CUtensorMap* u,
              CUtensorMap* dn) {
  if (w->layout == MOE_LAYOUT_TILED) return true;
  return map_weights(g, w->w_gate, d, dff, E) && map_weights(u, w->w_up, d, dff, E) &&
         map_weights(dn, w->w_down, dff, d, E);
}

// Per-kernel events for timing (moe_trace).  Every event sits between two
// kernels and costs the stream about a launch gap, so gemms_only keeps three
// per step: before the first GEMM and after each.
struct Tracer {
  moe_trace* t;
  cudaStream_t s;
  void begin() {
    if (!t) return;
    t->n_recorded = 0;
    t->n_launched = 0;
    if (t->gemms_only) return;
    if (t->n_events > 0 && cudaEventRecord(t->events[0], s) == cudaSuccess) t->n_recorded = 1;
  }
  void before_gemm() {
    if (!t || !t->gemms_only || t->n_recorded > 0) return;
    if (t->n_events > 0 && cudaEventRecord(t->events[0], s) == cudaSuccess) t->n_recorded = 1;
  }
  // after each launch step; `kernels` is how many kernels that step launched
  void after(const char* label, bool gemm = false, int kernels = 1) {
    if (t) t->n_launched += kernels;
    if (!t || t->n_recorded < 1 || (t->gemms_only && !gemm)) return;
    const int i = t->n_recorded;
    if (i >= t->n_events || i >= MOE_TRACE_MAX) return;
    t->labels[i - 1] = label;
    if (cudaEventRecord(t->events[i], s) == cudaSuccess) t->n_recorded = i + 1;
  }
};

#define MOE_CHECK_CUDA(expr)                    \
  do {                                          \
    if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

// Activation map of one GEMM pass: the 3-D map of 16-token tiles (rows
// interleaved with their term slots, box of 16 rows x the live terms), the f16
// panels of wide tiles (boxes of 32, 64, 96 and 128 rows x 64 values x two
// panels, so a tile's copy brings only its own rows rounded up to 32), or the
// planar FP8 codes of wide tiles (box of 128 rows x all terms).
struct ActMaps {
  CUtensorMap m16;
  CUtensorMap box;
  CUtensorMap box_rows[3];
  bool f16 = false;
  bool make(bool wide, bool fp8, const void* base, uint64_t K, uint64_t rows, int terms) {
    if (!wide) return map_act(&m16, base, K, rows, terms, kNTokSmall);
    if (fp8) {
      if (!map_act_planar(&box, base, K, rows, terms, kNTokWide)) return false;
    } else {
      f16 = true;
      for (int i = 0; i < 3; ++i)
        if (!map_rows_f16(&box_rows[i], base, K, rows, 32 * (i + 1))) return false;
      if (!map_rows_f16(&box, base, K, rows, kNTokWide)) return false;
    }
    m16 = box;
    return true;
  }
  void bind(GemmLaunch& g) const {
    g.act = &m16;
    g.act_box = &box;
    for (int i = 0; i < 3; ++i) g.act_box_rows[i] = f16 ? &box_rows[i] : nullptr;
  }
};

// Gate/up then down over `rows` sorted rows whose codes are already in xs (in
// the layout rows_layout gives, x_terms terms), tiles cut at tile_tokens(rows,
// experts) rows.  Down writes f16(topk_weight * o) to out[sorted_pos[row]]
// (identity and weight 1 when those are null).  fp8: dynamic FP8 activations
// (x and h one term each).
moe_status run_gemms(bool after_gather, bool fp8, const moe_weights* w, int64_t d, int64_t dff, int64_t experts,
                     int32_t rows, int x_terms,
                     uint8_t* xs, float* xs_inv, uint8_t* h, float* h_inv, TileDesc* tiles, int32_t* n_tiles,
                     const int32_t* sorted_pos, const float* topk_weight, void* out, uint32_t* err, cudaStream_t s,
                     Tracer& tr, const char* label_gateup, const char* label_down) {
  const int ntok = tile_tokens(rows, experts);
  const bool wide = ntok == kNTokWide;
  ActMaps mx, mh;
  const int h_terms = h_terms_of(fp8);
  if (!mx.make(wide, fp8, xs, d, rows, x_terms) || !mh.make(wide, fp8, h, dff, rows, h_terms)) return MOE_ERR_CUDA;
  CUtensorMap m_g, m_u, m_d;
  m_g = m_u = m_d = mx.m16;  // placeholders when the bank is tiled
  if (!map_bank(w, d, dff, experts, &m_g, &m_u, &m_d)) return MOE_ERR_CUDA;
  const bool tiled = w->layout == MOE_LAYOUT_TILED;
  GemmLaunch g{};
  g.ntok = ntok;
  g.terms = x_terms;
  g.fp8 = fp8;
  g.w0 = &m_g;
  g.w1 = &m_u;
  g.w_tiled = tiled ? w->w_gate : nullptr;
  mx.bind(g);
  g.s0 = w->s_gate;
  g.s1 = w->s_up;
  g.tiles = tiles;
  g.n_tiles = n_tiles;
  g.n_nb = static_cast<int32_t>(dff / 128);
  g.num_kb = static_cast<int32_t>(d / 128);
  g.act_inv = xs_inv;
  g.act_rows = rows;
  g.out = h;
  g.out_inv = h_inv;
  g.err = err;
  g.num_sms = num_sms();
  g.overlap = after_gather;
  // Wide tiles: the L2 prefetch ahead of the weight copies pays when an expert's
  // weights serve several token tiles (measured: -1.5 % at one tile per expert,
  // +1 to +4 % with several), so it is on from one full tile per expert.
  g.l2_prefetch = static_cast<int64_t>(rows) >= static_cast<int64_t>(kNTokWide) * experts;
  if (g.num_sms <= 0) return MOE_ERR_CUDA;
  tr.before_gemm();
  MOE_CHECK_CUDA(launch_gateup(g, s));
  tr.after(label_gateup, true);

  GemmLaunch q = g;
  q.overlap = false;
  q.terms = h_terms;
  q.w0 = &m_d;
  q.w1 = &m_d;
  q.w_tiled = tiled ? w->w_down : nullptr;
  mh.bind(q);
  q.s0 = w->s_down;
  q.s1 = w->s_down;
  q.n_nb = static_cast<int32_t>(d / 128);
  q.num_kb = static_cast<int32_t>(dff / 128);
  q.act_inv = h_inv;
  q.out = out;
  q.out_inv = nullptr;
  q.sorted_pos = sorted_pos;
  q.topk_weight = topk_weight;
  MOE_CHECK_CUDA(launch_down(q, s));
  tr.after(label_down, true);
  return MOE_OK;
}

// The expert pass on an already-sorted routing plan: gather, gate/up, down.
// `gather` selects the bf16 row gather (moe_experts_forward / moe_infer); the
// fused layer writes the sorted rows itself (RMSNorm scatter).  Either way the
// rows are bf16 values, which two e4m3 terms hold (one dynamic-FP8 term under
// that scheme).
// plan_ready: the routing kernel has already written the workspace's inv_pos (the
// inverse of sorted_pos) and tile list; otherwise they are derived here first.
moe_status experts_pass(const moe_dims* d, int64_t n, const void* x, const float* topk_weight,
                        const int32_t* offsets, const int32_t* sorted_pos, const moe_weights* w, void* rows,
                        void* ws, const Layout& L, bool gather, bool plan_ready, cudaStream_t s, Tracer& tr) {
  const int32_t R = static_cast<int32_t>(n * d->top_k);
  uint8_t* xs = at<uint8_t>(ws, L.xs);
  float* xs_inv = at<float>(ws, L.xs_inv);
  TileDesc* tiles = at<TileDesc>(ws, L.tiles);
  int32_t* n_tiles = at<int32_t>(ws, L.n_tiles);
  const bool fp8 = fp8_act(d);
  const int x_terms = x_terms_of(fp8);
  // The tile list is complete before the gather runs: the GEMMs are dependent launches
  // whose weight producer and MMA issuer read it without waiting.
  if (!plan_ready) {
    MOE_CHECK_CUDA(launch_build_tiles(offsets, d->num_experts, tile_tokens(R, d->num_experts), tiles, n_tiles, s));
    tr.after("build_tiles");
  }
  if (gather) {
    int32_t* ip = at<int32_t>(ws, L.inv_pos);
    if (!plan_ready) MOE_CHECK_CUDA(launch_invert_positions(sorted_pos, R, ip, s));
    MOE_CHECK_CUDA(launch_gather_rows(static_cast<const uint16_t*>(x), ip, static_cast<int32_t>(n), d->top_k, d->d,
                                      xs, rows_layout(R, d->num_experts, d->d, x_terms, fp8), xs_inv, s));
    tr.after("gather_rows");
  }
  return run_gemms(gather, fp8, w, d->d, d->d_ff, d->num_experts, R, x_terms, xs, xs_inv, at<uint8_t>(ws, L.h),
                   at<float>(ws, L.h_inv), tiles, n_tiles, sorted_pos, topk_weight, rows, at<uint32_t>(ws, L.err), s,
                   tr, "gateup_swiglu", "down_scatter");
}

// Shared expert on all n rows of xs_sh (identity order, weight 1) -> sh_out.
moe_status shared_pass(const moe_dims* d, int64_t n, const moe_weights* w, int32_t dff_sh, void* ws,
                       const Layout& L, cudaStream_t s, Tracer& tr) {
  TileDesc* tiles = at<TileDesc>(ws, L.tiles_sh);
  int32_t* n_tiles = at<int32_t>(ws, L.n_tiles) + 1;
  MOE_CHECK_CUDA(launch_identity_tiles(static_cast<int32_t>(n), tile_tokens(n, 1), tiles, n_tiles, s));
  tr.after("shared_tiles");
  const bool fp8 = fp8_act(d);
  return run_gemms(false, fp8, w, d->d, dff_sh, 1, static_cast<int32_t>(n), x_terms_of(fp8), at<uint8_t>(ws, L.xs_sh),
                   at<float>(ws, L.xs_sh_inv), at<uint8_t>(ws, L.h_sh), at<float>(ws, L.h_sh_inv), tiles, n_tiles,
                   nullptr, nullptr, at<uint16_t>(ws, L.sh_out), at<uint32_t>(ws, L.err), s, tr, "shared_gateup",
                   "shared_down");
}

}  // namespace
}  // namespace moe

// Scratch of moe_infer_static: a fixed device array in this library, so that
// entry point needs no workspace from its caller.  Every GPU that loads the
// library reserves it until the process exits.  Host code must not pass the
// symbol itself to a kernel (on the host it only names a stand-in object); the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t moe_static_scratch[MOE_STATIC_SCRATCH_BYTES];

namespace {

// Unique id of the calling thread's current CUDA context (cuCtxGetId), or 0
// when there is none or the driver does not offer the call.  Ids are never
// reused within a process, unlike context handles and device indices.
unsigned long long current_context_id() {
  using GetCurrentFn = CUresult (*)(CUcontext*);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long*);
  static std::once_flag once;
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of moe_static_scratch in the current device's context.  It is
// looked up (cudaGetSymbolAddress, with that device current) on the first call
// in each context and remembered with the context's id, so a context created
// again after cudaDeviceReset gets a fresh lookup instead of a stale address.
// nullptr if the lookup fails.
void* static_scratch_address() {
  struct Entry {
    unsigned long long ctx_id;
    void* addr;
  };
  static std::mutex mu;
  static Entry cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  const unsigned long long id = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (id != 0 && cache[dev].ctx_id == id && cache[dev].addr) return cache[dev].addr;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, moe_static_scratch) != cudaSuccess) return nullptr;
  // the lookup creates the context if this thread had none yet: key the entry on it
  cache[dev] = Entry{current_context_id(), p};
  return p;
}

}  // namespace

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_ROUTING: return "MOE_ERR_ROUTING";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_RANGE: return "MOE_ERR_RANGE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
  }
  return "MOE_ERR_UNKNOWN";
}

size_t moe_workspace_size(const moe_dims* dims, int64_t n_tokens, int32_t d_ff_shared) {
  Layout L;
  if (!make_layout(dims, n_tokens, d_ff_shared, &L)) return 0;
  return L.total;
}

size_t moe_permute_workspace_size(const moe_dims* dims, int64_t n_tokens) {
  Layout L;
  if (!make_layout(dims, n_tokens, 0, &L)) return 0;
  return L.route_end;
}

size_t moe_tiled_bytes(int32_t which, int32_t E, int32_t d, int32_t dff) {
  if (E < 1 || d <= 0 || dff <= 0 || d % 128 != 0 || dff % 128 != 0) return 0;
  if (which == 0) return static_cast<size_t>(pack_tile_count(E, dff, d, 0)) * 16384;
  if (which == 2) return static_cast<size_t>(pack_tile_count(E, d, dff, 1)) * 16384;
  return 0;
}

moe_status moe_pack_weights(int32_t E, int32_t d, int32_t dff, const moe_weights* src, const moe_weights* dst,
                            cudaStream_t s) {
  if (!src || !dst) return MOE_ERR_INVALID_ARG;
  if (E < 1 || d <= 0 || dff <= 0 || d % 128 != 0 || dff % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (src->layout != MOE_LAYOUT_ROW_MAJOR) return MOE_ERR_INVALID_ARG;
  const size_t mat = static_cast<size_t>(E) * d * dff;
  const uint8_t* in[3] = {src->w_gate, src->w_up, src->w_down};
  const uint8_t* out[2] = {dst->w_gate, dst->w_down};
  const size_t out_bytes[2] = {moe_tiled_bytes(0, E, d, dff), moe_tiled_bytes(2, E, d, dff)};
  for (int m = 0; m < 3; ++m)
    if (!in[m] || !aligned(in[m], 16)) return MOE_ERR_INVALID_ARG;
  for (int o = 0; o < 2; ++o) {
    if (!out[o] || !aligned(out[o], 16)) return MOE_ERR_INVALID_ARG;
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(out[o]);
    for (int m = 0; m < 3; ++m) {  // no source may overlap a destination
      const uintptr_t a0 = reinterpret_cast<uintptr_t>(in[m]);
      if (a0 < b0 + out_bytes[o] && b0 < a0 + mat) return MOE_ERR_INVALID_ARG;
    }
  }
  const uintptr_t g0 = reinterpret_cast<uintptr_t>(out[0]), d0 = reinterpret_cast<uintptr_t>(out[1]);
  if (g0 < d0 + out_bytes[1] && d0 < g0 + out_bytes[0]) return MOE_ERR_INVALID_ARG;
  if (launch_pack_tiles(in[0], in[1], const_cast<uint8_t*>(out[0]), E, dff, d, 0, s) != cudaSuccess ||
      launch_pack_tiles(in[2], nullptr, const_cast<uint8_t*>(out[1]), E, d, dff, 1, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_permute(const moe_dims* dims, int64_t n, const int32_t* topk_ids, int32_t* tokens_per_expert,
                       int32_t* expert_offsets, int32_t* sorted_pos, int32_t* inv_pos, int32_t validate,
                       void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (ws_bytes < L.route_end) return MOE_ERR_WORKSPACE;
  if (!tokens_per_expert || !expert_offsets) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!topk_ids || !sorted_pos)) return MOE_ERR_INVALID_ARG;
  uint32_t* err = at<uint32_t>(ws, L.err);
  if (launch_route_permute(topk_ids, static_cast<int32_t>(n), dims->top_k, dims->num_experts, tokens_per_expert,
                           expert_offsets, sorted_pos, inv_pos, validate, at<int32_t>(ws, L.route), err, 0, nullptr,
                           nullptr, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_experts_forward(const moe_dims* dims, int64_t n, const void* x, const float* topk_weight,
                               const int32_t* expert_offsets, const int32_t* sorted_pos, const moe_weights* w,
                               void* rows, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (n == 0) return MOE_OK;
  if (!x || !topk_weight || !expert_offsets || !sorted_pos || !rows || !weights_ok(w) || !aligned(x, 16) ||
      !aligned(rows, 16))
    return MOE_ERR_INVALID_ARG;
  Tracer tr{nullptr, s};
  return experts_pass(dims, n, x, topk_weight, expert_offsets, sorted_pos, w, rows, ws, L, true, false, s, tr);
}

moe_status moe_combine(const moe_dims* dims, int64_t n, const void* rows, const void* shared, const void* residual,
                       void* out, int32_t out_is_fp32, cudaStream_t s) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  if (!dims_ok(dims)) return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (!rows || !out || !aligned(rows, 16) || !aligned(out, 16) || (shared && !aligned(shared, 16)) ||
      (residual && !aligned(residual, 16)))
    return MOE_ERR_INVALID_ARG;
  if (launch_combine(static_cast<const uint16_t*>(rows), static_cast<const uint16_t*>(shared),
                     static_cast<const uint16_t*>(residual), static_cast<int32_t>(n), dims->top_k, dims->d, out,
                     out_is_fp32, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_infer(const moe_dims* dims, int64_t n, const void* x, const int32_t* topk_ids,
                     const float* topk_weight, const moe_weights* w, void* out, int32_t out_is_fp32, void* ws,
                     size_t ws_bytes, cudaStream_t s, moe_trace* trace) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (n == 0) return MOE_OK;
  if (!x || !topk_ids || !topk_weight || !out || !weights_ok(w) || !aligned(x, 16) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  Tracer tr{trace, s};
  tr.begin();
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* sp = at<int32_t>(ws, L.sorted_pos);
  int32_t* ip = at<int32_t>(ws, L.inv_pos);
  uint32_t* err = at<uint32_t>(ws, L.err);
  MOE_CHECK_CUDA(launch_route_permute(topk_ids, static_cast<int32_t>(n), dims->top_k, dims->num_experts, counts,
                                      offsets, sp, ip, 0, at<int32_t>(ws, L.route), err,
                                      tile_tokens(n * dims->top_k, dims->num_experts), at<TileDesc>(ws, L.tiles),
                                      at<int32_t>(ws, L.n_tiles), s));
  tr.after("route_permute", false, route_kernels(n * dims->top_k));
  void* rows = at<void>(ws, L.rows);
  moe_status st = experts_pass(dims, n, x, topk_weight, offsets, sp, w, rows, ws, L, true, true, s, tr);
  if (st != MOE_OK) return st;
  MOE_CHECK_CUDA(launch_combine(static_cast<const uint16_t*>(rows), nullptr, nullptr, static_cast<int32_t>(n),
                                dims->top_k, dims->d, out, out_is_fp32, s));
  tr.after("combine");
  return MOE_OK;
}

moe_status moe_layer_forward(const moe_dims* dims, int64_t n, const void* hidden, const void* gain, float eps,
                             const int32_t* topk_ids, const float* topk_weight, const moe_weights* routed,
                             const moe_weights* shared, int32_t dff_sh, void* out, int32_t out_is_fp32, void* ws,
                             size_t ws_bytes, cudaStream_t s, moe_trace* trace) {
  if (!dims || n < 0 || dff_sh < 0) return MOE_ERR_INVALID_ARG;
  if ((shared == nullptr) != (dff_sh == 0)) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, dff_sh, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (n == 0) return MOE_OK;
  if (!hidden || !gain || !topk_ids || !topk_weight || !out || !weights_ok(routed) ||
      (shared && !weights_ok(shared)) || !aligned(hidden, 16) || !aligned(gain, 16) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  if (!(eps >= 0.0f)) return MOE_ERR_INVALID_ARG;
  Tracer tr{trace, s};
  tr.begin();
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* sp = at<int32_t>(ws, L.sorted_pos);
  int32_t* ip = at<int32_t>(ws, L.inv_pos);
  uint32_t* err = at<uint32_t>(ws, L.err);
  MOE_CHECK_CUDA(launch_route_permute(topk_ids, static_cast<int32_t>(n), dims->top_k, dims->num_experts, counts,
                                      offsets, sp, ip, 0, at<int32_t>(ws, L.route), err,
                                      tile_tokens(n * dims->top_k, dims->num_experts), at<TileDesc>(ws, L.tiles),
                                      at<int32_t>(ws, L.n_tiles), s));
  tr.after("route_permute", false, route_kernels(n * dims->top_k));
  const int64_t R = n * dims->top_k;
  MOE_CHECK_CUDA(launch_rmsnorm_scatter(
      static_cast<const uint16_t*>(hidden), static_cast<const uint16_t*>(gain), eps, static_cast<int32_t>(n), dims->d,
      dims->top_k, ip, at<uint8_t>(ws, L.xs),
      rows_layout(R, dims->num_experts, dims->d, x_terms_of(fp8_act(dims)), fp8_act(dims)), at<float>(ws, L.xs_inv),
      shared ? at<uint8_t>(ws, L.xs_sh) : nullptr, rows_layout(n, 1, dims->d, x_terms_of(fp8_act(dims)), fp8_act(dims)),
      shared ? at<float>(ws, L.xs_sh_inv) : nullptr, s));
  tr.after("rmsnorm_scatter");
  void* rows = at<void>(ws, L.rows);
  moe_status st = experts_pass(dims, n, nullptr, topk_weight, offsets, sp, routed, rows, ws, L, false, true, s, tr);
  if (st != MOE_OK) return st;
  if (shared) {
    st = shared_pass(dims, n, shared, dff_sh, ws, L, s, tr);
    if (st != MOE_OK) return st;
  }
  MOE_CHECK_CUDA(launch_combine(static_cast<const uint16_t*>(rows),
                                shared ? at<uint16_t>(ws, L.sh_out) : nullptr, static_cast<const uint16_t*>(hidden),
                                static_cast<int32_t>(n), dims->top_k, dims->d, out, out_is_fp32, s));
  tr.after("combine");
  return MOE_OK;
}

moe_status moe_mlp_forward(const moe_dims* dims, int64_t n, const void* x, const moe_weights* w, void* out,
                           int32_t out_is_fp32, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  if (dims->num_experts != 1 || dims->top_k != 1) return MOE_ERR_UNSUPPORTED;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (n == 0) return MOE_OK;
  if (!x || !out || !weights_ok(w) || !aligned(x, 16) || !aligned(out, 16)) return MOE_ERR_INVALID_ARG;
  const bool fp8 = fp8_act(dims);
  const int32_t R = static_cast<int32_t>(n);
  TileDesc* tiles = at<TileDesc>(ws, L.tiles);
  int32_t* n_tiles = at<int32_t>(ws, L.n_tiles);
  uint8_t* xs = at<uint8_t>(ws, L.xs);
  float* xs_inv = at<float>(ws, L.xs_inv);
  Tracer tr{nullptr, s};
  // all n rows form one segment in their own order: identity tiles, identity gather
  MOE_CHECK_CUDA(launch_identity_tiles(R, tile_tokens(R, 1), tiles, n_tiles, s));
  MOE_CHECK_CUDA(launch_gather_rows(static_cast<const uint16_t*>(x), nullptr, R, 1, dims->d, xs,
                                    rows_layout(R, 1, dims->d, x_terms_of(fp8), fp8), xs_inv, s));
  void* rows = at<void>(ws, L.rows);
  moe_status st = run_gemms(true, fp8, w, dims->d, dims->d_ff, 1, R, x_terms_of(fp8), xs, xs_inv,
                            at<uint8_t>(ws, L.h), at<float>(ws, L.h_inv), tiles, n_tiles, nullptr, nullptr, rows,
                            at<uint32_t>(ws, L.err), s, tr, "mlp_gateup", "mlp_down");
  if (st != MOE_OK) return st;
  MOE_CHECK_CUDA(launch_combine(static_cast<const uint16_t*>(rows), nullptr, nullptr, R, 1, dims->d, out,
                                out_is_fp32, s));
  return MOE_OK;
}

moe_status moe_infer_static(const moe_dims* dims, int64_t n, const void* x, const int32_t* topk_ids,
                            const float* topk_weight, const moe_weights* w, void* out, int32_t out_is_fp32,
                            cudaStream_t s) {
  if (!dims || n < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (L.total > MOE_STATIC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;  // problem too big for the scratch
  if (n == 0) return MOE_OK;
  void* ws = static_scratch_address();
  if (!ws) return MOE_ERR_CUDA;
  // The same sequence as moe_infer; its first kernel resets the error word, the
  // only part of the scratch that must start at zero.
  return moe_infer(dims, n, x, topk_ids, topk_weight, w, out, out_is_fp32, ws, MOE_STATIC_SCRATCH_BYTES, s, nullptr);
}

// ---------------------------------------------------------------- expert parallelism

size_t moe_ep_plan_workspace_size(const moe_dims* dims, int64_t n_tokens) {
  Layout L;
  if (!make_layout(dims, n_tokens, 0, &L)) return 0;
  return L.xs;  // the error word, routing scratch, counts, offsets, sorted_pos and inv_pos
}

moe_status moe_ep_dispatch_plan(const moe_dims* dims, int32_t ep_size, int64_t n, const int32_t* topk_ids,
                                int32_t* tokens_per_expert, int32_t* send_counts, int32_t* tok_slot, int64_t capacity,
                                void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dims || n < 0 || capacity < 0) return MOE_ERR_INVALID_ARG;
  Layout L;
  if (!make_layout(dims, n, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (ep_size < 1 || ep_size > kMaxEpRanks || dims->num_experts % ep_size != 0) return MOE_ERR_UNSUPPORTED;
  if (capacity * ep_size >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.xs) return MOE_ERR_WORKSPACE;
  if (!tokens_per_expert || !send_counts) return MOE_ERR_INVALID_ARG;
  if (n > 0 && (!topk_ids || !tok_slot)) return MOE_ERR_INVALID_ARG;
  const int32_t R = static_cast<int32_t>(n * dims->top_k);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* ip = at<int32_t>(ws, L.inv_pos);
  uint32_t* err = at<uint32_t>(ws, L.err);
  if (launch_route_permute(topk_ids, static_cast<int32_t>(n), dims->top_k, dims->num_experts, tokens_per_expert,
                           offsets, at<int32_t>(ws, L.sorted_pos), ip, 0, at<int32_t>(ws, L.route), err, 0, nullptr,
                           nullptr, s) != cudaSuccess ||
      launch_ep_send_plan(topk_ids, R, dims->num_experts, ep_size, offsets, ip, capacity, send_counts, tok_slot, err,
                          s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_ep_gather(const moe_dims* dims, int64_t n, const void* x, const int32_t* tok_slot, int64_t n_slots,
                         void* send_rows, cudaStream_t s) {
  if (!dims || n < 0 || n_slots < 0) return MOE_ERR_INVALID_ARG;
  if (!dims_ok(dims) || n * dims->top_k >= (int64_t(1) << 31) || n_slots >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (!x || !tok_slot || !send_rows || !aligned(x, 16) || !aligned(send_rows, 16)) return MOE_ERR_INVALID_ARG;
  if (launch_ep_gather(static_cast<const uint16_t*>(x), tok_slot, static_cast<int32_t>(n), dims->top_k, dims->d,
                       n_slots, static_cast<uint16_t*>(send_rows), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

size_t moe_ep_regroup_workspace_size(int32_t experts_per_rank, int32_t ep_size) {
  if (experts_per_rank < 1 || ep_size < 1 || ep_size > kMaxEpRanks ||
      static_cast<int64_t>(experts_per_rank) * ep_size > kMaxExperts)
    return 0;
  return 256 + align_up(4 * static_cast<size_t>(ep_regroup_scratch_ints(experts_per_rank, ep_size)));
}

moe_status moe_ep_regroup(int32_t epr, int32_t ep_size, const int32_t* recv_counts, int64_t capacity, int64_t n_slots,
                          int32_t* local_counts, int32_t* local_offsets, int32_t* row_pos, int32_t* pos_row, void* ws,
                          size_t ws_bytes, cudaStream_t s) {
  if (capacity < 0 || n_slots < 0) return MOE_ERR_INVALID_ARG;
  const size_t need = moe_ep_regroup_workspace_size(epr, ep_size);
  if (need == 0 || n_slots >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < need) return MOE_ERR_WORKSPACE;
  if (!recv_counts || !local_counts || !local_offsets || (n_slots > 0 && (!row_pos || !pos_row)))
    return MOE_ERR_INVALID_ARG;
  if (launch_ep_regroup(recv_counts, epr, ep_size, capacity, n_slots, local_counts, local_offsets, row_pos, pos_row,
                        at<int32_t>(ws, 256), static_cast<uint32_t*>(ws), s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_ep_experts_forward(const moe_dims* dims, int64_t n_slots, const void* recv_rows,
                                  const int32_t* local_offsets, const int32_t* row_pos, const int32_t* pos_row,
                                  const moe_weights* w, void* out_rows, void* ws, size_t ws_bytes, cudaStream_t s) {
  if (!dims || n_slots < 0) return MOE_ERR_INVALID_ARG;
  if (dims->top_k != 1) return MOE_ERR_UNSUPPORTED;
  Layout L;
  if (!make_layout(dims, n_slots, 0, &L)) return MOE_ERR_UNSUPPORTED;
  if (!ws || !aligned(ws, 256) || ws_bytes < L.total) return MOE_ERR_WORKSPACE;
  if (n_slots == 0) return MOE_OK;
  if (!recv_rows || !local_offsets || !row_pos || !pos_row || !out_rows || !weights_ok(w) || !aligned(recv_rows, 16) ||
      !aligned(out_rows, 16))
    return MOE_ERR_INVALID_ARG;
  const int32_t R = static_cast<int32_t>(n_slots);
  const bool fp8 = fp8_act(dims);
  const int x_terms = x_terms_of(fp8);
  TileDesc* tiles = at<TileDesc>(ws, L.tiles);
  int32_t* n_tiles = at<int32_t>(ws, L.n_tiles);
  uint8_t* xs = at<uint8_t>(ws, L.xs);
  float* xs_inv = at<float>(ws, L.xs_inv);
  Tracer tr{nullptr, s};
  // tile list first (the GEMMs read it without waiting), then the received rows in expert order
  MOE_CHECK_CUDA(launch_build_tiles(local_offsets, dims->num_experts, tile_tokens(R, dims->num_experts), tiles,
                                    n_tiles, s));
  MOE_CHECK_CUDA(launch_gather_rows(static_cast<const uint16_t*>(recv_rows), row_pos, R, 1, dims->d, xs,
                                    rows_layout(R, dims->num_experts, dims->d, x_terms, fp8), xs_inv, s));
  // outputs unweighted (weight 1) to their received slot: out_rows[pos_row[sorted row]]
  return run_gemms(true, fp8, w, dims->d, dims->d_ff, dims->num_experts, R, x_terms, xs, xs_inv, at<uint8_t>(ws, L.h),
                   at<float>(ws, L.h_inv), tiles, n_tiles, pos_row, nullptr, out_rows, at<uint32_t>(ws, L.err), s, tr,
                   "ep_gateup", "ep_down");
}

moe_status moe_ep_combine(const moe_dims* dims, int64_t n, const void* back_rows, const int32_t* tok_slot,
                          int64_t n_slots, const float* topk_weight, void* out, int32_t out_is_fp32, cudaStream_t s) {
  if (!dims || n < 0 || n_slots < 0) return MOE_ERR_INVALID_ARG;
  if (!dims_ok(dims) || n * dims->top_k >= (int64_t(1) << 31) || n_slots >= (int64_t(1) << 31))
    return MOE_ERR_UNSUPPORTED;
  if (n == 0) return MOE_OK;
  if (!back_rows || !tok_slot || !topk_weight || !out || !aligned(back_rows, 16) || !aligned(out, 16))
    return MOE_ERR_INVALID_ARG;
  if (launch_ep_combine(static_cast<const uint16_t*>(back_rows), tok_slot, topk_weight, static_cast<int32_t>(n),
                        dims->top_k, dims->d, n_slots, out, out_is_fp32, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_check_bounded_wait(void* ws, cudaStream_t s) {
  if (!ws || !aligned(ws, 256)) return MOE_ERR_WORKSPACE;
  if (launch_bounded_wait_selftest(static_cast<uint32_t*>(ws), s) != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_get_error(void* ws, cudaStream_t s) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  uint32_t word = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpy(&word, ws, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  if (word == 0) return MOE_OK;
  if (cudaMemset(ws, 0, 4) != cudaSuccess) return MOE_ERR_CUDA;
  if (word & DEV_ERR_TIMEOUT) return MOE_ERR_TIMEOUT;
  if (word & DEV_ERR_ROUTING) return MOE_ERR_ROUTING;
  return MOE_ERR_RANGE;
}

}  // extern "C"
