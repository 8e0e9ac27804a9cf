/*
 * moe_ffn.h - C ABI of the GB300 routed-expert forward of a Kimi K2 MoE block.
 *
 * The operation (Kimi K2 model pages, pinned modeling_deepseek.py):
 *   "Mixture of experts" page, moe_infer: given token features x [n, d],
 *   router output topk_ids / topk_weight [n, k] and E SwiGLU experts, count
 *   the tokens of each expert, sort the flattened (token, slot) positions by
 *   expert, run every expert on its contiguous slice, put each output row
 *   back at its position and sum each token's k rows weighted by topk_weight.
 *   "SwiGLU output" page, MLP class: expert(x) = down(silu(gate x) * up x).
 *   "Element-wise product" page: h = silu(gate x) (.) (up x), [.., d_ff].
 *   "Input features" page, quantisation config: each linear weight is FP8
 *   e4m3 with one fp32 scale per 128 x 128 block (weight = code * scale).
 *   "Input features" page, decoder block + RMSNorm: the MoE block computes
 *   hidden + moe(RMSNorm(hidden)), RMSNorm(h) = gain * h / sqrt(mean(h^2) + eps)
 *   in fp32; "Mixture of experts" page, forward: plus one shared expert
 *   applied to every token.
 *
 * Conventions shared by every entry point
 *   - Buffers: all pointers except the dims/weights structs are DEVICE
 *     pointers owned by the caller.  The library never allocates or frees
 *     device memory and keeps no state between calls; scratch lives in the
 *     caller's workspace (see moe_workspace_size).  One exception:
 *     moe_infer_static takes no workspace and uses a fixed array inside the
 *     library that keeps the last call's contents (its Scratch and Sharing
 *     notes below).
 *   - Layouts are dense row-major.  Sizes: n tokens, d model width, d_ff
 *     expert width, E experts, k experts per token, R = n * k routed rows.
 *   - Types: activations bf16 (uint16 bit patterns), expert rows f16,
 *     router ids int32, router weights fp32, weights e4m3 bytes + fp32 scales.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream),
 *     performs no host synchronisation and can run inside stream capture.
 *     Errors that the host can see are returned at once and nothing is
 *     launched.  Errors only the device can see (an expert id outside
 *     [0, E), a duplicate id within one token when validation is on, a
 *     bounded wait that gave up, a value outside the f16 range) set a word in
 *     the workspace; the offending rows are skipped, never read or written
 *     out of bounds; moe_get_error reports and clears the word.
 *   - n = 0 is a no-op that returns MOE_OK.  Experts that no token selects
 *     cost nothing (they are skipped, as the page's loop skips them).
 *   - Limits: d and d_ff multiples of 128, 1 <= E <= 1024, 1 <= k <= 32,
 *     act_scheme one of the MOE_ACT_* values,
 *     n * k < 2^31.  Pointers handed to the tensor-memory-access engine
 *     (weights, x) must be 16-byte aligned; the workspace 256-byte aligned.
 *
 * Precision: the expert GEMMs run on the tensor cores into fp32 accumulators.
 * Under MOE_ACT_EXACT (the default; moe_dims below also offers dynamic FP8
 * activations) the operands depend on the tile width the batch gets (16-token
 * tiles while it averages fewer than 24 routed rows per expert, tiles of up to
 * 128 tokens from there on):
 *   16-token tiles: e4m3 weights x e4m3 activation terms.  Each activation row
 *     is carried as a sum of e4m3 terms sharing one power-of-two scale per 128
 *     columns: two terms hold a bf16 value exactly (x, and the bf16 RMSNorm
 *     output) unless it lies more than 2^10 below its block's maximum (then
 *     within 2^-18 of that maximum), three terms carry silu(g) * u (h, formed
 *     in fp32) to about 12 significant bits.  Each 128 x 128 weight block scale
 *     and the activation scale multiply the fp32 partial sum of their block.
 *   wide tiles: f16 x f16.  Each e4m3 weight code is widened to f16 exactly and
 *     multiplied by its block's scale times a power of two per weight row
 *     block (one f16 rounding, at most 2^-11 relative, while the block's scales
 *     along K lie within 2^10 of their largest); each activation row is the f16
 *     of the bf16 row times a power of two of its own, exact for every value
 *     within 2^28 of the row's largest magnitude; h is the f16 of
 *     silu(g) * u (at most 2^-11 relative from 2^-14 up, below that within
 *     2^-25 absolute).  The whole K extent accumulates in fp32 and the powers of
 *     two are undone in the epilogue.
 * Each weighted expert row is stored as f16, the k rows are summed in fp32 in
 * ascending slot order and the result is rounded once to bf16 (or kept in fp32
 * when out_is_fp32 is set).
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer where one is required, negative size, bad alignment */
    MOE_ERR_UNSUPPORTED = 2,   /* dims outside the limits above */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than moe_workspace_size */
    MOE_ERR_ROUTING = 4,       /* (device) expert id outside [0, E), or a duplicate id when validating */
    MOE_ERR_TIMEOUT = 5,       /* (device) a pipeline wait exceeded its bound; outputs are unspecified */
    MOE_ERR_RANGE = 6,         /* (device) an intermediate exceeded the f16 range; outputs hold inf */
    MOE_ERR_CUDA = 7           /* a CUDA runtime call or launch failed */
} moe_status;

/* Activation schemes ("Input features" page, quantisation config: fmt e4m3,
 * activation_scheme "dynamic", weight blocks of 128 x 128).
 *   MOE_ACT_EXACT        activations are never quantised to e4m3: every row
 *                        is carried as e4m3 split terms (16-token tiles) or
 *                        as a scaled f16 row (wide tiles), see Precision
 *                        above, so the result is the function of the FP8
 *                        weights to within those roundings and the f16 rows.
 *   MOE_ACT_FP8_DYNAMIC  every row entering a linear (x, the normalised row,
 *                        h) is quantised on the fly per group of 128
 *                        features: scale s = amax / 448 in fp32 (1 for an
 *                        all-zero group), code = e4m3 nearest to v / s (ties
 *                        to even, saturating at 448), the linear sees
 *                        code * s.  One e4m3 term per value: half the tensor
 *                        work of the exact scheme for gate/up, a third for
 *                        down, at the accuracy of e4m3 activations. */
#define MOE_ACT_EXACT 0
#define MOE_ACT_FP8_DYNAMIC 1

/* Problem dimensions: d = model width, d_ff = routed expert width,
 * num_experts = E, top_k = k, act_scheme = MOE_ACT_EXACT (0, what a
 * zero-initialised struct gives) or MOE_ACT_FP8_DYNAMIC. */
typedef struct {
    int32_t d;
    int32_t d_ff;
    int32_t num_experts;
    int32_t top_k;
    int32_t act_scheme;
} moe_dims;

/* Layout of the e4m3 codes of a bank. */
#define MOE_LAYOUT_ROW_MAJOR 0  /* [E][rows][cols], as the model stores them */
#define MOE_LAYOUT_TILED 1      /* moe_pack_weights output: 16 KB tiles, two per K block of a work unit */

/* One bank of FP8 SwiGLU experts (device pointers).
 *   w_gate, w_up : [E, d_ff, d] e4m3 codes;  s_gate, s_up : [E, d_ff/128, d/128] fp32
 *   w_down       : [E, d, d_ff] e4m3 codes;  s_down       : [E, d/128, d_ff/128] fp32
 * Element (r, c) of a matrix dequantises to e4m3(code[r][c]) * s[r/128][c/128].
 * With layout MOE_LAYOUT_TILED the codes are rearranged by moe_pack_weights:
 * w_gate holds gate and up together, w_up is not read (may be NULL), w_down
 * holds down (sizes from moe_tiled_bytes); the scales never change layout.
 * For the shared expert E = 1 and d_ff is the d_ff_shared argument. */
typedef struct {
    const uint8_t *w_gate, *w_up, *w_down;
    const float *s_gate, *s_up, *s_down;
    int32_t layout;         /* MOE_LAYOUT_ROW_MAJOR or MOE_LAYOUT_TILED */
} moe_weights;

/* Optional per-kernel timing.  The caller creates up to MOE_TRACE_MAX events;
 * a call that receives a trace records events[0] before its first kernel and
 * events[i + 1] after its i-th kernel on `stream`, sets labels[i] to a static
 * name for that kernel and n_recorded to the number of events recorded.  With
 * n_events = 0 nothing is recorded but n_launched is still set.  Pass NULL to
 * record and count nothing.  An event between two kernels costs the stream
 * about a launch gap, so timing a sample of calls disturbs the rest least. */
#define MOE_TRACE_MAX 16
typedef struct {
    cudaEvent_t events[MOE_TRACE_MAX];
    int32_t n_events;                   /* in: events usable */
    int32_t n_recorded;                 /* out */
    const char *labels[MOE_TRACE_MAX];  /* out */
    int32_t gemms_only;                 /* in: nonzero = events only around the grouped GEMMs:
                                           events[0] just before the first, events[i + 1] after the i-th */
    int32_t n_launched;                 /* out: kernels the call launched */
} moe_trace;

/* Bytes of workspace that every call below needs for n tokens (d_ff_shared =
 * width of the shared expert, 0 = none).  Returns 0 for unsupported dims. */
size_t moe_workspace_size(const moe_dims *dims, int64_t n_tokens, int32_t d_ff_shared);

/* Weight preparation for streaming (no counterpart on the pages: a storage
 * layout, not arithmetic).  The GEMMs work on units of one token tile times
 * two 128-row weight blocks: gate and up of the same rows, or down row blocks
 * 2p and 2p+1.  The tiled layout stores the two blocks' 128 x 128 tiles of one
 * K block (128 columns) next to each other, and consecutive K blocks one after
 * the other, so a unit streams one contiguous region and every copy moves
 * both blocks at once.  Each 16 KB tile holds row r of the tile at r * 128 with
 * its 16-byte chunk j at chunk position j ^ (r % 8) (the image a 128-byte-
 * swizzled TMA box leaves in shared memory).
 *   gate/up (dst->w_gate): tile (e, b, c, m) at (((e * d_ff/128 + b) * d/128 + c) * 2 + m) * 16384,
 *     m = 0 gate rows 128b.., m = 1 up rows 128b.., columns 128c..
 *   down (dst->w_down): with P = ceil(d/256) pairs, tile (e, p, c, m) at
 *     (((e * P + p) * d_ff/128 + c) * 2 + m) * 16384 holds down rows 128 (2p + m)..,
 *     columns 128c..; when d/128 is odd the last pair's second tile is zeros.
 *   num_experts, d, d_ff: the bank's sizes (d_ff = d_ff_shared for a shared expert)
 *   src: row-major codes; dst: caller-allocated buffers of moe_tiled_bytes bytes
 *        (dst->w_up, dst->s_* and dst->layout are not read).  src and dst must not overlap.
 * Asynchronous on `stream`; call once when the weights are loaded. */
moe_status moe_pack_weights(int32_t num_experts, int32_t d, int32_t d_ff, const moe_weights *src,
                            const moe_weights *dst, cudaStream_t stream);

/* Bytes of a tiled code buffer: which = 0 for w_gate (gate and up), 2 for
 * w_down.  0 for unsupported sizes or another `which`. */
size_t moe_tiled_bytes(int32_t which, int32_t num_experts, int32_t d, int32_t d_ff);

/* Routing plan ("Mixture of experts" page, moe_infer: the per-expert counts
 * and the sort of the flattened ids by expert).
 *   topk_ids          [n, k] int32 in
 *   tokens_per_expert [E]    int32 out: entries with id e
 *   expert_offsets    [E+1]  int32 out: exclusive prefix sum; offsets[E] = valid entries
 *   sorted_pos        [n*k]  int32 out: flat index t*k+j of the i-th entry in
 *                            (expert id, flat index) order - a stable sort; -1 past offsets[E]
 *   inv_pos           [n*k]  int32 out (may be NULL): inv_pos[sorted_pos[i]] = i; -1 for bad ids
 *   validate          nonzero: also flag a token that names one expert twice
 * Bad ids are counted nowhere and raise MOE_ERR_ROUTING on the device. */
moe_status moe_permute(const moe_dims *dims, int64_t n_tokens, const int32_t *topk_ids,
                       int32_t *tokens_per_expert, int32_t *expert_offsets, int32_t *sorted_pos,
                       int32_t *inv_pos, int32_t validate, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* moe_permute reads and writes only the first moe_permute_workspace_size bytes
 * of a workspace (the error word and, for large batches, per-chunk counts), so
 * a routing-only caller may pass a buffer of that size.  0 for unsupported dims. */
size_t moe_permute_workspace_size(const moe_dims *dims, int64_t n_tokens);

/* Expert pass ("Mixture of experts" page, moe_infer: gather the sorted token
 * rows, run each expert on its slice, write each output row back to its
 * position; "SwiGLU output" / "Element-wise product" pages for the expert).
 *   x               [n, d] bf16 in
 *   topk_weight     [n, k] fp32 in
 *   expert_offsets, sorted_pos: as produced by moe_permute for the same topk_ids
 *   weights         routed bank (struct on the host, tensors on the device)
 *   rows            [n, k, d] f16 out: rows[t][j] = topk_weight[t][j] * expert_{ids[t][j]}(x[t])
 * Rows of entries with bad ids are left unwritten. */
moe_status moe_experts_forward(const moe_dims *dims, int64_t n_tokens, const void *x, const float *topk_weight,
                               const int32_t *expert_offsets, const int32_t *sorted_pos,
                               const moe_weights *weights, void *rows, void *workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/* Combine ("Mixture of experts" page, moe_infer: weighted sum over the k
 * rows; forward: + shared expert; decoder block: + residual).
 *   out[t] = ((sum_{j=0..k-1} rows[t][j]) + shared[t]) + residual[t]
 * summed in fp32, j ascending.
 *   rows      [n, k, d] f16 in
 *   shared    [n, d] f16 in, or NULL
 *   residual  [n, d] bf16 in, or NULL
 *   out       [n, d] bf16, or fp32 when out_is_fp32 != 0 */
moe_status moe_combine(const moe_dims *dims, int64_t n_tokens, const void *rows, const void *shared,
                       const void *residual, void *out, int32_t out_is_fp32, cudaStream_t stream);

/* The whole routed-expert forward ("Mixture of experts" page, moe_infer):
 * moe_permute + moe_experts_forward + moe_combine with every intermediate in
 * the workspace.  out [n, d] bf16 (fp32 when out_is_fp32).  trace may be NULL. */
moe_status moe_infer(const moe_dims *dims, int64_t n_tokens, const void *x, const int32_t *topk_ids,
                     const float *topk_weight, const moe_weights *weights, void *out, int32_t out_is_fp32,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream, moe_trace *trace);

/* The MoE half of a decoder block ("Input features" page, decoder block and
 * RMSNorm; "Mixture of experts" page, forward):
 *   xn  = RMSNorm(hidden; gain, eps)                (fp32 arithmetic)
 *   out = hidden + ( sum_j topk_weight[t][j] * E_{ids[t][j]}(xn) + S(xn) )
 *   hidden [n, d] bf16, gain [d] bf16, routed bank, shared bank (E = 1,
 *   width d_ff_shared) or NULL with d_ff_shared = 0.  out as in moe_infer. */
moe_status moe_layer_forward(const moe_dims *dims, int64_t n_tokens, const void *hidden, const void *gain,
                             float eps, const int32_t *topk_ids, const float *topk_weight,
                             const moe_weights *routed, const moe_weights *shared, int32_t d_ff_shared,
                             void *out, int32_t out_is_fp32, void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, moe_trace *trace);

/* One SwiGLU MLP on every row ("SwiGLU output" page, MLP class: the same
 * module as each expert, which the model's dense feed-forward blocks also
 * use; their width is not printed on the pages, so d_ff is the caller's):
 *   out[t] = down( silu(gate x[t]) * up x[t] )
 * run through the same gather and grouped-GEMM kernels as a single expert
 * segment that holds all n rows in order, with weight 1.
 *   dims      num_experts = 1, top_k = 1 (else MOE_ERR_UNSUPPORTED); d_ff is
 *             the MLP's width; act_scheme as for moe_infer
 *   x         [n, d] bf16 in
 *   weights   one bank with E = 1 (either layout)
 *   out       [n, d] bf16, or fp32 when out_is_fp32 != 0
 *   workspace moe_workspace_size(dims, n, 0) bytes
 * Device-detected errors (f16 overflow, a timeout) accumulate in the
 * workspace's error word until moe_get_error reads it. */
moe_status moe_mlp_forward(const moe_dims *dims, int64_t n_tokens, const void *x, const moe_weights *weights,
                           void *out, int32_t out_is_fp32, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream);

/* ---------------------------------------------------------------- expert parallelism
 * "Input features" page, expert construction: with ep_size ranks, rank r holds
 * the experts [r * E/ep, (r + 1) * E/ep) (experts_per_rank = E / ep_size).
 * "Mixture of experts" page, moe_infer, ep_size > 1 branch: every rank sends
 * the rows it routes to rank r's experts to rank r, each rank groups what it
 * receives by local expert and runs its experts, the outputs return to their
 * source ranks and each token sums its k rows weighted by topk_weight.
 *
 * The two exchanges (an all-to-all of the per-expert counts, then of the rows
 * and back) are the caller's, e.g. NCCL through torch.distributed; the calls
 * below are the steps on either side of them, all asynchronous on `stream`
 * with no host synchronisation.  Rows travel in "slot" buffers:
 *   capacity = 0  rows for rank d follow those for ranks < d without gaps
 *                 (the pages' layout: the caller reads send_counts and the
 *                 received counts back to size the exchange);
 *   capacity = C  rows for rank d sit at slots d*C .. d*C + C - 1 (fixed split
 *                 sizes C, nothing to read back; a rank routing more than C
 *                 entries to one rank drops the rest and raises
 *                 MOE_ERR_ROUTING).
 * Sequence on each rank, for a batch of n tokens:
 *   1. moe_ep_dispatch_plan -> tokens_per_expert, send_counts, tok_slot
 *   2. moe_ep_gather        -> send rows (bf16, slot order)
 *   3. exchange tokens_per_expert [E] with equal splits of E/ep: rank r gets
 *      recv_counts [ep][E/ep] (source-major); exchange the rows
 *   4. moe_ep_regroup       -> local expert offsets, row_pos, pos_row
 *   5. moe_ep_experts_forward -> expert outputs in received slot order
 *   6. exchange the outputs back (the reverse of step 3's row exchange)
 *   7. moe_ep_combine       -> out [n, d]
 * Device-detected errors land in the error word at the start of each call's
 * workspace; moe_get_error reads it. */

/* Bytes of workspace moe_ep_dispatch_plan needs for n tokens (0: unsupported). */
size_t moe_ep_plan_workspace_size(const moe_dims *dims, int64_t n_tokens);

/* Step 1: the rank's routing plan (count and stable sort, as moe_permute) and
 * where each (token, slot) entry travels.
 *   dims              the full model: E = all routed experts, E % ep_size == 0
 *   ep_size           ranks, 1..256
 *   topk_ids          [n, k] int32 in
 *   tokens_per_expert [E] int32 out: entries per expert (what step 3 exchanges)
 *   send_counts       [ep] int32 out: entries for each rank (its split size)
 *   tok_slot          [n*k] int32 out: send slot of entry t*k+j, -1 when its id
 *                     is outside [0, E) (MOE_ERR_ROUTING) or dropped over capacity
 *   capacity          0 or C (see above) */
moe_status moe_ep_dispatch_plan(const moe_dims *dims, int32_t ep_size, int64_t n_tokens, const int32_t *topk_ids,
                                int32_t *tokens_per_expert, int32_t *send_counts, int32_t *tok_slot, int64_t capacity,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 2: send_rows[tok_slot[t*k+j]] = x[t] for every entry with a slot.
 *   x [n, d] bf16 in; send_rows [n_slots, d] bf16 out (slots without an entry are
 *   left as they are); n_slots = the send buffer's rows (n*k, or ep*C). */
moe_status moe_ep_gather(const moe_dims *dims, int64_t n_tokens, const void *x, const int32_t *tok_slot,
                         int64_t n_slots, void *send_rows, cudaStream_t stream);

/* Bytes of workspace moe_ep_regroup needs (0: unsupported sizes). */
size_t moe_ep_regroup_workspace_size(int32_t experts_per_rank, int32_t ep_size);

/* Step 4, on the receiving rank: the received rows grouped by local expert,
 * ties in received order (the page's regroup, taken stable).
 *   recv_counts   [ep][experts_per_rank] int32 in: rows from each source rank
 *                 for each local expert, as the count exchange delivers them
 *   capacity      0: the sources' rows follow each other without gaps; C: the
 *                 rows from source r start at slot r*C
 *   n_slots       rows of the received buffer; counts that do not fit are cut
 *                 (MOE_ERR_ROUTING)
 *   local_counts  [experts_per_rank] int32 out; local_offsets [experts_per_rank+1]
 *   row_pos       [n_slots] int32 out: position of received slot i in expert
 *                 order, -1 for an unused slot
 *   pos_row       [n_slots] int32 out: its inverse on the used positions */
moe_status moe_ep_regroup(int32_t experts_per_rank, int32_t ep_size, const int32_t *recv_counts, int64_t capacity,
                          int64_t n_slots, int32_t *local_counts, int32_t *local_offsets, int32_t *row_pos,
                          int32_t *pos_row, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Step 5: this rank's experts on the received rows ("SwiGLU output" page, MLP
 * class, each expert on its contiguous slice).
 *   dims          num_experts = experts_per_rank, top_k = 1 (else
 *                 MOE_ERR_UNSUPPORTED), d, d_ff, act_scheme as for moe_infer
 *   recv_rows     [n_slots, d] bf16 in (received slot order)
 *   local_offsets, row_pos, pos_row: from moe_ep_regroup
 *   weights       the rank's bank, E = experts_per_rank (global expert r*epr + e
 *                 at index e)
 *   out_rows      [n_slots, d] f16 out: expert(row) at the row's received slot,
 *                 not weighted; unused slots are left as they are
 *   workspace     moe_workspace_size(dims, n_slots, 0) bytes */
moe_status moe_ep_experts_forward(const moe_dims *dims, int64_t n_slots, const void *recv_rows,
                                  const int32_t *local_offsets, const int32_t *row_pos, const int32_t *pos_row,
                                  const moe_weights *weights, void *out_rows, void *workspace, size_t workspace_bytes,
                                  cudaStream_t stream);

/* Step 7: out[t] = sum_j topk_weight[t][j] * back_rows[tok_slot[t*k+j]] in fp32,
 * j ascending (entries without a slot add nothing).
 *   back_rows [n_slots, d] f16 in: the expert outputs returned to their send slots
 *   out       [n, d] bf16, or fp32 when out_is_fp32 != 0 */
moe_status moe_ep_combine(const moe_dims *dims, int64_t n_tokens, const void *back_rows, const int32_t *tok_slot,
                          int64_t n_slots, const float *topk_weight, void *out, int32_t out_is_fp32,
                          cudaStream_t stream);

/* moe_infer without a workspace, for callers that cannot allocate device
 * memory themselves: code that only receives input and output buffers from a
 * host framework (a plugin or an embedded runtime with its own memory
 * planner), code running inside another library's allocator or memory hooks,
 * and latency-critical paths where a cudaMalloc could synchronise the device.
 * The pages have no counterpart; it is a packaging of moe_infer.
 *   Scratch: a fixed array of MOE_STATIC_SCRATCH_BYTES inside this library,
 *   reserved on every GPU that loads it until the process exits.  Problems
 *   whose moe_workspace_size(dims, n, 0) exceeds it are rejected with
 *   MOE_ERR_WORKSPACE before anything runs (at K2 sizes, d 7168 / d_ff 2048 /
 *   k 8, that allows up to 24 tokens).
 *   Set-up: the first call in each device's CUDA context looks the array's
 *   device address up (cudaGetSymbolAddress) with that device current and
 *   remembers it for that context; make that first call before any stream
 *   capture (after cudaDeviceReset the new context's first call looks it up
 *   again).  No call allocates or frees memory.
 *   Sharing: every call on a device uses the same array, which keeps the last
 *   call's contents; calls that can overlap on the GPU (different streams
 *   without ordering, several host threads) race and corrupt each other's
 *   results, so order them.
 *   Errors: host-detectable errors are returned as by moe_infer.  Device-
 *   detected errors (bad expert ids, timeouts, f16 overflow) land in the shared
 *   array and are not reported; use moe_infer with a workspace to read them.
 * Arguments are those of moe_infer without workspace and trace. */
#define MOE_STATIC_SCRATCH_BYTES ((size_t)8 << 20)
moe_status moe_infer_static(const moe_dims *dims, int64_t n_tokens, const void *x, const int32_t *topk_ids,
                            const float *topk_weight, const moe_weights *weights, void *out, int32_t out_is_fp32,
                            cudaStream_t stream);

/* Diagnostic of the failure path (no counterpart on the pages): launches one
 * thread that waits on a barrier nothing will complete, through the same
 * bounded wait every GEMM pipeline stage uses.  After about one second it gives
 * up, records MOE_ERR_TIMEOUT in the workspace's error word and returns, so the
 * GPU context stays usable; moe_get_error then reports MOE_ERR_TIMEOUT.  Lets a
 * caller confirm that a stalled pipeline ends with a status, not a hang.
 *   workspace: any buffer of at least 256 bytes, 256-byte aligned. */
moe_status moe_check_bounded_wait(void *workspace, cudaStream_t stream);

/* Synchronises `stream`, returns the first device-detected error recorded in
 * `workspace` since the last call (MOE_OK if none) and clears it. */
moe_status moe_get_error(void *workspace, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
