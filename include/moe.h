/*
 * moe.h - C ABI of the sm_103a routed-expert FFN of one MoE layer.
 *
 * One MoE layer's routed-expert FFN over block-quantised expert weights held
 * in GPU memory: router top-k + softmax, a (token, expert) permutation grouped
 * by expert, then for every touched resident expert int4 dequant -> gate/up ->
 * SwiGLU -> down, and a deterministic weighted scatter back to the tokens, plus
 * an optional always-on shared expert. Experts absent from the expert-cache
 * slot map are skipped and reported as a list of ids.
 *
 * Passages of the Strata pages this follows (cited by page and section):
 *  - "extended-strata-moe reference", "Routing trace format": a token's routing
 *    is k expert ids and k fp32 weights;
 *  - "把 Strata 搬上 SGLang 引擎" post, TL;DR and section 3: one grouped call per
 *    layer does gather -> dequant -> gate/up -> SwiGLU -> down -> scatter over
 *    the packed expert bytes; section 2: only rows routed to an expert are
 *    computed (the expert-scoped layout);
 *  - Strata BATCHING, "Several requests at once": a window carries one or two
 *    rows per conversation and every expert shared by rows, and the shared
 *    expert, is read once per window;
 *  - "extended-strata-moe reference", "The mailbox": the GPU keeps its own
 *    copy of the slot map, computes the experts it holds and hands the others
 *    over; "C API": hits and misses count distinct experts per layer;
 *  - "PREFILL_HEAD_ALIAS": prompt chunks of up to 2,048 tokens.
 *
 * Conventions (all entry points):
 *  - Every pointer is a DEVICE pointer unless its comment says host. The
 *    caller owns every buffer; the library allocates no device memory.
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*,
 *    NULL = the legacy default stream) and never synchronise, except
 *    moe_read_status(). moe_route, moe_permute, moe_expert_ffn and
 *    moe_layer_forward may be captured into a CUDA graph; the first call of
 *    each on a device queries and sets kernel attributes and encodes tensor
 *    maps, so make one call before capturing (a warm-up call).
 *  - Argument errors found on the host return before anything is launched:
 *    MOE_ERR_INVALID (bad value or null pointer), MOE_ERR_UNSUPPORTED (a shape
 *    outside the limits below), MOE_ERR_WORKSPACE (workspace too small or not
 *    256-byte aligned). A failed launch returns MOE_ERR_CUDA.
 *  - Problems only the device can see are OR-ed into the status word at the
 *    start of the workspace; kernels never trap. Read it with
 *    moe_read_status(). Bits: 1 a non-finite router logit (that row's routing
 *    is unspecified); 2 a slot_map entry >= S, or an expert id outside [0, E)
 *    given to moe_expert_ffn (the entry is treated as not resident, the id is
 *    clamped); 4 a bounded wait expired after about a second (the call's
 *    results are incomplete); 8 an intermediate value beyond the fp16 range
 *    (an expert's SwiGLU output |h| >= 65504; the affected rows are
 *    unspecified); 16 a moe_decode_stack launch whose n_layers, T or
 *    workspace differ from its plan's (nothing ran).
 *  - Results are deterministic: run to run, and for the decode path (T <= 16)
 *    a row's output does not depend on the other rows of the window.
 *  - A workspace serves one call at a time: calls that share one must be
 *    ordered (one stream, or events). The one-launch decode kernel runs one
 *    CTA per SM; its work units go to whichever CTAs are running and its
 *    final reduction waits only for those units, so a CTA that starts late
 *    (SMs held by a kernel on another stream) delays the call without
 *    stalling the others. If a wait does expire (about a second; e.g. a
 *    workspace left inconsistent by an interrupted call), moe_read_status
 *    reports MOE_ERR_TIMEOUT: re-initialise the workspace and repeat the call.
 *
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), H and I (and shared_I)
 * multiples of 128 and at most 16384, T >= 0 (T = 0 is a no-op that reports
 * zero misses) with T*k <= 2^30 pairs (moe_workspace_bytes returns 0 beyond),
 * every q/scale pool, x and y 16-byte aligned. Three paths run a
 * layer: windows of T <= 16 rows with bf16 x, H a multiple of 512 up to 8192
 * and I, shared_I multiples of 256 take the one-launch decode kernel; T > 16
 * with bf16 x and H, I, shared_I multiples of 256 take the tensor-core
 * prefill kernels; every other call takes the separate-kernel path, which
 * holds a row block over all of H in shared memory and so takes H <= 11392.
 * The prefill and separate paths take T <= 65535 rows, and the separate path
 * at most 65535 work units (sum over experts of ceil(rows / 16), plus the
 * shared expert's). Calls beyond these limits return MOE_ERR_UNSUPPORTED
 * before anything is launched.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4,
  MOE_ERR_TIMEOUT = 5,
  MOE_ERR_DEVICE = 6
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* A block-quantised matrix pool, slot-major: for a matrix of `rows` rows and K
 * columns, slot s starts at q + s*rows*K/2 and scale + s*rows*K/32.
 *   q     [S][rows][K/2]  two's complement int4 codes in [-8, 7], column 2j in
 *                         the low nibble of byte j, column 2j+1 in the high one
 *   scale [S][rows][K/32] IEEE binary16 bit patterns, one per 32 columns
 * weight(r, c) = code(r, c) * scale(r, c/32). */
typedef struct {
  const uint8_t *q;
  const uint16_t *scale;
} moe_qmat;

/* One layer. gate and up have rows = I, K = H; down has rows = H, K = I.
 * The shared expert (shared_I > 0) has one slot of each, with I -> shared_I.
 * pick_counts: routing counters for an adaptive expert cache, counted inside
 * the engine ("extended-strata-moe reference", "The adaptive cache": picks per
 * (layer, expert), one per expert and window, large batches not counted).
 * Nullable device int32 [E], 4-byte aligned; when set, a moe_expert_ffn or
 * moe_layer_forward call of 1 <= T <= pick_max_rows rows adds 1 to
 * pick_counts[e] for every distinct expert e its window routes to, resident or
 * not (atomically, in the call's kernels). moe_cache_observe_device reads and
 * clears them. Zero-initialise the struct to leave counting off. */
typedef struct {
  int32_t H, I, E, k, S;
  moe_qmat gate, up, down;
  int32_t shared_I;
  moe_qmat shared_gate, shared_up, shared_down;
  int32_t *pick_counts;
  int32_t pick_max_rows;
} moe_layer_desc;

/* Router logits of the tiny configuration: logits[t][e] = sum_h x[t][h]*wg[h][e]
 * accumulated in float64 and rounded once to fp32 (so identical inputs give
 * the oracle's bits except at an fp32 rounding midpoint).
 * x [T][H] in x_dtype, wg [H][E] fp32, logits [T][E] fp32; T*E < 2^31
 * (MOE_ERR_UNSUPPORTED beyond). */
moe_status moe_router_logits(const void *x, moe_dtype x_dtype, const float *wg, int T, int H,
                             int E, float *logits, void *stream);

/* Router top-k and softmax ("extended-strata-moe reference", "Routing trace
 * format"; top-10 of 512 in the SGLang port post). Per row t of logits [T][E]:
 * ids[t][0..k) = the k largest logits in descending order, ties to the lower
 * expert id; w[t][j] = exp(l_j - l_0) / sum_i exp(l_i - l_0) over the k
 * selected, computed in float64 (sum in j order) and rounded once to fp32.
 * One warp per row. status: nullable device int32; a non-finite logit ORs 1
 * into it and the row's output is unspecified. */
moe_status moe_route(const float *logits, int T, int E, int k, int32_t *ids, float *w,
                     int32_t *status, void *stream);

/* Counting sort of the P = T*k pairs p = t*k + j by expert (SGLang port post,
 * section 2: rows grouped per expert). Outputs:
 *   offsets [E+1]       first sorted position of each expert, offsets[E] = P
 *   sorted_pair [P]     pair at each sorted position, p ascending within an expert
 *   pair_pos [P]        inverse of sorted_pair
 *   miss_ids [E]        distinct touched experts with slot_map[e] < 0, ascending
 *   n_miss [1]          their number ("C API": misses are distinct experts)
 * slot_map [E] nullable (= every expert resident in slot e); S = pool slots.
 * ws/ws_bytes: a workspace of at least moe_workspace_bytes() for (E, k, T).
 * A slot >= S ORs 2 into the workspace status word. */
moe_status moe_permute(const int32_t *ids, int T, int E, int k, const int32_t *slot_map, int S,
                       int32_t *offsets, int32_t *sorted_pair, int32_t *pair_pos,
                       int32_t *miss_ids, int32_t *n_miss, void *ws, size_t ws_bytes,
                       void *stream);

/* Routed-expert FFN given the routing (SGLang port post, section 3: gather ->
 * dequant -> gate/up -> SwiGLU -> down -> scatter in one call per layer):
 *   y[t] = sum_{j<k, slot(ids[t][j]) >= 0} w[t][j] * down(silu(gate x_t) * (up x_t))
 *          + shared(x_t)
 * summed in j order then the shared expert, fp32 out. x [T][H] in x_dtype,
 * ids/w [T][k] (from moe_route), slot_map [E] nullable, y [T][H] fp32,
 * miss_ids [E] and n_miss [1] as in moe_permute. Each touched resident
 * expert's packed bytes are streamed from the pool once per call. */
moe_status moe_expert_ffn(const moe_layer_desc *L, const void *x, moe_dtype x_dtype, int T,
                          const int32_t *ids, const float *w, const int32_t *slot_map, float *y,
                          int32_t *miss_ids, int32_t *n_miss, void *ws, size_t ws_bytes,
                          void *stream);

/* The whole layer from logits: moe_route then moe_expert_ffn. ids/w [T][k]
 * receive the routing. */
moe_status moe_layer_forward(const moe_layer_desc *L, const float *logits, const void *x,
                             moe_dtype x_dtype, int T, const int32_t *slot_map, float *y,
                             int32_t *ids, float *w, int32_t *miss_ids, int32_t *n_miss,
                             void *ws, size_t ws_bytes, void *stream);

/* ---- Several layers in one launch ----
 * The whole decode pass of a stack of MoE layers as one persistent kernel
 * (SGLang port post, section 3: the 48-layer pass captured as one graph; its
 * grouped-kernel figures show the per-launch cost a pass of 48 layers pays).
 * Each layer is moe_layer_forward on its own buffers: routing of its logits,
 * permutation, the held experts' FFN and the shared expert, the ordered
 * combine into its y (bitwise the same results as moe_layer_forward on that
 * layer). Layer l + 1 starts only after every CTA has finished layer l (a
 * grid-wide barrier), as a model whose next router input depends on this
 * layer's output requires. All layers take the one-launch decode kernel: bf16
 * x, 1 <= T <= 16, H a multiple of 512 up to 8192, I and shared_I multiples
 * of 256 (else MOE_ERR_UNSUPPORTED). */

/* One layer's DEVICE buffers, as moe_layer_forward takes them: logits [T][E]
 * fp32, x [T][H] bf16 (16-byte aligned), slot_map [E] (nullable = every
 * expert in slot e), y [T][H] fp32 (16-byte aligned), ids [T][k], w [T][k],
 * miss_ids [E], n_miss [1]. */
typedef struct {
  const float *logits;
  const void *x;
  const int32_t *slot_map;
  float *y;
  int32_t *ids;
  float *w;
  int32_t *miss_ids;
  int32_t *n_miss;
} moe_layer_io;

/* Bytes of a plan for n_layers layers (DEVICE memory the caller allocates,
 * 64-byte aligned); 0 if n_layers is out of 1 .. 124. */
size_t moe_decode_stack_plan_bytes(int32_t n_layers);

/* Build the plan of n_layers layers (layers and io: HOST arrays [n_layers])
 * for windows of T rows on workspace ws (at least moe_workspace_bytes of
 * every layer for T; shared by all layers): the per-layer kernel arguments
 * with their TMA descriptors, encoded on the host and copied into plan. It
 * synchronises `stream`: call it once, outside the hot path and outside any
 * stream capture. The plan holds the pointers given: it stays valid while
 * those buffers, the weight pools and ws do. Errors as moe_layer_forward,
 * plus MOE_ERR_INVALID for a plan smaller than moe_decode_stack_plan_bytes or
 * not 64-byte aligned. */
moe_status moe_decode_stack_prepare(const moe_layer_desc *layers, const moe_layer_io *io,
                                    int32_t n_layers, int32_t T, void *plan, size_t plan_bytes,
                                    void *ws, size_t ws_bytes, void *stream);

/* The same for a chained stack with the router in the launch (the whole
 * decode pass: the SGLang port post's section 3 runs the 48 layers, router
 * included, in one captured graph). router_w: HOST array [n_layers] of DEVICE
 * pointers to each layer's router weights [E][H] bf16 (16-byte aligned).
 * Layer l computes logits[t][e] = sum_h x_l[t][h] * W_r[e][h] (bf16 products,
 * fp32 sums in a fixed order: deterministic, within fp32 rounding of the
 * exact value) into io[l].logits, which is then an OUTPUT, routes them, and
 * runs the layer as above; its output also gives the next layer's input
 * x_{l+1}[t][h] = bf16_rne(x_l[t][h] + y_l[t][h]) (the residual add, one fp32
 * sum), written into io[l + 1].x. io[0].x is the caller's input; io[l].x for
 * l >= 1 are written by the launch. All layers take the same H. */
moe_status moe_decode_stack_prepare_routed(const moe_layer_desc *layers, const moe_layer_io *io,
                                           const uint16_t *const *router_w, int32_t n_layers,
                                           int32_t T, void *plan, size_t plan_bytes, void *ws,
                                           size_t ws_bytes, void *stream);

/* Run the prepared stack: one cooperative launch on `stream` (one CTA per SM,
 * all resident; MOE_ERR_CUDA if the device cannot hold them all). n_layers,
 * T and ws as prepared (the kernel checks them against the plan: a mismatch
 * ORs 16 into the status word of the ws given and runs nothing). Asynchronous and capturable
 * once the plan exists. Device-detected problems go to ws's status word as for
 * moe_layer_forward; a CTA that gives up (an expired bounded wait) ends the
 * launch after its layer, and the later layers' outputs are left unwritten. */
moe_status moe_decode_stack(const void *plan, int32_t n_layers, int32_t T, void *ws,
                            size_t ws_bytes, void *stream);

/* The routed-expert FFN for callers that cannot allocate device memory. The
 * Strata pages have no counterpart of this entry point: it exists for code
 * that cannot obtain a workspace (inside a framework whose allocator owns all
 * device memory, plugin code without an allocator handle, decode loops that
 * must not call cudaMalloc). Same arguments and results as moe_expert_ffn,
 * without ws/ws_bytes: the scratch is a fixed 16 MiB array inside the
 * library's device memory, reserved on every GPU that loads the library until
 * the process exits; nothing is allocated.
 *  - Returns MOE_ERR_UNSUPPORTED when moe_workspace_bytes(L, T) exceeds
 *    16 MiB (e.g. 2,048-token chunks): use moe_expert_ffn with a workspace.
 *  - Every call on a device shares the array and it keeps the last call's
 *    contents; the status word is cleared at each call. Calls that overlap on
 *    the GPU race on it: serialise them. Device-detected problems (an expired
 *    bounded wait, a slot beyond the pool, an id out of range, an h beyond the
 *    fp16 range) are OR-ed into the array's status word; read it with
 *    moe_static_read_status() after the call, before the next one.
 *  - The first call on a device looks up the array's address with that device
 *    current; make the first call before any stream capture. */
moe_status moe_expert_ffn_static(const moe_layer_desc *L, const void *x, moe_dtype x_dtype, int T,
                                 const int32_t *ids, const float *w, const int32_t *slot_map,
                                 float *y, int32_t *miss_ids, int32_t *n_miss, void *stream);

/* Status word of the last moe_expert_ffn_static call on the current device:
 * copies it on `stream` (after the call's kernels), waits for the stream and
 * stores the raw bits in *out. Returns MOE_OK (no bit set), MOE_ERR_TIMEOUT
 * (a bounded wait expired), MOE_ERR_DEVICE (other bits: 1 non-finite logit,
 * 2 bad slot or id, 8 h out of range), MOE_ERR_INVALID (null out) or
 * MOE_ERR_CUDA. Like moe_read_status, it synchronises: not for the hot path. */
moe_status moe_static_read_status(void *stream, int32_t *out);

/* Workspace bytes a call with this layer and T rows needs (256-byte aligned
 * base required); it also serves every call with fewer rows. L is a HOST
 * pointer. Returns 0 for an invalid desc or T (T < 0 or T*k > 2^30). */
size_t moe_workspace_bytes(const moe_layer_desc *L, int T);

/* Zero a workspace's status word and counters: once after allocating it, and
 * after any call that reported a device status (a timed-out call can leave the
 * counters non-zero). Needs ws_bytes >= 16,896. Asynchronous on stream. */
moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronise `stream`, then read the workspace status word into *out (HOST
 * pointer, the raw bits) and map it: 0 -> MOE_OK, a timeout -> MOE_ERR_TIMEOUT,
 * any other bit -> MOE_ERR_DEVICE. The word is sticky until moe_workspace_init. */
moe_status moe_read_status(const void *ws, void *stream, int32_t *out);

/* Static description of a status code (host string, never NULL). */
const char *moe_status_str(moe_status s);

/* Number of kernels the last call of this thread launched (host side count). */
int32_t moe_last_launch_count(void);

/* Kernel timing, a tracing aid (the pages' per-unit profilers, e.g. the SGLang
 * port post's env-gated per-expert-unit profiler, section 2). While enabled,
 * every kernel the library launches is bracketed by a pair of CUDA events
 * recorded on its own stream; on a stream being captured into a CUDA graph
 * they become external event-record nodes, re-recorded at every replay.
 *  moe_profile_enable(n): (re)arm with room for n launches, or disable (n = 0);
 *      resets the totals. MOE_ERR_CUDA if events cannot be created.
 *  moe_profile_collect(): wait for every recorded pair and add its elapsed time
 *      to the per-kind totals (call after each replay of a captured graph).
 *  moe_profile_forget(): drop the recorded pairs (before capturing anew).
 *  moe_profile_totals(kind, &ms, &count): the totals of one kernel kind.
 *  moe_profile_kind_name(kind): "route", "permute", "gateup", ... ("" if out of
 *      range). Kinds run from 0 while the name is non-empty. */
moe_status moe_profile_enable(int32_t max_launches);
moe_status moe_profile_collect(void);
moe_status moe_profile_forget(void);
moe_status moe_profile_totals(int32_t kind, double *total_ms, int64_t *count);
const char *moe_profile_kind_name(int32_t kind);

/* ---- Adaptive expert cache (host side) ----
 * "extended-strata-moe reference", "The adaptive cache": which experts occupy
 * a layer's pool slots is decided from the routing while decoding. A heat per
 * (layer, expert) counts one pick per expert and window (windows of more than
 * max_window_tokens rows do not count) and fades with a half-life in generated
 * tokens. Every fill_every_tokens, free slots take the hottest experts not held
 * (at most max_fills); every round_every_tokens, in a layer without free slots
 * the i-th hottest expert not held replaces the i-th coldest held one while
 * heat_in - in_picks > in_ratio * heat_out (at most max_swaps per round over
 * all layers, the hottest incoming first). Layers holding every expert are
 * left alone. The page's values: half-life 350 tokens, rounds every 32 tokens
 * with 64 swaps, fills every 8 tokens with 128, ratio 1.5 plus 2 picks, windows
 * of up to 32 tokens.
 *
 * The planner is host code on a HOST state buffer the caller owns (size from
 * moe_cache_state_bytes, 8-byte aligned); it only decides and keeps each
 * layer's slot map (int32 [E], -1 = not held, the moe_permute/moe_expert_ffn
 * slot_map). For each returned move the caller copies expert `expert_in`'s
 * codes and scales into pool slot `slot` of `layer` and uploads the layer's
 * slot map before the next window reads the pool. Calls on one state must not
 * run concurrently. Errors: MOE_ERR_INVALID (bad argument or not a state),
 * MOE_ERR_WORKSPACE (state buffer too small or misaligned); the int32/int64
 * returning calls give -1. */
typedef struct {
  int32_t n_layers, n_experts;     /* 1 .. 65536 each */
  double half_life_tokens;         /* > 0 */
  int32_t round_every_tokens;      /* >= 1 */
  int32_t max_swaps;               /* >= 0 */
  int32_t fill_every_tokens;       /* >= 1 */
  int32_t max_fills;               /* >= 0 */
  double in_ratio;                 /* >= 0 */
  double in_picks;
  int32_t max_window_tokens;       /* >= 1 */
  int32_t reserved;
} moe_cache_params;

/* One move of a round: expert_in takes slot `slot` of `layer`; expert_out is
 * the expert it evicts, -1 when the slot was free. */
typedef struct {
  int32_t layer, slot, expert_in, expert_out;
} moe_cache_swap;

/* Bytes of a state for these params and slots[n_layers] (HOST array, pool
 * slots per layer); 0 for invalid arguments. */
size_t moe_cache_state_bytes(const moe_cache_params *p, const int32_t *slots);
/* Initialise a state: every slot free, heat 0, clock 0. */
moe_status moe_cache_init(void *state, size_t bytes, const moe_cache_params *p, const int32_t *slots);
/* Place experts[0..n) (HOST, distinct) into slots 0..n-1 of a layer, freeing
 * the rest (e.g. a hottest-first start, or a layer held whole). */
moe_status moe_cache_set_resident(void *state, int32_t layer, const int32_t *experts, int32_t n);
/* Count one window's routing of a layer: ids (HOST int32 [T][k], e.g. moe_route's
 * output copied back) add one pick to every distinct expert. */
moe_status moe_cache_observe(void *state, int32_t layer, const int32_t *ids, int32_t T, int32_t k);
/* The same for every layer of a window at once: ids (HOST int32 [n_layers][T][k]).
 * Every id is validated before any layer is counted. */
moe_status moe_cache_observe_layers(void *state, const int32_t *ids, int32_t T, int32_t k);
/* Add picks counted elsewhere: counts (HOST int32 [n_layers][E], >= 0) are
 * added to the heats, counts[l][e] picks of expert e in layer l (the same as
 * that many moe_cache_observe windows picking it, with no advance between).
 * Every count is validated before any is added. */
moe_status moe_cache_observe_counts(void *state, const int32_t *counts);
/* The device-side counters of moe_layer_desc.pick_counts for every layer
 * (DEVICE int32 [n_layers][E], one layer's [E] per desc): copies them to the
 * host on `stream` (waits for it: call between windows, not in a captured
 * graph), clears them on `stream` and adds them as moe_cache_observe_counts
 * does. So the planner needs no per-window copy of the routing ids: the
 * counters accumulate on the GPU until the planner's next step. */
moe_status moe_cache_observe_device(void *state, int32_t *counts, void *stream);
/* Advance the clock by n_tokens generated tokens after a window: heats fade by
 * 2^(-n_tokens / half_life), then the fill round and the swap round run if
 * their clock has come (once each, fills first). swaps (HOST) receives the
 * moves; n_max must be at least max_fills + max_swaps. Returns the number of
 * moves. */
int32_t moe_cache_advance(void *state, int32_t n_tokens, moe_cache_swap *swaps, int32_t n_max);
/* A swap round now with at most max_swaps moves (n_max >= max_swaps), for
 * callers that decode in chunks. Returns the number of moves. */
int32_t moe_cache_rebalance(void *state, int32_t max_swaps, moe_cache_swap *swaps, int32_t n_max);
/* Copy out a layer's slot map (HOST int32 [E]) or its heats (HOST double [E]). */
moe_status moe_cache_slot_map(const void *state, int32_t layer, int32_t *slot_map);
moe_status moe_cache_heat(const void *state, int32_t layer, double *heat);
/* Experts brought into slots so far (fills and swaps). */
int64_t moe_cache_swapped_total(const void *state);

/* Expert profile ("Profile format (STRP)"), little-endian: "STRP", u32 version
 * 1, u32 n_layers, u32 n_expert, u32 slots (all layers), u32 n_ranked, then
 * n_ranked x (u16 layer, u16 expert) hottest first, then n_layers x n_expert x
 * i32 rank (-1 unranked). Write: the pairs with heat > 0, by heat, then layer,
 * then expert, into buf (HOST); n_max = 0 returns the size; returns the bytes
 * written or -1. Load: validates magic, version, dimensions against the state,
 * n_ranked and every pair, then fills each layer's slots with its pairs in
 * profile order (a repeated pair is skipped); the rank table is not read. */
int64_t moe_cache_profile_write(const void *state, uint8_t *buf, int64_t n_max);
moe_status moe_cache_profile_load(void *state, const uint8_t *buf, int64_t n);

/* ---- Mailbox: the missed experts, computed on the host ----
 * "extended-strata-moe reference", "The mailbox": the GPU computes the experts
 * its slot map holds and hands the rows routed to the others to host threads,
 * which compute those experts from the host copy of every expert and hand back
 * partial outputs; the GPU adds them to y in a fixed order. A job is one expert
 * over up to 8 of its rows (the multi-token CPU kernels of Strata BATCHING), so
 * a job reads the expert's weights once. The flow of one window:
 *   1. moe_layer_forward / moe_expert_ffn with the slot map (y holds the
 *      resident experts and the shared expert);
 *   2. copy ids, w (and x, if not on the host already) back; moe_mailbox_pairs
 *      lists the pairs p = t*k + j whose expert is not held, ascending;
 *   3. moe_mailbox_compute fills partial[i] = w_p * down(silu(gate x_t) * (up
 *      x_t)) for the i-th listed pair p, on the mailbox's threads (fp32);
 *   4. copy pairs and partials to the device; moe_mailbox_add adds, for every
 *      row t, its partials in list order (ascending j) to y[t].
 * The result is deterministic (each partial is one thread's fixed computation;
 * the sums run in list order).
 *  moe_mailbox_create(n_threads, timeout_ms): a pool of host threads; a compute
 *      call waits at most timeout_ms for its jobs. NULL for bad arguments.
 *  moe_mailbox_destroy: joins the threads.
 *  moe_mailbox_pairs: ids (HOST [T][k]), slot_map (HOST [E], -1 = not held) ->
 *      pairs (HOST, ascending) of the pairs whose expert is not held; returns
 *      their number (pairs NULL: only counts), or -1 (bad argument, an id
 *      outside [0, E), more than n_max pairs).
 *  moe_mailbox_compute: L describes a HOST store of every expert (slot = expert
 *      id: its gate/up/down q and scale pointers are host pointers, S >= E;
 *      shared expert ignored), x (HOST [T][H], x_dtype), ids and w (HOST
 *      [T][k]), pairs (HOST, strictly ascending, from moe_mailbox_pairs),
 *      partial (HOST [n_pairs][H] fp32, written). Returns MOE_OK, MOE_ERR_INVALID
 *      (bad argument or pair list), or MOE_ERR_TIMEOUT: a job did not come back
 *      in time (a stalled or lost thread); partial is then incomplete, no
 *      thread writes it or reads the caller's buffers after the call returns,
 *      and the mailbox serves the next call.
 *  moe_mailbox_inject(mb, mode): failure injection for tests, on the host: the
 *      next job taken stalls past the timeout (1) or is lost (2); 0 clears.
 *  moe_mailbox_add: partial (DEVICE [n][H] fp32, 16-byte aligned), pairs
 *      (DEVICE [n], ascending), y (DEVICE [T][H], 16-byte aligned): one kernel
 *      on `stream`; H a multiple of 4, T <= 65535. */
typedef struct moe_mailbox moe_mailbox;
moe_mailbox *moe_mailbox_create(int32_t n_threads, int32_t timeout_ms);
void moe_mailbox_destroy(moe_mailbox *mb);
int32_t moe_mailbox_pairs(const int32_t *ids, int32_t T, int32_t k, const int32_t *slot_map, int32_t E,
                          int32_t *pairs, int32_t n_max);
moe_status moe_mailbox_compute(moe_mailbox *mb, const moe_layer_desc *L, const void *x, moe_dtype x_dtype,
                               int32_t T, const int32_t *ids, const float *w, const int32_t *pairs,
                               int32_t n_pairs, float *partial);
moe_status moe_mailbox_inject(moe_mailbox *mb, int32_t mode);
moe_status moe_mailbox_add(const float *partial, const int32_t *pairs, int32_t n, int32_t T, int32_t k,
                           int32_t H, float *y, void *stream);

/* ---- Routing traces (host side) ----
 * "extended-strata-moe reference", "Routing trace format": one record per
 * token and layer, little-endian: int32 layer, int32 k, k x int32 expert id,
 * k x float32 weight.
 * moe_trace_write: records of one layer's T tokens from HOST ids/w [T][k] (w
 *   nullable: weights written as 0) into buf (HOST); n_max = 0 returns the
 *   size; returns the bytes written, or -1 (bad argument, buffer too small).
 * moe_trace_read: parses a buffer of records (any layers, any k <= k_max);
 *   n_max = 0 counts them; else fills layer[r], k_out[r], ids[r][k_max] and
 *   w[r][k_max] (HOST; slots past a record's k get id -1 and weight 0) for up
 *   to n_max records. Returns the number of records, or -1 for a truncated or
 *   malformed buffer (k < 1 or k > k_max) or more than n_max records. */
int64_t moe_trace_write(int32_t layer, const int32_t *ids, const float *w, int32_t T, int32_t k,
                        uint8_t *buf, int64_t n_max);
int64_t moe_trace_read(const uint8_t *buf, int64_t n, int32_t *layer, int32_t *k_out, int32_t *ids,
                       float *w, int32_t k_max, int64_t n_max);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
