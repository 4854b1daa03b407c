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
 *    moe_read_status().
 *  - Argument errors found on the host return before anything is launched:
 *    MOE_ERR_INVALID (bad value or null pointer), MOE_ERR_UNSUPPORTED (a shape
 *    outside the limits below), MOE_ERR_WORKSPACE (workspace too small or not
 *    256-byte aligned). A failed launch returns MOE_ERR_CUDA.
 *  - Problems only the device can see (non-finite logit, slot out of range, an
 *    expired bounded wait) are OR-ed into the status word at the start of the
 *    workspace; kernels never trap. Read it with moe_read_status().
 *  - Results are deterministic: run to run, and for the decode path (T <= 16)
 *    a row's output does not depend on the other rows of the window.
 *
 * Limits: 1 <= E <= 1024, 1 <= k <= min(E, 32), H and I (and shared_I)
 * multiples of 128 and at most 16384, T >= 0 (T = 0 is a no-op that reports
 * zero misses), every q/scale pool, x and y 16-byte aligned.
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
 * The shared expert (shared_I > 0) has one slot of each, with I -> shared_I. */
typedef struct {
  int32_t H, I, E, k, S;
  moe_qmat gate, up, down;
  int32_t shared_I;
  moe_qmat shared_gate, shared_up, shared_down;
} moe_layer_desc;

/* Router logits of the tiny configuration: logits[t][e] = sum_h x[t][h]*wg[h][e]
 * accumulated in float64 and rounded once to fp32 (so identical inputs give
 * the oracle's bits except at an fp32 rounding midpoint).
 * x [T][H] in x_dtype, wg [H][E] fp32, logits [T][E] fp32. */
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
 *    the GPU race on it: serialise them. moe_read_status() cannot reach this
 *    array; device-detected problems are not reported through it.
 *  - The first call on a device looks up the array's address with that device
 *    current; make the first call before any stream capture. */
moe_status moe_expert_ffn_static(const moe_layer_desc *L, const void *x, moe_dtype x_dtype, int T,
                                 const int32_t *ids, const float *w, const int32_t *slot_map,
                                 float *y, int32_t *miss_ids, int32_t *n_miss, void *stream);

/* Workspace bytes a call with this layer and T rows needs (256-byte aligned
 * base required). L is a HOST pointer. Returns 0 for an invalid desc. */
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

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
