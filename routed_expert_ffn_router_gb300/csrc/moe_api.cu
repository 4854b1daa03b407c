// C ABI of the routed-expert FFN library: argument validation, workspace
// layout and kernel sequencing. Declared in include/moe.h.
#include <climits>
#include <cstdio>
#include <mutex>
#include <vector>

#include "moe_internal.h"

namespace moe {

static thread_local int32_t g_launches = 0;

// ---- optional kernel timing: an event pair around every launch
namespace {
struct ProfPair {
  int kind;
  cudaEvent_t a, b;
};
struct Profiler {
  bool on = false;
  int cap = 0;
  std::vector<ProfPair> pairs;  // recorded since the last collect
  std::vector<cudaEvent_t> pool;
  size_t used = 0;
  double total_ms[K_NUM_KINDS] = {};
  int64_t count[K_NUM_KINDS] = {};
  int pending_kind = -1;
  cudaEvent_t pending = nullptr;
};
Profiler g_prof;
std::mutex g_prof_mu;

cudaEvent_t prof_event() {
  if (g_prof.used >= g_prof.pool.size()) return nullptr;
  return g_prof.pool[g_prof.used++];
}

void prof_record(cudaEvent_t ev, cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(st, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, st);
}
}  // namespace

void launch_begin(int kind, cudaStream_t st) {
  if (!g_prof.on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  cudaEvent_t ev = prof_event();
  if (!ev) return;
  prof_record(ev, st);
  g_prof.pending = ev;
  g_prof.pending_kind = kind;
}

void launch_end(cudaStream_t st) {
  ++g_launches;
  if (!g_prof.on) return;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  if (!g_prof.pending) return;
  cudaEvent_t ev = prof_event();
  if (!ev) return;
  prof_record(ev, st);
  g_prof.pairs.push_back({g_prof.pending_kind, g_prof.pending, ev});
  g_prof.pending = nullptr;
}

WsLayout ws_layout(int E, int k, int T, int H, int I, int shI) {
  WsLayout L{};
  const size_t P = (size_t)T * k;
  const int Imax = shI > I ? shI : I;
  size_t o = 0;
  L.P = (int)P;
  L.Imax = Imax;
  L.status = o;    o += 256;
  L.counters = o;  o += 256;
  L.sync = o;      o += (size_t)kSyncInts * 4;
  L.offsets = o;   o += align256(((size_t)E + 1) * 4);
  L.sorted_pair = o; o += align256((P ? P : 1) * 4);
  L.pair_pos = o;  o += align256((P ? P : 1) * 4);
  L.act = o;       o += align256(((P < (size_t)E ? P : (size_t)E) + 1) * sizeof(ActExpert));
  L.cu_max = cu_bound(T, E, k, shI > 0);
  L.cu = o;        o += align256((size_t)(L.cu_max > 0 ? L.cu_max : 1) * sizeof(int2));
  L.n_chunks = (int)((P + 1023) / 1024);
  L.hist = o;      o += L.n_chunks > 1 ? align256((size_t)L.n_chunks * E * 4) : 0;
  L.xhi = o;       o += align256((size_t)T * H * 2);
  L.xlo = o;       o += align256((size_t)T * H * 2);
  L.xcorr = o;     o += align256((size_t)T * (H / 32) * 4);
  const size_t rows = P + (size_t)T;
  L.hhi = o;       o += align256(rows * Imax * 2);
  L.hlo = o;       o += align256(rows * Imax * 2);
  L.hsum = o;      o += align256(rows * (Imax / 16) * 4);
  // The one-launch decode path keeps one partial per slice of I; a smaller
  // window may cut I finer, and a workspace sized for T serves every T' <= T.
  size_t prow = rows;
  for (int t = 1; t <= T && t <= 16; ++t) {
    const size_t r = (size_t)t * k + t;
    const size_t n = r * (size_t)fused_partial_slices(E, k, t, I, shI);
    prow = n > prow ? n : prow;
  }
  L.partial = o;   o += align256(prow * (size_t)H * 4);
  L.total = o;
  return L;
}

}  // namespace moe

namespace moe {
bool ffn_decode_supported(int H);  // moe_decode.cu: the separate-kernel path's H limit
}  // namespace moe

// (token, expert) pairs of a call at most: pair indices and counts are int32.
constexpr int64_t kMaxPairs = int64_t(1) << 30;
static bool pairs_ok(int T, int k) { return T >= 0 && (int64_t)T * k <= kMaxPairs; }

// Rows of a call, and work units of the separate-kernel path, index the second
// grid dimension of some launches (combine, x staging, gate/up, down).
constexpr int kMaxGridY = 65535;

// Whether the launches other than the one-launch decode kernel take this call:
// at most kMaxGridY rows, and on the separate-kernel path (not the tensor-core
// prefill) an H whose row block fits shared memory and at most kMaxGridY units.
static bool paths_take(const moe_layer_desc* Ld, int T, bool x_bf16, const moe::WsLayout& L) {
  if (T > kMaxGridY) return false;
  if (moe::prefill_tc_supported(Ld->H, Ld->I, Ld->shared_I, T, x_bf16)) return true;
  return moe::ffn_decode_supported(Ld->H) && L.cu_max <= kMaxGridY;
}

using namespace moe;

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static moe_status check_qmat(const moe_qmat& m) {
  if (!m.q || !m.scale) return MOE_ERR_INVALID;
  if (!aligned16(m.q) || !aligned16(m.scale)) return MOE_ERR_INVALID;
  return MOE_OK;
}

static moe_status check_dims(int E, int k) {
  if (E < 1 || k < 1) return MOE_ERR_INVALID;
  if (E > kMaxE || k > kMaxK || k > E) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

static moe_status check_desc(const moe_layer_desc* L) {
  if (!L) return MOE_ERR_INVALID;
  moe_status s = check_dims(L->E, L->k);
  if (s != MOE_OK) return s;
  if (L->H < 128 || L->I < 128 || L->S < 1 || L->shared_I < 0) return MOE_ERR_INVALID;
  if (L->H % 128 || L->I % 128 || L->shared_I % 128) return MOE_ERR_UNSUPPORTED;
  if (L->H > 16384 || L->I > 16384 || L->shared_I > 16384) return MOE_ERR_UNSUPPORTED;
  if ((s = check_qmat(L->gate)) != MOE_OK) return s;
  if ((s = check_qmat(L->up)) != MOE_OK) return s;
  if ((s = check_qmat(L->down)) != MOE_OK) return s;
  if (L->shared_I > 0) {
    if ((s = check_qmat(L->shared_gate)) != MOE_OK) return s;
    if ((s = check_qmat(L->shared_up)) != MOE_OK) return s;
    if ((s = check_qmat(L->shared_down)) != MOE_OK) return s;
  }
  if (L->pick_counts && ((reinterpret_cast<uintptr_t>(L->pick_counts) & 3u) || L->pick_max_rows < 0))
    return MOE_ERR_INVALID;
  return MOE_OK;
}

// The adaptive-cache counters of a call of T rows (nullptr: not counted).
static int32_t* picks_of(const moe_layer_desc* L, int T) {
  return L->pick_counts && T >= 1 && T <= L->pick_max_rows ? L->pick_counts : nullptr;
}

static moe_status check_ws(const void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return MOE_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_WORKSPACE;
  if (ws_bytes < need) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

static moe_status cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return MOE_OK;
  return MOE_ERR_CUDA;
}

template <typename T>
static T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

extern "C" {

const char* moe_status_str(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_WORKSPACE: return "workspace too small or misaligned";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "device-detected input error";
  }
  return "unknown status";
}

int32_t moe_last_launch_count(void) { return g_launches; }

moe_status moe_profile_enable(int32_t max_launches) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (cudaEvent_t e : g_prof.pool) cudaEventDestroy(e);
  g_prof.pool.clear();
  g_prof.pairs.clear();
  g_prof.used = 0;
  g_prof.pending = nullptr;
  for (int i = 0; i < K_NUM_KINDS; ++i) {
    g_prof.total_ms[i] = 0;
    g_prof.count[i] = 0;
  }
  g_prof.on = max_launches > 0;
  if (!g_prof.on) return MOE_OK;
  if (max_launches > (1 << 20)) return MOE_ERR_INVALID;
  for (int i = 0; i < 2 * max_launches; ++i) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) {
      g_prof.on = false;
      return MOE_ERR_CUDA;
    }
    g_prof.pool.push_back(e);
  }
  return MOE_OK;
}

moe_status moe_profile_collect(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  for (const ProfPair& p : g_prof.pairs) {
    float ms = 0.f;
    if (cudaEventSynchronize(p.b) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaEventElapsedTime(&ms, p.a, p.b) != cudaSuccess) return MOE_ERR_CUDA;
    g_prof.total_ms[p.kind] += ms;
    g_prof.count[p.kind] += 1;
  }
  return MOE_OK;
}

moe_status moe_profile_forget(void) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof.pairs.clear();
  g_prof.used = 0;
  return MOE_OK;
}

moe_status moe_profile_totals(int32_t kind, double* total_ms, int64_t* count) {
  if (kind < 0 || kind >= K_NUM_KINDS || !total_ms || !count) return MOE_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_prof_mu);
  *total_ms = g_prof.total_ms[kind];
  *count = g_prof.count[kind];
  return MOE_OK;
}

const char* moe_profile_kind_name(int32_t kind) {
  static const char* names[K_NUM_KINDS] = {"router_logits", "route", "permute", "x_prep",
                                           "gateup", "down", "combine", "fused_decode",
                                           "fused_stack"};
  if (kind < 0 || kind >= K_NUM_KINDS) return "";
  return names[kind];
}

size_t moe_workspace_bytes(const moe_layer_desc* L, int T) {
  if (check_desc(L) != MOE_OK || !pairs_ok(T, L->k)) return 0;
  return ws_layout(L->E, L->k, T, L->H, L->I, L->shared_I).total;
}

moe_status moe_workspace_init(void* ws, size_t ws_bytes, void* stream) {
  g_launches = 0;
  if (!ws || ws_bytes < kWsHeadBytes || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(ws, 0, kWsHeadBytes, static_cast<cudaStream_t>(stream)));
}

moe_status moe_read_status(const void* ws, void* stream, int32_t* out) {
  if (!ws || !out) return MOE_ERR_INVALID;
  int32_t v = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  *out = v;
  if (v == 0) return MOE_OK;
  if (v & DEV_TIMEOUT) return MOE_ERR_TIMEOUT;
  return MOE_ERR_DEVICE;
}

moe_status moe_router_logits(const void* x, moe_dtype x_dtype, const float* wg, int T, int H,
                             int E, float* logits, void* stream) {
  g_launches = 0;
  if (T < 0 || H < 1 || E < 1) return MOE_ERR_INVALID;
  if (x_dtype != MOE_F32 && x_dtype != MOE_BF16) return MOE_ERR_INVALID;
  if ((int64_t)T * E > INT32_MAX) return MOE_ERR_UNSUPPORTED;  // one thread per logit
  if (T == 0) return MOE_OK;
  if (!x || !wg || !logits) return MOE_ERR_INVALID;
  return cuda_status(launch_router_logits(x, x_dtype == MOE_BF16, wg, T, H, E, logits,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                     int32_t* status, void* stream) {
  g_launches = 0;
  moe_status s = check_dims(E, k);
  if (s != MOE_OK) return s;
  if (T < 0) return MOE_ERR_INVALID;
  if (T == 0) return MOE_OK;
  if (!logits || !ids || !w) return MOE_ERR_INVALID;
  return cuda_status(launch_route(logits, T, E, k, ids, w, status, static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute(const int32_t* ids, int T, int E, int k, const int32_t* slot_map, int S,
                       int32_t* offsets, int32_t* sorted_pair, int32_t* pair_pos,
                       int32_t* miss_ids, int32_t* n_miss, void* ws, size_t ws_bytes,
                       void* stream) {
  g_launches = 0;
  moe_status s = check_dims(E, k);
  if (s != MOE_OK) return s;
  if (T < 0 || S < 1) return MOE_ERR_INVALID;
  if (!pairs_ok(T, k)) return MOE_ERR_UNSUPPORTED;
  if (!offsets || !miss_ids || !n_miss) return MOE_ERR_INVALID;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the permutation needs no activation buffers: size its workspace for H = I = 128
  WsLayout L = ws_layout(E, k, T, 128, 128, 0);
  if ((s = check_ws(ws, ws_bytes, L.hist + (L.n_chunks > 1 ? (size_t)L.n_chunks * E * 4 : 0))) != MOE_OK)
    return s;
  if (T == 0) {
    cudaError_t e = cudaMemsetAsync(n_miss, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(offsets, 0, sizeof(int32_t) * (E + 1), st);
    return cuda_status(e);
  }
  if (!ids || !sorted_pair || !pair_pos) return MOE_ERR_INVALID;
  PermuteOut o;
  o.offsets = offsets;
  o.sorted_pair = sorted_pair;
  o.pair_pos = pair_pos;
  o.miss_ids = miss_ids;
  o.n_miss = n_miss;
  o.act = at<ActExpert>(ws, L.act);
  o.cu = at<int2>(ws, L.cu);
  o.counters = at<int32_t>(ws, L.counters);
  o.hist = at<int32_t>(ws, L.hist);
  o.status = at<int32_t>(ws, L.status);
  return cuda_status(launch_permute(ids, T, E, k, slot_map, S, false, o, st));
}

// The one-launch decode path: routing (when logits are given), permutation,
// gate/up, down and combine in one persistent kernel.
static moe_status fused_impl(const moe_layer_desc* Ld, const float* logits, const void* x, int T,
                             const int32_t* ids, const float* w, const int32_t* slot_map, float* y,
                             int32_t* ids_out, float* w_out, int32_t* miss_ids, int32_t* n_miss,
                             void* ws, const WsLayout& L, cudaStream_t st) {
  FusedLaunch f{};
  f.gq = Ld->gate.q; f.gs = Ld->gate.scale;
  f.uq = Ld->up.q;   f.us = Ld->up.scale;
  f.dq = Ld->down.q; f.ds = Ld->down.scale;
  if (Ld->shared_I > 0) {
    f.sgq = Ld->shared_gate.q; f.sgs = Ld->shared_gate.scale;
    f.suq = Ld->shared_up.q;   f.sus = Ld->shared_up.scale;
    f.sdq = Ld->shared_down.q; f.sds = Ld->shared_down.scale;
  }
  f.H = Ld->H; f.I = Ld->I; f.shI = Ld->shared_I; f.E = Ld->E; f.k = Ld->k; f.S = Ld->S;
  f.T = T; f.Imax = L.Imax; f.rows_cap = L.P + T;
  f.logits = logits; f.ids_in = ids; f.w_in = w;
  f.x = x; f.slot_map = slot_map;
  f.ids_out = ids_out; f.w_out = w_out; f.y = y; f.miss_ids = miss_ids; f.n_miss = n_miss;
  f.hhi = at<uint16_t>(ws, L.hhi);
  f.hlo = at<uint16_t>(ws, L.hlo);
  f.hcorr = at<float>(ws, L.hsum);
  f.partial = at<float>(ws, L.partial);
  f.status = at<int32_t>(ws, L.status);
  f.sync = at<int32_t>(ws, L.sync);
  f.picks = picks_of(Ld, T);
  return cuda_status(launch_fused_decode(f, st));
}

static moe_status expert_ffn_impl(const moe_layer_desc* Ld, const void* x, moe_dtype x_dtype, int T,
                                  const int32_t* ids, const float* w, const int32_t* slot_map,
                                  float* y, int32_t* miss_ids, int32_t* n_miss, void* ws,
                                  size_t ws_bytes, cudaStream_t st) {
  const WsLayout L = ws_layout(Ld->E, Ld->k, T, Ld->H, Ld->I, Ld->shared_I);
  moe_status s = check_ws(ws, ws_bytes, L.total);
  if (s != MOE_OK) return s;
  if (T == 0) return cuda_status(cudaMemsetAsync(n_miss, 0, sizeof(int32_t), st));
  if (!x || !ids || !w || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID;
  if (fused_decode_supported(Ld->H, Ld->I, Ld->shared_I, T, x_dtype == MOE_BF16))
    return fused_impl(Ld, nullptr, x, T, ids, w, slot_map, y, nullptr, nullptr, miss_ids, n_miss,
                      ws, L, st);
  if (!paths_take(Ld, T, x_dtype == MOE_BF16, L)) return MOE_ERR_UNSUPPORTED;
  const bool tc = prefill_tc_supported(Ld->H, Ld->I, Ld->shared_I, T, x_dtype == MOE_BF16);
  const bool has_shared = Ld->shared_I > 0;
  PermuteOut o;
  o.offsets = at<int32_t>(ws, L.offsets);
  o.sorted_pair = at<int32_t>(ws, L.sorted_pair);
  o.pair_pos = at<int32_t>(ws, L.pair_pos);
  o.miss_ids = miss_ids;
  o.n_miss = n_miss;
  o.act = at<ActExpert>(ws, L.act);
  o.cu = at<int2>(ws, L.cu);
  o.counters = at<int32_t>(ws, L.counters);
  o.hist = at<int32_t>(ws, L.hist);
  o.status = at<int32_t>(ws, L.status);
  cudaError_t e = launch_permute(ids, T, Ld->E, Ld->k, slot_map, Ld->S, has_shared, o, st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  if (int32_t* picks = picks_of(Ld, T))
    if ((e = launch_count_picks(o.offsets, Ld->E, picks, st)) != cudaSuccess) return MOE_ERR_CUDA;

  FfnArgs a{};
  a.gq = Ld->gate.q; a.gs = Ld->gate.scale;
  a.uq = Ld->up.q;   a.us = Ld->up.scale;
  a.dq = Ld->down.q; a.ds = Ld->down.scale;
  if (has_shared) {
    a.sgq = Ld->shared_gate.q; a.sgs = Ld->shared_gate.scale;
    a.suq = Ld->shared_up.q;   a.sus = Ld->shared_up.scale;
    a.sdq = Ld->shared_down.q; a.sds = Ld->shared_down.scale;
  }
  a.H = Ld->H; a.I = Ld->I; a.shI = Ld->shared_I; a.E = Ld->E; a.k = Ld->k; a.S = Ld->S;
  a.T = T; a.P = L.P; a.Imax = L.Imax;
  a.sorted_pair = o.sorted_pair;
  a.pair_pos = o.pair_pos;
  a.ids = ids;
  a.w = w;
  a.slot_map = slot_map;
  a.act = o.act;
  a.cu = o.cu;
  a.counters = o.counters;
  a.xhi = at<uint16_t>(ws, L.xhi);
  a.xlo = at<uint16_t>(ws, L.xlo);
  a.xcorr = at<float>(ws, L.xcorr);
  a.hhi = at<uint16_t>(ws, L.hhi);
  a.hlo = at<uint16_t>(ws, L.hlo);
  a.hsum = at<float>(ws, L.hsum);
  a.partial = at<float>(ws, L.partial);
  a.y = y;
  a.status = o.status;
  if (tc) {
    if ((e = launch_ffn_prefill_tc(a, x, st)) != cudaSuccess) return MOE_ERR_CUDA;
    return cuda_status(launch_combine(a, st));
  }
  return cuda_status(launch_ffn_decode(a, x, x_dtype == MOE_BF16, L.cu_max, st));
}

moe_status moe_expert_ffn(const moe_layer_desc* L, const void* x, moe_dtype x_dtype, int T,
                          const int32_t* ids, const float* w, const int32_t* slot_map, float* y,
                          int32_t* miss_ids, int32_t* n_miss, void* ws, size_t ws_bytes,
                          void* stream) {
  g_launches = 0;
  moe_status s = check_desc(L);
  if (s != MOE_OK) return s;
  if (T < 0 || (x_dtype != MOE_F32 && x_dtype != MOE_BF16)) return MOE_ERR_INVALID;
  if (!pairs_ok(T, L->k)) return MOE_ERR_UNSUPPORTED;
  if (!miss_ids || !n_miss) return MOE_ERR_INVALID;
  return expert_ffn_impl(L, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, ws, ws_bytes,
                         static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_forward(const moe_layer_desc* L, const float* logits, const void* x,
                             moe_dtype x_dtype, int T, const int32_t* slot_map, float* y,
                             int32_t* ids, float* w, int32_t* miss_ids, int32_t* n_miss, void* ws,
                             size_t ws_bytes, void* stream) {
  g_launches = 0;
  moe_status s = check_desc(L);
  if (s != MOE_OK) return s;
  if (T < 0 || (x_dtype != MOE_F32 && x_dtype != MOE_BF16)) return MOE_ERR_INVALID;
  if (!pairs_ok(T, L->k)) return MOE_ERR_UNSUPPORTED;
  if (!miss_ids || !n_miss) return MOE_ERR_INVALID;
  const WsLayout Lw = ws_layout(L->E, L->k, T, L->H, L->I, L->shared_I);
  if ((s = check_ws(ws, ws_bytes, Lw.total)) != MOE_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (T == 0) return cuda_status(cudaMemsetAsync(n_miss, 0, sizeof(int32_t), st));
  if (!logits || !ids || !w) return MOE_ERR_INVALID;
  if (!x || !y || !aligned16(x) || !aligned16(y)) return MOE_ERR_INVALID;
  if (fused_decode_supported(L->H, L->I, L->shared_I, T, x_dtype == MOE_BF16)) {
    return fused_impl(L, logits, x, T, nullptr, nullptr, slot_map, y, ids, w, miss_ids, n_miss, ws,
                      Lw, st);
  }
  if (!paths_take(L, T, x_dtype == MOE_BF16, Lw)) return MOE_ERR_UNSUPPORTED;
  cudaError_t e = launch_route(logits, T, L->E, L->k, ids, w, at<int32_t>(ws, Lw.status), st);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  return expert_ffn_impl(L, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, ws, ws_bytes, st);
}


size_t moe_decode_stack_plan_bytes(int32_t n_layers) {
  if (n_layers < 1 || n_layers > fused_stack_max_layers()) return 0;
  return fused_stack_plan_bytes(n_layers);
}

static moe_status stack_prepare(const moe_layer_desc* layers, const moe_layer_io* io,
                                const uint16_t* const* router_w, int32_t n_layers, int32_t T,
                                void* plan, size_t plan_bytes, void* ws, size_t ws_bytes,
                                void* stream) {
  g_launches = 0;
  if (!layers || !io || !plan) return MOE_ERR_INVALID;
  if (n_layers < 1 || T < 1) return MOE_ERR_INVALID;
  if (n_layers > fused_stack_max_layers()) return MOE_ERR_UNSUPPORTED;
  if (plan_bytes < fused_stack_plan_bytes(n_layers) || (reinterpret_cast<uintptr_t>(plan) & 63u))
    return MOE_ERR_INVALID;
  std::vector<FusedLaunch> fl((size_t)n_layers);
  for (int l = 0; l < n_layers; ++l) {
    const moe_layer_desc* Ld = &layers[l];
    const moe_layer_io& o = io[l];
    moe_status s = check_desc(Ld);
    if (s != MOE_OK) return s;
    if (!pairs_ok(T, Ld->k)) return MOE_ERR_UNSUPPORTED;
    if (!fused_decode_supported(Ld->H, Ld->I, Ld->shared_I, T, true)) return MOE_ERR_UNSUPPORTED;
    const WsLayout Lw = ws_layout(Ld->E, Ld->k, T, Ld->H, Ld->I, Ld->shared_I);
    if ((s = check_ws(ws, ws_bytes, Lw.total)) != MOE_OK) return s;
    if (!o.logits || !o.x || !o.y || !o.ids || !o.w || !o.miss_ids || !o.n_miss) return MOE_ERR_INVALID;
    if (!aligned16(o.x) || !aligned16(o.y)) return MOE_ERR_INVALID;
    if (router_w) {
      // chained: every layer the same H; layer l + 1's x is written by layer l
      if (!router_w[l] || !aligned16(router_w[l]) || Ld->H != layers[0].H) return MOE_ERR_INVALID;
      if (l + 1 < n_layers && !io[l + 1].x) return MOE_ERR_INVALID;
    }
    FusedLaunch& f = fl[(size_t)l];
    f.gq = Ld->gate.q; f.gs = Ld->gate.scale;
    f.uq = Ld->up.q;   f.us = Ld->up.scale;
    f.dq = Ld->down.q; f.ds = Ld->down.scale;
    if (Ld->shared_I > 0) {
      f.sgq = Ld->shared_gate.q; f.sgs = Ld->shared_gate.scale;
      f.suq = Ld->shared_up.q;   f.sus = Ld->shared_up.scale;
      f.sdq = Ld->shared_down.q; f.sds = Ld->shared_down.scale;
    }
    f.H = Ld->H; f.I = Ld->I; f.shI = Ld->shared_I; f.E = Ld->E; f.k = Ld->k; f.S = Ld->S;
    f.T = T; f.Imax = Lw.Imax; f.rows_cap = Lw.P + T;
    f.logits = o.logits;
    f.x = o.x; f.slot_map = o.slot_map;
    f.ids_out = o.ids; f.w_out = o.w; f.y = o.y; f.miss_ids = o.miss_ids; f.n_miss = o.n_miss;
    f.hhi = at<uint16_t>(ws, Lw.hhi);
    f.hlo = at<uint16_t>(ws, Lw.hlo);
    f.hcorr = at<float>(ws, Lw.hsum);
    f.partial = at<float>(ws, Lw.partial);
    f.status = at<int32_t>(ws, Lw.status);
    f.sync = at<int32_t>(ws, Lw.sync);
    f.picks = picks_of(Ld, T);
    if (router_w) {
      f.router_w = router_w[l];
      f.x_next = l + 1 < n_layers ? static_cast<uint16_t*>(const_cast<void*>(io[l + 1].x)) : nullptr;
    }
  }
  return cuda_status(fused_stack_prepare(fl.data(), n_layers, plan, static_cast<cudaStream_t>(stream)));
}

moe_status moe_decode_stack_prepare(const moe_layer_desc* layers, const moe_layer_io* io,
                                    int32_t n_layers, int32_t T, void* plan, size_t plan_bytes,
                                    void* ws, size_t ws_bytes, void* stream) {
  return stack_prepare(layers, io, nullptr, n_layers, T, plan, plan_bytes, ws, ws_bytes, stream);
}

moe_status moe_decode_stack_prepare_routed(const moe_layer_desc* layers, const moe_layer_io* io,
                                           const uint16_t* const* router_w, int32_t n_layers,
                                           int32_t T, void* plan, size_t plan_bytes, void* ws,
                                           size_t ws_bytes, void* stream) {
  if (!router_w) return MOE_ERR_INVALID;
  return stack_prepare(layers, io, router_w, n_layers, T, plan, plan_bytes, ws, ws_bytes, stream);
}

moe_status moe_decode_stack(const void* plan, int32_t n_layers, int32_t T, void* ws, size_t ws_bytes,
                            void* stream) {
  g_launches = 0;
  if (!plan || n_layers < 1 || T < 1 || T > 16) return MOE_ERR_INVALID;
  if (n_layers > fused_stack_max_layers()) return MOE_ERR_UNSUPPORTED;
  if (!ws || ws_bytes < kWsHeadBytes || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return MOE_ERR_WORKSPACE;
  const WsLayout Lw = ws_layout(1, 1, 1, 128, 128, 0);  // the head: status and counters
  return cuda_status(launch_fused_stack(plan, n_layers, T, at<int32_t>(ws, Lw.sync),
                                        at<int32_t>(ws, Lw.status), static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
