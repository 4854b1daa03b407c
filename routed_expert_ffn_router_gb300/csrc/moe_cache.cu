// Adaptive expert cache: the host-side planner that decides which experts
// occupy a layer's pool slots ("extended-strata-moe reference", "The adaptive
// cache"), and the STRP expert-profile format ("Profile format (STRP)").
//
// Rules, as the page states them:
//  * a heat per (layer, expert): one pick per expert and window (a window of
//    more than max_window_tokens rows does not count), old picks fading with a
//    half-life in generated tokens;
//  * every fill_every_tokens, free slots take the hottest experts not held, at
//    most max_fills per round;
//  * every round_every_tokens, the hottest experts not held replace the
//    coldest held ones, at most max_swaps per round, an expert coming in only
//    when its heat is more than in_ratio times the one it replaces plus
//    in_picks;
//  * layers held whole are left alone.
// Readings of the points the page leaves open are listed where they are used.
// The planner is plain host code: it decides and keeps the slot maps; the
// caller copies each swapped-in expert's bytes into its slot (between windows,
// before the next window reads the pool) and hands the slot map to the layer.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#include <algorithm>

#include "moe.h"

namespace {

constexpr uint32_t kStateMagic = 0x4d434143u;  // state buffer tag

// State buffer layout (host memory owned by the caller):
//   Header | int32 slots[L] | int32 slot_base[L] | int32 slot_map[L][E]
//   | int32 owner[total slots] | double heat[L][E]
struct Header {
  uint32_t magic;
  int32_t pad;
  moe_cache_params p;
  int64_t clock;       // generated tokens so far
  int64_t next_fill;   // clock of the next fill round
  int64_t next_round;  // clock of the next swap round
  int64_t n_swapped;   // experts brought in so far (fills and swaps)
  int32_t total_slots;
  int32_t pad2;
};

size_t align8(size_t v) { return (v + 7) & ~size_t(7); }

struct View {
  Header* h;
  int32_t* slots;
  int32_t* base;
  int32_t* map;    // [L][E]
  int32_t* owner;  // [total_slots]
  double* heat;    // [L][E]
};

size_t layout(const moe_cache_params* p, int total_slots, size_t off[5]) {
  const size_t L = (size_t)p->n_layers, E = (size_t)p->n_experts;
  size_t o = align8(sizeof(Header));
  off[0] = o; o = align8(o + 4 * L);                    // slots
  off[1] = o; o = align8(o + 4 * L);                    // slot_base
  off[2] = o; o = align8(o + 4 * L * E);                // slot_map
  off[3] = o; o = align8(o + 4 * (size_t)total_slots);  // owner
  off[4] = o; o = align8(o + 8 * L * E);                // heat
  return o;
}

bool params_ok(const moe_cache_params* p) {
  return p && p->n_layers >= 1 && p->n_layers <= 65536 && p->n_experts >= 1 && p->n_experts <= 65536 &&
         std::isfinite(p->half_life_tokens) && p->half_life_tokens > 0.0 && p->round_every_tokens >= 1 &&
         p->max_swaps >= 0 && p->fill_every_tokens >= 1 && p->max_fills >= 0 && std::isfinite(p->in_ratio) &&
         p->in_ratio >= 0.0 && std::isfinite(p->in_picks) && p->max_window_tokens >= 1;
}

int total_of(const moe_cache_params* p, const int32_t* slots) {
  if (!slots) return -1;
  int64_t t = 0;
  for (int l = 0; l < p->n_layers; ++l) {
    if (slots[l] < 0) return -1;
    t += slots[l];
  }
  return t > (int64_t)1 << 30 ? -1 : (int)t;
}

bool view_of(void* state, View* v) {
  if (!state) return false;
  Header* h = static_cast<Header*>(state);
  if (h->magic != kStateMagic) return false;
  size_t off[5];
  layout(&h->p, h->total_slots, off);
  uint8_t* b = static_cast<uint8_t*>(state);
  v->h = h;
  v->slots = reinterpret_cast<int32_t*>(b + off[0]);
  v->base = reinterpret_cast<int32_t*>(b + off[1]);
  v->map = reinterpret_cast<int32_t*>(b + off[2]);
  v->owner = reinterpret_cast<int32_t*>(b + off[3]);
  v->heat = reinterpret_cast<double*>(b + off[4]);
  return true;
}

int held_count(const View& v, int l) {
  int n = 0;
  for (int s = 0; s < v.slots[l]; ++s) n += v.owner[v.base[l] + s] >= 0 ? 1 : 0;
  return n;
}

// A layer is "held whole" when every expert has a slot; such a layer takes no
// part in rounds.
bool whole(const View& v, int l) { return held_count(v, l) >= v.h->p.n_experts; }

void place(View& v, int l, int slot, int e_in) {
  const int E = v.h->p.n_experts;
  const int prev = v.owner[v.base[l] + slot];
  if (prev >= 0) v.map[(size_t)l * E + prev] = -1;
  v.owner[v.base[l] + slot] = e_in;
  v.map[(size_t)l * E + e_in] = slot;
}

// The first `limit` of a list in the order `before` (a strict total order), in
// order: a round takes at most its cap from any layer, so only that many are
// sorted.
template <class Cmp>
void first_in_order(std::vector<int>& c, size_t limit, Cmp before) {
  if (c.size() > limit) {
    std::partial_sort(c.begin(), c.begin() + limit, c.end(), before);
    c.resize(limit);
  } else {
    std::sort(c.begin(), c.end(), before);
  }
}

// Experts of layer l not held and with heat > 0, hottest first (ties: lower
// id), at most `limit` of them.
std::vector<int> candidates_in(const View& v, int l, size_t limit, double above = 0.0) {
  const int E = v.h->p.n_experts;
  const double* ht = v.heat + (size_t)l * E;
  const int32_t* mp = v.map + (size_t)l * E;
  std::vector<int> c;
  for (int e = 0; e < E; ++e)
    if (mp[e] < 0 && ht[e] > 0.0 && ht[e] - above > 0.0) c.push_back(e);
  first_in_order(c, limit, [&](int a, int b) { return ht[a] > ht[b] || (ht[a] == ht[b] && a < b); });
  return c;
}

struct Move {
  double heat;
  int layer, e_in, e_out, slot;
};

// Global order of a round's moves: incoming heat descending, then layer, then
// expert id. Restricted to one layer it is that layer's candidate order, so
// a cap keeps a prefix of every layer's list.
void order_and_cap(std::vector<Move>& mv, int cap) {
  auto before = [](const Move& a, const Move& b) {
    if (a.heat != b.heat) return a.heat > b.heat;
    if (a.layer != b.layer) return a.layer < b.layer;
    return a.e_in < b.e_in;
  };
  if ((int)mv.size() > cap) {
    std::partial_sort(mv.begin(), mv.begin() + cap, mv.end(), before);
    mv.resize(cap);
  } else {
    std::sort(mv.begin(), mv.end(), before);
  }
}

// Fill round: free slots (ascending) take the hottest experts not held.
int fill_round(View& v, moe_cache_swap* out, int n_out) {
  std::vector<Move> mv;
  for (int l = 0; l < v.h->p.n_layers; ++l) {
    if (whole(v, l)) continue;
    std::vector<int> freeslots;
    for (int s = 0; s < v.slots[l]; ++s)
      if (v.owner[v.base[l] + s] < 0) freeslots.push_back(s);
    if (freeslots.empty()) continue;
    const std::vector<int> c =
        candidates_in(v, l, std::min(freeslots.size(), (size_t)std::max(v.h->p.max_fills, 0)));
    const size_t n = std::min(c.size(), freeslots.size());
    for (size_t i = 0; i < n; ++i)
      mv.push_back({v.heat[(size_t)l * v.h->p.n_experts + c[i]], l, c[i], -1, freeslots[i]});
  }
  // the cap keeps a prefix of each layer's list, so the kept moves of a layer
  // hold its lowest free slots in order
  order_and_cap(mv, v.h->p.max_fills);
  int n = 0;
  for (const Move& m : mv) {
    place(v, m.layer, m.slot, m.e_in);
    if (n < n_out) out[n] = {m.layer, m.slot, m.e_in, -1};
    ++n;
  }
  v.h->n_swapped += n;
  return n;
}

// Swap round: in a layer with no free slot (a layer with free slots is filled
// by fill rounds instead), the i-th hottest expert not held replaces the i-th
// coldest held one while heat_in - in_picks > in_ratio * heat_out: an incoming
// expert must beat in_ratio times the evicted one's heat by in_picks picks
// (1.5 and 2 on the page), so the held set does not flap. The comparison is
// written in this form (one product, one difference) wherever it is computed.
int swap_round(View& v, int cap, moe_cache_swap* out, int n_out) {
  const int E = v.h->p.n_experts;
  std::vector<Move> mv;
  for (int l = 0; l < v.h->p.n_layers; ++l) {
    if (v.slots[l] == 0 || whole(v, l) || held_count(v, l) < v.slots[l]) continue;
    const double* ht = v.heat + (size_t)l * E;
    const double picks = v.h->p.in_picks, ratio = v.h->p.in_ratio;
    // Exact shortcuts (the same decisions, less sorting): the test passes only
    // if heat_in - picks > ratio * heat_out >= 0, so an expert with
    // heat - picks <= 0 never comes in; and if the hottest expert outside
    // cannot replace the coldest held one, no pair of this layer can.
    double hmax = 0.0, hmin = 0.0;
    bool any_out = false;
    for (int e = 0; e < E; ++e) {
      const int32_t sm = v.map[(size_t)l * E + e];
      if (sm < 0 && ht[e] > 0.0) { hmax = any_out ? std::max(hmax, ht[e]) : ht[e]; any_out = true; }
    }
    for (int s = 0; s < v.slots[l]; ++s) {
      const double hv = ht[v.owner[v.base[l] + s]];
      hmin = s == 0 ? hv : std::min(hmin, hv);
    }
    if (!any_out || !(hmax - picks > ratio * hmin)) continue;
    const std::vector<int> in = candidates_in(v, l, (size_t)cap, picks);
    std::vector<int> held;
    for (int s = 0; s < v.slots[l]; ++s) held.push_back(v.owner[v.base[l] + s]);
    // coldest first (ties: lower id)
    first_in_order(held, in.size(), [&](int a, int b) { return ht[a] < ht[b] || (ht[a] == ht[b] && a < b); });
    const size_t n = std::min(in.size(), held.size());
    for (size_t i = 0; i < n; ++i) {
      const double hi = ht[in[i]], ho = ht[held[i]];
      if (!(hi - v.h->p.in_picks > v.h->p.in_ratio * ho)) break;
      mv.push_back({hi, l, in[i], held[i], v.map[(size_t)l * E + held[i]]});
    }
  }
  order_and_cap(mv, cap);
  int n = 0;
  for (const Move& m : mv) {
    place(v, m.layer, m.slot, m.e_in);
    if (n < n_out) out[n] = {m.layer, m.slot, m.e_in, m.e_out};
    ++n;
  }
  v.h->n_swapped += n;
  return n;
}

void put_u32(uint8_t* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
void put_u16(uint8_t* p, uint32_t v) {
  p[0] = (uint8_t)v;
  p[1] = (uint8_t)(v >> 8);
}
uint32_t get_u32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}
uint32_t get_u16(const uint8_t* p) { return (uint32_t)p[0] | ((uint32_t)p[1] << 8); }

}  // namespace

extern "C" {

size_t moe_cache_state_bytes(const moe_cache_params* p, const int32_t* slots) {
  if (!params_ok(p)) return 0;
  const int t = total_of(p, slots);
  if (t < 0) return 0;
  size_t off[5];
  return layout(p, t, off);
}

moe_status moe_cache_init(void* state, size_t bytes, const moe_cache_params* p, const int32_t* slots) {
  if (!state || !params_ok(p)) return MOE_ERR_INVALID;
  const int t = total_of(p, slots);
  if (t < 0) return MOE_ERR_INVALID;
  size_t off[5];
  const size_t need = layout(p, t, off);
  if (bytes < need || (reinterpret_cast<uintptr_t>(state) & 7)) return MOE_ERR_WORKSPACE;
  std::memset(state, 0, need);
  Header* h = static_cast<Header*>(state);
  h->magic = kStateMagic;
  h->p = *p;
  h->clock = 0;
  h->next_fill = p->fill_every_tokens;
  h->next_round = p->round_every_tokens;
  h->n_swapped = 0;
  h->total_slots = t;
  View v;
  view_of(state, &v);
  int b = 0;
  for (int l = 0; l < p->n_layers; ++l) {
    v.slots[l] = slots[l];
    v.base[l] = b;
    b += slots[l];
  }
  for (size_t i = 0; i < (size_t)p->n_layers * p->n_experts; ++i) v.map[i] = -1;
  for (int s = 0; s < t; ++s) v.owner[s] = -1;
  return MOE_OK;
}

moe_status moe_cache_set_resident(void* state, int32_t layer, const int32_t* experts, int32_t n) {
  View v;
  if (!view_of(state, &v)) return MOE_ERR_INVALID;
  const int E = v.h->p.n_experts;
  if (layer < 0 || layer >= v.h->p.n_layers || n < 0 || n > v.slots[layer] || (n > 0 && !experts))
    return MOE_ERR_INVALID;
  std::vector<char> seen(E, 0);
  for (int i = 0; i < n; ++i) {
    if (experts[i] < 0 || experts[i] >= E || seen[experts[i]]) return MOE_ERR_INVALID;
    seen[experts[i]] = 1;
  }
  for (int s = 0; s < v.slots[layer]; ++s) v.owner[v.base[layer] + s] = -1;
  for (int e = 0; e < E; ++e) v.map[(size_t)layer * E + e] = -1;
  for (int i = 0; i < n; ++i) place(v, layer, i, experts[i]);
  return MOE_OK;
}

moe_status moe_cache_observe(void* state, int32_t layer, const int32_t* ids, int32_t T, int32_t k) {
  View v;
  if (!view_of(state, &v)) return MOE_ERR_INVALID;
  const int E = v.h->p.n_experts;
  if (layer < 0 || layer >= v.h->p.n_layers || T < 0 || k < 1 || (T > 0 && !ids)) return MOE_ERR_INVALID;
  const size_t P = (size_t)T * k;
  for (size_t i = 0; i < P; ++i)
    if (ids[i] < 0 || ids[i] >= E) return MOE_ERR_INVALID;
  if (T > v.h->p.max_window_tokens) return MOE_OK;  // a large batch does not count
  std::vector<char> seen(E, 0);
  double* ht = v.heat + (size_t)layer * E;
  for (size_t i = 0; i < P; ++i)
    if (!seen[ids[i]]) {
      seen[ids[i]] = 1;
      ht[ids[i]] += 1.0;  // once per expert and window
    }
  return MOE_OK;
}

moe_status moe_cache_observe_layers(void* state, const int32_t* ids, int32_t T, int32_t k) {
  View v;
  if (!view_of(state, &v)) return MOE_ERR_INVALID;
  if (T < 0 || k < 1 || (T > 0 && !ids)) return MOE_ERR_INVALID;
  const size_t P = (size_t)T * k, E = (size_t)v.h->p.n_experts;
  const size_t all = P * (size_t)v.h->p.n_layers;
  for (size_t i = 0; i < all; ++i)  // validate every layer before counting any
    if (ids[i] < 0 || (size_t)ids[i] >= E) return MOE_ERR_INVALID;
  for (int l = 0; l < v.h->p.n_layers; ++l) {
    const moe_status s = moe_cache_observe(state, l, ids + (size_t)l * P, T, k);
    if (s != MOE_OK) return s;
  }
  return MOE_OK;
}

moe_status moe_cache_observe_counts(void* state, const int32_t* counts) {
  View v;
  if (!view_of(state, &v) || !counts) return MOE_ERR_INVALID;
  const size_t LE = (size_t)v.h->p.n_layers * v.h->p.n_experts;
  for (size_t i = 0; i < LE; ++i)  // validate every count before adding any
    if (counts[i] < 0) return MOE_ERR_INVALID;
  for (size_t i = 0; i < LE; ++i) v.heat[i] += (double)counts[i];
  return MOE_OK;
}

moe_status moe_cache_observe_device(void* state, int32_t* counts, void* stream) {
  View v;
  if (!view_of(state, &v) || !counts) return MOE_ERR_INVALID;
  const size_t LE = (size_t)v.h->p.n_layers * v.h->p.n_experts;
  std::vector<int32_t> host(LE);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(host.data(), counts, LE * sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(counts, 0, LE * sizeof(int32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return moe_cache_observe_counts(state, host.data());
}

int32_t moe_cache_advance(void* state, int32_t n_tokens, moe_cache_swap* swaps, int32_t n_max) {
  View v;
  if (!view_of(state, &v) || n_tokens < 0) return -1;
  const moe_cache_params& p = v.h->p;
  if (n_max < p.max_fills + p.max_swaps || (n_max > 0 && !swaps)) return -1;
  if (n_tokens > 0) {
    // old picks fade: heat *= 2^(-n / half_life)
    const double f = std::pow(2.0, -(double)n_tokens / p.half_life_tokens);
    const size_t LE = (size_t)p.n_layers * p.n_experts;
    for (size_t i = 0; i < LE; ++i) v.heat[i] = v.heat[i] * f;
  }
  v.h->clock += n_tokens;
  int n = 0;
  // Reading: a step that crosses one or more round boundaries runs each kind
  // of round once, the fill round first.
  if (v.h->clock >= v.h->next_fill) {
    n += fill_round(v, swaps + n, n_max - n);
    v.h->next_fill = (v.h->clock / p.fill_every_tokens + 1) * p.fill_every_tokens;
  }
  if (v.h->clock >= v.h->next_round) {
    n += swap_round(v, p.max_swaps, swaps + n, n_max - n);
    v.h->next_round = (v.h->clock / p.round_every_tokens + 1) * p.round_every_tokens;
  }
  return n;
}

int32_t moe_cache_rebalance(void* state, int32_t max_swaps, moe_cache_swap* swaps, int32_t n_max) {
  View v;
  if (!view_of(state, &v) || max_swaps < 0 || n_max < max_swaps || (n_max > 0 && !swaps)) return -1;
  return swap_round(v, max_swaps, swaps, n_max);
}

moe_status moe_cache_slot_map(const void* state, int32_t layer, int32_t* slot_map) {
  View v;
  if (!view_of(const_cast<void*>(state), &v) || !slot_map || layer < 0 || layer >= v.h->p.n_layers)
    return MOE_ERR_INVALID;
  std::memcpy(slot_map, v.map + (size_t)layer * v.h->p.n_experts, 4 * (size_t)v.h->p.n_experts);
  return MOE_OK;
}

moe_status moe_cache_heat(const void* state, int32_t layer, double* heat) {
  View v;
  if (!view_of(const_cast<void*>(state), &v) || !heat || layer < 0 || layer >= v.h->p.n_layers)
    return MOE_ERR_INVALID;
  std::memcpy(heat, v.heat + (size_t)layer * v.h->p.n_experts, 8 * (size_t)v.h->p.n_experts);
  return MOE_OK;
}

int64_t moe_cache_swapped_total(const void* state) {
  View v;
  if (!view_of(const_cast<void*>(state), &v)) return -1;
  return v.h->n_swapped;
}

// STRP, little-endian: "STRP", u32 version 1, u32 n_layers, u32 n_expert,
// u32 slots, u32 n_ranked, n_ranked x (u16 layer, u16 expert) hottest first,
// then n_layers x n_expert x i32 rank (-1 unranked). Ranked pairs: heat > 0,
// heat descending, then layer, then expert.
int64_t moe_cache_profile_write(const void* state, uint8_t* buf, int64_t n_max) {
  View v;
  if (!view_of(const_cast<void*>(state), &v) || n_max < 0) return -1;
  const int L = v.h->p.n_layers, E = v.h->p.n_experts;
  if (L > 65535 || E > 65535) return -1;  // u16 fields
  std::vector<Move> r;
  for (int l = 0; l < L; ++l)
    for (int e = 0; e < E; ++e) {
      const double hv = v.heat[(size_t)l * E + e];
      if (hv > 0.0) r.push_back({hv, l, e, -1, -1});
    }
  order_and_cap(r, (int)r.size());
  const int64_t size = 24 + 4 * (int64_t)r.size() + 4 * (int64_t)L * E;
  if (n_max == 0) return size;
  if (!buf || n_max < size) return -1;
  std::memcpy(buf, "STRP", 4);
  put_u32(buf + 4, 1);
  put_u32(buf + 8, (uint32_t)L);
  put_u32(buf + 12, (uint32_t)E);
  put_u32(buf + 16, (uint32_t)v.h->total_slots);
  put_u32(buf + 20, (uint32_t)r.size());
  uint8_t* q = buf + 24;
  std::vector<int32_t> rank((size_t)L * E, -1);
  for (size_t i = 0; i < r.size(); ++i, q += 4) {
    put_u16(q, (uint32_t)r[i].layer);
    put_u16(q + 2, (uint32_t)r[i].e_in);
    rank[(size_t)r[i].layer * E + r[i].e_in] = (int32_t)i;
  }
  for (size_t i = 0; i < rank.size(); ++i, q += 4) put_u32(q, (uint32_t)rank[i]);
  return size;
}

// Fill every layer's slots from a profile: the profile's pairs of that layer
// in order, as many as it has slots (a repeated pair is skipped). The header
// and every pair are validated first; the rank table is not read.
moe_status moe_cache_profile_load(void* state, const uint8_t* buf, int64_t n) {
  View v;
  if (!view_of(state, &v)) return MOE_ERR_INVALID;
  if (!buf || n < 24 || std::memcmp(buf, "STRP", 4) != 0 || get_u32(buf + 4) != 1) return MOE_ERR_INVALID;
  const uint32_t L = get_u32(buf + 8), E = get_u32(buf + 12), nr = get_u32(buf + 20);
  if (L != (uint32_t)v.h->p.n_layers || E != (uint32_t)v.h->p.n_experts) return MOE_ERR_INVALID;
  if ((uint64_t)nr > (uint64_t)L * E || n < 24 + 4 * (int64_t)nr) return MOE_ERR_INVALID;
  const uint8_t* q = buf + 24;
  for (uint32_t i = 0; i < nr; ++i)
    if (get_u16(q + 4 * i) >= L || get_u16(q + 4 * i + 2) >= E) return MOE_ERR_INVALID;
  std::vector<int> fill(L, 0);
  for (uint32_t l = 0; l < L; ++l) {
    for (int s = 0; s < v.slots[l]; ++s) v.owner[v.base[l] + s] = -1;
    for (uint32_t e = 0; e < E; ++e) v.map[(size_t)l * E + e] = -1;
  }
  for (uint32_t i = 0; i < nr; ++i) {
    const int l = (int)get_u16(q + 4 * i), e = (int)get_u16(q + 4 * i + 2);
    if (fill[l] >= v.slots[l] || v.map[(size_t)l * E + e] >= 0) continue;
    place(v, l, fill[l]++, e);
  }
  return MOE_OK;
}

}  // extern "C"
