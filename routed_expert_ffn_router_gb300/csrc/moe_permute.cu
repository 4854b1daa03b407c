// (token, expert) permutation: a deterministic counting sort of the P = T*k
// pairs by expert, stable in the pair index p = t*k + j (the expert-scoped
// layout of the SGLang port post, section 2), plus the slot-map lookup and the
// list of missing experts ("extended-strata-moe reference", "The mailbox"
// step 1; misses counted as distinct experts per layer, "C API").
//
// No order-dependent atomics decide a position: counts use integer atomics
// (order-free), positions come from prefix sums and an explicit rank of each
// pair among the earlier pairs of its expert.
#include "moe_internal.h"

namespace moe {

constexpr int kChunk = 1024;  // pairs per CTA in the chunked path

// Exclusive prefix sum over a 1024-thread block; *total receives the sum.
__device__ int block_excl_scan(int v, int* s_warp, int* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  __syncthreads();
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int wv = lane < nw ? s_warp[lane] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, wv, off);
      if (lane >= off) wv += y;
    }
    s_warp[lane] = wv;
    if (lane == 31) *s_total = wv;
  }
  __syncthreads();
  int base = warp > 0 ? s_warp[warp - 1] : 0;
  int res = base + x - v;
  __syncthreads();
  return res;
}

// Stable rank of this thread's pair among the earlier pairs of the 1024-thread
// block with the same expert e (valid: this thread holds a pair). Warp w
// counts its pairs per expert with a match (the lowest lane of each expert
// writes the count into cnt[e][w]); a pair's rank is the sum of its expert's
// counts in warps before w plus its position among the same-expert lanes of
// its own warp. cnt: [kMaxE][32] bytes.
__device__ int block_stable_rank(int e, bool valid, uint8_t (*cnt)[32]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < kMaxE * 8; i += blockDim.x) reinterpret_cast<uint32_t*>(cnt)[i] = 0;
  __syncthreads();
  const unsigned act = __ballot_sync(0xffffffffu, valid);
  const unsigned same = __match_any_sync(0xffffffffu, valid ? e : -1) & act;
  const unsigned lower = same & ((1u << lane) - 1u);
  if (valid && lower == 0) cnt[e][warp] = (uint8_t)__popc(same);
  __syncthreads();
  int r = __popc(lower);
  if (valid) {
    const uint4* row = reinterpret_cast<const uint4*>(cnt[e]);
    const uint4 a = row[0], b = row[1];
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int nb = min(max(warp - 4 * i, 0), 4);  // bytes of this word from warps before ours
      const uint32_t m = nb == 4 ? 0xffffffffu : ((1u << (8 * nb)) - 1u);
      r = (int)__dp4a(wd[i] & m, 0x01010101u, (unsigned)r);
    }
  }
  return r;
}

// Miss list, active-expert records and token-chunk work units, from the
// per-expert counts and offsets held in shared memory. Thread e handles
// expert e (blockDim >= E).
__device__ void build_lists(int E, int P, int T, int S, bool has_shared,
                            const int32_t* __restrict__ slot_map, const int* s_cnt,
                            const int* s_off, int* s_warp, int* s_total, const PermuteOut& o) {
  const int e = threadIdx.x;
  int c = e < E ? s_cnt[e] : 0;
  int slot = -1;
  if (c > 0) {
    slot = slot_map ? slot_map[e] : e;
    if (slot >= S) {
      atomicOr(o.status, DEV_BAD_SLOT);
      slot = -1;
    }
  }
  const int is_miss = (c > 0 && slot < 0) ? 1 : 0;
  const int is_act = (c > 0 && slot >= 0) ? 1 : 0;
  int mi = block_excl_scan(is_miss, s_warp, s_total);
  const int n_miss = *s_total;
  __syncthreads();
  int ai = block_excl_scan(is_act, s_warp, s_total);
  const int n_act = *s_total;
  __syncthreads();
  const int chunks = is_act ? (c + kTokTile - 1) / kTokTile : 0;
  int ci = block_excl_scan(chunks, s_warp, s_total);
  const int n_cu_routed = *s_total;
  __syncthreads();
  if (is_miss) o.miss_ids[mi] = e;
  if (is_act) {
    ActExpert r;
    r.e = e;
    r.slot = slot;
    r.off = s_off[e];
    r.cnt = c;
    o.act[ai] = r;
    for (int q = 0; q < chunks; ++q) o.cu[ci + q] = make_int2(ai, q);
  }
  const int sh_chunks = has_shared ? (T + kTokTile - 1) / kTokTile : 0;
  for (int q = threadIdx.x; q < sh_chunks; q += blockDim.x) o.cu[n_cu_routed + q] = make_int2(n_act, q);
  if (threadIdx.x == 0) {
    *o.n_miss = n_miss;
    if (has_shared) {
      ActExpert r;
      r.e = -1;
      r.slot = -1;
      r.off = P;
      r.cnt = T;
      o.act[n_act] = r;
    }
    o.counters[0] = n_act + (has_shared ? 1 : 0);
    o.counters[1] = n_cu_routed + sh_chunks;
  }
}

__device__ __forceinline__ int load_id(const int32_t* ids, int p, int E, int32_t* status) {
  int e = ids[p];
  if (e < 0 || e >= E) {
    atomicOr(status, DEV_BAD_SLOT);
    e = e < 0 ? 0 : E - 1;
  }
  return e;
}

// P <= 1024: everything in one CTA.
__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* __restrict__ ids, int T,
                                                             int E, int k,
                                                             const int32_t* __restrict__ slot_map,
                                                             int S, int has_shared, PermuteOut o) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ __align__(16) uint8_t s_rc[kMaxE][32];
  const int tid = threadIdx.x;
  const int P = T * k;
  int e = 0;
  if (tid < P) e = load_id(ids, tid, E, o.status);
  const int rank = block_stable_rank(e, tid < P, s_rc);
  if (tid < E) s_cnt[tid] = 0;
  __syncthreads();
  if (tid < P) atomicAdd(&s_cnt[e], 1);
  __syncthreads();
  int off = block_excl_scan(tid < E ? s_cnt[tid] : 0, s_warp, &s_total);
  if (tid < E) s_off[tid] = off;
  if (tid == 0) s_off[E] = P;
  __syncthreads();
  if (tid < P) {
    int pos = s_off[e] + rank;
    o.sorted_pair[pos] = tid;
    o.pair_pos[tid] = pos;
  }
  if (tid < E) o.offsets[tid] = s_off[tid];
  if (tid == 0) o.offsets[E] = P;
  build_lists(E, P, T, S, has_shared != 0, slot_map, s_cnt, s_off, s_warp, &s_total, o);
}

// Chunked path, step 1: per-chunk histograms hist[c][e].
__global__ void __launch_bounds__(1024) permute_hist_kernel(const int32_t* __restrict__ ids, int P,
                                                            int E, PermuteOut o) {
  __shared__ int s_cnt[kMaxE];
  const int tid = threadIdx.x;
  if (tid < E) s_cnt[tid] = 0;
  __syncthreads();
  int p = blockIdx.x * kChunk + tid;
  if (p < P) atomicAdd(&s_cnt[load_id(ids, p, E, o.status)], 1);
  __syncthreads();
  if (tid < E) o.hist[(size_t)blockIdx.x * E + tid] = s_cnt[tid];
}

// Step 2 (one CTA): per expert, chunk bases in chunk order (hist becomes the
// exclusive base), totals, offsets, then the lists.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int T, int E, int k, int n_chunks,
                                                            const int32_t* __restrict__ slot_map,
                                                            int S, int has_shared, PermuteOut o) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  const int tid = threadIdx.x;
  const int P = T * k;
  int run = 0;
  if (tid < E) {
    // 8 chunks' counts in flight at a time (the loads do not wait for the stores)
    for (int c0 = 0; c0 < n_chunks; c0 += 8) {
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = c0 + u < n_chunks ? __ldcg(o.hist + (size_t)(c0 + u) * E + tid) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < n_chunks) o.hist[(size_t)(c0 + u) * E + tid] = run;
        run += h[u];
      }
    }
    s_cnt[tid] = run;
  }
  __syncthreads();
  int off = block_excl_scan(tid < E ? run : 0, s_warp, &s_total);
  if (tid < E) s_off[tid] = off;
  if (tid == 0) s_off[E] = P;
  __syncthreads();
  if (tid < E) o.offsets[tid] = s_off[tid];
  if (tid == 0) o.offsets[E] = P;
  build_lists(E, P, T, S, has_shared != 0, slot_map, s_cnt, s_off, s_warp, &s_total, o);
}

// Step 3: position = offsets[e] + base of this chunk for e + rank inside the chunk.
__global__ void __launch_bounds__(1024) permute_scatter_kernel(const int32_t* __restrict__ ids,
                                                               int P, int E, PermuteOut o) {
  __shared__ __align__(16) uint8_t s_rc[kMaxE][32];
  const int tid = threadIdx.x;
  const int p0 = blockIdx.x * kChunk;
  const int n = min(kChunk, P - p0);
  int e = 0;
  if (tid < n) e = load_id(ids, p0 + tid, E, o.status);
  const int rank = block_stable_rank(e, tid < n, s_rc);
  if (tid < n) {
    int pos = o.offsets[e] + o.hist[(size_t)blockIdx.x * E + e] + rank;
    o.sorted_pair[pos] = p0 + tid;
    o.pair_pos[p0 + tid] = pos;
  }
}

// Steps 2 and 3 in one launch for up to kScanChunks chunks: every CTA derives
// its chunk's bases (the counts of the chunks before it) and the expert
// offsets from the histograms itself, then places its pairs; CTA 0 also
// writes the offsets and the lists.
constexpr int kScanChunks = 64;
__global__ void __launch_bounds__(1024) permute_place_kernel(const int32_t* __restrict__ ids, int T, int E,
                                                             int k, int n_chunks,
                                                             const int32_t* __restrict__ slot_map, int S,
                                                             int has_shared, PermuteOut o) {
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_off[kMaxE + 1];
  __shared__ int s_base[kMaxE];
  __shared__ int s_warp[32];
  __shared__ int s_total;
  __shared__ __align__(16) uint8_t s_rc[kMaxE][32];
  const int tid = threadIdx.x, c = blockIdx.x;
  const int P = T * k;
  const int p0 = c * kChunk;
  const int n = min(kChunk, P - p0);
  int e = 0;
  if (tid < n) e = load_id(ids, p0 + tid, E, o.status);
  int base = 0, tot = 0;
  if (tid < E) {
    for (int c0 = 0; c0 < n_chunks; c0 += 8) {  // 8 chunks' counts in flight at a time
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = c0 + u < n_chunks ? __ldcg(o.hist + (size_t)(c0 + u) * E + tid) : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        base += c0 + u < c ? h[u] : 0;
        tot += h[u];
      }
    }
    s_base[tid] = base;
    s_cnt[tid] = tot;
  }
  const int rank = block_stable_rank(e, tid < n, s_rc);  // syncs the block
  const int off = block_excl_scan(tid < E ? tot : 0, s_warp, &s_total);
  if (tid < E) s_off[tid] = off;
  if (tid == 0) s_off[E] = P;
  __syncthreads();
  if (tid < n) {
    const int pos = s_off[e] + s_base[e] + rank;
    o.sorted_pair[pos] = p0 + tid;
    o.pair_pos[p0 + tid] = pos;
  }
  if (c != 0) return;
  if (tid < E) o.offsets[tid] = s_off[tid];
  if (tid == 0) o.offsets[E] = P;
  build_lists(E, P, T, S, has_shared != 0, slot_map, s_cnt, s_off, s_warp, &s_total, o);
}

int cu_bound(int T, int E, int k, bool has_shared) {
  const int P = T * k;
  const int sh = has_shared ? (T + kTokTile - 1) / kTokTile : 0;
  if (T <= kTokTile) return (P < E ? P : E) + sh;
  // sum_e ceil(c_e/16) <= P/16 + (number of experts touched)
  return P / kTokTile + (P < E ? P : E) + sh;
}

cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, const int32_t* slot_map, int S,
                           bool has_shared, const PermuteOut& o, cudaStream_t st) {
  const int P = T * k;
  if (P <= kChunk) {
    launch_begin(K_PERMUTE, st);
    permute_small_kernel<<<1, 1024, 0, st>>>(ids, T, E, k, slot_map, S, has_shared ? 1 : 0, o);
    launch_end(st);
    return cudaGetLastError();
  }
  const int nc = (P + kChunk - 1) / kChunk;
  launch_begin(K_PERMUTE, st);
  permute_hist_kernel<<<nc, 1024, 0, st>>>(ids, P, E, o);
  launch_end(st);
  if (nc <= kScanChunks) {
    launch_begin(K_PERMUTE, st);
    permute_place_kernel<<<nc, 1024, 0, st>>>(ids, T, E, k, nc, slot_map, S, has_shared ? 1 : 0, o);
    launch_end(st);
    return cudaGetLastError();
  }
  launch_begin(K_PERMUTE, st);
  permute_scan_kernel<<<1, 1024, 0, st>>>(T, E, k, nc, slot_map, S, has_shared ? 1 : 0, o);
  launch_end(st);
  launch_begin(K_PERMUTE, st);
  permute_scatter_kernel<<<nc, 1024, 0, st>>>(ids, P, E, o);
  launch_end(st);
  return cudaGetLastError();
}

// Adaptive-cache routing counters ("extended-strata-moe reference", "The
// adaptive cache": picks per (layer, expert), one per expert and window): an
// expert with rows in the window's permutation gets one pick.
__global__ void count_picks_kernel(const int32_t* offsets, int E, int32_t* counts) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < E && offsets[e + 1] > offsets[e]) atomicAdd(counts + e, 1);
}

cudaError_t launch_count_picks(const int32_t* offsets, int E, int32_t* counts, cudaStream_t st) {
  launch_begin(K_PERMUTE, st);
  count_picks_kernel<<<(E + 255) / 256, 256, 0, st>>>(offsets, E, counts);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace moe
