// One persistent kernel per decode window (T <= 16 rows): routing, the
// (token, expert) permutation, gate/up + SwiGLU, down and the ordered combine.
//
// This is the grouped expert call of the SGLang port post (TL;DR and section
// 3: gather -> dequant -> gate/up -> SwiGLU -> down -> scatter in one call per
// layer) laid out for GB300:
//  * one CTA per SM; warp 0 streams jobs into a ring of shared-memory stages
//    with TMA tensor copies (full/empty mbarriers). A job is a tile of packed
//    weight rows (int4 codes in 128-byte-swizzled tiles, fp16 scales) together
//    with the activation rows it multiplies (a chunk of x, or the expert's
//    chunk of h): a handful of copies per job, and the 8 consumer warps never
//    wait on global memory. They split the job's columns and run the
//    exact-integer warp-MMA core (moe_decode.cu explains the 136 + q and
//    1032 + q code fragments);
//  * the per-block correction -magic * sum(B) comes from one more MMA whose A
//    operand is the constant -magic;
//  * every CTA computes the top-k ids and the permutation of the whole window
//    in shared memory, so no launch precedes the weight stream; CTA t computes
//    row t's float64 softmax weights;
//  * phase 1: gate/up units (32 rows of gate and of up, K in chunks), handed
//    out round-robin, write h = silu(g)*u as fp16 in fragment order; phase 2:
//    down units (R output rows, contiguous per CTA). The producer issues a
//    down job's weight copies at once and its h copy after the expert's
//    gate/up units are all done (a per-expert counter);
//  * the last CTA to finish a group of R output rows sums the routed partials
//    in j order, weighted, then adds the shared expert: y is deterministic;
//  * the last CTA to exit resets the cross-CTA counters for the next call.
// Every expert a window touches (and the shared expert, Strata BATCHING,
// "Several requests at once") is read from HBM exactly once.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "moe_internal.h"

namespace moe {
namespace fused {

constexpr int kCW = 8;                  // consumer warps
constexpr int kThreads = 32 * (kCW + 1);
constexpr int kNst = 4;                 // pipeline stages
constexpr int kGuRows = 32;             // rows of gate and of up per unit (one block of I)
constexpr int kMaxT = 16;               // largest window; x / h boxes hold TB = 8 or 16 rows
constexpr int kMaxMT = 4;               // m16 tiles per job
constexpr int kRed = 8 * 17;            // one (m-tile, n-tile) slab: 8 tokens x (16 rows + pad)
constexpr int kRedBytes = kCW * kMaxMT * 2 * kRed * 4;
constexpr int kChunkE = 4;              // experts per thread in the permutation scan
constexpr uint32_t kBf16NegMagic = 0xC308C308u;  // bf16 -136
constexpr uint32_t kF16NegMagic = 0xE408E408u;   // f16 -1032

// cross-CTA counters (int32 offsets in the workspace sync region)
constexpr int kSyncDone = 0, kSyncWReady = 1, kSyncReady = 16, kSyncRg = 16 + 1040;

struct Args {
  // TMA tensor maps (kernel parameters, read through their parameter address)
  CUtensorMap tm_gc, tm_uc, tm_dc;     // routed codes: gate, up [S*I][H/2]; down [S*H][I/2]
  CUtensorMap tm_gs, tm_us, tm_ds;     // routed scales
  CUtensorMap tm_sgc, tm_suc, tm_sdc;  // shared expert codes
  CUtensorMap tm_sgs, tm_sus, tm_sds;  // shared expert scales
  CUtensorMap tm_x;                    // x [T][H] bf16, 3D box (64, KC/64, 16)
  CUtensorMap tm_h, tm_hs;             // h [rows_cap][Imax] f16: routed / shared chunk boxes
  int H, I, shI, E, k, S, T, Imax;
  int KC;          // gate/up K chunk (columns per job)
  int KCd, KCds;   // down K chunk of the routed / shared experts
  int R;           // output rows per down unit
  int stage_bytes; // multiple of 1024
  int TB;          // rows of the x / h boxes (8 or 16, >= T)
  int rows_cap;    // rows of the h / partial buffers (P + T)
  const float* logits;     // non-null: route here (layer mode)
  const int32_t* ids_in;   // routing given (ffn mode)
  const float* w_in;
  const int32_t* slot_map;
  int32_t* ids_out;
  float* w_out;
  float* y;
  int32_t* miss_ids;
  int32_t* n_miss;
  uint16_t* h;             // f16 bits [rows_cap][Imax], fragment order
  float* partial;          // [rows_cap][H]
  int32_t* status;
  int32_t* sync;
};

// Dynamic shared memory: 1 KB of alignment slack, kNst stages, the cross-warp
// reduction buffer, barriers.
__host__ __device__ inline size_t smem_bytes(int stage_bytes) {
  return 1024 + (size_t)kNst * stage_bytes + kRedBytes + 2 * kNst * 8;
}

// Job stage layouts (byte offsets from the 1024-aligned stage base).
// gate/up: gate code tiles [KC/256][32 rows][128 B] (swizzled), up code tiles,
//          x box [TB rows][KC/64][128 B] (swizzled), gate scales [32][KC/32],
//          up scales [32][KC/32].
// down:    code tiles [KCd/256][R][128 B] (swizzled), h box [TB][KCd/64][128 B]
//          (swizzled), scales [R][KCd/32].
__host__ __device__ inline int gu_codes_bytes(int KC) { return (KC / 256) * kGuRows * 128; }
__host__ __device__ inline int gu_x(int KC) { return 2 * gu_codes_bytes(KC); }
__host__ __device__ inline int gu_scales(int KC, int TB) { return gu_x(KC) + TB * KC * 2; }
__host__ __device__ inline int gu_bytes(int KC, int TB) { return gu_scales(KC, TB) + 2 * kGuRows * (KC / 16); }
__host__ __device__ inline int dn_h(int R, int KCd) { return (KCd / 256) * R * 128; }
__host__ __device__ inline int dn_scales(int R, int KCd, int TB) { return dn_h(R, KCd) + TB * KCd * 2; }
__host__ __device__ inline int dn_bytes(int R, int KCd, int TB) { return dn_scales(R, KCd, TB) + R * (KCd / 16); }

__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0) u = 0;  // -0 and +0 are equal logits: same key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// n-th (0-based) set bit of a mask (mask has more than n bits set).
__device__ __forceinline__ int nth_bit(uint32_t m, int n) {
  for (int i = 0; i < n; ++i) m &= m - 1;
  return __ffs(m) - 1;
}

// Exclusive scan over all kThreads threads (unsigned: packed fields may use bit 31).
__device__ __forceinline__ uint32_t cta_excl_scan(uint32_t v, uint32_t* s_warp, uint32_t* s_total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t wv = lane < kCW + 1 ? s_warp[lane] : 0u;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      uint32_t y = __shfl_up_sync(0xffffffffu, wv, off);
      if (lane >= off) wv += y;
    }
    if (lane < kCW + 1) s_warp[lane] = wv;
    if (lane == kCW) *s_total = wv;
  }
  __syncthreads();
  const uint32_t base = warp > 0 ? s_warp[warp - 1] : 0u;
  const uint32_t r = base + x - v;
  __syncthreads();
  return r;
}


// Top-k of one row by one warp. Keys are 64-bit (order_key(logit) << 32 | ~id):
// unique, and larger means "earlier" (logit descending, ties to the lower id).
// The k-th largest of the 32 lane maxima bounds the k-th largest key from below
// (those k maxima are k distinct keys), so only keys at or above it can be
// selected; they are compacted and ranked by counting. If there are more than
// kTopkCand candidates (many top keys in few lanes) the warp falls back to k
// rounds of arg-max. Writes ids[0..k) in order and leaves the ranked keys in
// scr[kTopkRanked + r]. Returns true if a logit was not finite.
constexpr int kTopkCand = 256;
constexpr int kTopkRanked = 32 + kTopkCand;
constexpr int kTopkScratch = kTopkRanked + 32;  // 64-bit words per warp

template <int NPER>
__device__ bool topk_row(const float* l, int E, int k, unsigned long long* scr, int* ids) {
  const int lane = threadIdx.x & 31;
  unsigned long long key[NPER];
  unsigned long long mx = 0;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    const float v = e < E ? l[e] : 0.f;
    if (e < E && !isfinite(v)) bad = true;
    key[i] = e < E ? (((unsigned long long)order_key(v) << 32) | (uint32_t)(~e)) : 0ull;
    mx = key[i] > mx ? key[i] : mx;
  }
  bad = __any_sync(0xffffffffu, bad);
  scr[lane] = mx;
  __syncwarp();
  int rk = 0;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) rk += scr[i] > mx ? 1 : 0;
  const int kk = k < 32 ? k : 32;
  const unsigned sel = __ballot_sync(0xffffffffu, rk == kk - 1);
  const unsigned long long theta = __shfl_sync(0xffffffffu, mx, __ffs(sel) - 1);
  int c = 0;
#pragma unroll
  for (int i = 0; i < NPER; ++i) c += key[i] >= theta ? 1 : 0;
  int x = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  const int C = __shfl_sync(0xffffffffu, x, 31);
  unsigned long long* cand = scr + 32;
  unsigned long long* ranked = scr + kTopkRanked;
  if (C <= kTopkCand) {
    int pos = x - c;
#pragma unroll
    for (int i = 0; i < NPER; ++i)
      if (key[i] >= theta) cand[pos++] = key[i];
    __syncwarp();
    for (int q = lane; q < C; q += 32) {
      const unsigned long long me = cand[q];
      int r = 0;
      for (int i = 0; i < C; ++i) r += cand[i] > me ? 1 : 0;
      if (r < k) {
        ranked[r] = me;
        ids[r] = (int)(~(uint32_t)me);
      }
    }
  } else {
    unsigned long long best = 0;
#pragma unroll
    for (int i = 0; i < NPER; ++i) best = key[i] > best ? key[i] : best;
    for (int j = 0; j < k; ++j) {
      unsigned long long m = best;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
        m = o > m ? o : m;
      }
      if (m == best) {
        best = 0;
#pragma unroll
        for (int i = 0; i < NPER; ++i) {
          if (key[i] == m) key[i] = 0;
          best = key[i] > best ? key[i] : best;
        }
      }
      if (lane == j) {
        ranked[j] = m;
        ids[j] = (int)(~(uint32_t)m);
      }
    }
  }
  __syncwarp();
  return bad;
}


// One job's columns [b0, b1) (blocks of 32) for one consumer warp:
//   acc[m][nt] += sum_b scale(row, b) * (codes(row, b) . B(b, token slot))
// GU: gate/up job (bf16 x, 136 + q codes, m-tiles 0,1 gate / 2,3 up);
// otherwise a down job (f16 h, 1032 + q codes). All shared-memory loads of a
// block are issued before its arithmetic, so the MT x NT MMA chains overlap.
// Blocks b = cw, cw + 8, ... of the job: the blocks a warp sums, and their
// order, do not depend on how K is cut into chunks.
template <bool GU, int MT, int NT>
__device__ __forceinline__ void job_compute(const uint8_t* st, int kcols, int R, int TB, int cw,
                                            const int (&brow)[2], float (&acc)[kMaxMT][2][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  const int brow_bytes = kcols * 2;
  const uint8_t* bbox = st + (GU ? gu_x(kcols) : dn_h(R, kcols));
  const __half* scl =
      reinterpret_cast<const __half*>(st + (GU ? gu_scales(kcols, TB) : dn_scales(R, kcols, TB)));
  const int NB = kcols / 32;
  const int code_tile = (GU ? kGuRows : R) * 128;
  const int lines = kcols / 256;
  // every row this lane reads is g (mod 8): one swizzle for all of them
  const uint8_t* rowp[MT];
  const __half* sclp[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    const int mat = GU ? (m >> 1) : 0;
    const int r0 = GU ? (m & 1) * 16 + g : m * 16 + g;
    rowp[m] = st + (size_t)mat * lines * code_tile + r0 * 128 + c * 4;
    sclp[m] = scl + ((GU ? mat * kGuRows : 0) + r0) * NB;
  }
#pragma unroll 1
  for (int b = cw; b < NB; b += kCW) {
    const int line = b >> 3, chunk = b & 7;
    uint4 braw[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      braw[nt] = lds_v4(bbox + swz128((uint32_t)(brow[nt] * brow_bytes + b * 64 + c * 16)));
    const int coff = line * code_tile + ((chunk ^ g) << 4);
    uint32_t w[MT][2];
    float sc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      w[m][0] = *reinterpret_cast<const uint32_t*>(rowp[m] + coff);
      w[m][1] = *reinterpret_cast<const uint32_t*>(rowp[m] + coff + 8 * 128);
      sc[m][0] = __half2float(sclp[m][b]);
      sc[m][1] = __half2float(sclp[m][8 * NB + b]);
    }
    uint32_t bf[NT][4];
    float corr[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if (GU) {  // raw bf16 x: reorder to the fragment order
        bf[nt][0] = prmt(braw[nt].x, braw[nt].z, 0x5410);
        bf[nt][1] = prmt(braw[nt].x, braw[nt].z, 0x7632);
        bf[nt][2] = prmt(braw[nt].y, braw[nt].w, 0x5410);
        bf[nt][3] = prmt(braw[nt].y, braw[nt].w, 0x7632);
      } else {   // h is stored in fragment order
        bf[nt][0] = braw[nt].x; bf[nt][1] = braw[nt].y; bf[nt][2] = braw[nt].z; bf[nt][3] = braw[nt].w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) corr[nt][i] = 0.f;
      if (GU) {
        mma_bf16_16816(corr[nt], kBf16NegMagic, kBf16NegMagic, kBf16NegMagic, kBf16NegMagic, bf[nt][0], bf[nt][1]);
        mma_bf16_16816(corr[nt], kBf16NegMagic, kBf16NegMagic, kBf16NegMagic, kBf16NegMagic, bf[nt][2], bf[nt][3]);
      } else {
        mma_f16_16816(corr[nt], kF16NegMagic, kF16NegMagic, kF16NegMagic, kF16NegMagic, bf[nt][0], bf[nt][1]);
        mma_f16_16816(corr[nt], kF16NegMagic, kF16NegMagic, kF16NegMagic, kF16NegMagic, bf[nt][2], bf[nt][3]);
      }
    }
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      uint32_t d[4], e[4];
      if (GU) {
        dequant_word(w[m][0], d);
        dequant_word(w[m][1], e);
      } else {
        dequant_word_f16(w[m][0], d);
        dequant_word_f16(w[m][1], e);
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float t4[4] = {corr[nt][0], corr[nt][1], corr[nt][2], corr[nt][3]};
        if (GU) {
          mma_bf16_16816(t4, d[0], e[0], d[1], e[1], bf[nt][0], bf[nt][1]);
          mma_bf16_16816(t4, d[2], e[2], d[3], e[3], bf[nt][2], bf[nt][3]);
        } else {
          mma_f16_16816(t4, d[0], e[0], d[1], e[1], bf[nt][0], bf[nt][1]);
          mma_f16_16816(t4, d[2], e[2], d[3], e[3], bf[nt][2], bf[nt][3]);
        }
        acc[m][nt][0] = fmaf(sc[m][0], t4[0], acc[m][nt][0]);
        acc[m][nt][1] = fmaf(sc[m][0], t4[1], acc[m][nt][1]);
        acc[m][nt][2] = fmaf(sc[m][1], t4[2], acc[m][nt][2]);
        acc[m][nt][3] = fmaf(sc[m][1], t4[3], acc[m][nt][3]);
      }
    }
  }
}

struct Job {
  bool gu;        // gate/up (true) or down
  int d;          // active-expert index (D = the shared expert)
  int tile;       // gate/up: 32-row tile of I; down: R-row group of H
  int kc;         // K chunk
  bool first, last;
};

struct Plan {
  int nGu;        // gate/up units of this CTA (u = bid + i*G)
  int nKc, nKd;   // chunks per gate/up / down unit
  int v0, v1;     // down units of this CTA
  int nIu, D, nRg;
  __device__ int njobs() const { return nGu * nKc + (v1 - v0) * nKd; }
};

__device__ __forceinline__ Job decode_job(int j, const Plan& p, int bid, int G) {
  Job jb;
  if (j < p.nGu * p.nKc) {
    const int u = bid + (j / p.nKc) * G;
    jb.gu = true;
    jb.kc = j % p.nKc;
    if (u < p.D * p.nIu) {
      jb.d = u / p.nIu;
      jb.tile = u - jb.d * p.nIu;
    } else {
      jb.d = p.D;
      jb.tile = u - p.D * p.nIu;
    }
    jb.first = jb.kc == 0;
    jb.last = jb.kc == p.nKc - 1;
  } else {
    const int jj = j - p.nGu * p.nKc;
    const int v = p.v0 + jj / p.nKd;
    jb.gu = false;
    jb.kc = jj % p.nKd;
    jb.d = v / p.nRg;
    jb.tile = v - jb.d * p.nRg;
    jb.first = jb.kc == 0;
    jb.last = jb.kc == p.nKd - 1;
  }
  return jb;
}

__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(const __grid_constant__ Args a) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int s_ids[kMaxT][kMaxK];
  __shared__ uint32_t s_tokmask[kMaxE];
  __shared__ int16_t s_d_of_e[kMaxE];
  __shared__ int16_t s_act_e[kMaxE + 1];
  __shared__ int32_t s_act_slot[kMaxE + 1];
  __shared__ int16_t s_act_off[kMaxE + 1];
  __shared__ uint8_t s_act_cnt[kMaxE + 1];
  __shared__ uint32_t s_warp[32];
  __shared__ uint32_t s_total;
  __shared__ int s_abort;
  __shared__ int s_flag;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, bid = blockIdx.x;
  const int T = a.T, k = a.k, E = a.E, H = a.H;
  const bool layer_mode = a.logits != nullptr;
  const bool has_shared = a.shI > 0;
  // stages start at a 1024-byte boundary (the unit of the 128-byte swizzle)
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  float* const red = reinterpret_cast<float*>(smem + (size_t)kNst * a.stage_bytes);
  const uint32_t full0 = sbase + kNst * a.stage_bytes + kRedBytes, empty0 = full0 + kNst * 8;
  volatile int* abort_flag = &s_abort;  // read in loops without barriers

  for (int e = tid; e < E; e += kThreads) s_tokmask[e] = 0;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kNst; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kCW);
    }
    fence_barrier_init();
  }

  // ---- routing: ids of every row (all CTAs); weights of row bid (CTA bid < T).
  // The stage buffers are still idle: they hold the top-k scratch.
  if (layer_mode) {
    unsigned long long* scr = reinterpret_cast<unsigned long long*>(smem) + warp * kTopkScratch;
    for (int t = warp; t < T; t += kCW + 1) {
      const float* l = a.logits + (size_t)t * E;
      bool bad;
      if (E <= 128) bad = topk_row<4>(l, E, k, scr, &s_ids[t][0]);
      else if (E <= 256) bad = topk_row<8>(l, E, k, scr, &s_ids[t][0]);
      else if (E <= 512) bad = topk_row<16>(l, E, k, scr, &s_ids[t][0]);
      else bad = topk_row<32>(l, E, k, scr, &s_ids[t][0]);
      if (bad && lane == 0 && bid == 0) atomicOr(a.status, DEV_NONFINITE_LOGIT);
      if (bid == t) {
        // float64 softmax over the k selected, in rank order (the ranked keys are in scr)
        const float v = lane < k ? key_value((uint32_t)(scr[kTopkRanked + lane] >> 32)) : 0.f;
        const double m0 = (double)__shfl_sync(0xffffffffu, v, 0);
        const double ej = lane < k ? exp((double)v - m0) : 0.0;
        double sum = 0.0;
        for (int j = 0; j < k; ++j) sum += __shfl_sync(0xffffffffu, ej, j);
        if (lane < k) {
          a.ids_out[(size_t)t * k + lane] = s_ids[t][lane];
          a.w_out[(size_t)t * k + lane] = (float)(ej / sum);
        }
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(a.sync + kSyncWReady, 1);
      }
      __syncwarp();
    }
  } else {
    for (int i = tid; i < T * k; i += kThreads) {
      int e = a.ids_in[i];
      if (e < 0 || e >= E) {
        if (bid == 0) atomicOr(a.status, DEV_BAD_SLOT);
        e = e < 0 ? 0 : E - 1;
      }
      s_ids[i / k][i % k] = e;
    }
  }
  __syncthreads();  // the top-k scratch (stage memory) is released
  // ---- permutation: token masks (shared atomics), then one warp builds the
  // active-expert list (ascending id), the offsets and the miss list
  for (int p = tid; p < T * k; p += kThreads) atomicOr(&s_tokmask[s_ids[p / k][p % k]], 1u << (p / k));
  __syncthreads();
  if (warp == 1) {
    const int per = (E + 31) >> 5;
    const int e0 = lane * per, e1 = min(E, e0 + per);
    uint32_t pack = 0;  // active count | misses << 11 | routed rows << 22
    for (int e = e0; e < e1; ++e) {
      const uint32_t m = s_tokmask[e];
      if (!m) continue;
      int slot = a.slot_map ? a.slot_map[e] : e;
      if (slot >= a.S) slot = -1;
      pack += slot >= 0 ? 1u + ((uint32_t)__popc(m) << 22) : (1u << 11);
    }
    uint32_t x = pack;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    const uint32_t tot = __shfl_sync(0xffffffffu, x, 31);
    const uint32_t ex = x - pack;
    int ai = ex & 0x7ff, mi = (ex >> 11) & 0x7ff, off = (ex >> 22) & 0x3ff;
    for (int e = e0; e < e1; ++e) {
      int16_t dd = -1;
      const uint32_t m = s_tokmask[e];
      if (m) {
        int slot = a.slot_map ? a.slot_map[e] : e;
        if (slot >= a.S) {
          if (bid == 0) atomicOr(a.status, DEV_BAD_SLOT);
          slot = -1;
        }
        if (slot >= 0) {
          dd = (int16_t)ai;
          s_act_e[ai] = (int16_t)e;
          s_act_slot[ai] = slot;
          s_act_off[ai] = (int16_t)off;
          s_act_cnt[ai] = (uint8_t)__popc(m);
          off += __popc(m);
          ++ai;
        } else {
          if (bid == 0) a.miss_ids[mi] = e;
          ++mi;
        }
      }
      s_d_of_e[e] = dd;
    }
    if (lane == 0) {
      s_total = tot;
      const int Dw = tot & 0x7ff, Pw = (tot >> 22) & 0x3ff;
      if (bid == 0) *a.n_miss = (tot >> 11) & 0x7ff;
      if (has_shared) {
        s_act_e[Dw] = -1;
        s_act_slot[Dw] = -1;
        s_act_off[Dw] = (int16_t)Pw;
        s_act_cnt[Dw] = (uint8_t)T;
      }
    }
  }
  __syncthreads();
  const uint32_t tot = s_total;
  const int D = tot & 0x7ff, Pres = (tot >> 22) & 0x3ff;
  const int nDx = D + (has_shared ? 1 : 0);
  if (nDx == 0) {  // nothing resident and no shared expert: y = 0
    const int n = T * H;
    for (int i = bid * kThreads + tid; i < n; i += G * kThreads) a.y[i] = 0.f;
  }
  __syncthreads();

  // ---- work: gate/up units round-robin, then down units contiguous per CTA
  Plan pl;
  pl.nIu = a.I / kGuRows;
  pl.D = D;
  pl.nRg = H / a.R;
  pl.nKc = H / a.KC;
  pl.nKd = a.I / a.KCd;  // the shared expert's down has the same number of chunks
  const int nIs = a.shI / kGuRows;
  const int U1 = D * pl.nIu + (has_shared ? nIs : 0);
  pl.nGu = bid < U1 ? (U1 - bid + G - 1) / G : 0;
  const int U2 = nDx * pl.nRg;
  pl.v0 = (int)((long long)bid * U2 / G);
  pl.v1 = (int)((long long)(bid + 1) * U2 / G);
  const int njobs = pl.njobs();

  if (warp == 0) {
    // ================= producer (lane 0 issues; the warp stays converged) =================
    fence_proxy_async_shared();  // the top-k scratch in stage memory precedes the TMA writes
    int issued = 0;
    for (int j = 0; j < njobs; ++j) {
      if (*abort_flag) break;
      const Job jb = decode_job(j, pl, bid, G);
      const int slot = j % kNst;
      if (!mbar_wait_bounded(empty0 + 8 * slot, ((j / kNst) & 1) ^ 1, a.status)) {
        *abort_flag = 1;
        break;
      }
      const bool sh = jb.d == D;
      const int slotp = sh ? 0 : s_act_slot[jb.d];
      const uint32_t st = sbase + slot * a.stage_bytes;
      const uint32_t fb = full0 + 8 * slot;
      bool okh = true;
      if (lane == 0) {
        if (jb.gu) {
          const int KC = a.KC, nl = KC / 256;
          mbar_expect_tx(fb, (uint32_t)gu_bytes(KC, a.TB));
          const int row = (sh ? 0 : slotp * a.I) + jb.tile * kGuRows;
          const CUtensorMap* tq[2] = {sh ? &a.tm_sgc : &a.tm_gc, sh ? &a.tm_suc : &a.tm_uc};
          const CUtensorMap* ts[2] = {sh ? &a.tm_sgs : &a.tm_gs, sh ? &a.tm_sus : &a.tm_us};
          for (int mat = 0; mat < 2; ++mat) {
            for (int L = 0; L < nl; ++L)
              tma_load_2d(st + (mat * nl + L) * (kGuRows * 128), tq[mat],
                          jb.kc * (KC / 2) + L * 128, row, fb);
            tma_load_2d(st + gu_scales(KC, a.TB) + mat * kGuRows * (KC / 16), ts[mat], jb.kc * (KC / 32),
                        row, fb);
          }
          tma_load_3d(st + gu_x(KC), &a.tm_x, 0, jb.kc * (KC / 64), 0, fb);
        } else {
          const int KCd = sh ? a.KCds : a.KCd, nl = KCd / 256;
          mbar_expect_tx(fb, (uint32_t)dn_bytes(a.R, KCd, a.TB));
          const int row = (sh ? 0 : slotp * H) + jb.tile * a.R;
          const CUtensorMap* tq = sh ? &a.tm_sdc : &a.tm_dc;
          for (int L = 0; L < nl; ++L)
            tma_load_2d(st + L * (a.R * 128), tq, jb.kc * (KCd / 2) + L * 128, row, fb);
          tma_load_2d(st + dn_scales(a.R, KCd, a.TB), sh ? &a.tm_sds : &a.tm_ds, jb.kc * (KCd / 32), row,
                      fb);
          // the expert's h rows: only once all its gate/up units are done
          okh = wait_counter_bounded(a.sync + kSyncReady + jb.d, sh ? nIs : pl.nIu, a.status);
          if (okh) {
            fence_proxy_async_global();
            tma_load_3d(st + dn_h(a.R, KCd), sh ? &a.tm_hs : &a.tm_h, 0, jb.kc * (KCd / 64),
                        s_act_off[jb.d], fb);
          }
        }
      }
      issued = j + 1;
      if (!__shfl_sync(0xffffffffu, okh ? 1 : 0, 0)) {
        *abort_flag = 1;
        break;
      }
    }
    // no copy may still be in flight when the CTA exits (bounded)
    if (lane == 0)
      for (int j = issued - 1; j >= 0 && j >= issued - kNst; --j)
        mbar_wait_bounded(full0 + 8 * (j % kNst), (j / kNst) & 1, a.status);
  } else {
    // ================= consumers =================
    const int cw = warp - 1, ct = tid - 32;
    const int g = lane >> 2, c = lane & 3;
    float acc[kMaxMT][2][4];
    int brow[2] = {0, 0};  // row of token slot nt*8 + g in the x box (token) / h box (slot)
    int cnt = 0, ntiles = 1;
    for (int j = 0; j < njobs; ++j) {
      const Job jb = decode_job(j, pl, bid, G);
      const int slot = j % kNst;
      const bool sh = jb.d == D;
      if (jb.first) {
#pragma unroll
        for (int m = 0; m < kMaxMT; ++m)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[m][nt][i] = 0.f;
        cnt = s_act_cnt[jb.d];
        ntiles = cnt > 8 ? 2 : 1;
        const uint32_t mask = sh ? 0u : s_tokmask[s_act_e[jb.d]];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const int nb = min(nt * 8 + g, cnt - 1);
          brow[nt] = (jb.gu && !sh) ? nth_bit(mask, nb) : nb;
        }
      }
      const bool ok = !*abort_flag && mbar_wait_bounded(full0 + 8 * slot, (j / kNst) & 1, a.status);
      if (!ok) *abort_flag = 1;
      const uint8_t* st = smem + (size_t)slot * a.stage_bytes;
      const int MT = jb.gu ? 4 : a.R / 16;
      if (ok) {
        const int kcols = jb.gu ? a.KC : (sh ? a.KCds : a.KCd);
        const int TB = a.TB;
        if (jb.gu) {
          if (ntiles == 1) job_compute<true, 4, 1>(st, kcols, a.R, TB, cw, brow, acc);
          else job_compute<true, 4, 2>(st, kcols, a.R, TB, cw, brow, acc);
        } else {
          if (ntiles == 1) job_compute<false, 4, 1>(st, kcols, a.R, TB, cw, brow, acc);
          else job_compute<false, 4, 2>(st, kcols, a.R, TB, cw, brow, acc);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // this warp is done with the stage
      if (!jb.last) continue;

      // ---- unit epilogue: cross-warp reduction in fixed warp order
#pragma unroll
      for (int m = 0; m < kMaxMT; ++m)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
          if (m < MT && nt < ntiles) {
            float* slab = red + ((cw * kMaxMT + m) * 2 + nt) * kRed;
            slab[(2 * c) * 17 + g] = acc[m][nt][0];
            slab[(2 * c + 1) * 17 + g] = acc[m][nt][1];
            slab[(2 * c) * 17 + g + 8] = acc[m][nt][2];
            slab[(2 * c + 1) * 17 + g + 8] = acc[m][nt][3];
          }
      named_bar_sync(1, kCW * 32);
      const bool good = !*abort_flag;
      const int nl = ct >> 5, rl = ct & 31;
      const int base = s_act_off[jb.d];
      if (jb.gu) {
        float hv[2];
        const int mg = rl >> 4, rr = rl & 15;
        for (int nt = 0; nt < ntiles; ++nt) {
          float gs = 0.f, us = 0.f;
#pragma unroll
          for (int w = 0; w < kCW; ++w) {
            gs += red[((w * kMaxMT + mg) * 2 + nt) * kRed + nl * 17 + rr];
            us += red[((w * kMaxMT + 2 + mg) * 2 + nt) * kRed + nl * 17 + rr];
          }
          hv[nt] = gs / (1.0f + expf(-gs)) * us;
        }
        named_bar_sync(1, kCW * 32);  // red is read: the next unit may write it
        for (int nt = 0; nt < ntiles; ++nt) {
          const int n = nt * 8 + nl;
          if (good && n < cnt) {
            if (!(fabsf(hv[nt]) < 65504.f)) atomicOr(a.status, DEV_RANGE);
            const int col = jb.tile * kGuRows + rl;
            a.h[(size_t)(base + n) * a.Imax + (col & ~7) + perm8_pos(col & 7)] =
                __half_as_ushort(__float2half_rn(hv[nt]));
          }
        }
        named_bar_sync(1, kCW * 32);  // every h store of the unit is done (CTA scope)
        if (ct == 0) red_release_gpu_add(a.sync + kSyncReady + jb.d, 1);  // publish + count
      } else {
        float ov[2][2];
        for (int nt = 0; nt < ntiles; ++nt)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int r = rl + 32 * q;
            float o = 0.f;
            if (r < a.R) {
              const int m = r >> 4, rr = r & 15;
#pragma unroll
              for (int w = 0; w < kCW; ++w) o += red[((w * kMaxMT + m) * 2 + nt) * kRed + nl * 17 + rr];
            }
            ov[nt][q] = o;
          }
        named_bar_sync(1, kCW * 32);  // red is read: the next unit may write it
        for (int nt = 0; nt < ntiles; ++nt) {
          const int n = nt * 8 + nl;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int r = rl + 32 * q;
            if (good && n < cnt && r < a.R)
              a.partial[(size_t)(base + n) * H + (size_t)jb.tile * a.R + r] = ov[nt][q];
          }
        }
        named_bar_sync(1, kCW * 32);  // every partial store of the unit is done (CTA scope)
        if (ct == 0) {
          __threadfence();
          const bool last = atomicAdd(a.sync + kSyncRg + jb.tile, 1) == nDx - 1;
          if (last) __threadfence();  // acquire the other CTAs' partials
          s_flag = last;
        }
        named_bar_sync(1, kCW * 32);
        if (s_flag && good) {
          // last contribution to this row group: y = sum_j w_j o_j (j order) + shared
          bool wok = true;
          if (layer_mode) wok = wait_counter_bounded(a.sync + kSyncWReady, T, a.status);
          if (wok) {
            for (int idx = ct; idx < T * a.R; idx += kCW * 32) {
              const int t = idx / a.R, r = idx - t * a.R;
              const size_t col = (size_t)jb.tile * a.R + r;
              const float sv = has_shared ? ldg_cg_f32(a.partial + (size_t)(Pres + t) * H + col) : 0.f;
              float yv = 0.f;
              for (int j0 = 0; j0 < k; j0 += 8) {  // 8 pairs' loads in flight, summed in j order
                float pv[8], wv[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                  pv[q] = 0.f;
                  wv[q] = 0.f;
                  const int jj = j0 + q;
                  if (jj < k) {
                    const int e = s_ids[t][jj];
                    const int dd = s_d_of_e[e];
                    if (dd >= 0) {
                      const int pos = s_act_off[dd] + __popc(s_tokmask[e] & ((1u << t) - 1u));
                      wv[q] = layer_mode ? ldg_cg_f32(a.w_out + (size_t)t * k + jj)
                                         : a.w_in[(size_t)t * k + jj];
                      pv[q] = ldg_cg_f32(a.partial + (size_t)pos * H + col);
                    }
                  }
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                  if (j0 + q < k) yv = fmaf(wv[q], pv[q], yv);
              }
              a.y[(size_t)t * H + col] = yv + sv;
            }
          } else {
            *abort_flag = 1;
          }
          if (ct == 0) a.sync[kSyncRg + jb.tile] = 0;
        }
      }
    }
  }

  // ---- the last CTA out resets the cross-CTA counters for the next call
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.sync + kSyncDone, 1) == G - 1) {
      for (int d = 0; d <= D; ++d) a.sync[kSyncReady + d] = 0;
      for (int rg = 0; rg < pl.nRg; ++rg) a.sync[kSyncRg + rg] = 0;
      a.sync[kSyncWReady] = 0;
      a.sync[kSyncDone] = 0;
      __threadfence();
    }
  }
}

}  // namespace fused

// Host side -------------------------------------------------------------------
static int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess)
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

namespace {
struct FusedCfg {
  int KC, KCd, KCds, R, stage_bytes;
};

constexpr int kStageCap = 48 * 1024;

// Largest chunk c of K (a multiple of 256 dividing K, at most cap).
int chunk_of(int K, int cap) {
  for (int c = cap; c >= 256; c -= 256)
    if (K % c == 0) return c;
  return 0;
}

// The chunking: gate/up chunks of H, down rows per unit and down chunks of I
// such that one job (weights + TB activation rows) fits a stage. Warps take
// blocks b = w (mod 8) whatever the chunk size, and the down rows R do not
// depend on TB, so a row's arithmetic is the same in any window.
bool fused_cfg(int H, int I, int shI, int TB, FusedCfg* out) {
  FusedCfg f{};
  f.KC = chunk_of(H, 512);
  if (!f.KC) return false;
  int sb = fused::gu_bytes(f.KC, TB);
  f.R = 0;
  int Rfix = 0;  // the rows per down unit, fixed by the largest window
  for (int R = 64; R >= 64 && !Rfix; R /= 2) {  // the kernel handles 64-row down units only
    if (H % R) continue;
    for (int c = 256; c <= I; c += 256)
      if (I % c == 0 && fused::dn_bytes(R, c, fused::kMaxT) <= kStageCap) {
        Rfix = R;
        break;
      }
  }
  for (int R = Rfix; R == Rfix && R >= 16 && !f.R; R = 0) {
    for (int cap = 2048; cap >= 256; cap -= 256) {
      const int c = chunk_of(I, cap);
      if (!c) continue;
      const int nk = I / c;
      int bytes = fused::dn_bytes(R, c, TB);
      int cs = 0;
      if (shI > 0) {
        if (shI % nk) continue;
        cs = shI / nk;
        if (cs % 256) continue;
        const int bs = fused::dn_bytes(R, cs, TB);
        bytes = bytes > bs ? bytes : bs;
      }
      if (bytes <= kStageCap) {
        f.R = R;
        f.KCd = c;
        f.KCds = cs ? cs : c;
        sb = sb > bytes ? sb : bytes;
        break;
      }
    }
  }
  if (!f.R) return false;
  f.stage_bytes = (sb + 1023) & ~1023;
  if (fused::smem_bytes(f.stage_bytes) + 20 * 1024 > 227 * 1024) return false;
  *out = f;
  return true;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct MapKey {
  const void* ptr;
  uint64_t d0, d1, d2, s1, s2;
  uint32_t b0, b1, b2, dtype, swz;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof *this) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    const uint64_t* w = reinterpret_cast<const uint64_t*>(&k);
    uint64_t h = 1469598103934665603ull;
    for (size_t i = 0; i < sizeof k / 8; ++i) h = (h ^ w[i]) * 1099511628211ull;
    return (size_t)h;
  }
};

// Encode (or fetch from a small cache) a 2D or 3D tiled tensor map.
bool tensor_map(CUtensorMap* out, CUtensorMapDataType dt, const void* ptr, int rank,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box, bool swizzle) {
  static std::mutex mu;
  static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.ptr = ptr;
  key.d0 = dims[0]; key.d1 = dims[1]; key.d2 = rank > 2 ? dims[2] : 0;
  key.s1 = strides[0]; key.s2 = rank > 2 ? strides[1] : 0;
  key.b0 = box[0]; key.b1 = box[1]; key.b2 = rank > 2 ? box[2] : 0;
  key.dtype = (uint32_t)dt;
  key.swz = swizzle ? 1 : 0;
  std::lock_guard<std::mutex> lk(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  CUresult r = fn(&m, dt, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return true;
}

// Codes [rows][K/2] bytes: box 128 bytes x box_rows, 128-byte swizzle.
bool codes_map(CUtensorMap* m, const uint8_t* q, int K, int rows, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)rows};
  const uint64_t str[1] = {(uint64_t)K / 2};
  const uint32_t box[2] = {128, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 2, dims, str, box, true);
}
// Scales [rows][K/32] fp16: box (chunk/32) x box_rows, no swizzle.
bool scales_map(CUtensorMap* m, const uint16_t* s, int K, int rows, int chunk, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K / 32, (uint64_t)rows};
  const uint64_t str[1] = {(uint64_t)K / 16};
  const uint32_t box[2] = {(uint32_t)chunk / 32, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, 2, dims, str, box, false);
}
// 16-bit activations [rows][cols]: viewed as (64, cols/64, rows); box (64, chunk/64, box_rows).
bool act_map(CUtensorMap* m, const void* p, int cols, int rows, int chunk, int box_rows) {
  const uint64_t dims[3] = {64, (uint64_t)cols / 64, (uint64_t)rows};
  const uint64_t str[2] = {128, (uint64_t)cols * 2};
  const uint32_t box[3] = {64, (uint32_t)chunk / 64, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, p, 3, dims, str, box, true);
}
}  // namespace

static int box_rows(int T) { return T <= 8 ? 8 : 16; }

bool fused_decode_supported(int H, int I, int shI, int T, bool x_bf16) {
  if (!x_bf16 || T < 1 || T > fused::kMaxT) return false;
  if (H % 256 || I % 256 || shI % 256) return false;
  if (H > 8192 || T > num_sms()) return false;
  if (!encode_fn()) return false;
  FusedCfg f;
  return fused_cfg(H, I, shI, box_rows(T), &f);
}

cudaError_t launch_fused_decode(const FusedLaunch& f, cudaStream_t st) {
  FusedCfg cfg;
  const int TB = box_rows(f.T);
  if (!fused_cfg(f.H, f.I, f.shI, TB, &cfg)) return cudaErrorInvalidValue;
  fused::Args a;
  std::memset(&a, 0, sizeof a);
  a.H = f.H; a.I = f.I; a.shI = f.shI; a.E = f.E; a.k = f.k; a.S = f.S; a.T = f.T;
  a.Imax = f.Imax;
  a.KC = cfg.KC;
  a.KCd = cfg.KCd;
  a.KCds = cfg.KCds;
  a.R = cfg.R;
  a.stage_bytes = cfg.stage_bytes;
  a.TB = TB;
  a.rows_cap = f.rows_cap;
  const int H = f.H, I = f.I, S = f.S;
  bool ok = codes_map(&a.tm_gc, f.gq, H, S * I, fused::kGuRows) &&
            codes_map(&a.tm_uc, f.uq, H, S * I, fused::kGuRows) &&
            codes_map(&a.tm_dc, f.dq, I, S * H, cfg.R) &&
            scales_map(&a.tm_gs, f.gs, H, S * I, cfg.KC, fused::kGuRows) &&
            scales_map(&a.tm_us, f.us, H, S * I, cfg.KC, fused::kGuRows) &&
            scales_map(&a.tm_ds, f.ds, I, S * H, cfg.KCd, cfg.R) &&
            act_map(&a.tm_x, f.x, H, f.T, cfg.KC, TB) &&
            act_map(&a.tm_h, f.hhi, f.Imax, f.rows_cap, cfg.KCd, TB);
  if (ok && f.shI > 0)
    ok = codes_map(&a.tm_sgc, f.sgq, H, f.shI, fused::kGuRows) &&
         codes_map(&a.tm_suc, f.suq, H, f.shI, fused::kGuRows) &&
         codes_map(&a.tm_sdc, f.sdq, f.shI, H, cfg.R) &&
         scales_map(&a.tm_sgs, f.sgs, H, f.shI, cfg.KC, fused::kGuRows) &&
         scales_map(&a.tm_sus, f.sus, H, f.shI, cfg.KC, fused::kGuRows) &&
         scales_map(&a.tm_sds, f.sds, f.shI, H, cfg.KCds, cfg.R) &&
         act_map(&a.tm_hs, f.hhi, f.Imax, f.rows_cap, cfg.KCds, TB);
  if (!ok) return cudaErrorInvalidValue;
  a.logits = f.logits; a.ids_in = f.ids_in; a.w_in = f.w_in;
  a.slot_map = f.slot_map;
  a.ids_out = f.ids_out; a.w_out = f.w_out; a.y = f.y;
  a.miss_ids = f.miss_ids; a.n_miss = f.n_miss;
  a.h = f.hhi;
  a.partial = f.partial;
  a.status = f.status; a.sync = f.sync;
  const size_t smem = fused::smem_bytes(a.stage_bytes);
  static std::mutex mu;
  static size_t configured = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (smem > configured) {
      cudaError_t e = cudaFuncSetAttribute(fused::decode_layer_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
      }
      configured = smem;
    }
  }
  launch_begin(K_FUSED, st);
  fused::decode_layer_kernel<<<num_sms(), fused::kThreads, smem, st>>>(a);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace moe
