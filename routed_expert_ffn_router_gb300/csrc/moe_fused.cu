// One persistent kernel per decode window (T <= 16 rows): routing, the
// (token, expert) permutation, gate/up + SwiGLU, down and the ordered combine.
//
// This is the grouped expert call of the SGLang port post (TL;DR and section
// 3: gather -> dequant -> gate/up -> SwiGLU -> down -> scatter in one call per
// layer) laid out for GB300:
//  * one CTA per SM. Warp 0 (one thread) is the producer: it takes work units
//    from a grid-wide queue (one atomic per unit) and streams each unit's jobs
//    into a ring of shared-memory stages with TMA tensor copies (full/empty
//    mbarriers; the weights with an evict-first L2 policy). It also publishes
//    finished units, so no consumer waits on a gpu-scope fence;
//  * a unit is UI = 32 MT intermediate rows of one expert: its gate/up rows
//    over all of H (H / 256 jobs), then that slice of I's contribution to the
//    down projection (H / 256 jobs of 256 output rows). h never leaves the SM
//    and no unit waits for another CTA: the units stream back to back;
//  * the 8 consumer warps are 4 row warps x 2 column halves for gate/up (row
//    warp mw owns MT m16 tiles, half kh sums blocks 4kh..4kh+3 of each
//    256-column chunk) and 8 row warps for down. A row's summation order
//    depends only on H and I, never on the window;
//  * gate/up tiles interleave 8 gate rows and the same 8 up rows, so an MMA
//    accumulator holds g and u of one intermediate index side by side and
//    SwiGLU happens in registers; h is kept as fp16 in the down operand's
//    fragment order (h / 16 where it meets a high nibble). The exact-integer
//    warp-MMA core (moe_decode.cu explains the 136 + q and 1032 + q code
//    fragments; the down MMA takes high nibbles in place as 1152 + 16 q) gets
//    its per-block correction -magic * sum(B) from one more MMA whose A operand
//    is the constant -magic;
//  * every CTA computes the top-k ids and the permutation of the whole window
//    in shared memory, so no launch precedes the weight stream; a helper warp
//    computes the float64 softmax weights of the rows its CTA reduces (and
//    writes the routing of the rows whose first output block it owns), so no
//    CTA waits for another particular CTA: the reduction waits only for the
//    units, which the CTAs that are running take from the queue;
//  * once every unit is published, the CTAs share the reduction
//    y = sum_j w_j sum_g p(e_j, g) + sum_g p(shared, g) in a fixed order, so y is
//    deterministic; once past the wait for the units, each CTA counts itself
//    out, and the last one resets the cross-CTA counters.
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

constexpr int kCW = 8;                  // consumer warps: 4 row warps x 2 column halves
constexpr int kHelperWarp = kCW + 1;    // routing weights, off the weight stream's path
constexpr int kWarps = kCW + 2;         // producer, consumers, helper
constexpr int kThreads = 32 * kWarps;
constexpr int kKC = 256;                // columns of K per job
constexpr int kMaxNst = 8;              // stages in the ring at most
constexpr int kUnitRing = 16;           // units a producer may have unpublished
constexpr int kMaxT = 16;               // largest window; x boxes hold TB = 8 or 16 rows
constexpr int kDnRows = 512;            // output rows per down job (two 256-row boxes)
constexpr int kDnM = kDnRows / (kCW * 16);  // m16 tiles per warp in a down job
constexpr int kPubCount = kCW * 32;     // arrivals that publish a unit (every consumer lane)
constexpr int kPubBars = 4;             // publish barriers, used by units in turn
constexpr int kStgRow = 68;             // floats per token row of a warp's partial staging (64 + 4 pad)
constexpr int kRedBlock = kCW * 4;      // float4 outputs per CTA and step of the reduction
constexpr int kBarReduce = 6;           // named barrier: consumers + helper before the reduction
// Unrolling of the per-block loops of a job (the kernel holds the compute of
// three unit sizes; full unrolling of all of them crowds the instruction cache:
// measured on GB300, 2 takes 36.7 us per decode window where 4 takes 38.7 and 1 38.4).
constexpr int kBlockUnroll = 2;
constexpr int kMT = 4;                  // m16 tiles per row warp in a full unit
constexpr int kUI = 32 * kMT;           // intermediate rows of a full unit (a half unit has 64)
constexpr uint32_t kBf16NegMagic = 0xC308C308u;  // bf16 -136
constexpr uint32_t kF16NegMagic = 0xE408E408u;   // f16 -1032

// cross-CTA counters (int32 offsets in the workspace sync region)
// (the exit count has a cache line of its own: the units counter is still
// polled, and the queue drawn, while CTAs count themselves out)
constexpr int kSyncDone = 64, kSyncUnits = 1, kSyncQueue = 2;

// Jobs of full units (kUI intermediate rows) and half units (64): gate/up
// kind 2 s, down kind 2 s + 1 for unit size s = 0 (full), 1 (half).
enum JobKind : int { J_GU = 0, J_DN = 1, J_GUH = 2, J_DNH = 3, J_END = 4 };

struct Args {
  // TMA tensor maps (kernel parameters, read through their parameter address)
  CUtensorMap tm_gc, tm_uc, tm_dc;     // routed codes: gate, up [S*I][H/2]; down [S*H][I/2]
  CUtensorMap tm_gs, tm_us, tm_ds;     // routed scales
  CUtensorMap tm_sgc, tm_suc, tm_sdc;  // shared expert codes
  CUtensorMap tm_sgs, tm_sus, tm_sds;  // shared expert scales
  CUtensorMap tm_gch, tm_uch, tm_dch;  // the same in half-unit boxes (64 rows; 32-byte down rows)
  CUtensorMap tm_gsh, tm_ush;
  CUtensorMap tm_sgch, tm_such, tm_sdch;
  CUtensorMap tm_sgsh, tm_sush;
  CUtensorMap tm_x;                    // x [T][H] bf16, 3D box (64, 4, TB)
  int H, I, shI, E, k, S, T;
  int Gh;          // 64-column slices of I per partial row (max(I, shared I) / 64)
  int TB;          // rows of the x / h boxes (8 or 16, >= T)
  int nst;         // stages in the ring
  int stage_bytes; // multiple of 1024
  int rows_cap;    // rows of the partial buffer (P + T)
  const float* logits;     // non-null: route here (layer mode)
  const int32_t* ids_in;   // routing given (ffn mode)
  const float* w_in;
  const int32_t* slot_map;
  int32_t* ids_out;
  float* w_out;
  float* y;
  int32_t* miss_ids;
  int32_t* n_miss;
  // [rows_cap][Gh][H]: the down partials of each routed pair (and shared row):
  // a full unit's A + B at slice 2 g, a half unit's A or B at its own slice
  float* partial;
  int32_t* status;
  int32_t* sync;
  int32_t* picks;  // nullable: one pick per distinct expert of the window
  // a stack of chained layers with the router in the launch (else null):
  // logits = x W_r^T from router_w [E][H] bf16 into `logits` (which the
  // routing then reads), and x_next [T][H] bf16 = bf16(x + y) for the next layer
  const uint16_t* router_w;
  const uint16_t* xg;  // x [T][H] bf16 for the router and the residual add
  uint16_t* x_next;
  int stack_L;         // a stack plan's layer count (the launch checks it against its own)
};

// Stage layouts (byte offsets from the 1024-aligned stage base), UI = 32 MT
// (MT = 4 for full units, 2 for half units):
//  gate/up: gate codes [UI][128 B] (swizzled), up codes [UI][128 B], x box
//           [TB][4][128 B] (swizzled), gate scales [UI][8], up scales [UI][8];
//  down:    codes [512][UI/2 B] (swizzled by the row width, 64 or 32 bytes),
//           scales [512][8] (the 8 blocks
//           around the unit's UI columns).
__host__ __device__ constexpr int gu_job_bytes(int MT, int TB) { return 288 * 32 * MT + 512 * TB; }
__host__ __device__ constexpr int dn_job_bytes(int MT) { return kDnRows * 16 * MT + 16 * kDnRows; }
__host__ __device__ constexpr int stage_bytes_for(int MT, int TB) {
  return gu_job_bytes(MT, TB) > dn_job_bytes(MT) ? gu_job_bytes(MT, TB) : dn_job_bytes(MT);
}
__host__ __device__ constexpr int red_bytes(int MT, int NTX) { return 4 * (MT * NTX * 4) * 32 * 4; }
// two h buffers [kMaxT][UI + 8] f16 (the 16-byte pad keeps the B loads free of bank conflicts)
__host__ __device__ constexpr int hb_bytes(int MT) { return 2 * kMaxT * (64 * MT + 16); }
// per consumer warp, the down partials of its 64 rows: [TB][kStgRow] f32
__host__ __device__ constexpr int stg_bytes(int TB) { return kCW * TB * kStgRow * 4; }
// Dynamic shared memory: 1 KB of alignment slack, the stages, the exchange
// buffer of the two column halves, the h buffers, the partial staging rows.
__host__ __device__ inline size_t smem_bytes(int MT, int NTX, int nst, int stage_bytes, int TB) {
  return 1024 + (size_t)nst * stage_bytes + red_bytes(MT, NTX) + hb_bytes(MT) + stg_bytes(TB);
}
// The slot map's copy lives in stage memory during the routing (after the
// top-k scratch of every warp), before the first weight copy.
constexpr int kSlotMapOff = 32768;

// Four f16x2 registers from one word of int4 codes for the down MMA, without
// shifts per nibble: registers 0 and 2 hold the low nibbles of bytes (0, 2)
// and (1, 3) as 1032 + code, registers 1 and 3 the high nibbles as
// 1152 + 16 code (the nibble stays in place under the f16 constant 1024, bit 3
// of the nibble flipped). The h operand holds h / 16 at the high-nibble
// positions, so those products are (72 + code) h and the correction constant
// there is -1152 (times h / 16). Same register pairing as dequant_word_f16.
__device__ __forceinline__ void dequant_word_f16x16(uint32_t w, uint32_t (&d)[4]) {
  d[0] = lop3_and_xor(w, 0x000F000Fu, 0x64086408u);
  d[1] = lop3_and_xor(w, 0x00F000F0u, 0x64806480u);
  const uint32_t w8 = w >> 8;
  d[2] = lop3_and_xor(w8, 0x000F000Fu, 0x64086408u);
  d[3] = lop3_and_xor(w8, 0x00F000F0u, 0x64806480u);
}
constexpr uint32_t kF16NegMagicHi = 0xE480E480u;  // f16 -1152

// n-th (0-based) set bit of a mask (mask has more than n bits set).
__device__ __forceinline__ int nth_bit(uint32_t m, int n) {
  for (int i = 0; i < n; ++i) m &= m - 1;
  return __ffs(m) - 1;
}


// One job's share for one consumer warp (row warp mw, column half kh):
//   acc[m][nt] += sum_b scale(row, b) * (codes(row, b) . B(b, token slot))
// over blocks b = 4 kh .. 4 kh + 3 of the stage's 256-column chunk. All
// shared-memory loads of a block are issued before its arithmetic, so the
// MT x NT MMA chains overlap.
// GU: gate/up job (bf16 x, 136 + q codes); m-tile m holds gate rows
// 8 (mw MT + m) + 0..7 of the unit in A rows 0-7 and the same up rows in A
// rows 8-15. Otherwise a down job (f16 h, 1032 + q codes); m-tile m holds rows
// 16 (mw MT + m) + 0..15.
template <bool GU, int MT, int NT>
__device__ __forceinline__ void job_compute(uint32_t st, int mw, int kh, int TB,
                                            const int (&brow)[2], float (&acc)[MT][2][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr int UI = 32 * MT, R = 64 * MT;
  const uint32_t bbox = st + (GU ? 2 * UI * 128 : R * 128);
  const uint32_t scl0 = bbox + TB * 512;
  // the second code row of a lane: the up tile (gate/up), 8 rows further (down)
  constexpr int kRow2 = GU ? UI * 128 : 8 * 128;
  constexpr int kScl2 = GU ? UI * 16 : 8 * 16;
  // every row this lane reads is g (mod 8): one swizzle for all of them
  const int r0 = GU ? 8 * mw * MT + g : 16 * mw * MT + g;
  const uint32_t rowp = st + r0 * 128 + c * 4;
  const uint32_t sclp = scl0 + r0 * 16;
  constexpr int kMStep = GU ? 8 : 16;  // rows between m-tiles
#pragma unroll kBlockUnroll
  for (int i = 0; i < 4; ++i) {
    const int b = kh * 4 + i;
    uint4 braw[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
      braw[nt] = ld_s128(bbox + swz128((uint32_t)(brow[nt] * 512 + b * 64 + c * 16)));
    const int coff = (b ^ g) << 4;
    uint32_t w[MT][2];
    float sc[MT][2];
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      w[m][0] = ld_s32(rowp + m * kMStep * 128 + coff);
      w[m][1] = ld_s32(rowp + m * kMStep * 128 + kRow2 + coff);
      sc[m][0] = ld_s_half_as_float(sclp + m * kMStep * 16 + 2 * b);
      sc[m][1] = ld_s_half_as_float(sclp + m * kMStep * 16 + kScl2 + 2 * b);
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
      for (int q = 0; q < 4; ++q) corr[nt][q] = 0.f;
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

__device__ __forceinline__ float4 add4(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}

__device__ __forceinline__ float4 ldg_cg_f4(const float* p) {
  const uint4 v = ldg_cg_v4(p);
  return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                     __uint_as_float(v.w));
}

// One down job for one consumer warp: rows 64 cw + 16 m + (g, g + 8), m < 4,
// of the job's 512 output rows, over the unit's UI columns of I (MT blocks):
//   acc[m][nt] += sum_b scale(row, b) * (codes(row, b) . h(b, token slot))
// Codes: [512][UI/2 B] with the TMA swizzle of that row width (64-, 32-byte or
// none); scales [512][8] (the unit's blocks start at boff); h comes from the
// unit's shared-memory buffer [slot][UI + 8] f16 in fragment order.
// Blocks B0 .. B0 + NB - 1 of the unit's MT, summed in block order.
template <int MT, int NT, int B0, int NB>
__device__ __forceinline__ void dn_compute(uint32_t st, uint32_t hb, int cw, int boff,
                                           const int (&brow)[2], float (&acc)[kDnM][2][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  constexpr int UI = 32 * MT, RB = UI / 2;
  constexpr uint32_t kSwz = MT == 4 ? 3u : (MT == 2 ? 1u : 0u);
  constexpr int HB = UI * 2 + 16;
  const uint32_t scl = st + kDnRows * RB;
#pragma unroll kBlockUnroll
  for (int b = B0; b < B0 + NB; ++b) {
    uint32_t bf[NT][4];
    float corr[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint4 v = ld_s128(hb + brow[nt] * HB + b * 64 + c * 16);
      bf[nt][0] = v.x; bf[nt][1] = v.y; bf[nt][2] = v.z; bf[nt][3] = v.w;
#pragma unroll
      for (int q = 0; q < 4; ++q) corr[nt][q] = 0.f;
      // A rows: low-nibble positions (k = 2c, 2c + 1) -1032, high-nibble ones -1152
      mma_f16_16816(corr[nt], kF16NegMagic, kF16NegMagic, kF16NegMagicHi, kF16NegMagicHi, bf[nt][0], bf[nt][1]);
      mma_f16_16816(corr[nt], kF16NegMagic, kF16NegMagic, kF16NegMagicHi, kF16NegMagicHi, bf[nt][2], bf[nt][3]);
    }
    uint32_t w[kDnM][2];
    float sc[kDnM][2];
#pragma unroll
    for (int m = 0; m < kDnM; ++m) {
      const int r = 16 * (kDnM * cw + m) + g;
      const uint32_t o0 = r * RB + b * 16 + c * 4, o1 = o0 + 8 * RB;
      w[m][0] = ld_s32(st + (o0 ^ (((o0 >> 7) & kSwz) << 4)));
      w[m][1] = ld_s32(st + (o1 ^ (((o1 >> 7) & kSwz) << 4)));
      sc[m][0] = ld_s_half_as_float(scl + r * 16 + 2 * (boff + b));
      sc[m][1] = ld_s_half_as_float(scl + (r + 8) * 16 + 2 * (boff + b));
    }
#pragma unroll
    for (int m = 0; m < kDnM; ++m) {
      uint32_t d[4], e[4];
      dequant_word_f16x16(w[m][0], d);
      dequant_word_f16x16(w[m][1], e);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        float t4[4] = {corr[nt][0], corr[nt][1], corr[nt][2], corr[nt][3]};
        mma_f16_16816(t4, d[0], e[0], d[1], e[1], bf[nt][0], bf[nt][1]);
        mma_f16_16816(t4, d[2], e[2], d[3], e[3], bf[nt][2], bf[nt][3]);
        acc[m][nt][0] = fmaf(sc[m][0], t4[0], acc[m][nt][0]);
        acc[m][nt][1] = fmaf(sc[m][0], t4[1], acc[m][nt][1]);
        acc[m][nt][2] = fmaf(sc[m][1], t4[2], acc[m][nt][2]);
        acc[m][nt][3] = fmaf(sc[m][1], t4[3], acc[m][nt][3]);
      }
    }
  }
}

// The units of a window, in queue order. Group (d, g) is intermediate rows
// [g kUI, g kUI + kUI) of expert d, groups in the order: the shared expert's,
// then the routed experts' (expert order). The first nfull groups are full
// units; each later group is split into sf units of 128 / sf rows. A unit is
// its gate/up (H / 256 jobs) and its rows' share of the down projection
// (H / 512 jobs of 512 output rows).
//
// nfull balances the window over the G CTAs. Unsplit, U groups take M0 =
// ceil(U / G) rounds of full units. Splitting the R groups of the last round
// into halves instead takes M0 - 1 rounds plus ceil(2 R / G) rounds of half
// units, each costing about kHalfCostPct % of a full unit (measured: the fixed
// costs of a unit do not halve with its bytes); the cheaper plan is taken. The
// dynamic queue hands out the full units first, so the halves fill the CTAs
// that finish first. The results do not depend on the split: a group's down
// partial is A + B, A and B the scaled sums (fma chains) of its blocks 0-1 and
// 2-3, formed by one full unit or by its two halves, and added in the reduction.
constexpr int kHalfCostPct = 68;
struct Sched {
  int D;      // resident routed experts of the window (the shared expert is d = D)
  int nGs;    // groups of the shared expert (0 without one)
  int nGi;    // groups per routed expert
  int U;      // groups in all
  int nfull;  // groups that stay whole (the first nfull in queue order)
  int total;  // units in all
  __device__ void plan(int G) {
    U = nGs + D * nGi;
    const int M0 = (U + G - 1) / G;
    const int R = U - G * (M0 - 1);
    const int ch = 100 * (M0 - 1) + kHalfCostPct * ((2 * R + G - 1) / G);
    nfull = (U > 0 && ch < 100 * M0) ? U - R : U;
    total = nfull + 2 * (U - nfull);
  }
  __device__ int2 group(int u) const {  // (d, g) of group u
    if (u < nGs) return make_int2(D, u);
    const int d = (u - nGs) / nGi;
    return make_int2(d, u - nGs - d * nGi);
  }
  // unit t -> (d, its first 32-row slice of I: 4 g or 4 g + 2, size: 0 full, 1 half)
  __device__ int3 unit(int t) const {
    if (t < nfull) {
      const int2 dg = group(t);
      return make_int3(dg.x, 4 * dg.y, 0);
    }
    const int x = t - nfull;
    const int2 dg = group(nfull + (x >> 1));
    return make_int3(dg.x, 4 * dg.y + 2 * (x & 1), 1);
  }
  // group index of (d, g): d = D is the shared expert
  __device__ int group_index(int d, int g) const { return d == D ? g : nGs + d * nGi + g; }
};

// The producer thread's state and steps (always inlined: no call may make it
// wait for an atomic whose result it does not need yet).
struct Producer {
  const Args& a;
  uint32_t sbase, full0, empty0, pub0;
  int4* hdr;
  const int32_t* act_slot;
  int D;
  int nst, stage_bytes;
  uint64_t wpol;   // L2 policy of the weight copies
  int j;           // jobs issued
  int ui, pd;      // units taken, units published
  int slot, phase; // ring position of job j (slot = j mod nst, phase = (j / nst) & 1)

  // Count the units the consumer warps have published (never blocks).
  __device__ __forceinline__ void poll() {
    while (pd < ui && mbar_test(pub0 + 8 * (pd % kPubBars), (pd / kPubBars) & 1)) ++pd;
  }
  __device__ __forceinline__ bool timed_out(long long t0) {
    if (cycles_now() - t0 <= kWaitCycles) return false;
    atomicOr(a.status, DEV_TIMEOUT);
    return true;
  }
  // Free slot for job j (publishing meanwhile).
  // The thread sleeps in the barrier wait between polls: a spinning producer
  // would take issue slots from the consumer warps of its SM sub-partition.
  __device__ __forceinline__ bool acquire_slot() {
    const uint32_t par = phase ^ 1;
    if (mbar_test(empty0 + 8 * slot, par)) return true;
    const long long t0 = cycles_now();
    for (uint32_t it = 1;; ++it) {
      poll();
      if (mbar_try_wait_ns(empty0 + 8 * slot, par, 400)) return true;
      if ((it & 15) == 0 && timed_out(t0)) return false;
    }
  }
  // Sleep until the oldest unpublished unit's epilogue is done (or ~ns).
  __device__ __forceinline__ void wait_pub(uint32_t ns) {
    if (pd < ui) mbar_try_wait_ns(pub0 + 8 * (pd % kPubBars), (pd / kPubBars) & 1, ns);
  }
  // qi: the unit's first 32-row slice of the expert's I (4 g for a full unit)
  __device__ __forceinline__ bool issue(int kind, int d, int qi, int chunk) {
    if ((j & 3) == 0) poll();  // publications are also handled whenever the producer waits
    if (!acquire_slot()) return false;
    hdr[slot] = make_int4(kind, d, qi, chunk);
    const uint32_t st = sbase + slot * stage_bytes, fb = full0 + 8 * slot;
    ++j;
    if (++slot == nst) {
      slot = 0;
      phase ^= 1;
    }
    if (kind == J_END) {
      mbar_arrive(fb);
      return true;
    }
    const bool sh = d == D;
    const int slotp = sh ? 0 : act_slot[d];
    if ((kind & 1) == 0) {  // gate/up of a unit of size s: UI = kUI >> s rows
      const int sz = kind >> 1, UI = kUI >> sz;
      mbar_expect_tx(fb, (uint32_t)gu_job_bytes(kMT >> sz, a.TB));
      const int row = (sh ? 0 : slotp * a.I) + qi * 32;
      const uint32_t so = st + 2 * UI * 128 + a.TB * 512;
      const bool hf = sz == 1;
      tma_load_2d_hint(st, hf ? (sh ? &a.tm_sgch : &a.tm_gch) : (sh ? &a.tm_sgc : &a.tm_gc), chunk * 128,
                       row, fb, wpol);
      tma_load_2d_hint(st + UI * 128, hf ? (sh ? &a.tm_such : &a.tm_uch) : (sh ? &a.tm_suc : &a.tm_uc),
                       chunk * 128, row, fb, wpol);
      tma_load_2d_hint(so, hf ? (sh ? &a.tm_sgsh : &a.tm_gsh) : (sh ? &a.tm_sgs : &a.tm_gs), chunk * 8,
                       row, fb, wpol);
      tma_load_2d_hint(so + UI * 16, hf ? (sh ? &a.tm_sush : &a.tm_ush) : (sh ? &a.tm_sus : &a.tm_us),
                       chunk * 8, row, fb, wpol);
      tma_load_3d(st + 2 * UI * 128, &a.tm_x, 0, chunk * 4, 0, fb);
    } else {  // down: the unit's columns of 512 rows
      const int sz = kind >> 1;
      const int RB = (kUI / 2) >> sz;  // code bytes of a down row in the unit's columns
      mbar_expect_tx(fb, (uint32_t)dn_job_bytes(kMT >> sz));
      const int row = (sh ? 0 : slotp * a.H) + chunk * kDnRows;
      const uint32_t so = st + kDnRows * RB;
      const CUtensorMap* dc = sz == 0 ? (sh ? &a.tm_sdc : &a.tm_dc) : (sh ? &a.tm_sdch : &a.tm_dch);
#pragma unroll
      for (int h2 = 0; h2 < kDnRows / 256; ++h2) {  // boxes of 256 rows
        tma_load_2d_hint(st + h2 * 256 * RB, dc, qi * 16, row + 256 * h2, fb, wpol);
        tma_load_2d_hint(so + h2 * 256 * 16, sh ? &a.tm_sds : &a.tm_ds, qi & ~7, row + 256 * h2,
                         fb, wpol);
      }
    }
    return true;
  }
};

// Ring state a CTA carries from one layer to the next when one launch runs
// several layers: the producer's jobs issued, units taken and published; the
// consumers' ring position and units consumed.
struct RingState {
  int pj, pui, ppd;
  int cslot, cphase, ccs, cucnt;
};

// One layer's window (the whole work of decode_layer_kernel). `first`: the
// launch's first layer (barrier set-up, programmatic dependent launch);
// `count_out`: count the CTA out of the layer's cross-CTA counters after its
// reduction wait (the last CTA resets them); a launch of several layers
// resets them itself at its end.
// MAXNT: n8 token tiles at most (1 for windows of up to 8 rows, 2 beyond).
template <int MAXNT>
__device__ __forceinline__ bool layer_body(const Args& a, RingState& rs, bool first, bool count_out) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ int s_ids[kMaxT][kMaxK];
  __shared__ uint32_t s_tokmask[kMaxE];
  __shared__ int16_t s_d_of_e[kMaxE];
  // the selected logits of each row in rank order; the helper replaces those of
  // the rows this CTA reduces by their softmax weights
  __shared__ float s_rw[kMaxT][kMaxK];
  __shared__ int16_t s_act_e[kMaxE + 1];
  __shared__ int32_t s_act_slot[kMaxE + 1];
  __shared__ int16_t s_act_off[kMaxE + 1];
  __shared__ uint8_t s_act_cnt[kMaxE + 1];
  __shared__ __align__(8) uint64_t s_bar[2 * kMaxNst + kPubBars];  // full, empty, publish
  __shared__ int4 s_hdr[kMaxNst];                           // the job in each stage
  __shared__ uint32_t s_total;
  __shared__ uint32_t s_wsum[kWarps];  // warp sums of the permutation's prefix sum
  __shared__ int s_abort;
  __shared__ int s_reduce;  // set by consumer thread 0: the units are all published

  constexpr int MT = kMT, UI = kUI;  // full units; half units have MT = 2
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x, bid = blockIdx.x;
  const int T = a.T, k = a.k, E = a.E, H = a.H;
  const bool layer_mode = a.logits != nullptr;
  const bool has_shared = a.shI > 0;
  // stages start at a 1024-byte boundary (the unit of the 128-byte swizzle)
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  const uint32_t sbase = smem_u32(smem);
  float* const red = reinterpret_cast<float*>(smem + (size_t)a.nst * a.stage_bytes);
  uint8_t* const hbuf = smem + (size_t)a.nst * a.stage_bytes + red_bytes(MT, MAXNT);
  const uint32_t stg_s = smem_u32(hbuf) + hb_bytes(MT);
  int32_t* const s_slot = reinterpret_cast<int32_t*>(smem + kSlotMapOff);
  const uint32_t full0 = smem_u32(&s_bar[0]), empty0 = full0 + 8 * kMaxNst,
                 pub0 = empty0 + 8 * kMaxNst;
  volatile int* abort_flag = &s_abort;  // read in loops without barriers

  if (tid == 0) {
    if (first) {
      s_abort = 0;
      for (int i = 0; i < a.nst; ++i) {
        mbar_init(full0 + 8 * i, 1);
        mbar_init(empty0 + 8 * i, kCW);
      }
      for (int i = 0; i < kPubBars; ++i) mbar_init(pub0 + 8 * i, kPubCount);
      fence_barrier_init();
    }
    // the tensor maps' descriptors (kernel parameters or a plan in global
    // memory), fetched ahead of use
    const CUtensorMap* maps[] = {&a.tm_gc, &a.tm_uc, &a.tm_dc, &a.tm_gs, &a.tm_us, &a.tm_ds, &a.tm_x,
                                 &a.tm_gch, &a.tm_uch, &a.tm_dch, &a.tm_gsh, &a.tm_ush};
    for (const CUtensorMap* m : maps) prefetch_tensormap(m);
    if (has_shared) {
      const CUtensorMap* smaps[] = {&a.tm_sgc, &a.tm_suc, &a.tm_sdc, &a.tm_sgs, &a.tm_sus, &a.tm_sds,
                                    &a.tm_sgch, &a.tm_such, &a.tm_sdch, &a.tm_sgsh, &a.tm_sush};
      for (const CUtensorMap* m : smaps) prefetch_tensormap(m);
    }
    // the next kernel of the stream may be scheduled now: it takes an SM only
    // when a CTA of this one exits, and waits for this grid before reading
    if (first) griddep_launch_dependents();
  }
  for (int e = tid; e < E; e += kThreads) s_tokmask[e] = 0;
  // nothing above reads global memory: from here on the previous kernel of the
  // stream (which may have written the inputs or this workspace) is complete
  if (first) griddep_wait();
  // the slot map comes in by asynchronous copies while the routing runs
  for (int e = tid; e < E; e += kThreads) {
    if (a.slot_map) cp_async_4(&s_slot[e], a.slot_map + e);
    else s_slot[e] = e;
  }
  cp_async_commit();
  int ticket = 0;  // the producer's first unit (the atomic's latency overlaps the routing)
  if (tid == 0) ticket = atomicAdd(a.sync + kSyncQueue, 1);

  // ---- routing: ids of every row (all CTAs); weights of row bid (CTA bid < T).
  // The stage buffers are still idle: they hold the top-k scratch.
  if (layer_mode) {
    unsigned long long* scr = reinterpret_cast<unsigned long long*>(smem) + warp * kTopkScratch;
    for (int t = warp; t < T; t += kWarps) {
      const float* l = a.logits + (size_t)t * E;
      bool bad;
      if (E <= 128) bad = topk_row<4>(l, E, k, scr, &s_ids[t][0]);
      else if (E <= 256) bad = topk_row<8>(l, E, k, scr, &s_ids[t][0]);
      else if (E <= 512) bad = topk_row<16>(l, E, k, scr, &s_ids[t][0]);
      else bad = topk_row<32>(l, E, k, scr, &s_ids[t][0]);
      if (bad && lane == 0 && bid == 0) atomicOr(a.status, DEV_NONFINITE_LOGIT);
      if (lane < k) s_rw[t][lane] = key_value((uint32_t)(scr[kTopkRanked + lane] >> 32));
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
  cp_async_wait_all();
  __syncthreads();  // the top-k scratch (stage memory) is released; the slot map is in
  // ---- permutation: token masks (shared atomics), then the active-expert
  // list (ascending id), the offsets and the miss list: one expert per thread,
  // a prefix sum over the block of (active | misses << 11 | routed rows << 22)
  for (int p = tid; p < T * k; p += kThreads) atomicOr(&s_tokmask[s_ids[p / k][p % k]], 1u << (p / k));
  __syncthreads();
  {
    uint32_t base = 0;  // the pack of the experts of earlier rounds
    for (int r0 = 0; r0 < E; r0 += kThreads) {
      const int e = r0 + tid;
      uint32_t m = 0, pack = 0;
      int slot = -1;
      if (e < E) {
        m = s_tokmask[e];
        if (m) {
          slot = s_slot[e];
          if (slot >= a.S) {
            if (bid == 0) atomicOr(a.status, DEV_BAD_SLOT);
            slot = -1;
          }
          pack = slot >= 0 ? 1u + ((uint32_t)__popc(m) << 22) : (1u << 11);
        }
      }
      uint32_t x = pack;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
      }
      if (lane == 31) s_wsum[warp] = x;
      __syncthreads();
      uint32_t pre = base, rsum = 0;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t v = s_wsum[w];
        pre += w < warp ? v : 0u;
        rsum += v;
      }
      const uint32_t ex = pre + x - pack;
      if (e < E) {
        int16_t dd = -1;
        if (m) {
          const int ai = ex & 0x7ff, mi = (ex >> 11) & 0x7ff, off = (ex >> 22) & 0x3ff;
          if (slot >= 0) {
            dd = (int16_t)ai;
            s_act_e[ai] = (int16_t)e;
            s_act_slot[ai] = slot;
            s_act_off[ai] = (int16_t)off;
            s_act_cnt[ai] = (uint8_t)__popc(m);
          } else if (bid == 0) {
            a.miss_ids[mi] = e;
          }
        }
        s_d_of_e[e] = dd;
      }
      base += rsum;
      __syncthreads();  // s_wsum is read before the next round writes it
    }
    if (tid == 0) {
      s_total = base;
      const int Dw = base & 0x7ff, Pw = (base >> 22) & 0x3ff;
      if (bid == 0) *a.n_miss = (base >> 11) & 0x7ff;
      if (has_shared) {
        s_act_e[Dw] = -1;
        s_act_slot[Dw] = -1;
        s_act_off[Dw] = (int16_t)Pw;
        s_act_cnt[Dw] = (uint8_t)T;
      }
    }
  }
  __syncthreads();
  // adaptive-cache routing counters: one pick per distinct expert of the window
  if (a.picks && bid == 0)
    for (int e = tid; e < E; e += kThreads)
      if (s_tokmask[e]) atomicAdd(a.picks + e, 1);
  const uint32_t tot = s_total;
  Sched sc;
  sc.D = tot & 0x7ff;
  const int Pres = (tot >> 22) & 0x3ff;
  sc.nGs = has_shared ? a.shI / UI : 0;
  sc.nGi = a.I / UI;
  sc.plan(G);
  const int D = sc.D;
  const int nch = H / kKC;        // gate/up jobs (256 columns) per unit
  const int nchd = H / kDnRows;   // down jobs (512 rows) per unit
  // the reduction waits for every consumer warp's share of every unit
  const int target = sc.total * kCW;
  // reduction blocks of kRedBlock float4 outputs: block b is row b / nbr of y,
  // reduced by CTA b mod G (H is a multiple of 512, so a block never spans rows)
  const int nbr = H / (4 * kRedBlock), nblk = T * nbr;

  if (warp == 0) {
    if (lane == 0) {
      // ================= producer (one thread) =================
      fence_proxy_async_shared();  // the top-k scratch in stage memory precedes the TMA writes
      const int j0 = rs.pj;  // the layer's first job
      Producer P{a, sbase, full0, empty0, pub0, s_hdr, s_act_slot, D, a.nst, a.stage_bytes,
                     l2_evict_first_policy(), j0, rs.pui, rs.ppd, j0 % a.nst, (j0 / a.nst) & 1};
      bool ok = true;
      int next = ticket;
      while (ok && !*abort_flag && ticket < sc.total) {
        if (P.ui - P.pd >= kUnitRing) {  // bound the unpublished units
          const long long t0 = cycles_now();
          while (ok && P.ui - P.pd >= kUnitRing) {
            P.wait_pub(1000);
            P.poll();
            if (P.timed_out(t0)) ok = false;
          }
          if (!ok) break;
        }
        const int3 u = sc.unit(ticket);
        ++P.ui;
        next = atomicAdd(a.sync + kSyncQueue, 1);  // needed at the next unit only
        for (int ch = 0; ch < nch && ok; ++ch) {
          ok = P.issue(2 * u.z, u.x, u.y, ch);
          // the layer's first stage lands before the rest of the ring is
          // requested (all SMs ask at once; the consumers start one stage earlier)
          if (ok && P.j == j0 + 1)
            ok = mbar_wait_bounded(full0 + 8 * (j0 % a.nst), (j0 / a.nst) & 1, a.status);
        }
        for (int ch = 0; ch < nchd && ok; ++ch) ok = P.issue(2 * u.z + 1, u.x, u.y, ch);
        ticket = next;
      }
      if (ok) ok = P.issue(J_END, 0, 0, 0);
      // every unit published
      if (ok) {
        const long long t0 = cycles_now();
        for (uint32_t it = 1; ok && P.pd < P.ui; ++it) {
          P.wait_pub(1000);
          P.poll();
          if ((it & 15) == 0 && P.pd < P.ui && P.timed_out(t0)) ok = false;
        }
      }
      if (!ok) *abort_flag = 1;
      // no copy may still be in flight when the CTA exits (bounded)
      for (int jj = P.j - 1; jj >= 0 && jj >= P.j - a.nst; --jj)
        mbar_wait_bounded(full0 + 8 * (jj % a.nst), (jj / a.nst) & 1, a.status);
      rs.pj = P.j;
      rs.pui = P.ui;
      rs.ppd = P.pd;
    }
    __syncwarp();
  } else if (warp == kHelperWarp) {
    // ================= helper: routing weights of the rows this CTA reduces =================
    // softmax over the k selected logits in rank order, one rounding to fp32,
    // into s_rw; the routing of a row goes out from the CTA that reduces its
    // first block. Then the helper arrives at the reduction's barrier.
    if (layer_mode) {
      int prev = -1;
      for (int b = bid; b < nblk; b += G) {
        const int t = b / nbr;
        if (t == prev) continue;
        prev = t;
        const float v = lane < k ? s_rw[t][lane] : 0.f;
        const float wv = topk_softmax_weight(v, k);
        __syncwarp();
        if (lane < k) {
          s_rw[t][lane] = wv;
          if (b == t * nbr) {
            a.ids_out[(size_t)t * k + lane] = s_ids[t][lane];
            a.w_out[(size_t)t * k + lane] = wv;
          }
        }
      }
    }
    __syncwarp();
    // past this barrier the CTA's consumers no longer read the cross-CTA
    // counters and its producer draws no more units: count the CTA out, off
    // the reduction's path (the last CTA resets the counters for the next call)
    named_bar_sync(kBarReduce, kCW * 32 + 32);
    if (count_out && lane == 0 && atomicAdd(a.sync + kSyncDone, 1) == G - 1) {
      a.sync[kSyncUnits] = 0;
      a.sync[kSyncQueue] = 0;
      a.sync[kSyncDone] = 0;
    }
  } else {
    // ================= consumers =================
    const int cw = warp - 1, mw = cw & 3, kh = cw >> 2, ct = tid - 32;
    const int g = lane >> 2, c = lane & 3;
    float* const rw = red + mw * (MT * MAXNT * 4 * 32);  // this row warp's exchange area
    const uint32_t sw = stg_s + cw * (a.TB * kStgRow * 4);  // this warp's partial staging rows
    bool bulk_rd = false;   // this lane's bulk copies may still read its staging rows
    bool bulk_wr = false;   // ... or still be writing the partial buffer
    int pub_bar = -1;       // publish barrier of a unit whose partial copies may be in flight
    // A unit is published once its partial copies are complete (checked one
    // job later, when they have long landed): every consumer lane arrives.
    // Each warp publishes its share with a release add at gpu scope (after
    // its lanes' copies are complete), and tells the producer's unit ring.
    auto publish = [&]() {
      if (pub_bar < 0) return;
      if (bulk_wr) {
        bulk_wait_all();
        fence_proxy_async_global();
        bulk_wr = bulk_rd = false;
      }
      __syncwarp();
      if (lane == 0) red_release_gpu_add(a.sync + kSyncUnits, 1);
      mbar_arrive(pub0 + 8 * pub_bar);
      pub_bar = -1;
    };
    float acc[MT][2][4];
    float accd[kDnM][2][4];
    int browx[2] = {0, 0};  // x box row (token) of token slot nt*8 + g
    int browh[2] = {0, 0};  // h buffer row (slot) of token slot nt*8 + g
    int cnt = 0, ntiles = 1, ucnt = rs.cucnt;
    const int nst = a.nst;
    int slot = rs.cslot, phase = rs.cphase, cslot = rs.ccs;  // ring position of the job being consumed
    for (;;) {
      if (cslot >= 0 && ++slot == nst) {  // advance past the previous job
        slot = 0;
        phase ^= 1;
      }
      cslot = slot;
      if (*abort_flag) break;
      if (!mbar_wait_bounded(full0 + 8 * slot, phase, a.status)) {
        *abort_flag = 1;
        break;
      }
      const int4 hd = s_hdr[slot];
      if (hd.x == J_END) {
        // the stage is released too, for a launch whose next layer reuses it
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);
        publish();
        break;
      }
      const int kind = hd.x, d = hd.y, qi = hd.z, chunk = hd.w;
      const int sz = kind >> 1;               // 0 full, 1 half unit
      const int mta = MT >> sz;               // m16 tiles per row warp in this unit
      const int HB = 64 * mta + 16;           // bytes per token row of the h buffer
      const uint32_t st = sbase + slot * a.stage_bytes;
      uint8_t* hb = hbuf + (ucnt & 1) * (hb_bytes(MT) / 2);
      const uint32_t hbs = smem_u32(hb);
      if ((kind & 1) == 0) {
        if (chunk == 0) {
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int q = 0; q < 4; ++q) acc[m][nt][q] = 0.f;
          const bool sh = d == D;
          cnt = s_act_cnt[d];
          ntiles = cnt > 8 ? 2 : 1;
          const uint32_t mask = sh ? 0u : s_tokmask[s_act_e[d]];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int nb = min(nt * 8 + g, cnt - 1);
            browh[nt] = nb;
            browx[nt] = sh ? nb : nth_bit(mask, nb);
          }
        }
        float(&acc2)[2][2][4] = *reinterpret_cast<float(*)[2][2][4]>(&acc[0]);
        if (sz == 1) {
          if (MAXNT == 1 || ntiles == 1) job_compute<true, 2, 1>(st, mw, kh, a.TB, browx, acc2);
          else job_compute<true, 2, MAXNT>(st, mw, kh, a.TB, browx, acc2);
        } else {
          if (MAXNT == 1 || ntiles == 1) job_compute<true, MT, 1>(st, mw, kh, a.TB, browx, acc);
          else job_compute<true, MT, MAXNT>(st, mw, kh, a.TB, browx, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // this warp is done with the stage
        publish();
        if (chunk != nch - 1) continue;

        // ---- gate/up epilogue: half 1 hands its sums to half 0 (fixed order
        // h0 + h1); h = silu(g) u goes to the unit's shared-memory h buffer
        if (kh == 1) {
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int nt = 0; nt < MAXNT; ++nt)
              if (m < mta && nt < ntiles)
#pragma unroll
                for (int q = 0; q < 4; ++q) rw[((m * MAXNT + nt) * 4 + q) * 32 + lane] = acc[m][nt][q];
        }
        named_bar_sync(1 + mw, 64);
        if (kh == 0) {
#pragma unroll
          for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int nt = 0; nt < MAXNT; ++nt) {
              if (m >= mta || nt >= ntiles) continue;
              float v[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) v[q] = acc[m][nt][q] + rw[((m * MAXNT + nt) * 4 + q) * 32 + lane];
              // v = (g, g, u, u) of unit row il for token slots 2c, 2c+1
              const int il = 8 * (mw * mta + m) + g;
              const int col = (il & ~7) + perm8_pos(il & 7);
#pragma unroll
              for (int e2 = 0; e2 < 2; ++e2) {
                const int n = nt * 8 + 2 * c + e2;
                const float gv = v[e2];
                const float hv = gv / (1.0f + expf(-gv)) * v[2 + e2];
                if (n < cnt && !(fabsf(hv) < 65504.f)) atomicOr(a.status, DEV_RANGE);
                // odd rows of I meet high nibbles in the down MMA: stored as h / 16
                *reinterpret_cast<__half*>(hb + n * HB + 2 * col) = __float2half_rn((il & 1) ? hv * 0.0625f : hv);
              }
            }
        }
        named_bar_sync(5, kCW * 32);  // h is complete; the exchange area is free again
        continue;
      }

      // ---- down job: 512 output rows of this unit's columns of I. This warp's
      // 64 rows for the tokens < cnt are staged as [n][kStgRow] f32, then go
      // to the partial buffer by one 256-byte bulk copy per token. A full unit
      // sums A (blocks 0-1) and B (blocks 2-3) separately and stages A + B.
      auto zero_acc = [&]() {
#pragma unroll
        for (int m = 0; m < kDnM; ++m)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) accd[m][nt][q] = 0.f;
      };
      auto stage_out = [&]() {
        if (bulk_rd) {  // the previous job's copies have read the staging rows
          bulk_wait_read_all();
          bulk_rd = false;
        }
        __syncwarp();
#pragma unroll
        for (int m = 0; m < kDnM; ++m)
#pragma unroll
          for (int nt = 0; nt < MAXNT; ++nt) {
            if (nt >= ntiles) continue;
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int n = nt * 8 + 2 * c + e2;
              if (n < cnt) {
                const uint32_t o = sw + (uint32_t)(n * kStgRow + 16 * m + g) * 4u;
                st_s_f32(o, accd[m][nt][e2]);
                st_s_f32(o + 32, accd[m][nt][2 + e2]);
              }
            }
          }
      };
      const int boff = qi & 7;
      const bool nt1 = MAXNT == 1 || ntiles == 1;
      zero_acc();
      if (sz == 0) {
        float accb[kDnM][2][4];
#pragma unroll
        for (int m = 0; m < kDnM; ++m)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) accb[m][nt][q] = 0.f;
        if (nt1) {
          dn_compute<MT, 1, 0, 2>(st, hbs, cw, boff, browh, accd);
          dn_compute<MT, 1, 2, 2>(st, hbs, cw, boff, browh, accb);
        } else {
          dn_compute<MT, MAXNT, 0, 2>(st, hbs, cw, boff, browh, accd);
          dn_compute<MT, MAXNT, 2, 2>(st, hbs, cw, boff, browh, accb);
        }
#pragma unroll
        for (int m = 0; m < kDnM; ++m)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) accd[m][nt][q] += accb[m][nt][q];
      } else {  // half unit: A or B of its group
        if (nt1) dn_compute<2, 1, 0, 2>(st, hbs, cw, boff, browh, accd);
        else dn_compute<2, MAXNT, 0, 2>(st, hbs, cw, boff, browh, accd);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
      publish();
      {
        stage_out();
        fence_proxy_async_shared();
        __syncwarp();
        if (lane < cnt && !*abort_flag) {
          float* dst = a.partial + ((size_t)(s_act_off[d] + lane) * a.Gh + (qi >> 1)) * H + chunk * kDnRows + 64 * cw;
          bulk_s2g(dst, sw + (uint32_t)(lane * kStgRow) * 4u, 256);
          bulk_commit();
          bulk_rd = bulk_wr = true;
        }
      }
      if (chunk == nchd - 1) {
        pub_bar = ucnt % kPubBars;
        ++ucnt;
      }
    }

    if (bulk_wr) bulk_wait_all();

    // ---- reduction, once every unit of the window is published. Lane q of an
    // 8-lane group sums, for one output float4,
    //   v_q = sum_{j = q, q+8, ..} w_tj sum_g n(e_tj, g)[t] + sum_{g = q, q+8, ..} n(shared, g)[t]
    // (g in order; n the group's down partial, A + B from its halves if it was split),
    // and y = v_0 + ... + v_7 in lane order: a fixed order on every CTA, for any
    // window and any split.
    // One thread decides for all (the abort flag may still change meanwhile),
    // and every consumer and the helper meet at the barrier unconditionally.
    if (ct == 0) {
      bool go = !*abort_flag;
      if (go && !wait_counter_bounded(a.sync + kSyncUnits, target, a.status)) {
        *abort_flag = 1;
        go = false;
      }
      s_reduce = go ? 1 : 0;
    }
    named_bar_sync(kBarReduce, kCW * 32 + 32);
    // every consumer thread holds the same ring position; all of them have
    // read the layer's start position before this barrier
    if (ct == 0) {
      rs.cslot = slot;
      rs.cphase = phase;
      rs.ccs = cslot;
      rs.cucnt = ucnt;
    }
    {
      if (s_reduce) {
        const int q = ct & 7, H4 = H / 4, NO = T * H4;
        const size_t gstride = (size_t)a.Gh * H;
        for (int o0 = bid * kRedBlock; o0 < NO; o0 += G * kRedBlock) {
          const int o = o0 + (ct >> 3);
          const bool live = o < NO;
          const int t = live ? o / H4 : 0, col = live ? (o - t * H4) * 4 : 0;
          float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
          if (live) {
            // the first shared-expert group of this lane, in flight with the routed loads
            const float* psh = a.partial + (size_t)(Pres + t) * gstride + col;
            const float4 u0 = has_shared && q < sc.nGs ? ldg_cg_f4(psh + (size_t)(2 * q) * H) : make_float4(0.f, 0.f, 0.f, 0.f);
            for (int jj = q; jj < k; jj += 8) {
              const int e = s_ids[t][jj];
              const int dd = s_d_of_e[e];
              if (dd < 0) continue;
              const int pos = s_act_off[dd] + __popc(s_tokmask[e] & ((1u << t) - 1u));
              const float wv = layer_mode ? s_rw[t][jj] : a.w_in[(size_t)t * k + jj];
              const float* pp = a.partial + (size_t)pos * gstride + col;
              float4 sacc = make_float4(0.f, 0.f, 0.f, 0.f);
              for (int g0 = 0; g0 < sc.nGi; g0 += 8) {  // 8 groups' loads in flight
                float4 pv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  pv[u] = g0 + u < sc.nGi ? ldg_cg_f4(pp + (size_t)(2 * (g0 + u)) * H) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < 8; ++u)
                  if (g0 + u < sc.nGi && sc.group_index(dd, g0 + u) >= sc.nfull)
                    pv[u] = add4(pv[u], ldg_cg_f4(pp + (size_t)(2 * (g0 + u) + 1) * H));
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                  sacc.x += pv[u].x; sacc.y += pv[u].y; sacc.z += pv[u].z; sacc.w += pv[u].w;
                }
              }
              v.x = fmaf(wv, sacc.x, v.x); v.y = fmaf(wv, sacc.y, v.y);
              v.z = fmaf(wv, sacc.z, v.z); v.w = fmaf(wv, sacc.w, v.w);
            }
            if (has_shared && q < sc.nGs) {
              for (int gg = q; gg < sc.nGs; gg += 8) {
                float4 u4 = gg == q ? u0 : ldg_cg_f4(psh + (size_t)(2 * gg) * H);
                if (sc.group_index(D, gg) >= sc.nfull) u4 = add4(u4, ldg_cg_f4(psh + (size_t)(2 * gg + 1) * H));
                v.x += u4.x; v.y += u4.y; v.z += u4.z; v.w += u4.w;
              }
            }
          }
          // lanes q = 0..7 of the group, summed in lane order
          float4 y4 = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int s2 = 0; s2 < 8; ++s2) {
            y4.x += __shfl_sync(0xffffffffu, v.x, (lane & ~7) + s2);
            y4.y += __shfl_sync(0xffffffffu, v.y, (lane & ~7) + s2);
            y4.z += __shfl_sync(0xffffffffu, v.z, (lane & ~7) + s2);
            y4.w += __shfl_sync(0xffffffffu, v.w, (lane & ~7) + s2);
          }
          if (live && q == 0) {
            float* yp = a.y + (size_t)t * H + col;
            yp[0] = y4.x; yp[1] = y4.y; yp[2] = y4.z; yp[3] = y4.w;
            if (a.x_next) {  // the next layer's input: bf16(x + y), each sum in fp32
              const uint2 xv = __ldcg(reinterpret_cast<const uint2*>(a.xg + (size_t)t * H + col));
              const float s0 = bf16_to_f((uint16_t)(xv.x & 0xffffu)) + y4.x;
              const float s1 = bf16_to_f((uint16_t)(xv.x >> 16)) + y4.y;
              const float s2 = bf16_to_f((uint16_t)(xv.y & 0xffffu)) + y4.z;
              const float s3 = bf16_to_f((uint16_t)(xv.y >> 16)) + y4.w;
              uint2 o;
              o.x = (uint32_t)bf16_bits(s0) | ((uint32_t)bf16_bits(s1) << 16);
              o.y = (uint32_t)bf16_bits(s2) | ((uint32_t)bf16_bits(s3) << 16);
              *reinterpret_cast<uint2*>(a.x_next + (size_t)t * H + col) = o;
            }
          }
        }
      }
    }
  }
  // a launch of several layers learns here whether this CTA gave up
  if (count_out) return false;
  __syncthreads();
  return *abort_flag != 0;
}

// One window (T <= 16 rows) of one layer per launch.
template <int MAXNT>
__global__ void __launch_bounds__(kThreads, 1) decode_layer_kernel(const __grid_constant__ Args a) {
  RingState rs = {0, 0, 0, 0, 0, -1, 0};
  layer_body<MAXNT>(a, rs, true, true);
}

// Several layers in one launch, one window each (the whole decode pass in one
// call, as the SGLang port post's section 3 captures it in one graph): layer l
// is layer_body on plan[l] (the arguments in global memory, tensor maps
// 64-byte aligned; its cross-CTA counters at plan[l].sync), then a grid-wide
// barrier, so that no CTA starts layer l + 1's routing before every CTA has
// finished layer l (its output written, its partials read). The CTAs keep
// their barrier ring, shared memory and descriptors from layer to layer. One
// CTA per SM, all resident (a cooperative launch); every wait is bounded: a
// CTA that gave up, or a barrier that timed out, ends the launch after the
// layer (the status word says which).
// The router of a chained stack: logits[t][e] = sum_h x[t][h] * W_r[e][h],
// bf16 operands (products exact in fp32), fp32 sums in a fixed order: lane j
// of a warp takes h = 8 j .. 8 j + 7 (mod 256) in increasing h (one fma
// chain), then the 32 lane sums meet in the tree (a, a ^ 16), ..., (a, a ^ 1). CTA b computes the
// experts b, b + G, ...; its warps take the (expert, row) pairs in turn.
__device__ __forceinline__ void router_gemv(const Args& a, int G, int bid) {
  const int T = a.T, E = a.E, H = a.H;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (bid >= E) return;
  const int ne = (E - bid + G - 1) / G;
  for (int pi = warp; pi < ne * T; pi += kWarps) {
    const int e = bid + (pi / T) * G, t = pi - (pi / T) * T;
    const uint16_t* wr = a.router_w + (size_t)e * H;
    const uint16_t* xr = a.xg + (size_t)t * H;
    float s = 0.f;
    for (int hb = lane * 8; hb < H; hb += 8 * 256) {  // 8 steps' loads in flight together
      uint4 wv[8], xv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
        xv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (hb + 256 * u < H) {
          wv[u] = __ldg(reinterpret_cast<const uint4*>(wr + hb + 256 * u));
          // written in this launch by the layer before: read from L2
          xv[u] = __ldcg(reinterpret_cast<const uint4*>(xr + hb + 256 * u));
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (hb + 256 * u >= H) continue;
        const uint32_t wa[4] = {wv[u].x, wv[u].y, wv[u].z, wv[u].w};
        const uint32_t xa[4] = {xv[u].x, xv[u].y, xv[u].z, xv[u].w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s = fmaf(bf16_to_f((uint16_t)(xa[i] & 0xffffu)), bf16_to_f((uint16_t)(wa[i] & 0xffffu)), s);
          s = fmaf(bf16_to_f((uint16_t)(xa[i] >> 16)), bf16_to_f((uint16_t)(wa[i] >> 16)), s);
        }
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == 0) const_cast<float*>(a.logits)[(size_t)t * E + e] = s;
  }
}

constexpr int kStackBar = 96, kStackAbort = 97, kStackDone = 98;
constexpr int kStackBase = 128, kStackStride = 32;  // layer l's counters: sync + base + stride l

template <int MAXNT>
__global__ void __launch_bounds__(kThreads, 1)
decode_stack_kernel(const Args* __restrict__ plan, int L, int T, int nst,
                    int32_t* __restrict__ sync, int32_t* __restrict__ status) {
  __shared__ int s_stop;
  // the launch's layer count, rows, row tile, ring depth and workspace must be
  // the plan's (its shared-memory layout and counters are the plan's): else
  // nothing runs and the status word of the launch's workspace says so
  {
    const Args& p0 = plan[0];
    if (p0.stack_L != L || p0.T != T || p0.TB != (MAXNT == 1 ? 8 : 16) || p0.nst != nst ||
        p0.status != status) {
      if (threadIdx.x == 0 && blockIdx.x == 0) atomicOr(status, DEV_PLAN);
      return;
    }
  }
  // the ring state lives in shared memory between layers (each role reads it
  // at a layer's start and its owner writes it back at the end), so that no
  // register is held across the layers
  __shared__ RingState s_rs;
  if (threadIdx.x == 0) s_rs = RingState{0, 0, 0, 0, 0, -1, 0};
  __syncthreads();
  RingState& rs = s_rs;
  const int G = gridDim.x;
  const bool routed = plan[0].router_w != nullptr;  // chained layers, router in the launch
  int nbar = 0;  // grid barriers passed
  for (int l = 0; l < L; ++l) {
    if (routed) {
      // the router of layer l on its input (the caller's x for l = 0, else the
      // x_next the layer before wrote), then a barrier that publishes the logits
      if (l == 0) griddep_wait();
      router_gemv(plan[l], G, blockIdx.x);
      __syncthreads();
      if (threadIdx.x == 0) {
        red_release_gpu_add(sync + kStackBar, 1);
        s_stop = wait_counter_bounded(sync + kStackBar, (++nbar) * G, status) ? 0 : 1;
      }
      __syncthreads();
      if (s_stop) break;
    }
    const bool aborted = layer_body<MAXNT>(plan[l], rs, l == 0, false);
    if (threadIdx.x == 0) {
      // the next layer's descriptors, fetched while the barrier completes
      if (l + 1 < L) {
        const Args& n = plan[l + 1];
        const CUtensorMap* maps[] = {&n.tm_gc, &n.tm_uc, &n.tm_dc, &n.tm_gs, &n.tm_us, &n.tm_ds, &n.tm_x,
                                     &n.tm_gch, &n.tm_uch, &n.tm_dch, &n.tm_gsh, &n.tm_ush};
        for (const CUtensorMap* m : maps) prefetch_tensormap(m);
      }
      // unchained layers: a relaxed arrival, since nothing of layer l + 1
      // reads what layer l wrote in this launch (its y goes out at the
      // kernel's end; its partials were read into registers before the CTA
      // got here); an abort flag is ordered before the arrival that announces it
      if (aborted) {
        atomicOr(sync + kStackAbort, 1);
        __threadfence();
      }
      // chained layers: layer l's x_next is read by every CTA after this
      // barrier (generic loads, and the TMA of the next layer's x boxes)
      int stop;
      if (routed) {
        red_release_gpu_add(sync + kStackBar, 1);
        stop = wait_counter_bounded(sync + kStackBar, (++nbar) * G, status) ? 0 : 1;
        fence_proxy_async_global();
      } else {
        atomicAdd(sync + kStackBar, 1);
        stop = wait_counter_relaxed(sync + kStackBar, (++nbar) * G, status) ? 0 : 1;
      }
      if (ld_acquire_gpu(sync + kStackAbort)) stop = 1;
      s_stop = stop;
    }
    __syncthreads();
    if (s_stop) break;
  }
  // count out; the last CTA resets every counter the launch used
  if (threadIdx.x == 0 && atomicAdd(sync + kStackDone, 1) == G - 1) {
    for (int l = 0; l < L; ++l) {
      sync[kStackBase + kStackStride * l + kSyncUnits] = 0;
      sync[kStackBase + kStackStride * l + kSyncQueue] = 0;
    }
    sync[kStackBar] = 0;
    sync[kStackAbort] = 0;
    sync[kStackDone] = 0;
  }
}

}  // namespace fused

// Host side -------------------------------------------------------------------
// SM count of the current device (cached per device: the grid is one CTA per SM).
static int num_sms() {
  constexpr int kMaxDev = 64;
  static int n_of[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  if (dev < 0 || dev >= kMaxDev) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 1;
  }
  int n = __atomic_load_n(&n_of[dev], __ATOMIC_RELAXED);
  if (n == 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 1;
    }
    __atomic_store_n(&n_of[dev], n, __ATOMIC_RELAXED);
  }
  return n;
}

namespace {
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
// swz_bytes: the swizzle span (128, 64 or 32 bytes), anything else for none.
bool tensor_map(CUtensorMap* out, CUtensorMapDataType dt, const void* ptr, int rank,
                const uint64_t* dims, const uint64_t* strides, const uint32_t* box, int swz_bytes) {
  static std::mutex mu;
  static std::unordered_map<MapKey, CUtensorMap, MapKeyHash> cache;
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.ptr = ptr;
  key.d0 = dims[0]; key.d1 = dims[1]; key.d2 = rank > 2 ? dims[2] : 0;
  key.s1 = strides[0]; key.s2 = rank > 2 ? strides[1] : 0;
  key.b0 = box[0]; key.b1 = box[1]; key.b2 = rank > 2 ? box[2] : 0;
  key.dtype = (uint32_t)dt;
  key.swz = (uint32_t)swz_bytes;
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
                  swz_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                  : swz_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                  : swz_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                    : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return true;
}

// Codes [rows][K/2] bytes: box box_bytes x box_rows, swizzled by the box's row
// width (128, 64 or 32 bytes; 16-byte rows need none).
bool codes_map(CUtensorMap* m, const uint8_t* q, int K, int rows, int box_bytes, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)rows};
  const uint64_t str[1] = {(uint64_t)K / 2};
  const uint32_t box[2] = {(uint32_t)box_bytes, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, 2, dims, str, box, box_bytes);
}
// Scales [rows][K/32] fp16: box 8 (256 columns) x box_rows, no swizzle.
bool scales_map(CUtensorMap* m, const uint16_t* s, int K, int rows, int box_rows) {
  const uint64_t dims[2] = {(uint64_t)K / 32, (uint64_t)rows};
  const uint64_t str[1] = {(uint64_t)K / 16};
  const uint32_t box[2] = {8, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, 2, dims, str, box, 16);
}
// 16-bit activations [rows][cols]: viewed as (64, cols/64, rows); box (64, 4, box_rows).
bool act_map(CUtensorMap* m, const void* p, int cols, int rows, int box_rows) {
  const uint64_t dims[3] = {64, (uint64_t)cols / 64, (uint64_t)rows};
  const uint64_t str[2] = {128, (uint64_t)cols * 2};
  const uint32_t box[3] = {64, 4, (uint32_t)box_rows};
  return tensor_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, p, 3, dims, str, box, 128);
}
}  // namespace


static int box_rows(int T) { return T <= 8 ? 8 : 16; }

// Slices of I per partial row of the one-launch path: one per 64 intermediate
// columns (a full unit writes every second, a half unit its own).
int fused_partial_slices(int E, int k, int T, int I, int shI) {
  (void)E; (void)k; (void)T;
  return (I > shI ? I : shI) / 64;
}

// STACK: the kernel of several layers per launch (else one layer per launch).
template <int NTX, bool STACK = false>
static cudaError_t kernel_attrs(size_t* static_smem, int* optin) {
  static std::mutex mu;
  static size_t st = 0;
  static int opt = 0;
  std::lock_guard<std::mutex> lk(mu);
  if (opt == 0) {
    cudaFuncAttributes fa;
    cudaError_t e = STACK ? cudaFuncGetAttributes(&fa, fused::decode_stack_kernel<NTX>)
                          : cudaFuncGetAttributes(&fa, fused::decode_layer_kernel<NTX>);
    if (e != cudaSuccess) return e;
    int dev = 0, o = 0;
    e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&o, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    st = fa.sharedSizeBytes;
    opt = o;
  }
  *static_smem = st;
  *optin = opt;
  return cudaSuccess;
}

// Stages that fit next to the kernel's static shared memory (0: not even two).
template <int NTX, bool STACK = false>
static int stages_for(int TB) {
  constexpr int MT = fused::kMT;
  size_t st = 0;
  int optin = 0;
  if (kernel_attrs<NTX, STACK>(&st, &optin) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  const int stage = fused::stage_bytes_for(MT, TB);
  int n = fused::kMaxNst;
  while (n >= 2 && fused::smem_bytes(MT, NTX, n, stage, TB) + st > (size_t)optin) --n;
  // the routing's scratch and the slot map's copy live in the stages
  if ((size_t)n * stage < (size_t)fused::kSlotMapOff + 4 * kMaxE) return 0;
  return n >= 2 ? n : 0;
}

bool fused_decode_supported(int H, int I, int shI, int T, bool x_bf16) {
  if (!x_bf16 || T < 1 || T > fused::kMaxT) return false;
  if (H % fused::kDnRows || I % 256 || shI % 256) return false;
  if (H > 8192 || T > num_sms()) return false;
  if (!encode_fn()) return false;
  const int TB = box_rows(T);
  return TB == 8 ? stages_for<1>(TB) >= 2 : stages_for<2>(TB) >= 2;
}

template <int NTX>
static cudaError_t launch_nt(fused::Args& a, cudaStream_t st) {
  constexpr int MT = fused::kMT;
  a.stage_bytes = fused::stage_bytes_for(MT, a.TB);
  a.nst = stages_for<NTX>(a.TB);
  if (a.nst < 2) return cudaErrorInvalidValue;
  const size_t smem = fused::smem_bytes(MT, NTX, a.nst, a.stage_bytes, a.TB);
  // the shared-memory opt-in is a per-device attribute of the function
  static std::mutex mu;
  static size_t configured[64] = {};
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
      cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (smem > configured[dev]) {
      e = cudaFuncSetAttribute(fused::decode_layer_kernel<NTX>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
      }
      configured[dev] = smem;
    }
  }
  // programmatic dependent launch: the kernel's set-up overlaps the end of the
  // previous kernel in the stream (the kernel waits for it before reading)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(fused::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  launch_begin(K_FUSED, st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, fused::decode_layer_kernel<NTX>, a);
  launch_end(st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// The kernel arguments of one layer's window (tensor maps encoded on the host).
static bool build_args(const FusedLaunch& f, fused::Args& a) {
  const int TB = box_rows(f.T);
  const int UI = fused::kUI, HI = fused::kUI / 2, DR = 256;  // down boxes of 256 rows
  std::memset(&a, 0, sizeof a);
  a.H = f.H; a.I = f.I; a.shI = f.shI; a.E = f.E; a.k = f.k; a.S = f.S; a.T = f.T;
  a.Gh = fused_partial_slices(f.E, f.k, f.T, f.I, f.shI);
  a.TB = TB;
  a.rows_cap = f.rows_cap;
  const int H = f.H, I = f.I, S = f.S;
  bool ok = codes_map(&a.tm_gc, f.gq, H, S * I, 128, UI) &&
            codes_map(&a.tm_uc, f.uq, H, S * I, 128, UI) &&
            codes_map(&a.tm_dc, f.dq, I, S * H, UI / 2, DR) &&
            scales_map(&a.tm_gs, f.gs, H, S * I, UI) &&
            scales_map(&a.tm_us, f.us, H, S * I, UI) &&
            scales_map(&a.tm_ds, f.ds, I, S * H, DR) &&
            codes_map(&a.tm_gch, f.gq, H, S * I, 128, HI) &&
            codes_map(&a.tm_uch, f.uq, H, S * I, 128, HI) &&
            codes_map(&a.tm_dch, f.dq, I, S * H, HI / 2, DR) &&
            scales_map(&a.tm_gsh, f.gs, H, S * I, HI) &&
            scales_map(&a.tm_ush, f.us, H, S * I, HI) &&
            act_map(&a.tm_x, f.x, H, f.T, TB);
  if (ok && f.shI > 0)
    ok = codes_map(&a.tm_sgc, f.sgq, H, f.shI, 128, UI) &&
         codes_map(&a.tm_suc, f.suq, H, f.shI, 128, UI) &&
         codes_map(&a.tm_sdc, f.sdq, f.shI, H, UI / 2, DR) &&
         scales_map(&a.tm_sgs, f.sgs, H, f.shI, UI) &&
         scales_map(&a.tm_sus, f.sus, H, f.shI, UI) &&
         scales_map(&a.tm_sds, f.sds, f.shI, H, DR) &&
         codes_map(&a.tm_sgch, f.sgq, H, f.shI, 128, HI) &&
         codes_map(&a.tm_such, f.suq, H, f.shI, 128, HI) &&
         codes_map(&a.tm_sdch, f.sdq, f.shI, H, HI / 2, DR) &&
         scales_map(&a.tm_sgsh, f.sgs, H, f.shI, HI) &&
         scales_map(&a.tm_sush, f.sus, H, f.shI, HI);
  if (!ok) return false;
  a.logits = f.logits; a.ids_in = f.ids_in; a.w_in = f.w_in;
  a.slot_map = f.slot_map;
  a.ids_out = f.ids_out; a.w_out = f.w_out; a.y = f.y;
  a.miss_ids = f.miss_ids; a.n_miss = f.n_miss;
  a.partial = f.partial;
  a.status = f.status; a.sync = f.sync;
  a.picks = f.picks;
  a.router_w = f.router_w;
  a.xg = static_cast<const uint16_t*>(f.x);
  a.x_next = f.x_next;
  return true;
}

cudaError_t launch_fused_decode(const FusedLaunch& f, cudaStream_t st) {
  fused::Args a;
  if (!build_args(f, a)) return cudaErrorInvalidValue;
  return a.TB == 8 ? launch_nt<1>(a, st) : launch_nt<2>(a, st);
}

// ---- several layers per launch
size_t fused_stack_plan_bytes(int L) { return L > 0 ? (size_t)L * sizeof(fused::Args) : 0; }
int fused_stack_max_layers() {
  return (kSyncInts - fused::kStackBase) / fused::kStackStride;
}

cudaError_t fused_stack_prepare(const FusedLaunch* layers, int L, void* plan, cudaStream_t st) {
  if (L < 1 || L > fused_stack_max_layers() || !plan) return cudaErrorInvalidValue;
  const int TB = box_rows(layers[0].T);
  const int nst = TB == 8 ? stages_for<1, true>(TB) : stages_for<2, true>(TB);
  if (nst < 2) return cudaErrorInvalidValue;
  std::vector<fused::Args> h((size_t)L);
  for (int l = 0; l < L; ++l) {
    fused::Args& a = h[(size_t)l];
    std::memset(&a, 0, sizeof a);
    FusedLaunch f = layers[l];
    f.sync = layers[0].sync + fused::kStackBase + fused::kStackStride * l;
    if (f.T != layers[0].T || !build_args(f, a)) return cudaErrorInvalidValue;
    a.stage_bytes = fused::stage_bytes_for(fused::kMT, a.TB);
    a.nst = nst;
    a.stack_L = L;
  }
  cudaError_t e = cudaMemcpyAsync(plan, h.data(), h.size() * sizeof(fused::Args),
                                  cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);  // the host copy goes out of scope
  return e;
}

template <int NTX>
static cudaError_t launch_stack_nt(const fused::Args* plan, int L, int T, int TB, int nst,
                                   int32_t* sync, int32_t* status, cudaStream_t st) {
  constexpr int MT = fused::kMT;
  const size_t smem = fused::smem_bytes(MT, NTX, nst, fused::stage_bytes_for(MT, TB), TB);
  static std::mutex mu;
  static size_t configured[64] = {};
  {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
      cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (smem > configured[dev]) {
      e = cudaFuncSetAttribute(fused::decode_stack_kernel<NTX>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
      }
      configured[dev] = smem;
    }
  }
  // every CTA waits for every other at each layer's barrier: a cooperative
  // launch, which fails at launch instead of waiting when they cannot all be resident
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_sms());
  cfg.blockDim = dim3(fused::kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  launch_begin(K_FUSED_STACK, st);
  cudaError_t e = cudaLaunchKernelEx(&cfg, fused::decode_stack_kernel<NTX>, plan, L, T, nst, sync,
                                     status);
  launch_end(st);
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_fused_stack(const void* plan, int L, int T, int32_t* sync, int32_t* status,
                               cudaStream_t st) {
  if (L < 1 || L > fused_stack_max_layers() || !plan || T < 1 || T > fused::kMaxT)
    return cudaErrorInvalidValue;
  const int TB = box_rows(T);
  const int nst = TB == 8 ? stages_for<1, true>(TB) : stages_for<2, true>(TB);
  if (nst < 2) return cudaErrorInvalidValue;
  const fused::Args* p = static_cast<const fused::Args*>(plan);
  return TB == 8 ? launch_stack_nt<1>(p, L, T, TB, nst, sync, status, st)
                 : launch_stack_nt<2>(p, L, T, TB, nst, sync, status, st);
}

}  // namespace moe
