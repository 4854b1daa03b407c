// Shared device helpers of the sm_103a routed-expert FFN library.
//
// Inline PTX wrappers (mbarrier, bulk async copy, warp MMA, LOP3), the
// workspace layout and the device-status bits. Written for sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------- status bits
// Device-detected problems are OR-ed into the workspace status word; kernels
// never trap. moe_read_status() maps them back to moe_status codes.
enum : int32_t {
  DEV_NONFINITE_LOGIT = 1,   // a router logit was NaN or infinite
  DEV_BAD_SLOT = 2,          // slot_map[e] >= S (treated as not resident)
  DEV_TIMEOUT = 4,           // a bounded wait expired
  DEV_RANGE = 8,             // an activation outside the fp16 range (prefill path)
  DEV_PLAN = 16,             // a stack launch whose layers or rows differ from its plan's
};

constexpr int kMaxK = 32;
constexpr int kMaxE = 1024;
constexpr int kTokTile = 16;          // token slots per decode unit (two n8 MMA tiles)
constexpr int kRowTile = 16;          // weight rows per decode unit (one m16 MMA tile)
constexpr int kWarps = 8;             // warps per decode CTA (split K)
constexpr float kMagic = 136.0f;      // bf16 0x4300|n' = 128 + (q ^ 8) = 136 + q

// ---------------------------------------------------------------- workspace
// All offsets are 256-byte aligned. The layout depends only on (desc, T).
// The first kWsHeadBytes hold the status word, counters and the fused kernel's
// cross-CTA counters; moe_workspace_init zeroes exactly this head.
constexpr size_t kWsHeadBytes = 512 + 16384;
constexpr int kSyncInts = 4096;  // cross-CTA counters of the fused decode kernel

struct WsLayout {
  size_t status, counters, sync, offsets, sorted_pair, pair_pos, act, cu, hist;
  size_t xhi, xlo, xcorr, hhi, hlo, hsum, partial, total;
  int P, Imax, n_chunks, cu_max;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Per-active-expert record written by the permutation for the FFN kernels.
struct ActExpert {
  int32_t e;      // expert id (-1 for the shared expert)
  int32_t slot;   // pool slot (-1 for the shared expert)
  int32_t off;    // first row of this expert in the h / partial buffers
  int32_t cnt;    // rows routed to it
};

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// Bulk async copy global -> this CTA's shared memory, completing on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Time bound of every wait: about a second of SM clock cycles. The SM's own
// cycle counter is read in a few cycles (the global timer takes far longer),
// so a wait costs nothing when it does not have to wait.
constexpr long long kWaitCycles = 2000000000ll;
__device__ __forceinline__ long long cycles_now() { return clock64(); }

// Wait for phase `parity` of `bar`, giving up after about a second: then the
// status word gets DEV_TIMEOUT and the caller skips its work. Returns true on success.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  int32_t* status) {
  long long t0 = 0;
  for (uint32_t it = 0;; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (it == 0) t0 = cycles_now();
    else if ((it & 63) == 0 && cycles_now() - t0 > kWaitCycles) {
      if (status) atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

// Non-blocking test of phase `parity` of `bar` (true once that phase completed).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// 4-byte asynchronous copy global -> shared (completes at cp_async_wait_all).
__device__ __forceinline__ void cp_async_4(void* smem_dst, const void* gsrc) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(smem_dst)), "l"(gsrc)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Fetch a TMA descriptor (kernel parameter) ahead of its first use.
__device__ __forceinline__ void prefetch_tensormap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Programmatic dependent launch: let the stream's next kernel be scheduled;
// wait until the stream's previous kernel has completed (and its writes are visible).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Wait (suspended, up to about `ns` nanoseconds) for phase `parity` of `bar`;
// true once that phase completed. Leaves the issue slots to the other warps.
__device__ __forceinline__ bool mbar_try_wait_ns(uint32_t bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Bounded wait that sleeps in the barrier (up to ~hint_ns per try) instead of
// spinning: for warps that wait often, so that waiting leaves the issue slots
// to the warps that compute. Gives up after about a second (DEV_TIMEOUT).
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity, int32_t* status,
                                                uint32_t hint_ns = 1000) {
  if (mbar_try_wait_ns(bar, parity, hint_ns)) return true;
  const long long t0 = cycles_now();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_ns(bar, parity, hint_ns)) return true;
    if ((it & 15) == 0 && cycles_now() - t0 > kWaitCycles) {
      if (status) atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

// Bounded wait with a short sleep per try (for waits on fast pipeline stages).
__device__ __forceinline__ bool mbar_wait_short(uint32_t bar, uint32_t parity, int32_t* status) {
  return mbar_wait_sleep(bar, parity, status, 128);
}

// ---------------------------------------------------------------- top-k
__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t u = __float_as_uint(v);
  if ((u << 1) == 0) u = 0;  // -0 and +0 are equal logits: same key
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
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

// ---------------------------------------------------------------- routing weights
// Float-float numbers: an unevaluated sum h + l of two fp32 values (|l| at most
// half an ulp of h), about 48 significant bits. The error-free sum and product
// (Knuth's two-sum, Dekker's fast two-sum, the product error from one fused
// multiply-add) and the composite add and multiply follow the double-double
// algorithms of Hida, Li and Bailey ("Library for double-double and
// quad-double arithmetic", 2007), carried over to fp32 pairs.
struct FF {
  float h, l;
};
__device__ __forceinline__ FF ff_two_sum(float a, float b) {
  const float s = a + b, bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
__device__ __forceinline__ FF ff_fast_two_sum(float a, float b) {  // |a| >= |b| (or a = 0)
  const float s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ FF ff_add(FF a, FF b) {
  FF s = ff_two_sum(a.h, b.h);
  const FF t = ff_two_sum(a.l, b.l);
  s.l += t.h;
  s = ff_fast_two_sum(s.h, s.l);
  s.l += t.l;
  return ff_fast_two_sum(s.h, s.l);
}
__device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = a.h * b.h;
  float e = fmaf(a.h, b.h, -p);
  e = fmaf(a.h, b.l, e);
  e = fmaf(a.l, b.h, e);
  return ff_fast_two_sum(p, e);
}

// exp(d) = E * 2^n for a float-float d <= 0 with d.h >= -80: n = round(d / ln 2),
// r = d - n ln 2 with ln 2 = L1 + L2 + L3 (L1 holds 17 significant bits, so n L1
// is exact; |r| <= ln2 / 2 + tiny), and E = the Taylor series of exp(r) to
// degree 12 (truncation below 2^-52 for |r| <= 0.35): the terms from r^9 on in
// fp32, the rest by float-float Horner steps. Coefficients: 1/i! split into
// two fp32 values.
__device__ __forceinline__ FF ff_exp_scaled(FF d, int& n_out) {
  constexpr float kL1 = 0x1.62e4p-1f, kL2 = 0x1.7f7d1cp-20f, kL3 = 0x1.ef357ap-45f;
  constexpr float kLog2e = 0x1.715476p+0f;
  const float n = rintf(d.h * kLog2e);
  const float t = fmaf(-n, kL1, d.h);  // exact: n L1 is exact and close to d.h
  FF r = ff_two_sum(t, d.l);
  const float p2 = -n * kL2;
  r = ff_add(r, FF{p2, fmaf(-n, kL2, -p2)});
  r = ff_add(r, FF{-n * kL3, 0.f});
  constexpr float ch[9] = {1.f, 1.f, 0x1p-1f, 0x1.555556p-3f, 0x1.555556p-5f, 0x1.111112p-7f,
                           0x1.6c16c2p-10f, 0x1.a01a02p-13f, 0x1.a01a02p-16f};
  constexpr float cl[9] = {0.f, 0.f, 0.f, -0x1.555556p-28f, -0x1.555556p-30f, -0x1.dddddep-32f,
                           -0x1.27d27ep-35f, -0x1.7f97fap-39f, -0x1.7f97fap-42f};
  float tail = 0x1.1eed8ep-29f;  // 1/12!
  tail = fmaf(tail, r.h, 0x1.ae6456p-26f);  // 1/11!
  tail = fmaf(tail, r.h, 0x1.27e4fcp-22f);  // 1/10!
  tail = fmaf(tail, r.h, 0x1.71de3ap-19f);  // 1/9!
  FF acc{tail, 0.f};
#pragma unroll
  for (int i = 8; i >= 0; --i) acc = ff_add(ff_mul(acc, r), FF{ch[i], cl[i]});
  n_out = (int)n;
  return acc;
}

// Softmax over the k selected logits of one row, one warp: lane j < k holds
// logit v_j in rank order (v_0 the largest) and receives
//   w_j = fp32( exp(v_j - v_0) / sum_{i < k} exp(v_i - v_0) ),  the sum in i order,
// the reference evaluated in float64. Here in float-float, to about 2^-42
// relative, so the one rounding to fp32 agrees with float64 except for values
// within that distance of an fp32 rounding midpoint (float64 itself is slow on
// this GPU). Rows with a difference below -80 (a weight near fp32 underflow) or
// a non-finite logit take the float64 evaluation. Call with all 32 lanes.
__device__ __forceinline__ float topk_softmax_weight_f64(float v, int k) {
  const int lane = threadIdx.x & 31;
  const double m0 = (double)__shfl_sync(0xffffffffu, v, 0);
  const double ej = lane < k ? exp((double)v - m0) : 0.0;
  double s = 0.0;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ej, j);
  return (float)(ej / s);
}
__device__ __forceinline__ float topk_softmax_weight(float v, int k) {
  const int lane = threadIdx.x & 31;
  const bool act = lane < k;
  const float v0 = __shfl_sync(0xffffffffu, v, 0);
  const FF d = ff_two_sum(v, -v0);  // v - v0, exactly
  const bool slow = act && !(d.h >= -80.f && d.h <= 0.f && isfinite(d.l));
  if (__any_sync(0xffffffffu, slow)) return topk_softmax_weight_f64(v, k);
  int n = 0;
  FF e{0.f, 0.f};
  if (act) e = ff_exp_scaled(d, n);
  const float eh = ldexpf(e.h, n), el = ldexpf(e.l, n);
  FF s{0.f, 0.f};
  for (int i = 0; i < k; ++i)
    s = ff_add(s, FF{__shfl_sync(0xffffffffu, eh, i), __shfl_sync(0xffffffffu, el, i)});
  // q = e / s: the quotient of the leading parts, corrected by the remainder
  const float qh = __fdiv_rn(e.h, s.h);
  const FF p = ff_mul(FF{qh, 0.f}, s);
  const FF rem = ff_add(e, FF{-p.h, -p.l});
  const float q = qh + __fdiv_rn(rem.h, s.h);
  return ldexpf(q, n);  // exact: q 2^n stays a normal fp32 number for n >= -116
}

// f = (a & b) ^ c
__device__ __forceinline__ uint32_t lop3_and_xor(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Four bf16x2 registers from one 32-bit word of int4 codes (nibble i = column
// 8c+i of the block). Register r holds (column 8c+r, column 8c+r+4) as the
// bf16 values 136 + code: lop3 drops nibble r and r+4 into the low mantissa bits
// of the bf16 constant 128 (0x4300) and flips bit 3, which maps a two's
// complement code q to q + 8.
__device__ __forceinline__ void dequant_word(uint32_t w, uint32_t (&d)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x43084308u;
  d[0] = lop3_and_xor(w, mask, magic);
  d[1] = lop3_and_xor(w >> 4, mask, magic);
  d[2] = lop3_and_xor(w >> 8, mask, magic);
  d[3] = lop3_and_xor(w >> 12, mask, magic);
}

// D += A(16x16 bf16, row) * B(16x8 bf16, col), fp32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A(16x16 f16, row) * B(16x8 f16, col), fp32 accumulate.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four f16x2 registers from one word of int4 codes, holding 1032 + code: the
// nibble lands in the low mantissa bits of the f16 constant 1024 (0x6400)
// and bit 3 is flipped (q -> q + 8). Same column order as dequant_word.
__device__ __forceinline__ void dequant_word_f16(uint32_t w, uint32_t (&d)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x64086408u;
  d[0] = lop3_and_xor(w, mask, magic);
  d[1] = lop3_and_xor(w >> 4, mask, magic);
  d[2] = lop3_and_xor(w >> 8, mask, magic);
  d[3] = lop3_and_xor(w >> 12, mask, magic);
}

// TMA tensor loads into this CTA's shared memory, completing on `bar`. The
// innermost coordinate times the element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, int c0, int c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// L2 policy for data read once per call (the expert weights): evicted before
// anything else, so the stream does not push the kernel's code and the small
// per-call buffers out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const void* tmap, int c0, int c1,
                                                 uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(
          dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

// Byte offset inside a region written by a 128-byte-swizzled TMA box whose base
// is 1024-byte aligned: the 16-byte chunk index is XOR-ed with the 128-byte row.
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bulk asynchronous copy shared -> global in this thread's bulk async-group
// (both addresses 16-byte aligned, bytes a multiple of 16), the group commit,
// and the waits: until the sources may be overwritten (.read) or until the
// writes are complete.
__device__ __forceinline__ void bulk_s2g(void* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_s_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}

// Shared-memory loads by 32-bit shared-window address.
__device__ __forceinline__ uint32_t ld_s32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint4 ld_s128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float ld_s_half_as_float(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.b16 %0, [%1];" : "=h"(v) : "r"(a));
  return __half2float(__ushort_as_half(v));
}

__device__ __forceinline__ uint4 lds_v4(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// L2-only 16-byte load (bypasses L1): for data other CTAs wrote during the
// same kernel, read after an acquire.
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ float ldg_cg_f32(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Spin until *p >= target (acquire), giving up after about a second with
// DEV_TIMEOUT. Each poll is one load's round trip (the thread waits for its
// value), so the loop needs no sleep: one thread per CTA polls.
__device__ __forceinline__ bool wait_counter_bounded(const int* p, int target, int32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = cycles_now();
  for (uint32_t it = 1;; ++it) {
    if (ld_acquire_gpu(p) >= target) return true;
    if ((it & 15) == 0 && cycles_now() - t0 > kWaitCycles) {
      if (status) atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ int ld_relaxed_gpu(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// The same wait without acquire ordering (for counters that order nothing
// but their own value).
__device__ __forceinline__ bool wait_counter_relaxed(const int* p, int target, int32_t* status) {
  if (ld_relaxed_gpu(p) >= target) return true;
  const long long t0 = cycles_now();
  for (uint32_t it = 1;; ++it) {
    if (ld_relaxed_gpu(p) >= target) return true;
    if ((it & 15) == 0 && cycles_now() - t0 > kWaitCycles) {
      if (status) atomicOr(status, DEV_TIMEOUT);
      return false;
    }
  }
}

// Release-ordered atomic add at GPU scope: this thread's earlier writes, and
// those it observed through a CTA barrier, are visible before the add.
__device__ __forceinline__ void red_release_gpu_add(int* p, int v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier over `count` threads (a multiple of 32).
__device__ __forceinline__ void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Arrive at named barrier `id` without waiting (the threads that sync on it
// see this thread's earlier shared-memory writes once it completes).
__device__ __forceinline__ void named_bar_arrive(int id, int count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Position of column j (0..7) of an 8-column group in the fragment order
// [0,4,1,5,2,6,3,7] used for the MMA B operand.
__host__ __device__ __forceinline__ int perm8_pos(int j) { return 2 * (j & 3) + (j >> 2); }

__device__ __forceinline__ uint16_t bf16_bits(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ float bf16_to_f(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace moe
