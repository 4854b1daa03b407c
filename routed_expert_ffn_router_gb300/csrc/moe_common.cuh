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

// Spin until *p >= target (acquire), giving up after about a second with DEV_TIMEOUT.
__device__ __forceinline__ bool wait_counter_bounded(const int* p, int target, int32_t* status) {
  if (ld_acquire_gpu(p) >= target) return true;
  const long long t0 = cycles_now();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ld_acquire_gpu(p) >= target) return true;
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
