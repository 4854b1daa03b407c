// Prefill path (prompt chunks): the routed experts' gate/up + SwiGLU and down
// as grouped GEMMs on the 5th-generation tensor cores (tcgen05, TMEM
// accumulators), over int4 blocks dequantised in shared memory.
//
// The pages' prompt path is a batched quantised GEMM in which a token batch
// shares one weight read, grouped by expert (SGLang port post, section 2, the
// expert-scoped layout that computes only the rows routed to each expert, and
// section 3, the MMQ-class kernel); the grouping here is the (token, expert)
// permutation: an expert's tokens are consecutive rows of the sorted order.
//
// Two persistent kernels, one per GEMM, each a warp-specialised pipeline:
//   warp 12 (one thread) streams a job's int4 codes and fp16 scales (TMA tensor
//   copies, 256 columns of K per raw stage);
//   16 warps dequantise a raw stage, q = (1024 + (q ^ 8)) - 1032 exactly, then
//   q * s with the fp16 scale, rounded once (2^-12): one thread per weight row
//   writes 64 columns of K per step into tensor memory (tcgen05.st, a ring of
//   4 steps; a warp reaches its TMEM lane quarter, the warps of a quarter split
//   the two matrices of a job (gate and up, or two down row tiles) and the
//   even and odd steps);
//   warp 13 (one thread) streams the job's token rows of the expert-sorted x
//   or h (a TMA box of 16, 32, 64 or 128 rows by the job's token count);
//   warp 14 (the whole warp, its elected lane issuing) runs tcgen05.mma with
//   each 128-row weight matrix as A, from tensor memory, and the job's tokens
//   as B (N = tokens rounded to 16), K = 16, and commits each stage back to its
//   producers. Keeping the weight tiles in tensor memory takes their write and
//   read (64 KB per step) off the shared-memory port;
//   8 epilogue warps (TMEM lanes = weight rows) drain the accumulators: each
//   thread holds one weight row's outputs for the job's tokens and writes
//   h = silu(g) u in fp16 (gate/up: gate and up rows meet on the same lane;
//   jobs of up to 128 tokens, those of up to 64 in alternating accumulators)
//   or w * (W_d h) as fp32
//   partials (down: two accumulators in turn, jobs of up to 64 tokens); the
//   weight ring takes the tensor memory's other 256 columns. h is stored with
//   the columns of each group of 8 in the order (0, 4, 1, 5, 2, 6, 3, 7), the
//   order in which the down dequantisation yields the codes.
// Both operands are fp16: the tensor cores take one type for A and B, and fp16
// keeps q * s and h to 2^-12 where bf16 would round to 2^-9. x enters as
// x / 2^e_t in fp16, written once per routed pair in the expert-sorted row
// order, the columns of each group of 8 in the order (0, 4, 1, 5, 2, 6, 3, 7)
// in which the gate/up dequantisation yields the codes (x16_prep_kernel; e_t is the smallest power of two that keeps the row
// below 2^15, 0 for ordinary activations): exact for every bf16 value in
// range, and the gate/up epilogue multiplies g and u back by 2^e_t.
// A job is (active expert, 128 gate and 128 up rows, or 256 down rows, up to
// 128 of its tokens); both kernels derive the job list from the permutation,
// large token blocks first, and each CTA takes every G-th position of it
// (gate/up: in alternating directions), no CTA waiting for another. The
// ordered combine (moe_decode.cu) then sums the partials in
// j order and adds the shared expert, which enters as one more expert with all
// T tokens.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "moe_internal.h"

namespace moe {
namespace pf {

constexpr int kBM = 128;              // weight rows per tile (two tiles per job)
constexpr int kNT = 128;              // tokens per gate/up job at most (the MMA's N); down: 64
constexpr int kRawSt = 2, kBSt = 4;
// The dequantised weight tiles live in tensor memory, a ring of 4 steps from
// column kTmA on, per step two matrices of 128 lanes x 32 columns (64 fp16 of
// K). Columns 0-255: gate/up two accumulator buffers of 128 columns, a job of
// up to 64 tokens taking one (gate at +0, up at +64) and a larger job both
// (gate at 0, up at 128); down two (at 0 and 128), each holding its two row
// tiles at +0 and +64.
constexpr int kTmA = 256, kTmAStage = 64, kTmAMat = 32, kAStTm = 4;
template <bool GU>
__host__ __device__ constexpr int a_stages() { return kAStTm; }
// tokens per job at most: gate/up 128 (one accumulator of 256 columns), down 64
// (two accumulators of two 64-column row tiles)
template <bool GU>
__host__ __device__ constexpr int job_nt() { return GU ? kNT : kNT / 2; }
// warps 0-3 and 15-18 epilogue, 4-11 and 19-26 dequant, 12-13 producers, 14 MMA
constexpr int kThreads = 864;
constexpr int kDqWarps = 16;          // 8 per weight tile: one 16-row band each
constexpr int kEpiWarps = 8;          // two per TMEM lane quarter, each for half of the weight rows
constexpr int kMaxAct = kMaxE + 1;
constexpr int kJobCap = 64;           // jobs per CTA decoded at the start (later ones on the fly)
constexpr int kCodeBox = 128 * 128;   // one raw code box: 128 rows x 128 bytes (256 columns)
constexpr int kScaleBox = 128 * 16;   // one raw scale box: 128 rows x 8 fp16
constexpr int kBTile = kNT * 128;     // one fp16 token tile: 128 rows x 64 columns

struct Args {
  CUtensorMap tm_c[2], tm_s[2];       // routed codes / scales (gate, up; or down)
  CUtensorMap tm_sc[2], tm_ss[2];     // the shared expert's
  CUtensorMap tm_b[4];                // expert-sorted x16 [rows][H] or h [rows][Imax], fp16,
                                      // boxes of 16, 32, 64 and 128 rows
  int H, I, shI, k, T, P, Imax;
  const ActExpert* act;
  const int32_t* counters;            // [0]: active experts including the shared one
  const int32_t* sorted_pair;
  const float* w;
  const float* xscale;                // 2^e_t per token (gate/up)
  uint16_t* h;                        // fp16 [rows][Imax], expert-sorted rows
  float* partial;                     // [rows][H]
  int32_t* status;
};

// Two A tiles per stage: gate and up (gate/up), or two row tiles (down).
template <bool GU>
__host__ __device__ constexpr int nmat() { return 2; }
template <bool GU>
__host__ __device__ constexpr int job_rows() { return GU ? kBM : 2 * kBM; }
template <bool GU>
__host__ __device__ constexpr int raw_bytes() { return nmat<GU>() * (kCodeBox + kScaleBox); }
template <bool GU>
__host__ __device__ constexpr size_t smem_bytes() {
  return 1024 + (size_t)kRawSt * raw_bytes<GU>() + (size_t)kBSt * kBTile;
}

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  // K-major, 128-byte swizzle: start address, leading offset 16 B (unused),
  // 1024 B between 8-row groups, descriptor version 1, layout SWIZZLE_128B
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// kind::f16 instruction descriptor: fp32 accumulator, fp16 A and B, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
// The issue forms used by the MMA warps: the whole warp runs the issue loop
// (its operands stay warp-uniform) and the elected lane issues (lead != 0).
// Measured on GB300: a converged warp with an elected issuer takes about two
// thirds of the issue time of a lone lane in a divergent branch.
__device__ __forceinline__ uint32_t elect_lane() {
  uint32_t r;
  asm volatile("{\n .reg .pred p;\n elect.sync _|p, 0xffffffff;\n selp.u32 %0, 1, 0, p;\n}" : "=r"(r));
  return r;
}
__device__ __forceinline__ void tc_mma_el(uint32_t d, uint64_t ad, uint64_t bd, uint32_t idesc, uint32_t acc,
                                          uint32_t lead) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d),
      "l"(ad), "l"(bd), "r"(idesc), "r"(acc), "r"(lead));
}
// A from tensor memory (K-major: row i in TMEM lane i, two fp16 of K per column)
__device__ __forceinline__ void tc_mma_ts_el(uint32_t d, uint32_t at, uint64_t bd, uint32_t idesc, uint32_t acc,
                                             uint32_t lead) {
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.b32 p, %4, 0;\n setp.ne.b32 q, %5, 0;\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}" ::"r"(d),
      "r"(at), "l"(bd), "r"(idesc), "r"(acc), "r"(lead));
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tc_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_commit_el(uint32_t bar, uint32_t lead) {
  asm volatile(
      "{\n .reg .pred q;\n setp.ne.b32 q, %1, 0;\n"
      " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}" ::"r"(bar), "r"(lead)
      : "memory");
}
__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void st_s128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}

// One 32-bit word of codes (columns 8c..8c+7, nibble i = column 8c+i) -> four
// f16x2 registers holding q * s for columns (0,1), (2,3), (4,5), (6,7).
__device__ __forceinline__ void dequant_word_h(uint32_t wd, __half2 s2, uint32_t (&o)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x64086408u;  // f16 1024 + (q ^ 8) = 1032 + q
  const uint32_t x0 = lop3_and_xor(wd, mask, magic), x1 = lop3_and_xor(wd >> 4, mask, magic);
  const uint32_t x2 = lop3_and_xor(wd >> 8, mask, magic), x3 = lop3_and_xor(wd >> 12, mask, magic);
  const uint32_t p[4] = {prmt(x0, x1, 0x5410), prmt(x2, x3, 0x5410), prmt(x0, x1, 0x7632), prmt(x2, x3, 0x7632)};
  const __half2 m1032 = __floats2half2_rn(1032.f, 1032.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = *reinterpret_cast<const __half2*>(&p[i]);
    v = __hmul2(__hsub2(v, m1032), s2);  // q exactly, then one rounding of q * s
    o[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// One word of codes (columns 8c..8c+7) -> four f16x2 registers of q * s in the
// order the nibbles come out: (0, 4), (1, 5), (2, 6), (3, 7). The gate/up B
// operand (x16) holds its columns in the same order within each group of 8.
__device__ __forceinline__ void dequant_word_h_perm(uint32_t wd, __half2 s2, uint32_t (&o)[4]) {
  const uint32_t mask = 0x000F000Fu, magic = 0x64086408u;  // f16 1024 + (q ^ 8) = 1032 + q
  const uint32_t x[4] = {lop3_and_xor(wd, mask, magic), lop3_and_xor(wd >> 4, mask, magic),
                         lop3_and_xor(wd >> 8, mask, magic), lop3_and_xor(wd >> 12, mask, magic)};
  const __half2 m1032 = __floats2half2_rn(1032.f, 1032.f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __half2 v = *reinterpret_cast<const __half2*>(&x[i]);
    v = __hmul2(__hsub2(v, m1032), s2);  // q exactly, then one rounding of q * s
    o[i] = *reinterpret_cast<const uint32_t*>(&v);
  }
}

// Gate/up accumulators: two buffers of 128 TMEM columns. A job of up to 64
// tokens takes one (gate at +0, up at +64), buffers in turn by small-job count;
// a job of more tokens takes both (gate at 0, up at 128). The MMA warp and the
// epilogue walk the same job sequence and keep the same use counts per buffer.
struct AccUse {
  int nsmall;   // small jobs so far
  int u0, u1;   // uses of buffers 0 and 1 so far
  __device__ int use(int b) const { return b ? u1 : u0; }
  __device__ void used(int b) {
    if (b) ++u1;
    else ++u0;
  }
  __device__ void next(int np, int& b0, int& b1, uint32_t& gbase, uint32_t& uoff) {
    if (np <= 64) {
      b0 = b1 = nsmall++ & 1;
      gbase = 128u * (uint32_t)b0;
      uoff = 64;
    } else {
      b0 = 0;
      b1 = 1;
      gbase = 0;
      uoff = 128;
    }
  }
};

struct Job {
  int mt, n0, nn, np;      // row tile, first token slot, tokens, tokens rounded to 16
  int bsel;                // token box of 16 << bsel rows; a token slot holds 8 >> bsel boxes
  int off, slot;           // first sorted row of the expert; pool slot (-1: shared)
  bool sh;
};

template <bool GU>
__global__ void __launch_bounds__(kThreads, 1) pf_kernel(const __grid_constant__ Args a) {
  constexpr int NM = nmat<GU>();
  extern __shared__ __align__(128) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t s_bar[2 * kRawSt + 2 * kAStTm + 2 * kBSt + 4];
  __shared__ int s_js[2][kMaxAct + 1];   // first job of each active entry, per job class
  __shared__ int4 s_job[kJobCap];        // the CTA's first kJobCap jobs, decoded once
  __shared__ int s_off[kMaxAct], s_cnt[kMaxAct], s_slot[kMaxAct];
  __shared__ float s_colf[2][kNT];       // down: the routing weight of each token column of a job
  __shared__ float s_cfw[kEpiWarps][kNT];  // gate/up: each epilogue warp's token prescales
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, bid = blockIdx.x;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  // token ring first: a step's 128-row tile may start inside the last slot and
  // read past the ring's end, into the raw ring (those rows are never used)
  const uint32_t sB = smem_u32(smem);
  const uint32_t sraw = sB + kBSt * kBTile;
  const uint32_t sA = sraw + kRawSt * raw_bytes<GU>();
  const uint32_t bar0 = smem_u32(&s_bar[0]);
  const uint32_t raw_full = bar0, raw_empty = raw_full + 8 * kRawSt;
  const uint32_t a_full = raw_empty + 8 * kRawSt, a_empty = a_full + 8 * kAStTm;
  const uint32_t b_full = a_empty + 8 * kAStTm, b_empty = b_full + 8 * kBSt;
  const uint32_t acc_full = b_empty + 8 * kBSt, acc_empty = acc_full + 16;
  volatile int* abort_flag = &s_abort;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kRawSt; ++i) {
      mbar_init(raw_full + 8 * i, 1);
      mbar_init(raw_empty + 8 * i, kDqWarps);  // one arrival per dequantising warp
    }
    for (int i = 0; i < a_stages<GU>(); ++i) {
      mbar_init(a_full + 8 * i, kDqWarps / 2);  // the 8 dequantising warps of the step's parity
      mbar_init(a_empty + 8 * i, 1);
    }
    for (int i = 0; i < kBSt; ++i) {
      mbar_init(b_full + 8 * i, 1);
      mbar_init(b_empty + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(acc_full + 8 * i, 1);
      mbar_init(acc_empty + 8 * i, kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == 14) {  // the whole TMEM (512 columns): two accumulator buffers of 256
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  // the job list: per active entry, (rows / 128) row tiles x ceil(tokens / 128)
  const int n_act = min(a.counters[0], kMaxAct);
  const int P = a.P;
  for (int i = tid; i < n_act; i += kThreads) {
    const ActExpert e = a.act[i];
    s_off[i] = e.off;
    s_cnt[i] = e.cnt;
    s_slot[i] = e.slot;
  }
  __syncthreads();
  // Two job classes: token blocks of more than half the job size (the full
  // blocks of an entry and a large last block), then the small last blocks,
  // each class in entry order; per entry and class, the row tiles of one token
  // block are consecutive. The large jobs, which take longer, come first.
  if (warp < 2) {
    const int cls = warp;
    const int per = (n_act + 31) / 32, i0 = lane * per, i1 = min(n_act, i0 + per);
    auto njob = [&](int i) {
      const int rows = GU ? (s_slot[i] < 0 ? a.shI : a.I) : a.H;
      const int nt = job_nt<GU>(), rem = s_cnt[i] % nt;
      const int nb = cls == 0 ? s_cnt[i] / nt + (rem > nt / 2 ? 1 : 0) : (rem > 0 && rem <= nt / 2 ? 1 : 0);
      return (rows / job_rows<GU>()) * nb;
    };
    int sum = 0;
    for (int i = i0; i < i1; ++i) sum += njob(i);
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    int run = x - sum;
    for (int i = i0; i < i1; ++i) {
      s_js[cls][i] = run;
      run += njob(i);
    }
    if (lane == 31) s_js[cls][n_act] = x;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int nfirst = s_js[0][n_act];
  const int njobs = nfirst + s_js[1][n_act];
  // CTA b's jobs: gate/up takes list positions b, 2G - 1 - b, 2G + b,
  // 4G - 1 - b, ... (each round of G positions in the opposite CTA order to the
  // one before), down positions b, b + G, b + 2G, ... (measured on GB300: the
  // order of least time for each kernel)
  auto next_pos = [&](int j) { return GU ? j + 2 * G - 1 - 2 * (j % G) : j + G; };

  auto job_of = [&](int j) {
    const int cls = j < nfirst ? 0 : 1;
    if (cls) j -= nfirst;
    const int* js = s_js[cls];
    int lo = 0, hi = n_act - 1;  // last entry with js <= j
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (js[mid] <= j) lo = mid;
      else hi = mid - 1;
    }
    Job jb;
    jb.sh = s_slot[lo] < 0;
    const int rows = GU ? (jb.sh ? a.shI : a.I) : a.H;
    const int nM = rows / job_rows<GU>();
    const int loc = j - js[lo];
    jb.mt = loc % nM;
    jb.n0 = (cls == 0 ? loc / nM : s_cnt[lo] / job_nt<GU>()) * job_nt<GU>();
    jb.nn = min(job_nt<GU>(), s_cnt[lo] - jb.n0);
    jb.np = (jb.nn + 15) & ~15;
    jb.bsel = jb.np <= 16 ? 0 : jb.np <= 32 ? 1 : jb.np <= 64 ? 2 : 3;
    jb.off = s_off[lo];
    jb.slot = s_slot[lo];
    return jb;
  };
  auto k_of = [&](const Job& jb) { return GU ? a.H : (jb.sh ? a.shI : a.I); };
  // The CTA's i-th job: from the table decoded below for i < kJobCap (every
  // role walks the same sequence; one decode instead of one per warp)
  auto job_at = [&](int i, int j) {
    if (i >= kJobCap) return job_of(j);
    const int4 v = s_job[i];
    Job jb;
    jb.off = v.x;
    jb.slot = v.y;
    jb.sh = v.y < 0;
    jb.n0 = v.z;
    jb.mt = v.w >> 8;
    jb.nn = v.w & 255;
    jb.np = (jb.nn + 15) & ~15;
    jb.bsel = jb.np <= 16 ? 0 : jb.np <= 32 ? 1 : jb.np <= 64 ? 2 : 3;
    return jb;
  };
  if (warp < 2) {  // two of the epilogue warps, before their first job
    for (int i = tid; i < kJobCap; i += 64) {
      int j = bid;
      for (int r = 0; r < i && j < njobs; ++r) j = next_pos(j);
      if (j < njobs) {
        const Job jb = job_of(j);
        s_job[i] = make_int4(jb.off, jb.slot, jb.n0, (jb.mt << 8) | jb.nn);
      }
    }
  }
  __syncthreads();

  if (warp == 12) {
    // ================= raw producer: codes and scales =================
    if (lane == 0) {
      int rcnt = 0;
      for (int j = bid, ji = 0; j < njobs && !*abort_flag; j = next_pos(j), ++ji) {
        const Job jb = job_at(ji, j);
        const int K = k_of(jb);
        const int row0 = (jb.sh ? 0 : jb.slot * (GU ? a.I : a.H)) + jb.mt * job_rows<GU>();
        bool ok = true;
        for (int kr = 0; kr < K / 256; ++kr) {
          const int rs = rcnt % kRawSt;
          if (!(ok = mbar_wait_short(raw_empty + 8 * rs, ((rcnt / kRawSt) & 1) ^ 1, a.status))) break;
          const uint32_t st = sraw + rs * raw_bytes<GU>(), fb = raw_full + 8 * rs;
          mbar_expect_tx(fb, raw_bytes<GU>());
#pragma unroll
          for (int m = 0; m < NM; ++m) {  // gate/up: two matrices; down: two row tiles of one
            const int mi = GU ? m : 0, rm = GU ? row0 : row0 + m * kBM;
            tma_load_2d(st + m * kCodeBox, jb.sh ? &a.tm_sc[mi] : &a.tm_c[mi], kr * 128, rm, fb);
            tma_load_2d(st + NM * kCodeBox + m * kScaleBox, jb.sh ? &a.tm_ss[mi] : &a.tm_s[mi], kr * 8, rm,
                        fb);
          }
          ++rcnt;
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 13) {
    // ================= token producer: the job's rows of x or h =================
    // a 16 KB slot holds the boxes of 8 >> bsel consecutive steps (16 << bsel
    // rows each); the 128-row tile of a step starts at its box, and the rows
    // after the box (later steps' boxes, stale data) only reach accumulator
    // lanes that are never read
    if (lane == 0) {
      int bcnt = 0;
      for (int j = bid, ji = 0; j < njobs && !*abort_flag; j = next_pos(j), ++ji) {
        const Job jb = job_at(ji, j);
        const uint32_t bbytes = (16u << jb.bsel) * 128;  // one box
        const int spb = 8 >> jb.bsel;                      // boxes per slot
        bool ok = true;
        for (int kb = 0; kb < k_of(jb) / 64; kb += spb) {
          const int bs = bcnt % kBSt;
          if (!(ok = mbar_wait_short(b_empty + 8 * bs, ((bcnt / kBSt) & 1) ^ 1, a.status))) break;
          const uint32_t dst = sB + bs * kBTile, bb = b_full + 8 * bs;
          mbar_expect_tx(bb, bbytes * spb);
          for (int u = 0; u < spb; ++u)
            tma_load_2d(dst + u * bbytes, &a.tm_b[jb.bsel], (kb + u) * 64, jb.off + jb.n0, bb);
          ++bcnt;
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
    }
    __syncwarp();
  } else if (warp == 14) {
    // ================= MMA issuer (whole warp, elected lane issues) =================
    // D[weight row][token] += W(128 x 16) . X(np x 16)^T per matrix: eight MMAs per step
    const uint32_t lead = elect_lane();
    // descriptors of the first tiles; the others differ by their address / 16
    // in the low field (no carry: shared addresses < 256 KB)
    const uint64_t xd0 = sdesc_sw128(sB);
    int acnt = 0, bcnt = 0, jcnt = 0;
    AccUse au{0, 0, 0};
    for (int j = bid; j < njobs && !*abort_flag; j = next_pos(j), ++jcnt) {
      const Job jb = job_at(jcnt, j);
      const int ab = GU ? 0 : jcnt & 1;
      int gb0 = 0, gb1 = 0;
      uint32_t gbase = 0, uoff = 128;
      bool accok;
      if constexpr (GU) {
        au.next(jb.np, gb0, gb1, gbase, uoff);
        accok = mbar_wait_short(acc_empty + 8 * gb0, (au.use(gb0) & 1) ^ 1, a.status) &&
                (gb1 == gb0 || mbar_wait_short(acc_empty + 8 * gb1, (au.use(gb1) & 1) ^ 1, a.status));
      } else {
        accok = mbar_wait_short(acc_empty + 8 * ab, ((jcnt >> 1) & 1) ^ 1, a.status);
      }
      if (!__all_sync(0xffffffffu, accok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int nkb = k_of(jb) / 64;
      const int spb = 8 >> jb.bsel;
      const uint32_t bbytes = (16u << jb.bsel) * 128;
      // each 128-row weight matrix (gate/up: gate and up, from tensor memory;
      // down: two row tiles, from shared memory) as A, the job's tokens as B
      const uint32_t idesc = idesc_f16(kBM, jb.np);
      bool ok = true;
      for (int kb = 0, u = 0; kb < nkb; ++kb) {  // u = kb mod spb (a power of two)
        const int as = acnt % a_stages<GU>(), bs = bcnt % kBSt;
        const uint32_t apar = (acnt / a_stages<GU>()) & 1;
        // a ready stage is the common case: test once before the sleeping wait
        ok = (mbar_test(a_full + 8 * as, apar) || mbar_wait_short(a_full + 8 * as, apar, a.status)) &&
             (u != 0 || mbar_test(b_full + 8 * bs, (bcnt / kBSt) & 1) ||
              mbar_wait_short(b_full + 8 * bs, (bcnt / kBSt) & 1, a.status));
        if (!(ok = __all_sync(0xffffffffu, ok))) break;
        tc_fence_after();
        const uint64_t xdk = xd0 + ((uint32_t)(bs * kBTile + u * bbytes) >> 4);
        if constexpr (GU) {
          const uint32_t ta = tmem + kTmA + as * kTmAStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int m = 0; m < NM; ++m)  // K = 16: 8 TMEM columns of A
              tc_mma_ts_el(tmem + gbase + m * uoff, ta + m * kTmAMat + kk * 8, xdk + ((kk * 32) >> 4), idesc,
                           (kb > 0 || kk > 0) ? 1u : 0u, lead);
        } else {
          const uint32_t ta = tmem + kTmA + as * kTmAStage;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int m = 0; m < NM; ++m)  // accumulator ab: row tile m at 64 m
              tc_mma_ts_el(tmem + ab * 128 + m * 64, ta + m * kTmAMat + kk * 8, xdk + ((kk * 32) >> 4), idesc,
                           (kb > 0 || kk > 0) ? 1u : 0u, lead);
        }
        tc_commit_el(a_empty + 8 * as, lead);  // the tiles are free once these MMAs are done
        ++acnt;
        // a slot is free after its last step; a job's last slot may hold fewer
        // than spb steps (K / 64 not a multiple of spb)
        if (++u == spb || kb == nkb - 1) {
          tc_commit_el(b_empty + 8 * bs, lead);
          ++bcnt;
          u = 0;
        }
      }
      if (!ok) {
        *abort_flag = 1;
        break;
      }
      // the job's accumulators are complete
      if constexpr (GU) {
        tc_commit_el(acc_full + 8 * gb0, lead);
        au.used(gb0);
        if (gb1 != gb0) {
          tc_commit_el(acc_full + 8 * gb1, lead);
          au.used(gb1);
        }
      } else {
        tc_commit_el(acc_full + 8 * ab, lead);
      }
    }
    __syncwarp();
  } else if ((warp >= 4 && warp <= 11) || warp >= 19) {
    // ================= dequantisation (16 warps: tile m = wd / 8, rows 16 (wd mod 8) ..) =================
    // Thread: row r, 32-column block h of each 64-column step. The 8 lanes of a
    // quarter-warp read 8 consecutive rows of one block: 8 different 16-byte
    // chunks of the swizzled raw rows, no bank conflict.
    {
    // Thread = one weight row r of matrix m (gate/up: gate or up; down: row tile), which is TMEM lane r of the A
    // tiles (a warp reaches lane quarter warp mod 4); the warps of each quarter
    // split the matrices and the even and odd steps. Per step of 64 columns:
    // 32 code bytes (two 16-byte chunks of the swizzled raw row) and the scales
    // of its two 32-column blocks, 32 registers of fp16 pairs to the step's
    // TMEM columns.
    const int q4 = warp & 3;
    const int idx = warp <= 11 ? (warp - 4) >> 2 : 2 + ((warp - 19) >> 2);
    const int m = idx & 1, par = idx >> 1;
    const int r = 32 * q4 + lane;
    const uint32_t rsw = (uint32_t)(r & 7);
    const uint32_t trow = tmem + ((uint32_t)(32 * q4) << 16) + kTmA + m * kTmAMat;
    int rcnt = 0, acnt = 0;
    for (int j = bid, ji = 0; j < njobs && !*abort_flag; j = next_pos(j), ++ji) {
      const Job jb = job_at(ji, j);
      const int K = k_of(jb);
      bool ok = true;
      for (int kr = 0; kr < K / 256 && ok; ++kr) {
        const int rs = rcnt % kRawSt;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait_short(raw_full + 8 * rs, (rcnt / kRawSt) & 1, a.status))))
          break;
        const uint32_t st = sraw + rs * raw_bytes<GU>();
        const uint32_t crow = st + m * kCodeBox + r * 128;
        const uint32_t srow = st + NM * kCodeBox + m * kScaleBox + r * 16;
        for (int s4 = 0; s4 < 4 && ok; ++s4, ++acnt) {
          if ((s4 & 1) != par) continue;  // the other warps of the quarter take this step
          const int as = acnt % kAStTm;
          if (!(ok = __all_sync(0xffffffffu,
                                mbar_wait_short(a_empty + 8 * as, ((acnt / kAStTm) & 1) ^ 1, a.status))))
            break;
          tc_fence_after();
          const uint4 c0 = ld_s128(crow + (((uint32_t)(2 * s4) ^ rsw) << 4));
          const uint4 c1 = ld_s128(crow + (((uint32_t)(2 * s4 + 1) ^ rsw) << 4));
          const uint32_t sc = ld_s32(srow + 4 * s4);  // blocks 2 s4 (low half) and 2 s4 + 1
          const uint32_t s0u = prmt(sc, 0u, 0x1010), s1u = prmt(sc, 0u, 0x3232);
          const __half2 s0 = *reinterpret_cast<const __half2*>(&s0u);
          const __half2 s1 = *reinterpret_cast<const __half2*>(&s1u);
          uint32_t o[8][4];
          dequant_word_h_perm(c0.x, s0, o[0]);
          dequant_word_h_perm(c0.y, s0, o[1]);
          dequant_word_h_perm(c0.z, s0, o[2]);
          dequant_word_h_perm(c0.w, s0, o[3]);
          dequant_word_h_perm(c1.x, s1, o[4]);
          dequant_word_h_perm(c1.y, s1, o[5]);
          dequant_word_h_perm(c1.z, s1, o[6]);
          dequant_word_h_perm(c1.w, s1, o[7]);
          tc_st32(trow + as * kTmAStage, *reinterpret_cast<const uint32_t(*)[32]>(&o[0][0]));
          tc_st_wait();
          tc_fence_before();  // the MMA warp reads the tile after the barrier
          __syncwarp();
          if (lane == 0) mbar_arrive(a_full + 8 * as);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(raw_empty + 8 * rs);
        ++rcnt;
      }
      if (!ok) *abort_flag = 1;
    }
    }
  } else {
    // ================= epilogue (warps 0-3 and 15-18) =================
    // A warp reaches the TMEM lane quarter warp mod 4; the two warps of a
    // quarter split the accumulator's columns (gate/up) or its two weight row
    // tiles (down).
    const int qw = warp & 3, half = warp >= 15 ? 1 : 0;
    int jcnt = 0;
    if constexpr (GU) {
    // Gate/up: thread = one intermediate row of the job's 128 (TMEM lane); the
    // columns are the job's tokens, gate at 0 and up at 128. The two warps of
    // a quarter take alternate 16-token chunks; each warp store is 32
    // consecutive fp16 of one token's h row.
    const int row = qw * 32 + lane;
    AccUse au{0, 0, 0};
    for (int j = bid; j < njobs && !*abort_flag; j = next_pos(j), ++jcnt) {
      const Job jb = job_at(jcnt, j);
      int gb0, gb1;
      uint32_t gbase, uoff;
      au.next(jb.np, gb0, gb1, gbase, uoff);
      // the x prescale of each token column (this warp's own copy: no barrier
      // with the other epilogue warps), fetched while the job's MMAs run
      float* colf = s_cfw[qw + 4 * half];
      __syncwarp();  // the previous job's reads of colf are done
      for (int e = lane; e < jb.nn; e += 32) {
        const size_t s = (size_t)jb.off + jb.n0 + e;
        colf[e] = jb.sh ? __ldg(a.xscale + (s - P)) : __ldg(a.xscale + a.sorted_pair[s] / a.k);
      }
      __syncwarp();
      const bool fok = mbar_wait_short(acc_full + 8 * gb0, au.use(gb0) & 1, a.status) &&
                       (gb1 == gb0 || mbar_wait_short(acc_full + 8 * gb1, au.use(gb1) & 1, a.status));
      if (!__all_sync(0xffffffffu, fok)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(qw * 32) << 16) + gbase;
      bool range_ok = true;
      // the columns of h in each group of 8 in the order (0, 4, 1, 5, 2, 6, 3, 7),
      // the order in which the down dequantisation yields the codes
      uint16_t* hcol = a.h + (size_t)(jb.off + jb.n0) * a.Imax + jb.mt * kBM + (row & ~7) + perm8_pos(row & 7);
#pragma unroll 1
      for (int c0 = half * 16; c0 < jb.np; c0 += 32) {
        uint32_t g[16], u[16];
        tc_ld16(tb + c0, g);
        tc_ld16(tb + uoff + c0, u);
        tc_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = c0 + i;
          if (c < jb.nn) {  // undo the token's power-of-two prescale of x (exact)
            const float cf = colf[c];
            const float gv = __uint_as_float(g[i]) * cf, uv = __uint_as_float(u[i]) * cf;
            const float hv = __fdividef(gv, 1.0f + __expf(-gv)) * uv;  // rounded to fp16 below
            range_ok = range_ok && fabsf(hv) < 65504.f;
            hcol[(size_t)c * a.Imax] = __half_as_ushort(__float2half_rn(hv));
          }
        }
      }
      if (!range_ok) atomicOr(a.status, DEV_RANGE);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(acc_empty + 8 * gb0);
        if (gb1 != gb0) mbar_arrive(acc_empty + 8 * gb1);
      }
      au.used(gb0);
      if (gb1 != gb0) au.used(gb1);
    }
    } else {
    // Down: thread = one output row of weight tile `half` (TMEM lane), the
    // columns are the job's tokens; each warp store is a contiguous 128-byte
    // segment of one token's partial row.
    const int row = qw * 32 + lane;
    for (int j = bid; j < njobs && !*abort_flag; j = next_pos(j), ++jcnt) {
      const Job jb = job_at(jcnt, j);
      const int ab = jcnt & 1;
      // the routing weights of the job's pairs, fetched while its MMAs run
      float* colf = s_colf[ab];
      const int e = half * kBM + row;
      if (e < jb.nn) colf[e] = jb.sh ? 1.0f : __ldg(a.w + a.sorted_pair[jb.off + jb.n0 + e]);
      named_bar_sync(1, 32 * kEpiWarps);
      if (!__all_sync(0xffffffffu, mbar_wait_short(acc_full + 8 * ab, (jcnt >> 1) & 1, a.status))) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem + ((uint32_t)(qw * 32) << 16) + ab * 128 + half * 64;
      float* pcol = a.partial + (size_t)(jb.off + jb.n0) * a.H + jb.mt * (2 * kBM) + half * kBM + row;
      for (int c0 = 0; c0 < jb.np; c0 += 16) {
        uint32_t v[16];
        tc_ld16(tb + c0, v);
        tc_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (c0 + i < jb.nn) pcol[(size_t)(c0 + i) * a.H] = colf[c0 + i] * __uint_as_float(v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty + 8 * ab);
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 14) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

// Row t of x, as fp16(x[t] / 2^e_t), to every sorted row of token t (its k
// routed pairs, pair_pos, and the shared expert's row P + t); xscale[t] = 2^e_t
// with e_t >= 0 smallest such that max|x[t]| / 2^e_t < 2^15. Dividing a bf16
// value by a power of two and storing it as fp16 is exact while the result
// stays a normal fp16 number.
__global__ void __launch_bounds__(256) x16_prep_kernel(const uint16_t* __restrict__ x, int H, int k, int P,
                                                      const int32_t* __restrict__ pair_pos, int copies,
                                                      uint16_t* __restrict__ x16, float* __restrict__ xscale) {
  __shared__ float s_red[8];
  const int t = blockIdx.x;
  const uint16_t* xr = x + (size_t)t * H;
  float m = 0.f;
  for (int i = threadIdx.x; i < H; i += 256) m = fmaxf(m, fabsf(bf16_to_f(xr[i])));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = m;
  __syncthreads();
  m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, s_red[i]);
  int e = 0;
  if (isfinite(m))
    while (m >= 32768.f) {  // at most 113 halvings for a finite bf16 value
      m *= 0.5f;
      ++e;
    }
  const float inv = exp2f((float)-e);
  if (threadIdx.x == 0) xscale[t] = exp2f((float)e);
  for (int i = threadIdx.x * 8; i < H; i += 256 * 8) {  // 8 columns (16 bytes) per thread and step
    const uint4 v = *reinterpret_cast<const uint4*>(xr + i);
    const uint32_t in[4] = {v.x, v.y, v.z, v.w};
    // columns (q, q + 4) of the group of 8 in register q, the order of the
    // gate/up dequantisation's nibble pairs
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t a0 = in[q >> 1], a1 = in[(q >> 1) + 2];
      const float lo = __uint_as_float((q & 1) ? (a0 & 0xFFFF0000u) : (a0 << 16)) * inv;
      const float hi = __uint_as_float((q & 1) ? (a1 & 0xFFFF0000u) : (a1 << 16)) * inv;
      const __half2 h2 = __floats2half2_rn(lo, hi);
      o[q] = *reinterpret_cast<const uint32_t*>(&h2);
    }
    const uint4 ov = make_uint4(o[0], o[1], o[2], o[3]);
    for (int c = 0; c < copies; ++c) {
      const int s = c < k ? pair_pos[(size_t)t * k + c] : P + t;
      *reinterpret_cast<uint4*>(x16 + (size_t)s * H + i) = ov;
    }
  }
}

}  // namespace pf

// Host side -------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 pf_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

bool map2d(CUtensorMap* m, CUtensorMapDataType dt, const void* p, uint64_t inner, uint64_t rows,
           uint64_t row_bytes, uint32_t bx, uint32_t by, bool swz) {
  auto fn = pf_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t str[1] = {row_bytes};
  const cuuint32_t box[2] = {bx, by};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(p), dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swz ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// codes [rows][K/2] u8: box 128 bytes (256 columns) x 128 rows, 128-byte swizzle
bool pf_codes(CUtensorMap* m, const uint8_t* q, int K, int rows) {
  return map2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, (uint64_t)K / 2, rows, (uint64_t)K / 2, 128, 128, true);
}
// scales [rows][K/32] fp16: box 8 (256 columns) x 128 rows
bool pf_scales(CUtensorMap* m, const uint16_t* s, int K, int rows) {
  return map2d(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, (uint64_t)K / 32, rows, (uint64_t)K / 16, 8, 128, false);
}

// fp16 [rows][cols] B operand: boxes of 64 columns x 16, 32, 64 and 128 rows
bool b_maps(CUtensorMap* m, const void* p, int cols, int rows) {
  for (int i = 0; i < 4; ++i)
    if (!map2d(&m[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, p, cols, rows, (uint64_t)cols * 2, 64, 16u << i, true))
      return false;
  return true;
}

template <bool GU>
cudaError_t pf_launch(pf::Args& a, cudaStream_t st) {
  const size_t smem = pf::smem_bytes<GU>();
  // the shared-memory opt-in is a per-device attribute of the function
  static std::mutex mu;
  static bool configured[64] = {};
  int dev = 0, sms = 0;
  {
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
      cudaGetLastError();
      return e != cudaSuccess ? e : cudaErrorInvalidDevice;
    }
    std::lock_guard<std::mutex> lk(mu);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(pf::pf_kernel<GU>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) {
        cudaGetLastError();
        return e;
      }
      configured[dev] = true;
    }
  }
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  launch_begin(GU ? K_GATEUP : K_DOWN, st);
  pf::pf_kernel<GU><<<sms > 0 ? sms : 1, pf::kThreads, smem, st>>>(a);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(int H, int I, int shI, int T, bool x_bf16) {
  if (!x_bf16 || T <= 16) return false;
  if (H % 256 || I % 256 || shI % 256) return false;  // raw stages of 256 columns, down jobs of 256 rows
  return pf_encode_fn() != nullptr;
}

cudaError_t launch_ffn_prefill_tc(const FfnArgs& f, const void* x, cudaStream_t st) {
  const int H = f.H, I = f.I, shI = f.shI, S = f.S;
  const int rows = f.P + f.T;
  // the expert-sorted fp16 x lives in the partial buffer: only the down kernel,
  // which runs after the gate/up kernel, writes partials
  uint16_t* x16s = reinterpret_cast<uint16_t*>(f.partial);
  pf::Args g;
  std::memset(&g, 0, sizeof g);
  g.H = H; g.I = I; g.shI = shI; g.k = f.k; g.T = f.T; g.P = f.P; g.Imax = f.Imax;
  g.act = f.act; g.counters = f.counters; g.sorted_pair = f.sorted_pair; g.w = f.w;
  g.h = f.hhi; g.partial = f.partial; g.status = f.status;
  g.xscale = f.xcorr;
  pf::Args d = g;
  bool ok = pf_codes(&g.tm_c[0], f.gq, H, S * I) && pf_codes(&g.tm_c[1], f.uq, H, S * I) &&
            pf_scales(&g.tm_s[0], f.gs, H, S * I) && pf_scales(&g.tm_s[1], f.us, H, S * I) &&
            b_maps(g.tm_b, x16s, H, rows) &&
            pf_codes(&d.tm_c[0], f.dq, I, S * H) && pf_scales(&d.tm_s[0], f.ds, I, S * H) &&
            b_maps(d.tm_b, f.hhi, f.Imax, rows);
  if (ok && shI > 0)
    ok = pf_codes(&g.tm_sc[0], f.sgq, H, shI) && pf_codes(&g.tm_sc[1], f.suq, H, shI) &&
         pf_scales(&g.tm_ss[0], f.sgs, H, shI) && pf_scales(&g.tm_ss[1], f.sus, H, shI) &&
         pf_codes(&d.tm_sc[0], f.sdq, shI, H) && pf_scales(&d.tm_ss[0], f.sds, shI, H);
  if (!ok) return cudaErrorInvalidValue;
  launch_begin(K_X_PREP, st);
  pf::x16_prep_kernel<<<f.T, 256, 0, st>>>(static_cast<const uint16_t*>(x), H, f.k, f.P, f.pair_pos,
                                           f.k + (shI > 0 ? 1 : 0), x16s, const_cast<float*>(f.xcorr));
  launch_end(st);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = pf_launch<true>(g, st);
  if (e != cudaSuccess) return e;
  return pf_launch<false>(d, st);
}

}  // namespace moe
