// Expert FFN over block-quantised int4 weights: gate/up + SwiGLU, down with a
// weighted scatter, and the ordered combine (SGLang port post, TL;DR and
// section 3: gather -> dequant -> gate/up -> SwiGLU -> down -> scatter over the
// packed expert bytes; Strata BATCHING: an expert shared by several rows of a
// window is read once for all of them).
//
// Work unit: (touched resident expert or the shared expert, 16 weight rows,
// up to 16 token slots). A CTA pulls its 16 rows of packed codes into shared
// memory with bulk async copies (one per row, into rows padded by 16 bytes so
// the fragment reads below are free of bank conflicts), then 8 warps split the
// reduction dimension and run warp MMAs m16n8k16 (bf16 in, fp32 accumulate):
// A = 16 weight rows, B = 8 token slots.
//
// Exact integer codes: a 32-bit word of 8 codes becomes 4 bf16x2 registers
// holding 136 + q (lop3 into the mantissa of 128, see dequant_word). Per block
// of 32 columns the MMA accumulator starts at -136 * sum(B over the block), so
// it ends at sum(q * B) exactly up to fp32 accumulation; it is then scaled by
// the block's fp16 scale and added to the running sum. No weight is ever
// rounded. Activations enter as bf16; fp32 values (the tiny case's x and the
// intermediate h) enter as a pair hi = bf16(v), lo = bf16(v - hi), two MMAs.
//
// Within a block the k order is permuted (column 8c+i of the block sits in the
// order [0,4,1,5,2,6,3,7] of each 8-group) so that one 16-byte load yields a
// lane's B registers for both k-steps; A follows the same order by construction.
#include <mutex>
#include <vector>

#include "moe_internal.h"

namespace moe {

__host__ __device__ inline int sc_words(int K) {
  int sw = K / 64;
  if (sw % 8 == 0) sw += 4;  // row stride in 32-bit words, never 0 mod 8: no bank conflicts
  return sw;
}

struct UnitSmem {
  int qstride;     // bytes per padded code row
  int sw;          // 32-bit words per padded scale row
  size_t q_off, s_off, c_off, e_off, bar_off, total;
};

template <int NMAT>
__host__ __device__ inline UnitSmem unit_smem(int K, int Kmax) {
  UnitSmem u;
  u.qstride = K / 2 + 16;
  u.sw = sc_words(K);
  const int qsm = Kmax / 2 + 16;
  size_t q = (size_t)NMAT * kRowTile * qsm;
  size_t red = (size_t)kWarps * NMAT * 2 * 128 * 4;
  u.q_off = 0;
  u.s_off = align256(q > red ? q : red);
  u.c_off = u.s_off + align256((size_t)NMAT * kRowTile * (Kmax / 64 + 4) * 4);
  u.e_off = u.c_off + align256((size_t)(Kmax / 32) * 16 * 4);
  u.bar_off = u.e_off + align256(16 * 17 * 4);
  u.total = u.bar_off + 64;
  return u;
}

// ---------------------------------------------------------------- x staging
// Per row: bf16 hi (and lo for fp32 input) in fragment order, plus
// xcorr[t][b] = -136 * sum over block b of (hi + lo).
template <bool XBF16>
__global__ void __launch_bounds__(256) x_prep_kernel(const void* __restrict__ x, int T, int H,
                                                     uint16_t* __restrict__ xhi,
                                                     uint16_t* __restrict__ xlo,
                                                     float* __restrict__ xcorr) {
  const int t = blockIdx.y;
  const int gi = blockIdx.x * 256 + threadIdx.x;  // 8-column group
  const int ng = H / 8;                             // multiple of 16
  const bool active = gi < ng;
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = 0.f;
  if (active) {
    if (XBF16) {
      uint4 r = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(x) + (size_t)t * H +
                                                (size_t)gi * 8);
      uint32_t wds[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[2 * j] = __uint_as_float(wds[j] << 16);
        v[2 * j + 1] = __uint_as_float(wds[j] & 0xFFFF0000u);
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(x) +
                                                        (size_t)t * H + (size_t)gi * 8);
      float4 a = p[0], b = p[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
  }
  uint16_t ho[8], lo[8];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    uint16_t h = bf16_bits(v[j]);
    float hf = bf16_to_f(h);
    uint16_t l = XBF16 ? (uint16_t)0 : bf16_bits(v[j] - hf);
    ho[perm8_pos(j)] = h;
    lo[perm8_pos(j)] = l;
    s += hf + bf16_to_f(l);
  }
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  if (active) {
    uint4 oh, ol;
    oh.x = ho[0] | ((uint32_t)ho[1] << 16); oh.y = ho[2] | ((uint32_t)ho[3] << 16);
    oh.z = ho[4] | ((uint32_t)ho[5] << 16); oh.w = ho[6] | ((uint32_t)ho[7] << 16);
    ol.x = lo[0] | ((uint32_t)lo[1] << 16); ol.y = lo[2] | ((uint32_t)lo[3] << 16);
    ol.z = lo[4] | ((uint32_t)lo[5] << 16); ol.w = lo[6] | ((uint32_t)lo[7] << 16);
    *reinterpret_cast<uint4*>(xhi + (size_t)t * H + (size_t)gi * 8) = oh;
    *reinterpret_cast<uint4*>(xlo + (size_t)t * H + (size_t)gi * 8) = ol;
    if ((gi & 3) == 0) xcorr[(size_t)t * (H / 32) + gi / 4] = -kMagic * s;
  }
}

// ---------------------------------------------------------------- MMA core
// acc[m][nt][*] += sum over blocks [kb0, kb1) of scale * (codes . B) for the
// lane's accumulator cells (rows g, g+8; token slots nt*8 + 2c, 2c+1).
template <int NMAT, bool SPLIT>
__device__ __forceinline__ void unit_mma(const uint8_t* __restrict__ sq, int qstride,
                                         const uint32_t* __restrict__ ssw, int sw,
                                         const float* __restrict__ corr_s,
                                         const uint16_t* const (&bhi)[2],
                                         const uint16_t* const (&blo)[2], int ntiles, int kb0,
                                         int kb1, float (&acc)[NMAT][2][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
  for (int b = kb0; b < kb1; ++b) {
    uint4 bh[2], bl[2];
    float2 cc[2];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      if (nt < ntiles) {
        bh[nt] = ldg_nc_v4(bhi[nt] + b * 32 + c * 8);
        if (SPLIT) bl[nt] = ldg_nc_v4(blo[nt] + b * 32 + c * 8);
        cc[nt] = *reinterpret_cast<const float2*>(corr_s + b * 16 + nt * 8 + 2 * c);
      }
    }
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      const uint8_t* qm = sq + (size_t)m * kRowTile * qstride + b * 16 + c * 4;
      uint32_t w0 = *reinterpret_cast<const uint32_t*>(qm + g * qstride);
      uint32_t w1 = *reinterpret_cast<const uint32_t*>(qm + (g + 8) * qstride);
      uint32_t d[4], e[4];
      dequant_word(w0, d);
      dequant_word(w1, e);
      const __half* sh = reinterpret_cast<const __half*>(ssw + (size_t)m * kRowTile * sw);
      const float s0 = __half2float(sh[g * 2 * sw + b]);
      const float s1 = __half2float(sh[(g + 8) * 2 * sw + b]);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        if (nt < ntiles) {
          float t[4] = {cc[nt].x, cc[nt].y, cc[nt].x, cc[nt].y};
          mma_bf16_16816(t, d[0], e[0], d[1], e[1], bh[nt].x, bh[nt].y);
          mma_bf16_16816(t, d[2], e[2], d[3], e[3], bh[nt].z, bh[nt].w);
          if (SPLIT) {
            mma_bf16_16816(t, d[0], e[0], d[1], e[1], bl[nt].x, bl[nt].y);
            mma_bf16_16816(t, d[2], e[2], d[3], e[3], bl[nt].z, bl[nt].w);
          }
          acc[m][nt][0] = fmaf(s0, t[0], acc[m][nt][0]);
          acc[m][nt][1] = fmaf(s0, t[1], acc[m][nt][1]);
          acc[m][nt][2] = fmaf(s1, t[2], acc[m][nt][2]);
          acc[m][nt][3] = fmaf(s1, t[3], acc[m][nt][3]);
        }
      }
    }
  }
}

// Issue the bulk copies of 16 code rows of NMAT matrices and load their scales.
template <int NMAT>
__device__ __forceinline__ void unit_load(uint8_t* smem, const UnitSmem& L, uint32_t bar, int K,
                                          const uint8_t* const (&q)[NMAT],
                                          const uint16_t* const (&sc)[NMAT]) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_expect_tx(bar, (uint32_t)(NMAT * kRowTile * (K / 2)));
#pragma unroll
    for (int m = 0; m < NMAT; ++m)
      for (int r = 0; r < kRowTile; ++r)
        bulk_g2s(smem_u32(smem + L.q_off + (size_t)(m * kRowTile + r) * L.qstride),
                 q[m] + (size_t)r * (K / 2), (uint32_t)(K / 2), bar);
  }
  const int nsw = K / 64;  // scale words per row
  uint32_t* ssw = reinterpret_cast<uint32_t*>(smem + L.s_off);
  for (int idx = tid; idx < NMAT * kRowTile * nsw; idx += blockDim.x) {
    int m = idx / (kRowTile * nsw);
    int rem = idx - m * kRowTile * nsw;
    int r = rem / nsw, wd = rem - r * nsw;
    ssw[(m * kRowTile + r) * L.sw + wd] =
        reinterpret_cast<const uint32_t*>(sc[m] + (size_t)r * (K / 32))[wd];
  }
}

// Gate/up + SwiGLU: h = silu(gate x) * (up x) for 16 intermediate rows and up
// to 16 token slots; h is stored as bf16 hi/lo in fragment order, and the
// sum of each 16-row half block goes to hsum for the down kernel's correction.
template <bool SPLIT>
__global__ void __launch_bounds__(256) gateup_kernel(FfnArgs a) {
  const int u = blockIdx.y;
  if (u >= a.counters[1]) return;
  const int2 cu = a.cu[u];
  const ActExpert ex = a.act[cu.x];
  const bool shared = ex.e < 0;
  const int Ie = shared ? a.shI : a.I;
  const int rt = blockIdx.x;
  if (rt * kRowTile >= Ie) return;
  const int K = a.H;
  const int n0 = cu.y * kTokTile;
  const int ntok = min(kTokTile, ex.cnt - n0);
  const int ntiles = ntok > 8 ? 2 : 1;

  extern __shared__ __align__(128) uint8_t smem[];
  const UnitSmem L = unit_smem<2>(K, K);
  const uint32_t bar = smem_u32(smem + L.bar_off);
  __shared__ int s_tok[kTokTile];
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  const size_t qslot = (size_t)Ie * (K / 2), sslot = (size_t)Ie * (K / 32);
  const uint8_t* q[2] = {
      (shared ? a.sgq : a.gq + (size_t)ex.slot * qslot) + (size_t)rt * kRowTile * (K / 2),
      (shared ? a.suq : a.uq + (size_t)ex.slot * qslot) + (size_t)rt * kRowTile * (K / 2)};
  const uint16_t* sc[2] = {
      (shared ? a.sgs : a.gs + (size_t)ex.slot * sslot) + (size_t)rt * kRowTile * (K / 32),
      (shared ? a.sus : a.us + (size_t)ex.slot * sslot) + (size_t)rt * kRowTile * (K / 32)};
  unit_load<2>(smem, L, bar, K, q, sc);

  if (tid < kTokTile) {
    int n = n0 + (tid < ntok ? tid : 0);
    s_tok[tid] = shared ? n : a.sorted_pair[ex.off + n] / a.k;
  }
  __syncthreads();
  const int NB = K / 32;
  float* corr_s = reinterpret_cast<float*>(smem + L.c_off);
  for (int idx = tid; idx < NB * kTokTile; idx += blockDim.x) {
    int b = idx >> 4, n = idx & 15;
    corr_s[idx] = a.xcorr[(size_t)s_tok[n] * NB + b];
  }
  __syncthreads();

  const int lane = tid & 31, warp = tid >> 5, g = lane >> 2;
  const uint16_t* bhi[2];
  const uint16_t* blo[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    int tok = s_tok[nt * 8 + g];
    bhi[nt] = a.xhi + (size_t)tok * K;
    blo[nt] = a.xlo + (size_t)tok * K;
  }
  const int per = (NB + kWarps - 1) / kWarps;
  const int kb0 = min(NB, warp * per), kb1 = min(NB, kb0 + per);
  float acc[2][2][4] = {};
  const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, a.status)) != 0;
  if (ok)
    unit_mma<2, SPLIT>(smem + L.q_off, L.qstride, reinterpret_cast<const uint32_t*>(smem + L.s_off),
                       L.sw, corr_s, bhi, blo, ntiles, kb0, kb1, acc);
  __syncthreads();
  if (!ok) return;
  float* red = reinterpret_cast<float*>(smem + L.q_off);  // [warp][m][nt][128]
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int i = 0; i < 4; ++i) red[((warp * 2 + m) * 2 + nt) * 128 + lane * 4 + i] = acc[m][nt][i];
  __syncthreads();
  const int r = tid >> 4, n = tid & 15, nt = n >> 3, nn = n & 7;
  const int cell = ((r & 7) * 4 + (nn >> 1)) * 4 + (r >> 3) * 2 + (nn & 1);
  float gs = 0.f, us = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    gs += red[((w * 2 + 0) * 2 + nt) * 128 + cell];
    us += red[((w * 2 + 1) * 2 + nt) * 128 + cell];
  }
  const float h = gs / (1.0f + expf(-gs)) * us;
  const uint16_t hi = bf16_bits(h);
  const uint16_t lo = bf16_bits(h - bf16_to_f(hi));
  float* epi = reinterpret_cast<float*>(smem + L.e_off);
  epi[n * 17 + r] = bf16_to_f(hi) + bf16_to_f(lo);
  if (n < ntok) {
    const size_t row = (size_t)(ex.off + n0 + n);
    const int col = rt * kRowTile + r;
    const size_t pos = row * a.Imax + (col & ~7) + perm8_pos(col & 7);
    a.hhi[pos] = hi;
    a.hlo[pos] = lo;
  }
  __syncthreads();
  if (tid < ntok) {
    float s = 0.f;
    for (int rr = 0; rr < kRowTile; ++rr) s += epi[tid * 17 + rr];
    a.hsum[(size_t)(ex.off + n0 + tid) * (a.Imax / 16) + rt] = s;
  }
}

// Down projection: partial[row] = w * (W_down h) for 16 output rows and up to
// 16 token slots; row = the pair's sorted position (P + t for the shared expert).
__global__ void __launch_bounds__(256) down_kernel(FfnArgs a) {
  const int u = blockIdx.y;
  if (u >= a.counters[1]) return;
  const int2 cu = a.cu[u];
  const ActExpert ex = a.act[cu.x];
  const bool shared = ex.e < 0;
  const int K = shared ? a.shI : a.I;
  const int rt = blockIdx.x;
  const int n0 = cu.y * kTokTile;
  const int ntok = min(kTokTile, ex.cnt - n0);
  const int ntiles = ntok > 8 ? 2 : 1;

  extern __shared__ __align__(128) uint8_t smem[];
  const UnitSmem L = unit_smem<1>(K, a.Imax);
  const uint32_t bar = smem_u32(smem + L.bar_off);
  const int tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  const size_t qslot = (size_t)a.H * (K / 2), sslot = (size_t)a.H * (K / 32);
  const uint8_t* q[1] = {(shared ? a.sdq : a.dq + (size_t)ex.slot * qslot) +
                         (size_t)rt * kRowTile * (K / 2)};
  const uint16_t* sc[1] = {(shared ? a.sds : a.ds + (size_t)ex.slot * sslot) +
                           (size_t)rt * kRowTile * (K / 32)};
  unit_load<1>(smem, L, bar, K, q, sc);

  const int NB = K / 32;
  const int hs_stride = a.Imax / 16;
  float* corr_s = reinterpret_cast<float*>(smem + L.c_off);
  for (int idx = tid; idx < NB * kTokTile; idx += blockDim.x) {
    int b = idx >> 4, n = idx & 15;
    size_t row = (size_t)(ex.off + n0 + (n < ntok ? n : 0));
    corr_s[idx] = -kMagic * (a.hsum[row * hs_stride + 2 * b] + a.hsum[row * hs_stride + 2 * b + 1]);
  }
  __syncthreads();
  const int lane = tid & 31, warp = tid >> 5, g = lane >> 2;
  const uint16_t* bhi[2];
  const uint16_t* blo[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    int n = nt * 8 + g;
    size_t row = (size_t)(ex.off + n0 + (n < ntok ? n : 0));
    bhi[nt] = a.hhi + row * a.Imax;
    blo[nt] = a.hlo + row * a.Imax;
  }
  const int per = (NB + kWarps - 1) / kWarps;
  const int kb0 = min(NB, warp * per), kb1 = min(NB, kb0 + per);
  float acc[1][2][4] = {};
  const bool ok = __syncthreads_and(mbar_wait_bounded(bar, 0, a.status)) != 0;
  if (ok)
    unit_mma<1, true>(smem + L.q_off, L.qstride, reinterpret_cast<const uint32_t*>(smem + L.s_off),
                      L.sw, corr_s, bhi, blo, ntiles, kb0, kb1, acc);
  __syncthreads();
  if (!ok) return;
  float* red = reinterpret_cast<float*>(smem + L.q_off);  // [warp][nt][128]
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(warp * 2 + nt) * 128 + lane * 4 + i] = acc[0][nt][i];
  __syncthreads();
  const int r = tid >> 4, n = tid & 15, nt = n >> 3, nn = n & 7;
  const int cell = ((r & 7) * 4 + (nn >> 1)) * 4 + (r >> 3) * 2 + (nn & 1);
  float v = 0.f;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) v += red[(w * 2 + nt) * 128 + cell];
  if (n < ntok) {
    const int s = ex.off + n0 + n;
    const float wt = shared ? 1.0f : a.w[a.sorted_pair[s]];
    a.partial[(size_t)s * a.H + rt * kRowTile + r] = wt * v;
  }
}

// y[t] = sum_{j<k, resident} partial[pair_pos[t*k+j]] (j order) + partial[P+t].
// The routing entries and partial rows of 8 picks are loaded before any is
// summed, so a thread has 8 partial loads in flight instead of one.
__global__ void __launch_bounds__(256) combine_kernel(FfnArgs a, int has_shared) {
  const int t = blockIdx.y;
  const int c4 = blockIdx.x * 256 + threadIdx.x;
  if (c4 * 4 >= a.H) return;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < a.k; j0 += 8) {
    int pos[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      pos[u] = -1;
      const int j = j0 + u;
      if (j < a.k) {
        const int p = t * a.k + j;
        const int e = a.ids[p];
        if (e >= 0 && e < a.E) {
          const int slot = a.slot_map ? a.slot_map[e] : e;
          if (slot >= 0 && slot < a.S) pos[u] = a.pair_pos[p];
        }
      }
    }
    float4 v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      v[u] = pos[u] >= 0 ? *reinterpret_cast<const float4*>(a.partial + (size_t)pos[u] * a.H + (size_t)c4 * 4)
                         : zero;
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (pos[u] >= 0) {
        acc.x += v[u].x; acc.y += v[u].y; acc.z += v[u].z; acc.w += v[u].w;
      }
  }
  if (has_shared) {
    const float4 v =
        *reinterpret_cast<const float4*>(a.partial + (size_t)(a.P + t) * a.H + (size_t)c4 * 4);
    acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
  }
  *reinterpret_cast<float4*>(a.y + (size_t)t * a.H + (size_t)c4 * 4) = acc;
}

// Raise a kernel's dynamic shared-memory limit to the opt-in maximum of the
// device minus the kernel's static shared memory, once per kernel and process
// (the first call normally precedes any graph capture). A failure is consumed
// from the runtime's last-error slot so that it cannot surface in a later call.
static cudaError_t set_smem(const void* fn, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  static std::mutex mu;
  static std::vector<std::pair<const void*, size_t>> done;
  std::lock_guard<std::mutex> lk(mu);
  for (const auto& f : done)
    if (f.first == fn) return bytes <= f.second ? cudaSuccess : cudaErrorInvalidValue;
  int dev = 0, optin = 0;
  cudaFuncAttributes fa{};
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  const size_t limit = optin > (int)fa.sharedSizeBytes ? optin - fa.sharedSizeBytes : 0;
  if (e == cudaSuccess && bytes > limit) e = cudaErrorInvalidValue;
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)limit);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  done.emplace_back(fn, limit);
  return cudaSuccess;
}

// Whether the separate-kernel path takes hidden size H: its gate/up CTA holds 16
// rows of gate and up codes over all of H with their scales and block
// corrections (unit_smem<2>(H, H).total bytes, plus 128 bytes of static shared
// memory) within the 227 KB of shared memory a CTA may opt into on sm_103a.
// That is H <= 11,392 in multiples of 128; the down kernel's rows are I long
// and fit for every I the library takes.
bool ffn_decode_supported(int H) {
  return unit_smem<2>(H, H).total + 128 <= (size_t)227 * 1024;
}

cudaError_t launch_ffn_decode(const FfnArgs& a, const void* x, bool x_bf16, int cu_max,
                              cudaStream_t st) {
  cudaError_t err;
  {
    dim3 grid((a.H / 8 + 255) / 256, a.T);
    launch_begin(K_X_PREP, st);
    if (x_bf16)
      x_prep_kernel<true><<<grid, 256, 0, st>>>(x, a.T, a.H, const_cast<uint16_t*>(a.xhi),
                                                const_cast<uint16_t*>(a.xlo),
                                                const_cast<float*>(a.xcorr));
    else
      x_prep_kernel<false><<<grid, 256, 0, st>>>(x, a.T, a.H, const_cast<uint16_t*>(a.xhi),
                                                 const_cast<uint16_t*>(a.xlo),
                                                 const_cast<float*>(a.xcorr));
    launch_end(st);
  }
  {
    const size_t smem = unit_smem<2>(a.H, a.H).total;
    const int Igu = a.shI > a.I ? a.shI : a.I;
    dim3 grid(Igu / kRowTile, cu_max);
    if ((err = set_smem(x_bf16 ? (const void*)gateup_kernel<false> : (const void*)gateup_kernel<true>,
                        smem)) != cudaSuccess)
      return err;
    launch_begin(K_GATEUP, st);
    if (x_bf16)
      gateup_kernel<false><<<grid, 256, smem, st>>>(a);
    else
      gateup_kernel<true><<<grid, 256, smem, st>>>(a);
    launch_end(st);
  }
  {
    const size_t smem = unit_smem<1>(a.Imax, a.Imax).total;
    dim3 grid(a.H / kRowTile, cu_max);
    if ((err = set_smem((const void*)down_kernel, smem)) != cudaSuccess) return err;
    launch_begin(K_DOWN, st);
    down_kernel<<<grid, 256, smem, st>>>(a);
    launch_end(st);
  }
  {
    dim3 grid((a.H / 4 + 255) / 256, a.T);
    launch_begin(K_COMBINE, st);
    combine_kernel<<<grid, 256, 0, st>>>(a, a.shI > 0 ? 1 : 0);
    launch_end(st);
  }
  return cudaGetLastError();
}

// The ordered combine alone (the prefill path runs its own GEMM kernels first).
cudaError_t launch_combine(const FfnArgs& a, cudaStream_t st) {
  dim3 grid((a.H / 4 + 255) / 256, a.T);
  launch_begin(K_COMBINE, st);
  combine_kernel<<<grid, 256, 0, st>>>(a, a.shI > 0 ? 1 : 0);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace moe
