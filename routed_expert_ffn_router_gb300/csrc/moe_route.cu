// Router kernels: fp64-accumulated router GEMV (tiny configuration) and the
// warp-per-row top-k + softmax.
//
// Routing follows "extended-strata-moe reference", "Routing trace format" (a
// token's routing is k expert ids plus k fp32 weights) and the top-10-of-512
// router of the SGLang port post. Order: logit descending, ties to the lower
// id; weights: softmax over the k selected, float64, one rounding to fp32.
#include "moe_internal.h"

namespace moe {

// logits[t][e] = fp32(sum_h x[t][h] * wg[h][e]); the sum runs in h order in
// float64. Each product of two fp32 (or bf16 x fp32) values is exact in
// float64, so the fused multiply-add below rounds exactly like a separate
// multiply and add: the result is reproducible bit for bit.
template <bool XBF16>
__global__ void router_logits_kernel(const void* __restrict__ x, const float* __restrict__ wg,
                                     int T, int H, int E, float* __restrict__ logits) {
  int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= T * E) return;
  int t = idx / E, e = idx % E;
  double s = 0.0;
  for (int h = 0; h < H; ++h) {
    double xv = XBF16 ? (double)bf16_to_f(static_cast<const uint16_t*>(x)[(size_t)t * H + h])
                      : (double)static_cast<const float*>(x)[(size_t)t * H + h];
    s = fma(xv, (double)wg[(size_t)h * E + e], s);
  }
  logits[idx] = (float)s;
}

// One warp per row. Each lane owns experts e = lane + 32*i (i < ceil(E/32));
// its taken flags live in one register. k rounds of a warp arg-max pick the
// experts in order; a candidate beats another if its logit is larger, or equal
// with a lower id. Weights: lane j holds e_j = exp(l_j - l_0) in float64; every
// lane forms s = e_0 + e_1 + ... in j order through shuffles, then
// w_j = fp32(e_j / s).
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w,
                                                    int32_t* __restrict__ status) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  const int nper = (E + 31) >> 5;  // <= 32
  float v[32];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    int e = lane + 32 * i;
    v[i] = (i < nper && e < E) ? l[e] : 0.f;
    if (i < nper && e < E && !isfinite(v[i])) bad = true;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0 && status) atomicOr(status, DEV_NONFINITE_LOGIT);
  uint32_t taken = 0;
  float my_v = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      int e = lane + 32 * i;
      if (i < nper && e < E && !((taken >> i) & 1u)) {
        if (be == 0x7fffffff || v[i] > bv) {  // ascending e: strict '>' keeps the lower id
          bv = v[i];
          be = e;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oe = __shfl_xor_sync(0xffffffffu, be, off);
      bool take = (be == 0x7fffffff) || (oe != 0x7fffffff && (ov > bv || (ov == bv && oe < be)));
      if (take) {
        bv = ov;
        be = oe;
      }
    }
    if (be == 0x7fffffff) be = 0;  // only with non-finite input (already flagged)
    if ((be & 31) == lane) taken |= 1u << (be >> 5);
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const double m = (double)__shfl_sync(0xffffffffu, my_v, 0);
  double ej = (lane < k) ? exp((double)my_v - m) : 0.0;
  double s = 0.0;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xffffffffu, ej, j);
  if (lane < k) {
    ids[(size_t)t * k + lane] = my_e;
    w[(size_t)t * k + lane] = (float)(ej / s);
  }
}

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wg, int T, int H, int E,
                                 float* logits, cudaStream_t st) {
  int n = T * E;
  dim3 grid((n + 255) / 256);
  launch_begin(K_ROUTER_LOGITS, st);
  if (x_bf16)
    router_logits_kernel<true><<<grid, 256, 0, st>>>(x, wg, T, H, E, logits);
  else
    router_logits_kernel<false><<<grid, 256, 0, st>>>(x, wg, T, H, E, logits);
  launch_end(st);
  return cudaGetLastError();
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         int32_t* status, cudaStream_t st) {
  dim3 grid((T + 7) / 8);
  launch_begin(K_ROUTE, st);
  route_kernel<<<grid, 256, 0, st>>>(logits, T, E, k, ids, w, status);
  launch_end(st);
  return cudaGetLastError();
}

}  // namespace moe
