// Router kernels: fp64-accumulated router GEMV (tiny configuration) and the
// warp-per-row top-k + softmax.
//
// Routing follows "extended-strata-moe reference", "Routing trace format" (a
// token's routing is k expert ids plus k fp32 weights) and the top-10-of-512
// router of the SGLang port post. Order: logit descending, ties to the lower
// id; weights: softmax over the k selected, one rounding to fp32 (float-float
// arithmetic standing in for float64, see topk_softmax_weight).
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

// One warp per row: topk_row (ids in rank order, ties to the lower id; the
// threshold of the lane maxima, then ranking by counting), then
// topk_softmax_weight with lane j holding the j-th pick's logit.
template <int NPER>
__device__ __forceinline__ void route_row(const float* l, int E, int k, unsigned long long* scr, int* sid,
                                          int32_t* ids, float* w, int32_t* status) {
  const int lane = threadIdx.x & 31;
  const bool bad = topk_row<NPER>(l, E, k, scr, sid);
  if (bad && lane == 0 && status) atomicOr(status, DEV_NONFINITE_LOGIT);
  const float v = lane < k ? key_value((uint32_t)(scr[kTopkRanked + lane] >> 32)) : 0.f;
  const float wv = topk_softmax_weight(v, k);
  if (lane < k) {
    ids[lane] = sid[lane];
    w[lane] = wv;
  }
}

__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ ids,
                                                    float* __restrict__ w,
                                                    int32_t* __restrict__ status) {
  __shared__ unsigned long long s_scr[8][kTopkScratch];
  __shared__ int s_id[8][kMaxK];
  const int wp = threadIdx.x >> 5;
  const int t = blockIdx.x * 8 + wp;
  if (t >= T) return;
  const float* l = logits + (size_t)t * E;
  int32_t* ir = ids + (size_t)t * k;
  float* wr = w + (size_t)t * k;
  if (E <= 128) route_row<4>(l, E, k, s_scr[wp], s_id[wp], ir, wr, status);
  else if (E <= 256) route_row<8>(l, E, k, s_scr[wp], s_id[wp], ir, wr, status);
  else if (E <= 512) route_row<16>(l, E, k, s_scr[wp], s_id[wp], ir, wr, status);
  else route_row<32>(l, E, k, s_scr[wp], s_id[wp], ir, wr, status);
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
