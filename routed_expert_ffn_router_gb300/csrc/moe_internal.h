// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe_common.cuh"

namespace moe {

// Kernel kinds for the optional event timing (moe_profile_*).
enum KernelKind : int {
  K_ROUTER_LOGITS = 0, K_ROUTE, K_PERMUTE, K_X_PREP, K_GATEUP, K_DOWN, K_COMBINE, K_FUSED,
  K_FUSED_STACK,
  K_NUM_KINDS
};

// Every kernel launch is bracketed by these: they count launches and, when
// timing is enabled, record a CUDA event pair on the launching stream.
void launch_begin(int kind, cudaStream_t st);
void launch_end(cudaStream_t st);

// Sizes the host validated; everything a launch needs besides pointers.
struct Shape {
  int H, I, shI, E, k, S, T, P, Imax;
};

WsLayout ws_layout(int E, int k, int T, int H, int I, int shI);

struct PermuteOut {
  int32_t* offsets;
  int32_t* sorted_pair;
  int32_t* pair_pos;
  int32_t* miss_ids;
  int32_t* n_miss;
  ActExpert* act;
  int2* cu;          // column units: (active index, token chunk of 16)
  int32_t* counters;  // [0] active experts incl. shared, [1] column units
  int32_t* hist;      // chunked path scratch [n_chunks][E]
  int32_t* status;
};

struct FfnArgs {
  const uint8_t *gq, *uq, *dq;
  const uint16_t *gs, *us, *ds;
  const uint8_t *sgq, *suq, *sdq;
  const uint16_t *sgs, *sus, *sds;
  int H, I, shI, E, k, S, T, P, Imax;
  const int32_t* sorted_pair;
  const int32_t* pair_pos;
  const int32_t* ids;
  const float* w;
  const int32_t* slot_map;
  const ActExpert* act;
  const int2* cu;
  const int32_t* counters;
  const uint16_t* xhi;
  const uint16_t* xlo;
  const float* xcorr;
  uint16_t* hhi;
  uint16_t* hlo;
  float* hsum;
  float* partial;
  float* y;
  int32_t* status;
};

cudaError_t launch_router_logits(const void* x, bool x_bf16, const float* wg, int T, int H, int E,
                                 float* logits, cudaStream_t st);
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* ids, float* w,
                         int32_t* status, cudaStream_t st);
cudaError_t launch_permute(const int32_t* ids, int T, int E, int k, const int32_t* slot_map, int S,
                           bool has_shared, const PermuteOut& o, cudaStream_t st);
cudaError_t launch_ffn_decode(const FfnArgs& a, const void* x, bool x_bf16, int cu_max,
                              cudaStream_t st);
// counts[e] += 1 for every expert with rows in the permutation (offsets [E+1]).
cudaError_t launch_count_picks(const int32_t* offsets, int E, int32_t* counts, cudaStream_t st);

int cu_bound(int T, int E, int k, bool has_shared);
cudaError_t launch_combine(const FfnArgs& a, cudaStream_t st);

// The prefill path on the tcgen05 tensor cores (moe_prefill.cu): gate/up +
// SwiGLU into expert-sorted h, down into weighted partials; launch_combine
// then forms y.
bool prefill_tc_supported(int H, int I, int shI, int T, bool x_bf16);
cudaError_t launch_ffn_prefill_tc(const FfnArgs& a, const void* x, cudaStream_t st);

// The one-launch decode path (moe_fused.cu).
struct FusedLaunch {
  const uint8_t *gq, *uq, *dq;
  const uint16_t *gs, *us, *ds;
  const uint8_t *sgq, *suq, *sdq;
  const uint16_t *sgs, *sus, *sds;
  int H, I, shI, E, k, S, T, Imax, rows_cap;
  const float* logits;     // layer mode when non-null
  const int32_t* ids_in;
  const float* w_in;
  const void* x;
  const int32_t* slot_map;
  int32_t* ids_out;
  float* w_out;
  float* y;
  int32_t* miss_ids;
  int32_t* n_miss;
  uint16_t* hhi;
  uint16_t* hlo;
  float* hcorr;
  float* partial;
  int32_t* status;
  int32_t* sync;
  int32_t* picks;  // nullable: +1 per distinct routed expert (adaptive-cache counters)
  // a chained stack with the router in the launch (else null): router weights
  // [E][H] bf16 (logits written to `logits`), and the next layer's input
  const uint16_t* router_w;
  uint16_t* x_next;
};
bool fused_decode_supported(int H, int I, int shI, int T, bool x_bf16);
// Slices of I per partial row of the one-launch path (the partial buffer holds
// rows x slices x H floats).
int fused_partial_slices(int E, int k, int T, int I, int shI);
cudaError_t launch_fused_decode(const FusedLaunch& f, cudaStream_t st);
// Several layers' windows in one launch: a plan of per-layer kernel arguments
// in device memory (fused_stack_plan_bytes(L) bytes, 64-byte aligned), built
// from the layers' launches (same T; the cross-CTA counters of layer l at
// layers[0].sync + a per-layer offset) and copied there synchronously.
size_t fused_stack_plan_bytes(int L);
int fused_stack_max_layers();
cudaError_t fused_stack_prepare(const FusedLaunch* layers, int L, void* plan, cudaStream_t st);
cudaError_t launch_fused_stack(const void* plan, int L, int T, int32_t* sync, int32_t* status,
                               cudaStream_t st);

}  // namespace moe
