// moe_expert_ffn_static: the routed-expert FFN for callers that cannot
// allocate device memory.
//
// Some callers have no way to obtain a workspace: code that runs inside a
// host framework whose allocator owns all device memory and forbids raw
// cudaMalloc, plugin or driver-level code without an allocator handle, and
// latency-critical decode loops where a cudaMalloc/cudaFree could synchronise
// the device. For them this entry point takes the same inputs and outputs as
// moe_expert_ffn but uses, as its scratch, a fixed array in the library's own
// device memory (kStaticScratchBytes, reserved on every GPU that loads the
// library until the process exits). It calls no allocating routine.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the status word at its start is cleared on each call and read
// back by moe_static_read_status. Calls that
// overlap on the GPU (other streams, other host threads) race on the array and
// must be serialised by the caller. The first call on a device looks up the
// array's device address (once, with that device current); make that first
// call before any stream capture.
#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

std::mutex g_static_mu;
void* g_static_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (nullptr on error).
// In host code the array's name is only a host-side handle; the address the
// kernels need comes from cudaGetSymbolAddress, once per device.
void* static_scratch_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return nullptr;
    }
    g_static_ptr[dev] = p;
  }
  return g_static_ptr[dev];
}

}  // namespace

extern "C" moe_status moe_expert_ffn_static(const moe_layer_desc* L, const void* x,
                                            moe_dtype x_dtype, int T, const int32_t* ids,
                                            const float* w, const int32_t* slot_map, float* y,
                                            int32_t* miss_ids, int32_t* n_miss, void* stream) {
  const size_t need = moe_workspace_bytes(L, T);
  if (need == 0 || T < 0)  // invalid desc or T: let the regular entry point report which
    return moe_expert_ffn(L, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, nullptr, 0,
                          stream);
  if (need > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
  void* ws = static_scratch_ptr();
  if (!ws) return MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the previous call's status bits and counters must not leak into this one
  if (cudaMemsetAsync(ws, 0, moe::kWsHeadBytes, st) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return moe_expert_ffn(L, x, x_dtype, T, ids, w, slot_map, y, miss_ids, n_miss, ws,
                        kStaticScratchBytes, stream);
}

extern "C" moe_status moe_static_read_status(void* stream, int32_t* out) {
  if (!out) return MOE_ERR_INVALID;
  void* ws = static_scratch_ptr();
  if (!ws) return MOE_ERR_CUDA;
  return moe_read_status(ws, stream, out);
}
