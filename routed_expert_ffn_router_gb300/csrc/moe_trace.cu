// Routing traces ("extended-strata-moe reference", "Routing trace format"): a
// dump of the routing, one record per token and layer, little-endian:
// int32 layer, int32 k, k x int32 expert id, k x float32 weight. Host code on
// host buffers (the routing is copied back from moe_route / moe_layer_forward
// first); the page's dumping tool writes the weights as 0, which a null
// weight array reproduces.
#include <cstdint>
#include <cstring>

#include "moe.h"

namespace {

void put32(uint8_t* p, uint32_t v) {
  for (int i = 0; i < 4; ++i) p[i] = (uint8_t)(v >> (8 * i));
}
uint32_t get32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

}  // namespace

extern "C" {

int64_t moe_trace_write(int32_t layer, const int32_t* ids, const float* w, int32_t T, int32_t k, uint8_t* buf,
                        int64_t n_max) {
  if (T < 0 || k < 1 || k > 1 << 20 || (T > 0 && !ids) || n_max < 0) return -1;
  const int64_t rec = 8 + 8 * (int64_t)k, size = rec * T;
  if (n_max == 0) return size;
  if (!buf || n_max < size) return -1;
  uint8_t* q = buf;
  for (int32_t t = 0; t < T; ++t) {
    put32(q, (uint32_t)layer);
    put32(q + 4, (uint32_t)k);
    q += 8;
    for (int32_t j = 0; j < k; ++j, q += 4) put32(q, (uint32_t)ids[(size_t)t * k + j]);
    for (int32_t j = 0; j < k; ++j, q += 4) {
      uint32_t bits = 0;
      if (w) std::memcpy(&bits, &w[(size_t)t * k + j], 4);
      put32(q, bits);
    }
  }
  return size;
}

int64_t moe_trace_read(const uint8_t* buf, int64_t n, int32_t* layer, int32_t* k_out, int32_t* ids, float* w,
                       int32_t k_max, int64_t n_max) {
  if (!buf || n < 0 || k_max < 1 || n_max < 0) return -1;
  if (n_max > 0 && (!layer || !k_out || !ids || !w)) return -1;
  int64_t off = 0, r = 0;
  while (off < n) {
    if (n - off < 8) return -1;  // a truncated record
    const int32_t lay = (int32_t)get32(buf + off), k = (int32_t)get32(buf + off + 4);
    if (k < 1 || k > k_max || n - off < 8 + 8 * (int64_t)k) return -1;
    if (n_max > 0) {
      if (r >= n_max) return -1;
      layer[r] = lay;
      k_out[r] = k;
      for (int32_t j = 0; j < k_max; ++j) {
        ids[r * k_max + j] = j < k ? (int32_t)get32(buf + off + 8 + 4 * j) : -1;
        uint32_t bits = j < k ? get32(buf + off + 8 + 4 * (int64_t)k + 4 * j) : 0u;
        std::memcpy(&w[r * k_max + j], &bits, 4);
      }
    }
    off += 8 + 8 * (int64_t)k;
    ++r;
  }
  return r;
}

}  // extern "C"
