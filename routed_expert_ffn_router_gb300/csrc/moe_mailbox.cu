// The mailbox: experts the slot map does not hold, computed on the host.
//
// "extended-strata-moe reference", "The mailbox": the GPU keeps its own slot
// map, computes the experts it holds and hands the rows routed to the others
// to host threads; they compute those experts from the host copy of the
// weights and hand back partial outputs, which the GPU adds to the layer output
// in a fixed order. The CPU experts are the pages' multi-token CPU kernels
// (Strata BATCHING): one job is one expert over up to 8 of its rows, so the
// expert's weights are read once per job.
//
// Here the hand-over is stream-ordered: the caller reads the miss list and the
// routing back after the layer call, moe_mailbox_compute runs the jobs on the
// mailbox's threads and waits for them (bounded), the caller copies the
// partials to the device and moe_mailbox_add sums them into y. Host code on
// host buffers, except moe_mailbox_add (one kernel).
#include <algorithm>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstring>
#include <deque>
#include <mutex>
#include <thread>
#include <vector>

#include "moe_internal.h"

namespace {

constexpr int kRowsPerJob = 8;

// IEEE binary16 bit pattern -> float (the format's definition: sign, 5-bit
// exponent with bias 15, 10-bit fraction; subnormals, infinities, NaN).
float half_bits_to_float(uint16_t h) {
  const uint32_t s = (uint32_t)(h >> 15) << 31, e = (h >> 10) & 31u, f = h & 1023u;
  uint32_t bits;
  if (e == 0) {
    if (f == 0) {
      bits = s;
    } else {  // subnormal: f * 2^-24, exact in float
      float v = (float)f * 5.9604644775390625e-8f;
      std::memcpy(&bits, &v, 4);
      bits |= s;
    }
  } else if (e == 31) {
    bits = s | 0x7F800000u | (f << 13);
  } else {
    bits = s | ((e + 112u) << 23) | (f << 13);
  }
  float out;
  std::memcpy(&out, &bits, 4);
  return out;
}

float bf16_bits_to_float(uint16_t b) {
  const uint32_t bits = (uint32_t)b << 16;
  float out;
  std::memcpy(&out, &bits, 4);
  return out;
}

// Row r of a block-quantised matrix with K columns, dequantised into out[K].
void dequant_row(const moe_qmat& m, size_t r, int K, float* out) {
  const uint8_t* q = m.q + r * (size_t)(K / 2);
  const uint16_t* sc = m.scale + r * (size_t)(K / 32);
  for (int b = 0; b < K / 32; ++b) {
    const float s = half_bits_to_float(sc[b]);
    for (int j = 0; j < 16; ++j) {
      const uint8_t byte = q[b * 16 + j];
      const int lo = (int)(byte & 15u) - ((byte & 8u) ? 16 : 0);
      const int hi = (int)(byte >> 4) - ((byte & 128u) ? 16 : 0);
      out[b * 32 + 2 * j] = s * (float)lo;
      out[b * 32 + 2 * j + 1] = s * (float)hi;
    }
  }
}

struct Job {
  int64_t gen;
  int e;       // expert id (its slot in the host store)
  int first;   // first entry of the call's expert-sorted pair list
  int count;   // rows (<= kRowsPerJob)
};

// What one compute call hands to the workers (valid while the call waits).
struct Task {
  moe_layer_desc L;
  const void* x;
  bool x_bf16;
  int k;
  const float* w;
  const int32_t* order;  // pair indices sorted by (expert, pair)
  const int32_t* where;  // position of each listed pair in the caller's list
  float* partial;
};

}  // namespace

struct moe_mailbox {
  std::vector<std::thread> workers;
  std::mutex mu;
  std::condition_variable cv_job, cv_done;
  std::deque<Job> queue;
  int64_t gen = 0;
  int pending = 0;  // jobs of the current call not yet finished
  int active = 0;   // jobs being computed now (any call)
  bool stop = false;
  int timeout_ms = 1000;
  int inject = 0;   // test hook: 1 the next job stalls, 2 the next job is dropped
  Task task{};

  void run() {
    std::vector<float> wrow, xr, g, u, h, o;
    for (;;) {
      Job j;
      Task t;
      {
        std::unique_lock<std::mutex> lk(mu);
        cv_job.wait(lk, [&] { return stop || !queue.empty(); });
        if (stop) return;
        j = queue.front();
        queue.pop_front();
        int inj = inject;
        inject = 0;
        if (inj == 2) continue;  // a peer that dies with the job: nothing comes back
        if (inj == 1) {          // a peer that stalls past the call's limit
          lk.unlock();
          std::this_thread::sleep_for(std::chrono::milliseconds(2 * timeout_ms + 50));
          lk.lock();
        }
        if (j.gen != gen) continue;  // the call gave up: never touch its buffers
        t = task;
        ++active;
      }
      compute(t, j, wrow, xr, g, u, h, o);
      {
        std::lock_guard<std::mutex> lk(mu);
        --active;
        if (j.gen == gen) {
          const int H = t.L.H;
          for (int r = 0; r < j.count; ++r)
            std::memcpy(t.partial + (size_t)t.where[j.first + r] * H, o.data() + (size_t)r * H,
                        sizeof(float) * H);
          --pending;
        }
      }
      cv_done.notify_all();
    }
  }

  // One expert over up to kRowsPerJob rows: g = W_g x, u = W_u x, h = silu(g) u,
  // o = w * (W_d h), fp32 arithmetic, each weight row dequantised once.
  void compute(const Task& t, const Job& j, std::vector<float>& wrow, std::vector<float>& xr,
               std::vector<float>& g, std::vector<float>& u, std::vector<float>& h,
               std::vector<float>& o) {
    const int H = t.L.H, I = t.L.I, n = j.count;
    wrow.resize(std::max(H, I));
    xr.resize((size_t)n * H);
    g.assign((size_t)n * I, 0.f);
    u.assign((size_t)n * I, 0.f);
    h.resize((size_t)n * I);
    o.assign((size_t)n * H, 0.f);
    for (int r = 0; r < n; ++r) {
      const int p = t.order[j.first + r], tok = p / t.k;
      for (int c = 0; c < H; ++c)
        xr[(size_t)r * H + c] =
            t.x_bf16 ? bf16_bits_to_float(static_cast<const uint16_t*>(t.x)[(size_t)tok * H + c])
                     : static_cast<const float*>(t.x)[(size_t)tok * H + c];
    }
    const size_t e = (size_t)j.e;
    for (int i = 0; i < I; ++i) {
      dequant_row(t.L.gate, e * I + i, H, wrow.data());
      for (int r = 0; r < n; ++r) {
        const float* xv = xr.data() + (size_t)r * H;
        float s = 0.f;
        for (int c = 0; c < H; ++c) s += wrow[c] * xv[c];
        g[(size_t)r * I + i] = s;
      }
      dequant_row(t.L.up, e * I + i, H, wrow.data());
      for (int r = 0; r < n; ++r) {
        const float* xv = xr.data() + (size_t)r * H;
        float s = 0.f;
        for (int c = 0; c < H; ++c) s += wrow[c] * xv[c];
        u[(size_t)r * I + i] = s;
      }
    }
    for (size_t i = 0; i < (size_t)n * I; ++i) h[i] = g[i] / (1.f + std::exp(-g[i])) * u[i];
    for (int c = 0; c < H; ++c) {
      dequant_row(t.L.down, e * H + c, I, wrow.data());
      for (int r = 0; r < n; ++r) {
        const float* hv = h.data() + (size_t)r * I;
        float s = 0.f;
        for (int i = 0; i < I; ++i) s += wrow[i] * hv[i];
        o[(size_t)r * H + c] = s;
      }
    }
    for (int r = 0; r < n; ++r) {
      const float wv = t.w[t.order[j.first + r]];
      for (int c = 0; c < H; ++c) o[(size_t)r * H + c] *= wv;
    }
  }
};

namespace moe {

// y[t] += sum of the partials of row t's listed pairs, in list order (ascending
// pair index p = t * k + j). One thread per (row, 4 columns).
__global__ void mailbox_add_kernel(const float* __restrict__ partial, const int32_t* __restrict__ pairs,
                                   int n, int k, int H, float* __restrict__ y) {
  const int c4 = blockIdx.x * blockDim.x + threadIdx.x, t = blockIdx.y;
  if (c4 * 4 >= H) return;
  // the pairs of row t are a contiguous run of the ascending list
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pairs[mid] < t * k) lo = mid + 1;
    else hi = mid;
  }
  float4 acc = reinterpret_cast<float4*>(y + (size_t)t * H)[c4];
  for (int i = lo; i < n && pairs[i] < (t + 1) * k; ++i) {
    const float4 v = reinterpret_cast<const float4*>(partial + (size_t)i * H)[c4];
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  reinterpret_cast<float4*>(y + (size_t)t * H)[c4] = acc;
}

}  // namespace moe

extern "C" {

moe_mailbox* moe_mailbox_create(int32_t n_threads, int32_t timeout_ms) {
  if (n_threads < 1 || n_threads > 1024 || timeout_ms < 1) return nullptr;
  moe_mailbox* mb = new (std::nothrow) moe_mailbox();
  if (!mb) return nullptr;
  mb->timeout_ms = timeout_ms;
  try {
    for (int i = 0; i < n_threads; ++i) mb->workers.emplace_back([mb] { mb->run(); });
  } catch (...) {
    moe_mailbox_destroy(mb);
    return nullptr;
  }
  return mb;
}

void moe_mailbox_destroy(moe_mailbox* mb) {
  if (!mb) return;
  {
    std::lock_guard<std::mutex> lk(mb->mu);
    mb->stop = true;
    ++mb->gen;
  }
  mb->cv_job.notify_all();
  for (std::thread& th : mb->workers)
    if (th.joinable()) th.join();
  delete mb;
}

int32_t moe_mailbox_pairs(const int32_t* ids, int32_t T, int32_t k, const int32_t* slot_map, int32_t E,
                          int32_t* pairs, int32_t n_max) {
  if (T < 0 || k < 1 || E < 1 || (T > 0 && !ids) || !slot_map || n_max < 0) return -1;
  const int64_t P = (int64_t)T * k;
  int32_t n = 0;
  for (int64_t p = 0; p < P; ++p) {
    const int32_t e = ids[p];
    if (e < 0 || e >= E) return -1;
    if (slot_map[e] >= 0) continue;
    if (pairs) {
      if (n >= n_max) return -1;
      pairs[n] = (int32_t)p;
    }
    ++n;
  }
  return n;
}

moe_status moe_mailbox_compute(moe_mailbox* mb, const moe_layer_desc* L, const void* x, moe_dtype x_dtype,
                               int32_t T, const int32_t* ids, const float* w, const int32_t* pairs,
                               int32_t n_pairs, float* partial) {
  if (!mb || !L || T < 0 || n_pairs < 0 || (x_dtype != MOE_F32 && x_dtype != MOE_BF16))
    return MOE_ERR_INVALID;
  if (L->E < 1 || L->k < 1 || L->H < 32 || L->I < 32 || L->H % 32 || L->I % 32) return MOE_ERR_INVALID;
  if (n_pairs == 0) return MOE_OK;
  if (!x || !ids || !w || !pairs || !partial || !L->gate.q || !L->gate.scale || !L->up.q || !L->up.scale ||
      !L->down.q || !L->down.scale)
    return MOE_ERR_INVALID;
  const int64_t P = (int64_t)T * L->k;
  for (int32_t i = 0; i < n_pairs; ++i) {
    if (pairs[i] < 0 || pairs[i] >= P || (i > 0 && pairs[i] <= pairs[i - 1])) return MOE_ERR_INVALID;
    const int32_t e = ids[pairs[i]];
    if (e < 0 || e >= L->E) return MOE_ERR_INVALID;
  }
  // jobs: the listed pairs grouped by expert (pair order within an expert), at
  // most kRowsPerJob rows each
  std::vector<int32_t> order(pairs, pairs + n_pairs), where(n_pairs);
  std::stable_sort(order.begin(), order.end(),
                   [&](int32_t a, int32_t b) { return ids[a] < ids[b]; });
  for (int32_t i = 0; i < n_pairs; ++i)
    where[i] = (int32_t)(std::lower_bound(pairs, pairs + n_pairs, order[i]) - pairs);
  std::unique_lock<std::mutex> lk(mb->mu);
  const int64_t g = ++mb->gen;
  mb->task = Task{*L, x, x_dtype == MOE_BF16, L->k, w, order.data(), where.data(), partial};
  int njobs = 0;
  for (int32_t i = 0; i < n_pairs;) {
    const int32_t e = ids[order[i]];
    int32_t j = i;
    while (j < n_pairs && ids[order[j]] == e && j - i < kRowsPerJob) ++j;
    mb->queue.push_back(Job{g, e, i, j - i});
    ++njobs;
    i = j;
  }
  mb->pending = njobs;
  mb->cv_job.notify_all();
  const bool done = mb->cv_done.wait_for(lk, std::chrono::milliseconds(mb->timeout_ms),
                                         [&] { return mb->pending == 0; });
  if (done) return MOE_OK;
  // give up: no worker starts or reports a job of this call from now on; the
  // jobs being computed stop reading the caller's buffers before it returns
  ++mb->gen;
  mb->queue.clear();
  mb->cv_done.wait(lk, [&] { return mb->active == 0; });
  return MOE_ERR_TIMEOUT;
}

moe_status moe_mailbox_inject(moe_mailbox* mb, int32_t mode) {
  if (!mb || mode < 0 || mode > 2) return MOE_ERR_INVALID;
  std::lock_guard<std::mutex> lk(mb->mu);
  mb->inject = mode;
  return MOE_OK;
}

moe_status moe_mailbox_add(const float* partial, const int32_t* pairs, int32_t n, int32_t T, int32_t k,
                           int32_t H, float* y, void* stream) {
  if (n < 0 || T < 0 || k < 1 || H < 4 || H % 4) return MOE_ERR_INVALID;
  if (n == 0 || T == 0) return MOE_OK;
  if (!partial || !pairs || !y || (reinterpret_cast<uintptr_t>(partial) & 15u) ||
      (reinterpret_cast<uintptr_t>(y) & 15u))
    return MOE_ERR_INVALID;
  if (T > 65535) return MOE_ERR_UNSUPPORTED;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dim3 grid((H / 4 + 127) / 128, T);
  moe::launch_begin(moe::K_COMBINE, st);
  moe::mailbox_add_kernel<<<grid, 128, 0, st>>>(partial, pairs, n, k, H, y);
  moe::launch_end(st);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
