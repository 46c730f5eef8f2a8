// C-ABI entry points of libtw (declared and documented in include/tw.h).
// Validation happens here, before any CUDA call; kernels are in fused_kernel.cu.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "tw.h"
#include "tw_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether [a, a + na) and [b, b + nb) share a byte.
bool overlap(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + static_cast<uintptr_t>(nb) && y < x + static_cast<uintptr_t>(na);
}

// Checks that do not look at pointers (shared by the launch-shape query).
int validate_shape(int N, float eps, int64_t T, int64_t H, int sm_budget) {
  if (N < 1 || N > TW_MAX_PARTIALS) return TW_ERR_INVALID_ARG;
  if (T < 0 || H <= 0) return TW_ERR_INVALID_ARG;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return TW_ERR_INVALID_ARG;
  if (sm_budget < 0) return TW_ERR_INVALID_ARG;
  if (H % 8 != 0) return TW_ERR_ALIGN;
  if (H > TW_MAX_HIDDEN) return TW_ERR_UNSUPPORTED;
  if (T > (INT64_MAX / 4) / H) return TW_ERR_INVALID_ARG;  // T * H * 2 bytes must not overflow
  return TW_OK;
}

// Full validation of one fused call over rows [0, T); fills the kernel args.
int validate(const void* const* partials, int N, void* residual, const void* gamma, float eps,
             int64_t T, int64_t H, void* out, int sm_budget, tw::FusedArgs* a) {
  int st = validate_shape(N, eps, T, H, sm_budget);
  if (st != TW_OK) return st;
  if (T == 0) return TW_OK;
  if (!partials || !residual || !gamma || !out) return TW_ERR_INVALID_ARG;
  for (int r = 0; r < N; ++r)
    if (!partials[r]) return TW_ERR_INVALID_ARG;
  for (int r = 0; r < N; ++r)
    if (!aligned16(partials[r])) return TW_ERR_ALIGN;
  if (!aligned16(residual) || !aligned16(gamma) || !aligned16(out)) return TW_ERR_ALIGN;
  const int64_t bytes = T * H * 2;
  // The two written tensors may overlap nothing else (inputs may alias each
  // other), except that out may be exactly one partial's buffer: a row's
  // partial chunks are all staged before the row's output is written, and
  // staging runs ahead only into later rows.
  if (overlap(residual, bytes, out, bytes)) return TW_ERR_INVALID_ARG;
  for (void* w : {residual, out}) {
    if (overlap(w, bytes, gamma, H * 2)) return TW_ERR_INVALID_ARG;
    for (int r = 0; r < N; ++r)
      if (overlap(w, bytes, partials[r], bytes) && !(w == out && out == partials[r]))
        return TW_ERR_INVALID_ARG;
  }
  for (int r = 0; r < N; ++r) a->partials[r] = partials[r];
  a->n = N;
  a->residual = residual;
  a->gamma = gamma;
  a->out = out;
  a->eps = eps;
  a->rows = T;
  a->hidden = H;
  return TW_OK;
}

// The split's fork and join events: one pair per (host thread, device), taken
// from a process-wide pool on the thread's first split call on that device and
// handed back to the pool when the thread exits. A pair is reused only after
// the stream waits that consumed its previous records were enqueued, so reuse
// keeps the ordering. Handing back makes no CUDA call (the context may already
// be gone at thread or process exit); pooled events live until the process
// ends, so their number is bounded by the most threads that ever called at
// once, however many short-lived threads call over time.
constexpr int kMaxDevices = 64;
struct EventPair {
  cudaEvent_t fork = nullptr;
  cudaEvent_t join = nullptr;
};
struct EventPool {
  std::mutex mutex;
  std::vector<EventPair> free[kMaxDevices];
};
EventPool& event_pool() {
  static EventPool* pool = new EventPool;  // never destroyed: used by thread-exit hand-backs
  return *pool;
}
struct ThreadEvents {
  EventPair pair[kMaxDevices];
  ~ThreadEvents() {
    EventPool& pool = event_pool();
    std::lock_guard<std::mutex> lock(pool.mutex);
    for (int d = 0; d < kMaxDevices; ++d)
      if (pair[d].fork) pool.free[d].push_back(pair[d]);
  }
};
thread_local ThreadEvents t_events;

int split_events(cudaEvent_t* fork, cudaEvent_t* join) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TW_ERR_CUDA;
  EventPair& mine = t_events.pair[dev];
  if (!mine.fork) {
    EventPair got;
    {
      EventPool& pool = event_pool();
      std::lock_guard<std::mutex> lock(pool.mutex);
      if (!pool.free[dev].empty()) {
        got = pool.free[dev].back();
        pool.free[dev].pop_back();
      }
    }
    if (!got.fork) {
      if (cudaEventCreateWithFlags(&got.fork, cudaEventDisableTiming) != cudaSuccess)
        return TW_ERR_CUDA;
      if (cudaEventCreateWithFlags(&got.join, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(got.fork);
        return TW_ERR_CUDA;
      }
    }
    mine = got;
  }
  *fork = mine.fork;
  *join = mine.join;
  return TW_OK;
}

// Rows [row0, row0 + rows) of a validated call.
tw::FusedArgs slice(const tw::FusedArgs& a, int64_t row0, int64_t rows) {
  tw::FusedArgs s = a;
  const int64_t off = row0 * a.hidden * 2;
  for (int r = 0; r < a.n; ++r) s.partials[r] = static_cast<const char*>(a.partials[r]) + off;
  s.residual = static_cast<char*>(a.residual) + off;
  s.out = static_cast<char*>(a.out) + off;
  s.rows = rows;
  return s;
}

}  // namespace

extern "C" int tw_fused_reduce_residual_rmsnorm(const void* const* partials, int N, void* residual,
                                                const void* gamma, float eps, int64_t T, int64_t H,
                                                void* out, tw_stream_t stream, int sm_budget) {
  try {
    tw::FusedArgs a;
    const int st = validate(partials, N, residual, gamma, eps, T, H, out, sm_budget, &a);
    if (st != TW_OK || T == 0) return st;
    return tw::launch_fused(a, reinterpret_cast<cudaStream_t>(stream), sm_budget, nullptr);
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_fused_debug_smid(const void* const* partials, int N, void* residual,
                                   const void* gamma, float eps, int64_t T, int64_t H, void* out,
                                   tw_stream_t stream, int sm_budget, int* smid_out) {
  try {
    if (!smid_out) return TW_ERR_INVALID_ARG;
    tw::FusedArgs a;
    const int st = validate(partials, N, residual, gamma, eps, T, H, out, sm_budget, &a);
    if (st != TW_OK || T == 0) return st;
    return tw::launch_fused(a, reinterpret_cast<cudaStream_t>(stream), sm_budget, smid_out);
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

namespace {

// The split runner on validated arguments (`a` is filled only when T > 0),
// prefix_tokens in [0, T].
int run_split(const tw::FusedArgs& a, int64_t T, int64_t prefix_tokens, tw_stream_t stream_a,
              tw_stream_t stream_b, int sm_budget) {
  if (T == 0) return TW_OK;
  cudaStream_t sa = reinterpret_cast<cudaStream_t>(stream_a);
  cudaStream_t sb = reinterpret_cast<cudaStream_t>(stream_b);
  const int64_t suffix = T - prefix_tokens;
  int st = TW_OK;
  if (suffix == 0 || sa == sb) {
    if (prefix_tokens > 0 &&
        (st = tw::launch_fused(slice(a, 0, prefix_tokens), sa, sm_budget, nullptr)) != TW_OK)
      return st;
    if (suffix > 0)
      return tw::launch_fused(slice(a, prefix_tokens, suffix), sa, sm_budget, nullptr);
    return TW_OK;
  }
  cudaEvent_t fork = nullptr, join = nullptr;
  if ((st = split_events(&fork, &join)) != TW_OK) return st;
  if (cudaEventRecord(fork, sa) != cudaSuccess || cudaStreamWaitEvent(sb, fork, 0) != cudaSuccess)
    return TW_ERR_CUDA;
  if (prefix_tokens > 0 &&
      (st = tw::launch_fused(slice(a, 0, prefix_tokens), sa, sm_budget, nullptr)) != TW_OK)
    return st;
  if ((st = tw::launch_fused(slice(a, prefix_tokens, suffix), sb, sm_budget, nullptr)) != TW_OK)
    return st;
  if (cudaEventRecord(join, sb) != cudaSuccess || cudaStreamWaitEvent(sa, join, 0) != cudaSuccess)
    return TW_ERR_CUDA;
  return TW_OK;
}

}  // namespace

extern "C" int tw_run_split(int64_t prefix_tokens, const void* const* partials, int N,
                            void* residual, const void* gamma, float eps, int64_t T, int64_t H,
                            void* out, tw_stream_t stream_a, tw_stream_t stream_b, int sm_budget) {
  try {
    tw::FusedArgs a;
    const int st = validate(partials, N, residual, gamma, eps, T, H, out, sm_budget, &a);
    if (st != TW_OK) return st;
    if (prefix_tokens < 0 || prefix_tokens > T) return TW_ERR_INVALID_ARG;
    return run_split(a, T, prefix_tokens, stream_a, stream_b, sm_budget);
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_run_wave_split(int64_t ctas_unsplit, int num_sms, const tw_split_opts* opts,
                                 const void* const* partials, int N, void* residual,
                                 const void* gamma, float eps, int64_t T, int64_t H, void* out,
                                 tw_stream_t stream_a, tw_stream_t stream_b, int sm_budget,
                                 int64_t* prefix_tokens, int64_t* suffix_tokens) {
  try {
    tw::FusedArgs a;
    int st = validate(partials, N, residual, gamma, eps, T, H, out, sm_budget, &a);
    if (st != TW_OK) return st;
    int64_t prefix = 0, suffix = 0;
    if ((st = tw_wave_split(T, ctas_unsplit, num_sms, opts, &prefix, &suffix)) != TW_OK) return st;
    if (prefix_tokens) *prefix_tokens = prefix;
    if (suffix_tokens) *suffix_tokens = suffix;
    return run_split(a, T, prefix, stream_a, stream_b, sm_budget);
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_run_split_after(int64_t prefix_tokens, const void* const* partials, int N,
                                  void* residual, const void* gamma, float eps, int64_t T,
                                  int64_t H, void* out, tw_stream_t stream, tw_event_t prefix_ready,
                                  tw_event_t suffix_ready, int sm_budget) {
  try {
    tw::FusedArgs a;
    int st = validate(partials, N, residual, gamma, eps, T, H, out, sm_budget, &a);
    if (st != TW_OK) return st;
    if (prefix_tokens < 0 || prefix_tokens > T) return TW_ERR_INVALID_ARG;
    if (T == 0) return TW_OK;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int64_t suffix = T - prefix_tokens;
    if (prefix_ready &&
        cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(prefix_ready), 0) != cudaSuccess)
      return TW_ERR_CUDA;
    if (prefix_tokens > 0 &&
        (st = tw::launch_fused(slice(a, 0, prefix_tokens), s, sm_budget, nullptr)) != TW_OK)
      return st;
    if (suffix_ready &&
        cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(suffix_ready), 0) != cudaSuccess)
      return TW_ERR_CUDA;
    if (suffix > 0) return tw::launch_fused(slice(a, prefix_tokens, suffix), s, sm_budget, nullptr);
    return TW_OK;
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_reduce_partials(const void* const* partials, int N, int64_t T, int64_t H,
                                  void* sum_out, tw_stream_t stream) {
  try {
    int st = validate_shape(N, 0.0f, T, H, 0);
    if (st != TW_OK || T == 0) return st;
    if (!partials || !sum_out) return TW_ERR_INVALID_ARG;
    for (int r = 0; r < N; ++r)
      if (!partials[r]) return TW_ERR_INVALID_ARG;
    for (int r = 0; r < N; ++r)
      if (!aligned16(partials[r])) return TW_ERR_ALIGN;
    if (!aligned16(sum_out)) return TW_ERR_ALIGN;
    const int64_t bytes = T * H * 2;
    for (int r = 0; r < N; ++r)
      if (overlap(sum_out, bytes, partials[r], bytes)) return TW_ERR_INVALID_ARG;
    return tw::launch_reduce(partials, N, T, H, sum_out, reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_add_rmsnorm(const void* sum, void* residual, const void* gamma, float eps,
                              int64_t T, int64_t H, void* out, tw_stream_t stream) {
  try {
    int st = validate_shape(1, eps, T, H, 0);
    if (st != TW_OK || T == 0) return st;
    if (!sum || !residual || !gamma || !out) return TW_ERR_INVALID_ARG;
    if (!aligned16(sum) || !aligned16(residual) || !aligned16(gamma) || !aligned16(out))
      return TW_ERR_ALIGN;
    const int64_t bytes = T * H * 2;
    if (overlap(residual, bytes, out, bytes) || overlap(residual, bytes, sum, bytes))
      return TW_ERR_INVALID_ARG;
    if (overlap(residual, bytes, gamma, H * 2) || overlap(out, bytes, gamma, H * 2))
      return TW_ERR_INVALID_ARG;
    if (sum != out && overlap(sum, bytes, out, bytes)) return TW_ERR_INVALID_ARG;  // same buffer is fine
    return tw::launch_add_rmsnorm(sum, residual, gamma, eps, T, H, out,
                                  reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_launch_shape(int64_t T, int64_t H, int N, int sm_budget, int* grid, int* threads,
                               int* smem_bytes, int* stages) {
  try {
    const int st = validate_shape(N, 0.0f, T, H, sm_budget);
    if (st != TW_OK) return st;
    tw::LaunchShape s;
    const int q = tw::plan_launch(T, H, N, sm_budget, &s);
    if (q != TW_OK) return q;
    if (grid) *grid = s.grid;
    if (threads) *threads = s.threads;
    if (smem_bytes) *smem_bytes = s.smem_bytes;
    if (stages) *stages = s.stages;
    return TW_OK;
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_device_status(int reset, int* code) {
  try {
    if (!code) return TW_ERR_INVALID_ARG;
    return tw::read_device_error(reset, code);
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" int tw_debug_wait_timeout(int64_t limit_ns, tw_stream_t stream) {
  try {
    if (limit_ns < 1000 || limit_ns > 2000000000ll) return TW_ERR_INVALID_ARG;
    return tw::launch_wait_probe(limit_ns, reinterpret_cast<cudaStream_t>(stream));
  } catch (...) {
    return TW_ERR_CUDA;
  }
}

extern "C" const char* tw_strerror(int status) {
  switch (status) {
    case TW_OK: return "TW_OK: success";
    case TW_ERR_INVALID_ARG: return "TW_ERR_INVALID_ARG: invalid argument";
    case TW_ERR_ALIGN: return "TW_ERR_ALIGN: H must be a multiple of 8 and pointers 16-byte aligned";
    case TW_ERR_UNSUPPORTED: return "TW_ERR_UNSUPPORTED: hidden size above TW_MAX_HIDDEN";
    case TW_ERR_CUDA: return "TW_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case TW_ERR_DEVICE: return "TW_ERR_DEVICE: a kernel gave up on a bounded wait";
    default: return "unknown tw_status";
  }
}
