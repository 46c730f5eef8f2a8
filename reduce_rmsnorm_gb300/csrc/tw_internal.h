// Internal interface between the C-ABI layer (abi.cpp) and the kernels
// (fused_kernel.cu). Not installed; not part of the public boundary.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "tw.h"

namespace tw {

// Arguments of one fused launch, already validated by the ABI layer.
struct FusedArgs {
  const void* partials[TW_MAX_PARTIALS];
  int n;
  void* residual;
  const void* gamma;
  void* out;
  float eps;
  int64_t rows;
  int64_t hidden;
};

struct LaunchShape {
  int grid;        // CTAs (one per SM)
  int threads;     // threads per CTA
  int smem_bytes;  // dynamic shared memory per CTA
  int stages;      // staging-ring depth
  int kmax;        // row chunks held in registers (template instance)
};

// Launch shape on the current device (queries and caches device attributes).
int plan_launch(int64_t rows, int64_t hidden, int n, int sm_budget, LaunchShape* shape);

// Enqueue the fused kernel on `stream`. smid_out: optional device int32[grid].
int launch_fused(const FusedArgs& a, cudaStream_t stream, int sm_budget, int* smid_out);

// Unfused baseline (unfused_kernels.cu): S = bf16(sum of partials), then the
// residual add + RMSNorm of the stored residual.
int launch_reduce(const void* const* partials, int n, int64_t rows, int64_t hidden, void* sum,
                  cudaStream_t stream);
int launch_add_rmsnorm(const void* sum, void* residual, const void* gamma, float eps, int64_t rows,
                       int64_t hidden, void* out, cudaStream_t stream);

// Diagnostic kernel: a bounded wait on an mbarrier nothing completes.
int launch_wait_probe(long long limit_ns, cudaStream_t stream);

// Read (and optionally clear) the device-side error word of the current device.
int read_device_error(int reset, int* code);

}  // namespace tw
