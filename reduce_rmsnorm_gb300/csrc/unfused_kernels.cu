// Unfused baseline for sm_103a: the one-GPU analogue of the pipeline the fused
// step replaces, an all-reduce that writes its result to memory followed by a
// separate RMSNorm kernel.
//
// [W] = "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
// Arithmetic, Not Finer Tiles", "Fix two": vLLM runs RMSNorm after the
// all-reduce has written its result to memory. [G] = "TokenWeave Guide:
// Compute-Communication Overlap for LLMs", "The Standard RMSNorm Memory
// Round-Trip": the reduced tensor is written to HBM and read back by a
// separate normalisation kernel.
//
//   reduce_kernel       S = bf16( ((P_0 + P_1) + ...) + P_{N-1} )        fp32 adds
//   add_rmsnorm_kernel  x = fp32(S) + fp32(R);  R = bf16(x);
//                       Y = bf16( (R * rsqrt(sum R^2 / H + eps)) * gamma ) on the stored R
//
// Both are plain streaming kernels with 16-byte vector loads (ld.global.nc,
// evict-first) and many threads in flight; they are tuned as a baseline in
// their own right, so that the measured fusion gain is the HBM round trip of
// S (write + read) and one launch, not a weak baseline. Like the fused kernel,
// both use programmatic dependent launch: a kernel's blocks may start while
// the previous kernel on the stream drains, and wait (griddepcontrol.wait)
// before their first global-memory access (-10% per pair back to back at
// T = 1024, H = 8192, N = 8; -45% at T = 128, H = 4096, N = 2).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "tw_internal.h"

namespace tw {
namespace {

constexpr int kReduceThreads = 512;
constexpr int kNormThreads = 256;

struct ReduceParams {
  const uint4* partials[TW_MAX_PARTIALS];
  uint4* sum;
  long long vectors;  // T * H / 8
  int n_partials;
};

struct NormParams {
  const uint4* sum;
  uint4* residual;
  const uint4* gamma;
  uint4* out;
  long long rows;
  int vec_per_row;
  float eps;
  float hidden;
};

__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack(const uint4 q, float a[8]) {
  a[0] = lo16(q.x); a[1] = hi16(q.x); a[2] = lo16(q.y); a[3] = hi16(q.y);
  a[4] = lo16(q.z); a[5] = hi16(q.z); a[6] = lo16(q.w); a[7] = hi16(q.w);
}

__device__ __forceinline__ void accumulate(const uint4 q, float a[8]) {
  a[0] += lo16(q.x); a[1] += hi16(q.x); a[2] += lo16(q.y); a[3] += hi16(q.y);
  a[4] += lo16(q.z); a[5] += hi16(q.z); a[6] += lo16(q.w); a[7] += hi16(q.w);
}

__device__ __forceinline__ uint32_t pack(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float a[8]) {
  return make_uint4(pack(a[0], a[1]), pack(a[2], a[3]), pack(a[4], a[5]), pack(a[6], a[7]));
}

// Programmatic dependent launch: wait until the previous kernel on the stream
// has completed and its writes are visible; then let the next one launch.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Grid-stride over 16-byte vectors of the flattened [T, H] tensors.
template <int NT>
__global__ void __launch_bounds__(kReduceThreads) reduce_kernel(const __grid_constant__ ReduceParams p) {
  grid_dependency_wait();
  grid_launch_dependents();
  const int n = NT > 0 ? NT : p.n_partials;
  const long long stride = static_cast<long long>(gridDim.x) * kReduceThreads;
  for (long long i = static_cast<long long>(blockIdx.x) * kReduceThreads + threadIdx.x;
       i < p.vectors; i += stride) {
    float a[8];
    if constexpr (NT > 0) {
      uint4 q[NT];
#pragma unroll
      for (int r = 0; r < NT; ++r) q[r] = __ldcs(p.partials[r] + i);
      unpack(q[0], a);
#pragma unroll
      for (int r = 1; r < NT; ++r) accumulate(q[r], a);
    } else {
      unpack(__ldcs(p.partials[0] + i), a);
      for (int r = 1; r < n; ++r) accumulate(__ldcs(p.partials[r] + i), a);
    }
    p.sum[i] = pack8(a);
  }
}

// One CTA per token row at a time (rows stride over the grid); thread t owns
// vectors t, t + 256, ... (KMAX of them).
template <int KMAX>
__global__ void __launch_bounds__(kNormThreads) add_rmsnorm_kernel(const __grid_constant__ NormParams p) {
  __shared__ float warp_ss[2][kNormThreads / 32];
  grid_dependency_wait();
  grid_launch_dependents();
  const int t = threadIdx.x;
  const int vpr = p.vec_per_row;
  int buf = 0;
  for (long long row = blockIdx.x; row < p.rows; row += gridDim.x, buf ^= 1) {
    const uint4* s_row = p.sum + row * vpr;
    uint4* r_row = p.residual + row * vpr;
    float x[KMAX][8];
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int v = k * kNormThreads + t;
      if (v < vpr) {
        float a[8];
        unpack(__ldcs(s_row + v), a);
        accumulate(__ldcs(r_row + v), a);
        const uint4 stored = pack8(a);
        r_row[v] = stored;
        unpack(stored, x[k]);  // the norm reads the stored bf16 residual
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(x[k][i], x[k][i], ss);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    // two buffers: a thread can only write buffer b again after every thread
    // has passed the next row's barrier, i.e. has finished reading buffer b
    if ((t & 31) == 0) warp_ss[buf][t >> 5] = ss;
    __syncthreads();
    float total = 0.0f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) total += warp_ss[buf][w];
    const float rs = rsqrtf(total / p.hidden + p.eps);
    uint4* o_row = p.out + row * vpr;
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int v = k * kNormThreads + t;
      if (v < vpr) {
        float g[8], y[8];
        unpack(__ldg(p.gamma + v), g);
#pragma unroll
        for (int i = 0; i < 8; ++i) y[i] = (x[k][i] * rs) * g[i];
        o_row[v] = pack8(y);
      }
    }
  }
}

using ReduceFn = void (*)(ReduceParams);
using NormFn = void (*)(NormParams);
const ReduceFn kReduce[4] = {reduce_kernel<0>, reduce_kernel<2>, reduce_kernel<4>, reduce_kernel<8>};
const NormFn kNorm[5] = {add_rmsnorm_kernel<1>, add_rmsnorm_kernel<2>, add_rmsnorm_kernel<4>,
                         add_rmsnorm_kernel<8>, add_rmsnorm_kernel<16>};

std::atomic<int> g_sm_count[64];  // static storage: starts at 0 (not yet queried)

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  int sms = g_sm_count[dev].load(std::memory_order_relaxed);
  if (sms == 0) {
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_sm_count[dev].store(sms, std::memory_order_relaxed);
  }
  return sms;
}

// Launch with programmatic stream serialization (the kernels wait on
// griddepcontrol.wait before touching global memory).
template <typename P>
int launch_programmatic(void (*fn)(P), unsigned grid, int threads, cudaStream_t stream,
                        const P& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, fn, p) != cudaSuccess) {
    cudaGetLastError();
    return TW_ERR_CUDA;
  }
  return TW_OK;
}

}  // namespace

int launch_reduce(const void* const* partials, int n, int64_t rows, int64_t hidden, void* sum,
                  cudaStream_t stream) {
  ReduceParams p;
  for (int r = 0; r < TW_MAX_PARTIALS; ++r)
    p.partials[r] = r < n ? static_cast<const uint4*>(partials[r]) : nullptr;
  p.sum = static_cast<uint4*>(sum);
  p.vectors = rows * (hidden / 8);
  p.n_partials = n;
  const int sms = sm_count();
  if (sms <= 0) return TW_ERR_CUDA;
  long long blocks = (p.vectors + kReduceThreads - 1) / kReduceThreads;
  const long long cap = static_cast<long long>(sms) * 4;  // 4 x 512 threads per SM
  if (blocks > cap) blocks = cap;
  const int ni = n == 2 ? 1 : n == 4 ? 2 : n == 8 ? 3 : 0;
  return launch_programmatic(kReduce[ni], static_cast<unsigned>(blocks), kReduceThreads, stream, p);
}

int launch_add_rmsnorm(const void* sum, void* residual, const void* gamma, float eps, int64_t rows,
                       int64_t hidden, void* out, cudaStream_t stream) {
  NormParams p;
  p.sum = static_cast<const uint4*>(sum);
  p.residual = static_cast<uint4*>(residual);
  p.gamma = static_cast<const uint4*>(gamma);
  p.out = static_cast<uint4*>(out);
  p.rows = rows;
  p.vec_per_row = static_cast<int>(hidden / 8);
  p.eps = eps;
  p.hidden = static_cast<float>(hidden);
  const int slots = (p.vec_per_row + kNormThreads - 1) / kNormThreads;
  int k = 0;
  while ((1 << k) < slots) ++k;
  if (k > 4) return TW_ERR_UNSUPPORTED;  // H <= TW_MAX_HIDDEN keeps k <= 4
  const int sms = sm_count();
  if (sms <= 0) return TW_ERR_CUDA;
  // one row per CTA up to 16 resident CTAs per SM; larger batches loop
  const long long cap = static_cast<long long>(sms) * 16;
  const long long grid = rows < cap ? rows : cap;
  return launch_programmatic(kNorm[k], static_cast<unsigned>(grid), kNormThreads, stream, p);
}

}  // namespace tw
