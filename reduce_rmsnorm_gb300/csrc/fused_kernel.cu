// Fused reduce + residual + RMSNorm kernel for sm_103a.
//
// [W] = "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
// Arithmetic, Not Finer Tiles", section "Fix two: RMSNorm was never
// insignificant": per CTA, load-and-reduce the ranks' vectors, add the
// residual in the same pass, take the sum of squares on the register-resident
// result (no HBM re-read), scale by rsqrt(variance / hidden_size + eps) and the
// weight, store once. On one GPU the ranks' contributions are N local buffers.
//
// GB300 design (not the pages' multimem kernel, which targets NVSwitch):
//   * Persistent: one CTA per SM (it asks for ~216 KB of shared memory, so no
//     second CTA of this kernel fits), each owning a contiguous range of token
//     rows ([W]'s tokens_per_cta = ceil(num_tokens / gridDim.x), balanced).
//     The grid size is the SM budget. With one row per CTA the ring holds just
//     that row, so a small row leaves room for the next launch's CTAs; the
//     direct form (below) holds no ring at all, and on the whole GPU runs one
//     CTA per row while all of them fit on the GPU at once.
//   * Warp-specialised: the producer warp streams each row, in chunks of 8 KiB
//     (N <= 8) or 4 KiB of every source (N partials + residual), from HBM into
//     a ring of shared-memory stages with 1-D TMA bulk copies (cp.async.bulk,
//     mbarrier completion); lane r issues source r's copy, so the N + 1
//     copies of a stage go out in parallel (one lane issuing 4 KiB copies in
//     turn capped an SM under an SM budget near 57 GB/s; now 8 KiB copies
//     reach ~128 GB/s and 4 KiB copies 80-95 GB/s). Eight consumer warps
//     read a chunk (one or two 16-byte vectors per thread per source), sum in
//     fp32 in rank order (packed f32x2 adds), add the residual, store the
//     updated residual, and keep z in registers.
//   * After a row's last chunk: warp xor-shuffle sum of squares, a fixed-order
//     combine of the 8 warp sums, rsqrtf, and Y = (z * r) * gamma stored with
//     16-byte stores. The per-row arithmetic depends only on H, so every grid
//     size (SM budget), split and shard gives bitwise the same rows.
//   * Two more forms serve an SM budget, where each SM must stream as much as
//     it can: two independent pipelines per CTA (each its own producer lanes,
//     half of the ring and 8 consumer warps) for N <= 4, where the consumers'
//     work per byte caps an SM; and the row ring (rowring_kernel), one bulk
//     copy per source row, for N >= 9, where 4 KiB copies cap it. And with
//     one row per CTA (decode-sized batches) the direct form (direct_kernel)
//     loads each thread's vectors straight into registers, with no ring. Each
//     thread owns the same vectors and adds in the same order in every form,
//     so the forms give bitwise the same rows; select_kernel picks one by
//     speed.
//   * L2 policy per call: evict-first loads and a streaming output when no
//     CTA owns more than one row and that row is over 144 KiB, for N <= 2 or
//     N >= 9 with an output of at most an eighth of the L2, and for N <= 2
//     with an output of at least 7/16 of it; otherwise the normal policy.
//   * Programmatic dependent launch: the CTAs set up their barriers while the
//     previous kernel in the stream drains, ask L2 for the first ~144 KiB of
//     their rows (a prefetch hint, when a CTA owns more than one row or its
//     one row fits in it), then wait (griddepcontrol.wait) before reading or
//     writing global memory.
//   * Every wait on an mbarrier is bounded (time and iterations); on giving up
//     the CTA sets a device error word and finishes without further waits.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "tw_internal.h"

namespace tw {

// Device-side error word (bit 0: consumer wait, bit 1: producer wait,
// bit 2: final drain). Read and cleared by read_device_error().
__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
// A "slot" is one 16-byte vector per consumer thread: 256 vectors, 4 KiB of a
// source row. A chunk (the unit of one bulk copy per source) is VPT slots.
constexpr int kSlotVec = kConsumerThreads;
constexpr int kSlotBytes = kSlotVec * 16;
constexpr int kMaxStages = 32;
constexpr int kConsumerBarrierId = 1;            // named barrier of the consumer warps

constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // give up after 2 s
constexpr uint32_t kWaitLimitPolls = 1u << 26;
constexpr unsigned long long kDrainLimitNs = 200000000ull;  // 0.2 s per stage
// L2 warm-up before the dependency wait: bytes per CTA over all sources, and
// the size of one prefetch instruction. Measured on T = 512-8192, H = 4096-16384,
// N = 2-16: best or within 1% of the best of 4-24 KiB per source.
constexpr uint32_t kPrefetchPerCta = 144u * 1024u;
constexpr uint32_t kPrefetchPiece = 32u * 1024u;

struct Params {
  const uint4* partials[TW_MAX_PARTIALS];
  const uint4* gamma;
  uint4* residual;
  uint4* out;
  int* smid_out;
  int l2_stream;    // 1: evict-first loads and streaming output stores (see launch_fused)
  uint32_t prefetch_bytes;  // per source, from the CTA's first row: L2 warm-up before the
                            // dependency wait (multiple of 16; 0 = none)
  long long rows;
  int vec_per_row;  // H / 8
  int n_partials;
  int chunks;       // ceil(vec_per_row / (kSlotVec * VPT))
  int stages;       // stages of the ring (of pipeline 0 with two pipelines)
  int stages1;      // two pipelines: pipeline 1's stages
  int split_num;    // two pipelines: pipeline 0 owns split_num / split_den of the
  int split_den;    // CTA's rows
  float eps;
  float hidden;
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// 1-D TMA bulk copy global -> shared, completing `bytes` on the mbarrier.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// Asks L2 to fetch [src, src + bytes) (16-byte aligned, bytes a multiple of
// 16). A hint only: nothing is returned to the thread and no memory is written.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t id;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(id));
  return id;
}

// Wait for the phase of the given parity of *bar to complete. Bounded: gives
// up after limit_ns (kWaitLimitNs in the kernels) or kWaitLimitPolls polls,
// then sets *abort and the device error word. Returns false at once while
// *abort is set.
__device__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort, unsigned code,
                           unsigned long long limit_ns = kWaitLimitNs) {
  if (*abort) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1; i < kWaitLimitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > limit_ns) break;
    }
  }
  *abort = 1;
  atomicOr(&g_device_error, code);
  return false;
}

// Bounded wait that ignores the abort flag (used to drain in-flight copies).
__device__ bool drain_phase(uint64_t* bar, uint32_t parity) {
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 0; i < kWaitLimitPolls; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u && global_timer_ns() - t0 > kDrainLimitNs) break;
  }
  atomicOr(&g_device_error, 4u);
  return false;
}

// Waits (bounded) until every bulk copy a producer issued into its ring of
// `stages` stages has landed: `issued` items went out in order, item i on
// stage i % stages in phase i / stages, so the last item of each stage
// completes after all earlier ones there. The producer owns this drain, on
// the normal path too (where it returns as the consumers' waits complete),
// so no CTA exits with copies into its shared memory in flight, even if a
// consumer gives up a wait after the producer has left its issue loop.
__device__ void drain_ring(uint64_t* full, int stages, long long issued) {
  const long long last = issued - 1;
  for (int st = 0; st < stages && st <= last; ++st) {
    const long long it_last = last - ((last - st) % stages);
    drain_phase(&full[st], static_cast<uint32_t>((it_last / stages) & 1));
  }
}

// ------------------------------------------------------------------ bf16 x 8

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void load8(const uint4 q, float a[8]) {
  a[0] = bf16_lo(q.x); a[1] = bf16_hi(q.x);
  a[2] = bf16_lo(q.y); a[3] = bf16_hi(q.y);
  a[4] = bf16_lo(q.z); a[5] = bf16_hi(q.z);
  a[6] = bf16_lo(q.w); a[7] = bf16_hi(q.w);
}

// a[2i], a[2i+1] += the two bf16 values of word w, as one packed fp32x2 add
// (add.rn.f32x2: two independent IEEE round-to-nearest fp32 additions, the
// same results as two scalar adds, in one instruction).
__device__ __forceinline__ void add2(float& lo, float& hi, uint32_t w) {
  uint64_t acc, v;
  asm("mov.b64 %0, {%1, %2};" : "=l"(acc) : "f"(lo), "f"(hi));
  asm("mov.b64 %0, {%1, %2};" : "=l"(v) : "r"(w << 16), "r"(w & 0xffff0000u));
  asm("add.rn.f32x2 %0, %0, %1;" : "+l"(acc) : "l"(v));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(acc));
}

__device__ __forceinline__ void add8(const uint4 q, float a[8]) {
  add2(a[0], a[1], q.x);
  add2(a[2], a[3], q.y);
  add2(a[4], a[5], q.z);
  add2(a[6], a[7], q.w);
}

// y[i] = (z[i] * rs) * gamma[i] for the 8 bf16 gamma values of q, as packed
// fp32x2 multiplies (mul.rn.f32x2: two IEEE round-to-nearest products per
// instruction, the same results as scalar multiplies in the same order).
__device__ __forceinline__ void scale8(const float z[8], float rs, const uint4 q, float y[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint64_t r2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r2) : "f"(rs));
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint64_t a, g;
    asm("mov.b64 %0, {%1, %2};" : "=l"(a) : "f"(z[2 * k]), "f"(z[2 * k + 1]));
    asm("mov.b64 %0, {%1, %2};" : "=l"(g) : "r"(w[k] << 16), "r"(w[k] & 0xffff0000u));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(r2));
    asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(a) : "l"(g));
    asm("mov.b64 {%0, %1}, %2;" : "=f"(y[2 * k]), "=f"(y[2 * k + 1]) : "l"(a));
  }
}

// Sum of the 8 warp partials in warp order, read as two 16-byte loads.
__device__ __forceinline__ float warp_total(const float* w8) {
  const float4 a = *reinterpret_cast<const float4*>(w8);
  const float4 b = *reinterpret_cast<const float4*>(w8 + 4);
  return ((((((a.x + a.y) + a.z) + a.w) + b.x) + b.y) + b.z) + b.w;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const float a[8]) {
  return make_uint4(pack2(a[0], a[1]), pack2(a[2], a[3]), pack2(a[4], a[5]), pack2(a[6], a[7]));
}

// ------------------------------------------------------------------ the kernel

// Sum of the N partials and the residual for one 16-byte vector column of a
// staged chunk, in rank order, residual last. `src` addresses the column in
// source 0's chunk; source r's chunk is `cbytes` further per r. NT > 0: N is a
// compile-time constant and all N + 1 shared loads issue before the first
// add; NT == 0: runtime N, loads issued in groups of up to four.
template <int NT>
__device__ __forceinline__ void reduce_vector(uint32_t src, uint32_t cbytes, int n, float a[8]) {
  if constexpr (NT > 0) {
    uint4 q[NT + 1];
#pragma unroll
    for (int r = 0; r <= NT; ++r) q[r] = lds128(src + r * cbytes);
    load8(q[0], a);
#pragma unroll
    for (int r = 1; r <= NT; ++r) add8(q[r], a);
  } else {
    // Sources 1..n (source n is the residual) in groups of four whose loads
    // issue together, then the last one to three together, so no load waits
    // alone. The adds keep rank order, so the sum is bitwise the same.
    load8(lds128(src), a);
    int r = 1;
    for (; r + 3 <= n; r += 4) {
      const uint4 q0 = lds128(src + r * cbytes), q1 = lds128(src + (r + 1) * cbytes);
      const uint4 q2 = lds128(src + (r + 2) * cbytes), q3 = lds128(src + (r + 3) * cbytes);
      add8(q0, a); add8(q1, a); add8(q2, a); add8(q3, a);
    }
    const int left = n + 1 - r;  // 0..3 sources after the full groups
    if (left == 3) {
      const uint4 q0 = lds128(src + r * cbytes), q1 = lds128(src + (r + 1) * cbytes);
      const uint4 q2 = lds128(src + (r + 2) * cbytes);
      add8(q0, a); add8(q1, a); add8(q2, a);
    } else if (left == 2) {
      const uint4 q0 = lds128(src + r * cbytes), q1 = lds128(src + (r + 1) * cbytes);
      add8(q0, a); add8(q1, a);
    } else if (left == 1) {
      add8(lds128(src + r * cbytes), a);
    }
  }
}

// The end of a row, shared by every kernel form: the sum of squares is
// reduced across the warp (xor shuffle) and then across the pipeline's 8
// warps in warp order (through `wsum`, this row's 8 floats), r = rsqrt(mean +
// eps), and Y = (z * r) * gamma is stored as bf16. With evict-first loads the
// output is stored streaming too, so its lines drain during this launch; with
// normal loads the store policy measured within 0.2%. A kernel that reads Y
// right after still finds it unless L2 needs the room. The residual keeps the
// default policy (evict-first there measured -1%).
template <int KMAX, bool EXACT, int GN>
__device__ __forceinline__ void finish_row(const Params& p, float ss, const float (&z)[KMAX][8],
                                           const uint4 (&g_reg)[GN], float* wsum, int bar_id,
                                           int lane, int wg, int t, int vpr, long long row) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) wsum[wg] = ss;
  asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kConsumerThreads) : "memory");
  const float total = warp_total(wsum);
  const float rs = rsqrtf(total / p.hidden + p.eps);
  uint4* out_row = p.out + row * vpr;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const int v = j * kSlotVec + t;
    if (EXACT || v < vpr) {
      float y[8];
      if constexpr (GN == KMAX) scale8(z[j], rs, g_reg[j], y);
      else scale8(z[j], rs, __ldg(p.gamma + v), y);
      if (p.l2_stream) __stcs(out_row + v, pack8(y));
      else out_row[v] = pack8(y);
    }
  }
}

// KMAX:  slots of a row held in registers (ceil(H/8 / 256) rounded up to a
//        power of two, >= VPT).
// VPT:   slots per chunk (1: 4 KiB copies; 2: 8 KiB copies).
// NT:    compile-time partial count, or 0 for any N.
// EXACT: H/8 == KMAX * 256 (H = 4096, 8192, 16384, 32768 with 8 KiB chunks):
//        every chunk is full and the chunk count is a constant, so the
//        ragged-edge checks compile away (~5% per SM under an SM budget).
// Thread t of the consumers owns vectors t, t + 256, t + 512, ... of every row
// (slot j = vector j * 256 + t) whatever VPT is, so the per-row arithmetic,
// including the order of the sum of squares, depends only on H.
// G:     independent pipelines sharing the CTA (1 or 2). Pipeline g owns a
//        contiguous part of the CTA's rows, G-th of the ring, producer lanes
//        16 g .. 16 g + N and consumer warps 8 g .. 8 g + 7; a second pipeline
//        overlaps one row's epilogue with another row's reduction where the
//        consumer work per byte caps an SM (small N under an SM budget).
template <int KMAX, int VPT, int NT, bool EXACT, int G = 1>
__global__ void __launch_bounds__(G * kConsumerThreads + 32, 1)
    fused_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(16) float warp_ss[G][2][kConsumerWarps];
  __shared__ int abort_flag;

  constexpr int kChunkVec = kSlotVec * VPT;
  constexpr uint32_t kChunkBytes = kSlotBytes * VPT;
  constexpr int kProducerWarp = G * kConsumerWarps;
  static_assert(KMAX % VPT == 0, "slots must fill whole chunks");
  // G = 2 is instantiated only with a compile-time N of 1..4 (kChunkTwo): each
  // pipeline's producer group is lanes 16 g .. 16 g + N.
  static_assert(G == 1 || NT <= 15, "two pipelines take at most 16 producer lanes each");
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long grid = gridDim.x;
  const long long row0 = static_cast<long long>(blockIdx.x) * p.rows / grid;
  const long long row1 = static_cast<long long>(blockIdx.x + 1) * p.rows / grid;
  const int n = NT > 0 ? NT : p.n_partials;
  const int vpr = EXACT ? KMAX * kSlotVec : p.vec_per_row;
  const int chunks = EXACT ? KMAX / VPT : p.chunks;
  const int st0 = p.stages, st1 = G == 1 ? 0 : p.stages1;  // stages of pipelines 0 and 1
  const uint32_t stage_bytes = static_cast<uint32_t>(n + 1) * kChunkBytes;
  // rows of pipeline g: [part(g), part(g + 1)); pipeline 0 owns split_num /
  // split_den of the CTA's rows (half, or more when its ring is deeper)
  auto part = [&](int g) {
    if constexpr (G == 1) return row0 + (row1 - row0) * g;
    else return g == 0 ? row0 : (g == G ? row1 : row0 + (row1 - row0) * p.split_num / p.split_den);
  };

  if (tid == 0) {
    for (int s = 0; s < st0 + st1; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Producer lane -> (pipeline, source): lane r for G = 1; lane 16 g + r for
  // G = 2.
  const int pg = G == 1 ? 0 : lane >> 4;
  const int src_lane = G == 1 ? lane : (lane & 15);
  // Programmatic dependent launch: this CTA may be resident before the
  // previous kernel in the stream has finished. Nothing above read or wrote
  // global memory. A CTA that lands on an SM the previous kernel has already
  // left asks L2 for the first bytes of its rows, so HBM works through the
  // previous kernel's tail instead of idling. This is a hint: the step's data
  // is read only by the copies issued after the wait, through the L2, which
  // is the device's point of coherence and so holds the previous kernel's
  // writes. Then wait until that kernel has completed and its writes are
  // visible, and allow the next kernel in the stream to start launching.
  if (p.prefetch_bytes != 0 && warp == kProducerWarp && src_lane <= n && pg < G) {
    const long long ra = part(pg), rb = part(pg + 1);
    if (rb > ra) {
      const char* src = reinterpret_cast<const char*>(
          (src_lane < n ? p.partials[src_lane] : p.residual) + ra * vpr);
      const long long avail = (rb - ra) * vpr * 16;
      const uint32_t want = (p.prefetch_bytes / G) & ~15u;
      const uint32_t total =
          static_cast<uint32_t>(static_cast<long long>(want) < avail ? want : avail);
      for (uint32_t off = 0; off < total; off += kPrefetchPiece)
        prefetch_l2(src + off, total - off < kPrefetchPiece ? total - off : kPrefetchPiece);
    }
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (tid == 0 && p.smid_out) p.smid_out[blockIdx.x] = static_cast<int>(sm_id());
  volatile int* abort = &abort_flag;

  if (warp == kProducerWarp) {
    // ---------------- producer: lanes 0..N of pipeline g stream its (row,
    // chunk) items into its part of the ring; lane r < N copies partial r,
    // lane N the residual.
    if (src_lane > n || pg >= G) return;
    const unsigned lanes = (n + 1 == 32 ? 0xffffffffu : ((1u << (n + 1)) - 1u)) << (16 * pg);
    const int lead = 16 * pg;  // the pipeline's first lane
    const int stages = (G == 1 || pg == 0) ? st0 : st1;
    const int first = pg == 0 ? 0 : st0;  // the pipeline's first stage
    uint64_t* full = full_bar + first;
    uint64_t* empty = empty_bar + first;
    unsigned char* my_ring = ring + static_cast<size_t>(first) * stage_bytes;
    // Evict-first or normal L2 policy for the loads, chosen per call on the
    // host (launch_fused).
    const uint64_t policy = p.l2_stream ? l2_evict_first_policy() : l2_evict_normal_policy();
    const uint4* src_base = src_lane < n ? p.partials[src_lane] : p.residual;
    const long long ra = part(pg), rb = part(pg + 1);
    const long long items = (rb - ra) * chunks;
    long long issued = 0;
    long long row = ra;
    int chunk = 0, s = 0;
    uint32_t round_parity = 0;  // parity of the current pass over the ring
    bool first_pass = true;
    for (long long it = 0; it < items; ++it) {
      int ok = 1;
      const int v0 = chunk * kChunkVec;
      const int nvec = EXACT ? kChunkVec : min(kChunkVec, vpr - v0);
      const uint32_t bytes = static_cast<uint32_t>(nvec) * 16u;
      if (src_lane == 0) {
        if (!first_pass) ok = wait_phase(&empty[s], round_parity ^ 1u, abort, 2u);
        if (ok) mbar_arrive_expect_tx(&full[s], bytes * static_cast<uint32_t>(n + 1));
      }
      if (!__shfl_sync(lanes, ok, lead)) break;
      bulk_load(my_ring + static_cast<size_t>(s) * stage_bytes + src_lane * kChunkBytes,
                src_base + row * vpr + v0, bytes, &full[s], policy);
      ++issued;
      if (++chunk == chunks) { chunk = 0; ++row; }
      if (++s == stages) { s = 0; round_parity ^= 1u; first_pass = false; }
    }
    if (src_lane == 0) drain_ring(full, stages, issued);
    return;
  }

  // ---------------- consumers: 8 warps per pipeline; thread t owns slots j
  // (vector j*256 + t)
  const int g = warp / kConsumerWarps;
  const int wg = warp % kConsumerWarps;
  const int t = tid - g * kConsumerThreads;
  const int stages = (G == 1 || g == 0) ? st0 : st1;
  const int first = G == 1 ? g * st0 : (g == 0 ? 0 : st0);  // the pipeline's first stage
  uint64_t* full = full_bar + first;
  uint64_t* empty = empty_bar + first;
  const uint32_t ring_base = smem_addr(ring) + static_cast<uint32_t>(first) * stage_bytes +
                             static_cast<uint32_t>(t) * 16u;
  // gamma stays in registers for the CTA's whole row range (read once per CTA)
  constexpr bool kGammaRegs = KMAX <= 8;
  uint4 g_reg[kGammaRegs ? KMAX : 1];
  if constexpr (kGammaRegs) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int v = j * kSlotVec + t;
      g_reg[j] = (EXACT || v < vpr) ? __ldg(p.gamma + v) : make_uint4(0, 0, 0, 0);
    }
  }
  int s = 0;
  uint32_t parity = 0;
  float z[KMAX][8];
  const long long ra = part(g), rb = part(g + 1);
  for (long long row = ra; row < rb; ++row) {
    float ss = 0.0f;
    uint4* res_row = p.residual + row * vpr;
#pragma unroll
    for (int c = 0; c < KMAX / VPT; ++c) {
      if (c < chunks) {
        wait_phase(&full[s], parity, abort, 1u);
        const uint32_t stage = ring_base + static_cast<uint32_t>(s) * stage_bytes;
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
          const int j = c * VPT + u;
          if (EXACT || j * kSlotVec + t < vpr)
            reduce_vector<NT>(stage + u * kSlotBytes, kChunkBytes, n, z[j]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
        for (int u = 0; u < VPT; ++u) {
          const int j = c * VPT + u;
          const int v = j * kSlotVec + t;
          if (EXACT || v < vpr) {
#pragma unroll
            for (int i = 0; i < 8; ++i) ss = fmaf(z[j][i], z[j][i], ss);
            res_row[v] = pack8(z[j]);
          }
        }
        if (++s == stages) { s = 0; parity ^= 1u; }
      }
    }
    // the two row buffers of warp sums alternate, so a warp can post row i + 1
    // while slower warps still read row i's
    finish_row<KMAX, EXACT>(p, ss, z, g_reg, warp_ss[g][(row - ra) & 1], kConsumerBarrierId + g,
                            lane, wg, t, vpr, row);
  }
}

// Direct form, for launches of one row per CTA of at most 8 slots (H <= 16384)
// and a compile-time N <= 8. KMAX is the slot count rounded up to a power of
// two; EXACT rows fill it (H = 2048, 4096, 8192, 16384), other rows check
// each vector against the row's end, as fused_kernel does.
// Consumer thread t loads its own vectors t + 256 j of every source straight
// into registers, so each byte crosses the SM's L1 once; the ring forms write
// it into shared memory with a bulk copy and read it back. With one row per
// CTA there is no later row for a ring to stage ahead, and the row is already
// in L2 from the prefetch before the dependency wait. Thread t owns the same
// vectors and adds the sources in the same rank order, then the residual, as
// in fused_kernel, and the end of the row is finish_row, so rows are bitwise
// those of the ring forms. No producer warp, no dynamic shared memory, no
// mbarrier: the only wait is the CTA barrier inside finish_row.
template <int KMAX, int NT, bool EXACT>
__global__ void __launch_bounds__(kConsumerThreads, 1)
    direct_kernel(const __grid_constant__ Params p) {
  __shared__ __align__(16) float warp_ss[kConsumerWarps];
  static_assert(KMAX == 1 || KMAX == 2 || KMAX == 4 || KMAX == 8, "one to eight slots");
  static_assert(NT >= 1 && NT <= 8, "compile-time N of 1..8");
  const int vpr = EXACT ? KMAX * kSlotVec : p.vec_per_row;
  const int t = threadIdx.x;
  const int lane = t & 31;
  const int wg = t >> 5;
  const long long row = blockIdx.x;  // grid = rows
  // L2 warm-up of the whole row before the dependency wait, as in
  // fused_kernel: lane r of warp 0 asks for source r's row (r = N: the
  // residual).
  if (p.prefetch_bytes != 0 && wg == 0 && lane <= NT) {
    const char* src =
        reinterpret_cast<const char*>((lane < NT ? p.partials[lane] : p.residual) + row * vpr);
    const uint32_t total = p.prefetch_bytes < static_cast<uint32_t>(vpr * 16)
                               ? p.prefetch_bytes
                               : static_cast<uint32_t>(vpr * 16);
    for (uint32_t off = 0; off < total; off += kPrefetchPiece)
      prefetch_l2(src + off, total - off < kPrefetchPiece ? total - off : kPrefetchPiece);
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (t == 0 && p.smid_out) p.smid_out[blockIdx.x] = static_cast<int>(sm_id());
  uint4 g_reg[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const int v = j * kSlotVec + t;
    g_reg[j] = (EXACT || v < vpr) ? __ldg(p.gamma + v) : make_uint4(0, 0, 0, 0);
  }
  // Every load of the row issues before the first add. The partials are
  // loaded evict-first (their lines are not read again); the residual with
  // the default policy, since this thread writes it back below.
  uint4 q[KMAX][NT + 1];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const int v = j * kSlotVec + t;
    if (EXACT || v < vpr) {
#pragma unroll
      for (int r = 0; r < NT; ++r) q[j][r] = __ldcs(p.partials[r] + row * vpr + v);
      q[j][NT] = p.residual[row * vpr + v];
    }
  }
  float z[KMAX][8];
  float ss = 0.0f;
  uint4* res_row = p.residual + row * vpr;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const int v = j * kSlotVec + t;
    if (EXACT || v < vpr) {
      load8(q[j][0], z[j]);
#pragma unroll
      for (int r = 1; r <= NT; ++r) add8(q[j][r], z[j]);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss = fmaf(z[j][i], z[j][i], ss);
      res_row[v] = pack8(z[j]);
    }
  }
  finish_row<KMAX, EXACT>(p, ss, z, g_reg, warp_ss, kConsumerBarrierId, lane, wg, t, vpr, row);
}

// Row-ring form: one bulk copy per (row, source), so a stage holds one
// source's whole row (KMAX 4 KiB slots: 16-64 KiB), and G independent
// pipelines share the CTA. Pipeline g owns a contiguous part of the CTA's rows,
// producer lane g, its own part of the ring (p.stages stages) and consumer
// warps 8g .. 8g + 7; each pipeline is consumed in order by its own warps, as
// in fused_kernel. Against fused_kernel it issues (N + 1) copies per row
// instead of (N + 1) * chunks, of 16 KiB and more (the TMA issue cost is
// nearly flat in size up to 8 KiB, so small copies cap an SM under an SM
// budget), and with G = 2 two rows are reduced at once (the consumer work per
// byte is what caps an SM at small N). Thread t of a pipeline owns the same
// vectors t + 256 j as in fused_kernel and adds the sources in the same rank
// order, then the residual, so rows are bitwise those of fused_kernel.
template <int KMAX, int G, int NT, bool EXACT>
__global__ void __launch_bounds__(G * kConsumerThreads + 32, 1)
    rowring_kernel(const __grid_constant__ Params p) {
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(16) float warp_ss[G][2][kConsumerWarps];
  __shared__ int abort_flag;

  constexpr uint32_t kStageBytes = KMAX * kSlotBytes;
  constexpr int kProducerWarp = G * kConsumerWarps;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long grid = gridDim.x;
  const long long row0 = static_cast<long long>(blockIdx.x) * p.rows / grid;
  const long long row1 = static_cast<long long>(blockIdx.x + 1) * p.rows / grid;
  const int n = NT > 0 ? NT : p.n_partials;
  const int vpr = EXACT ? KMAX * kSlotVec : p.vec_per_row;
  const int spp = p.stages;  // stages of each pipeline
  // rows of pipeline g: [part(g), part(g + 1))
  auto part = [&](int g) { return row0 + (row1 - row0) * g / G; };

  if (tid == 0) {
    for (int s = 0; s < G * spp; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // L2 warm-up before the dependency wait, as in fused_kernel: lane r asks for
  // the first bytes of source r's rows of each pipeline.
  if (p.prefetch_bytes != 0 && warp == kProducerWarp && lane <= n) {
    const uint4* base = lane < n ? p.partials[lane] : p.residual;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const long long ra = part(g), rb = part(g + 1);
      if (rb <= ra) continue;
      const char* src = reinterpret_cast<const char*>(base + ra * vpr);
      const long long avail = (rb - ra) * vpr * 16;
      const uint32_t want = (p.prefetch_bytes / G) & ~15u;
      const uint32_t total =
          static_cast<uint32_t>(static_cast<long long>(want) < avail ? want : avail);
      for (uint32_t off = 0; off < total; off += kPrefetchPiece)
        prefetch_l2(src + off, total - off < kPrefetchPiece ? total - off : kPrefetchPiece);
    }
  }
  grid_dependency_wait();
  grid_launch_dependents();
  if (tid == 0 && p.smid_out) p.smid_out[blockIdx.x] = static_cast<int>(sm_id());
  volatile int* abort = &abort_flag;

  if (warp == kProducerWarp) {
    // ---------------- producer lane g feeds pipeline g: items (row, source),
    // sources 0..N-1 then the residual, one whole-row bulk copy each.
    if (lane >= G) return;
    const int g = lane;
    uint64_t* full = full_bar + g * spp;
    uint64_t* empty = empty_bar + g * spp;
    unsigned char* my_ring = ring + static_cast<size_t>(g) * spp * kStageBytes;
    const uint64_t policy = p.l2_stream ? l2_evict_first_policy() : l2_evict_normal_policy();
    const uint32_t bytes = static_cast<uint32_t>(vpr) * 16u;
    const long long ra = part(g), rb = part(g + 1);
    const long long items = (rb - ra) * (n + 1);
    long long issued = 0;
    long long row = ra;
    int r = 0, s = 0;
    uint32_t round_parity = 0;
    bool first_pass = true;
    for (long long it = 0; it < items; ++it) {
      if (!first_pass && !wait_phase(&empty[s], round_parity ^ 1u, abort, 2u)) break;
      mbar_arrive_expect_tx(&full[s], bytes);
      const uint4* src = r < n ? p.partials[r] : p.residual;
      bulk_load(my_ring + static_cast<size_t>(s) * kStageBytes, src + row * vpr, bytes, &full[s],
                policy);
      ++issued;
      if (++r > n) { r = 0; ++row; }
      if (++s == spp) { s = 0; round_parity ^= 1u; first_pass = false; }
    }
    drain_ring(full, spp, issued);
    return;
  }

  // ---------------- consumers: pipeline g = warp / 8; thread t owns slots j
  // (vector j * 256 + t) of every row of the pipeline
  const int g = warp / kConsumerWarps;
  const int wg = warp % kConsumerWarps;
  const int t = tid - g * kConsumerThreads;
  uint64_t* full = full_bar + g * spp;
  uint64_t* empty = empty_bar + g * spp;
  const uint32_t ring_base = smem_addr(ring) + static_cast<uint32_t>(g * spp) * kStageBytes +
                             static_cast<uint32_t>(t) * 16u;
  constexpr bool kGammaRegs = KMAX <= 8;
  uint4 g_reg[kGammaRegs ? KMAX : 1];
  if constexpr (kGammaRegs) {
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int v = j * kSlotVec + t;
      g_reg[j] = (EXACT || v < vpr) ? __ldg(p.gamma + v) : make_uint4(0, 0, 0, 0);
    }
  }
  int s = 0;
  uint32_t parity = 0;
  float z[KMAX][8];
  const long long ra = part(g), rb = part(g + 1);
  for (long long row = ra; row < rb; ++row) {
    // source r's whole row is one stage: z = P_0, then += P_1 .. P_{N-1}, += R
    auto take = [&](bool first) {
      wait_phase(&full[s], parity, abort, 1u);
      const uint32_t stage = ring_base + static_cast<uint32_t>(s) * kStageBytes;
      // loads of up to 8 slots issue together, then their adds
      constexpr int kBatch = KMAX < 8 ? KMAX : 8;
#pragma unroll
      for (int j0 = 0; j0 < KMAX; j0 += kBatch) {
        uint4 q[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (EXACT || (j0 + u) * kSlotVec + t < vpr) q[u] = lds128(stage + (j0 + u) * kSlotBytes);
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (EXACT || (j0 + u) * kSlotVec + t < vpr) {
            if (first) load8(q[u], z[j0 + u]);
            else add8(q[u], z[j0 + u]);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (++s == spp) { s = 0; parity ^= 1u; }
    };
    take(true);
    if constexpr (NT > 0) {
#pragma unroll
      for (int r = 1; r <= NT; ++r) take(false);
    } else {
      for (int r = 1; r <= n; ++r) take(false);
    }
    float ss = 0.0f;
    uint4* res_row = p.residual + row * vpr;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      const int v = j * kSlotVec + t;
      if (EXACT || v < vpr) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(z[j][i], z[j][i], ss);
        res_row[v] = pack8(z[j]);
      }
    }
    finish_row<KMAX, EXACT>(p, ss, z, g_reg, warp_ss[g][(row - ra) & 1], kConsumerBarrierId + g,
                            lane, wg, t, vpr, row);
  }
}

// Diagnostic: one CTA waits, with the kernels' bounded wait, on an mbarrier
// phase that nothing completes (one pending arrival that never comes). The
// wait gives up after limit_ns and reports through the device error word.
__global__ void wait_timeout_probe(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) wait_phase(&bar, 0u, &abort_flag, 1u, limit_ns);
}

// ------------------------------------------------------------------ host side

constexpr int kMaxDevices = 64;
constexpr int kStaticSmemReserve = 2048;  // barriers, warp sums, flag, slack

using KernelFn = void (*)(Params);

// Kernel instances. VPT = 2 (8 KiB copies) serves N <= 8 with a compile-time
// N for every N at H <= 8192 (KMAX 2 and 4) and for 1, 2, 4, 8 at larger H;
// VPT = 1 (4 KiB copies) serves N = 9..16, whose stages would not fit three
// deep at 8 KiB, with a compile-time N for 16. Other shapes use a runtime-N
// instance. Every shape exists in a general and an EXACT (whole-chunk rows)
// form. Columns of kVpt2: N = runtime, 1, 2, 4, 8, 3, 5, 6, 7.
#define TW_V2S(K, E) {fused_kernel<K, 2, 0, E>, fused_kernel<K, 2, 1, E>, fused_kernel<K, 2, 2, E>, \
                      fused_kernel<K, 2, 4, E>, fused_kernel<K, 2, 8, E>, fused_kernel<K, 2, 3, E>, \
                      fused_kernel<K, 2, 5, E>, fused_kernel<K, 2, 6, E>, fused_kernel<K, 2, 7, E>}
#define TW_V2L(K, E) {fused_kernel<K, 2, 0, E>, fused_kernel<K, 2, 1, E>, fused_kernel<K, 2, 2, E>, \
                      fused_kernel<K, 2, 4, E>, fused_kernel<K, 2, 8, E>, fused_kernel<K, 2, 0, E>, \
                      fused_kernel<K, 2, 0, E>, fused_kernel<K, 2, 0, E>, fused_kernel<K, 2, 0, E>}
// KMAX 16: N = 4 takes the runtime-N instance (the compile-time one spilled
// at the 168-register cap of a 9-warp CTA).
#define TW_V2XL(E) {fused_kernel<16, 2, 0, E>, fused_kernel<16, 2, 1, E>, fused_kernel<16, 2, 2, E>, \
                    fused_kernel<16, 2, 0, E>, fused_kernel<16, 2, 8, E>, fused_kernel<16, 2, 0, E>, \
                    fused_kernel<16, 2, 0, E>, fused_kernel<16, 2, 0, E>, fused_kernel<16, 2, 0, E>}
const KernelFn kVpt2[2][4][9] = {
    {TW_V2S(2, false), TW_V2S(4, false), TW_V2L(8, false), TW_V2XL(false)},
    {TW_V2S(2, true), TW_V2S(4, true), TW_V2L(8, true), TW_V2XL(true)}};
#undef TW_V2S
#undef TW_V2L
#undef TW_V2XL
#define TW_V1(K, E) {fused_kernel<K, 1, 0, E>, fused_kernel<K, 1, 16, E>}
const KernelFn kVpt1[2][5][2] = {
    {TW_V1(1, false), TW_V1(2, false), TW_V1(4, false), TW_V1(8, false), TW_V1(16, false)},
    {TW_V1(1, true), TW_V1(2, true), TW_V1(4, true), TW_V1(8, true), TW_V1(16, true)}};
#undef TW_V1
// Two-pipeline instances, all at KMAX = 4 (H/8 in 513..1024). The chunk ring
// with 8 KiB chunks for N = 1..4 (N = 4 only for whole-chunk rows: the ragged
// form spills at the two-pipeline register cap of 96), and the row ring for
// whole-chunk rows (H = 8192) with N = 9..15 (runtime N) and 16.
const KernelFn kChunkTwo[2][4] = {
    {fused_kernel<4, 2, 1, false, 2>, fused_kernel<4, 2, 2, false, 2>,
     fused_kernel<4, 2, 3, false, 2>, nullptr},
    {fused_kernel<4, 2, 1, true, 2>, fused_kernel<4, 2, 2, true, 2>,
     fused_kernel<4, 2, 3, true, 2>, fused_kernel<4, 2, 4, true, 2>}};
const KernelFn kRowTwo[2] = {rowring_kernel<4, 2, 0, true>, rowring_kernel<4, 2, 16, true>};
// Direct-form instances (one row per CTA): ragged and EXACT, KMAX = 1, 2, 4,
// 8, N = 1..8. The ragged KMAX = 8 instances for N = 6..8 spilled (96-440
// bytes of stack at the 255-register limit) and are not built: those shapes
// keep the chunk ring.
#define TW_DIRECT(K, E) {direct_kernel<K, 1, E>, direct_kernel<K, 2, E>, direct_kernel<K, 3, E>, \
                         direct_kernel<K, 4, E>, direct_kernel<K, 5, E>, direct_kernel<K, 6, E>, \
                         direct_kernel<K, 7, E>, direct_kernel<K, 8, E>}
const KernelFn kDirect[2][4][8] = {
    {TW_DIRECT(1, false), TW_DIRECT(2, false), TW_DIRECT(4, false),
     {direct_kernel<8, 1, false>, direct_kernel<8, 2, false>, direct_kernel<8, 3, false>,
      direct_kernel<8, 4, false>, direct_kernel<8, 5, false>, nullptr, nullptr, nullptr}},
    {TW_DIRECT(1, true), TW_DIRECT(2, true), TW_DIRECT(4, true), TW_DIRECT(8, true)}};
#undef TW_DIRECT
constexpr int kNumKernels = 92 + 8 + 2 + 64;

// The kernel instance for a launch, and what its launch needs.
struct Choice {
  KernelFn fn;
  int index;    // attribute-cache slot
  int kmax;
  int rowring;  // 0: chunk ring (fused_kernel); 1: row ring (rowring_kernel)
  int direct;   // 1: direct form (direct_kernel), no ring
  int groups;   // pipelines per CTA
  int vpt;      // chunk ring: slots per chunk
  int stages1;  // set by shape_for: two pipelines, pipeline 1's stages
  int split_num, split_den;  // set by shape_for: pipeline 0's share of the rows
};

// Per-device attributes, queried once; the launch path reads them without a
// lock once `ready` is set (the flags live in static storage, so they start
// false).
struct DeviceInfo {
  std::atomic<bool> ready;
  int sms;
  int smem_optin;
  int l2_bytes;
  int regs_per_sm;
  std::atomic<bool> attr_done[kNumKernels];
};

DeviceInfo g_devices[kMaxDevices];
std::mutex g_mutex;

int log2_pow2_at_least(int x) {
  int k = 0;
  while ((1 << k) < x) ++k;
  return k;
}

// Column of the instance tables for N (0: runtime N).
int partials_index_vpt2(int n) {
  switch (n) {
    case 1: return 1;
    case 2: return 2;
    case 4: return 3;
    case 8: return 4;
    case 3: return 5;
    case 5: return 6;
    case 6: return 7;
    case 7: return 8;
    default: return 0;
  }
}
int partials_index_vpt1(int n) { return n == 16 ? 1 : 0; }

int vpt_for(int n) { return n <= 8 ? 2 : 1; }

// Which instance serves a launch of `rows` rows of H/8 = vpr vectors over
// `grid` CTAs on a GPU of `sms` SMs. Every form gives bitwise the same rows
// (same thread-to-vector map, same order of every sum), so the choice is by
// speed alone. Measured back to back, interleaved, at H = 8192:
//  * N <= 4, some CTA owning >= 4 rows (>= 3 for N <= 2): the chunk ring
//    with two pipelines. Per SM at an 8-SM budget (T = 4096) N = 1 78 -> 102
//    GB/s, 2: 88 -> 116, 3: 98 -> 121, 4: 107 -> 108; at full GPU 0-5%
//    faster for T >= 1024, but 6% slower with ~3 rows per CTA (T = 512,
//    N = 4), hence the row floor; for N <= 2 with 3-4 rows per CTA
//    (T = 512-600, H = 8192) 3-7% faster back to back.
//  * N >= 9, whole-chunk rows, a grid of at most half the SMs, more rows than
//    CTAs: the row ring with two pipelines, whose 16 KiB copies lift the
//    per-SM rate from 83-95 to 112 GB/s at an 8-SM budget. At full GPU, where
//    an SM needs ~45 GB/s, the chunk ring is 2-4% faster. With one row per
//    CTA one of the two pipelines idles and the chunk ring, with every
//    source's chunks in flight, is 10-20% faster (T = 16-76, N = 9-16).
//  * one row per CTA, N <= 8, H <= 16384 (but not N >= 6 with H over 8192
//    and short of 16384): the direct form, with no staging in shared memory. Interleaved against the
//    one-pipeline chunk ring at T = 32-152 (H = 4096, 8192; N = 2, 8): per
//    launch up to 25% faster and never slower; back to back 8-17% faster at
//    T = 128-152 and within 3% at T <= 64; from one CUDA graph 11-23% faster,
//    except at H = 8192, N = 8, T <= 64 (-3% to +4%). At H = 16384 (N = 2, 4,
//    8) never slower per launch; back to back 9-22% faster at N = 2, 3-7% at
//    N = 8, unchanged at N = 4. Ragged rows (H = 1024, 3072, 5120, 6144,
//    7168, 12288; N = 2, 8; T = 32-152): never slower per launch, from one
//    CUDA graph 5-30% faster, back to back mostly 5-17% faster.
//  * otherwise the chunk ring with one pipeline.
Choice select_kernel(int vpr, int n, int64_t rows, int grid, int sms) {
  Choice c;
  c.direct = 0;
  const int dk = log2_pow2_at_least((vpr + kSlotVec - 1) / kSlotVec);  // direct KMAX = 2^dk
  const int dexact = vpr == (1 << dk) * kSlotVec ? 1 : 0;
  if (rows <= grid && n <= 8 && dk <= 3 && kDirect[dexact][dk][n - 1] != nullptr) {
    c.direct = 1;
    c.kmax = 1 << dk;
    c.rowring = 0;
    c.groups = 1;
    c.vpt = 1;  // unused
    c.index = 102 + dexact * 32 + dk * 8 + (n - 1);
    c.fn = kDirect[dexact][dk][n - 1];
    return c;
  }
  const int vpt = vpt_for(n);
  const int chunks = (vpr + kSlotVec * vpt - 1) / (kSlotVec * vpt);
  const int k = log2_pow2_at_least(chunks * vpt);  // KMAX = 2^k
  c.kmax = 1 << k;
  c.rowring = 0;
  c.groups = 1;
  c.vpt = vpt;
  const int exact = vpr == (1 << k) * kSlotVec ? 1 : 0;
  const bool enough_rows = rows >= (n <= 2 ? 3 : 4) * static_cast<int64_t>(grid);
  if (vpt == 2 && k == 2 && enough_rows && (n <= 3 || (n == 4 && exact))) {
    c.groups = 2;
    c.index = 92 + exact * 4 + (n - 1);
    c.fn = kChunkTwo[exact][n - 1];
    return c;
  }
  if (n >= 9 && vpr == 4 * kSlotVec && 2 * grid <= sms && rows > grid) {
    c.rowring = 1;
    c.groups = 2;
    c.kmax = 4;
    c.index = 100 + (n == 16 ? 1 : 0);
    c.fn = kRowTwo[n == 16 ? 1 : 0];
    return c;
  }
  if (vpt == 2) {
    const int ki = k - 1, ni = partials_index_vpt2(n);  // KMAX 2..16
    c.index = exact * 36 + ki * 9 + ni;
    c.fn = kVpt2[exact][ki][ni];
  } else {
    const int ni = partials_index_vpt1(n);  // KMAX 1..16
    c.index = 72 + exact * 10 + k * 2 + ni;
    c.fn = kVpt1[exact][k][ni];
  }
  return c;
}

int device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TW_ERR_CUDA;
  DeviceInfo& d = g_devices[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return TW_ERR_CUDA;
      if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
          cudaSuccess)
        return TW_ERR_CUDA;
      if (cudaDeviceGetAttribute(&d.l2_bytes, cudaDevAttrL2CacheSize, dev) != cudaSuccess)
        return TW_ERR_CUDA;
      if (cudaDeviceGetAttribute(&d.regs_per_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) !=
          cudaSuccess)
        return TW_ERR_CUDA;
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return TW_OK;
}

// One CTA per SM, at most sm_budget (0: all) and at most one per row.
int grid_for(const DeviceInfo& d, int64_t rows, int sm_budget) {
  int grid = d.sms;
  if (sm_budget > 0 && sm_budget < grid) grid = sm_budget;
  if (rows < grid) grid = static_cast<int>(rows);
  return grid;
}

// Registers per thread of each instance, queried once (0: not yet known).
// They are a property of the compiled code, the same on every device.
std::atomic<int> g_kernel_regs[kNumKernels];

// Whether two CTAs of a direct-form instance fit in one SM's registers
// (allocated per warp in units of 8 registers a thread), which also caches
// the instance's register count.
bool two_direct_ctas_fit(const DeviceInfo& d, const Choice& c) {
  int r = g_kernel_regs[c.index].load(std::memory_order_relaxed);
  if (r == 0) {
    cudaFuncAttributes a;
    if (cudaFuncGetAttributes(&a, c.fn) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    r = a.numRegs;
    g_kernel_regs[c.index].store(r, std::memory_order_relaxed);
  }
  const int per_cta = (r + 7) / 8 * 8 * kConsumerThreads;
  return 2 * per_cta <= d.regs_per_sm;
}
// How many CTAs of a direct-form instance an SM holds at once: by registers,
// and at most 8 (2048 threads of 256).
int direct_ctas_per_sm(const DeviceInfo& d, const Choice& c) {
  if (!two_direct_ctas_fit(d, c)) return 1;
  const int r = g_kernel_regs[c.index].load(std::memory_order_relaxed);
  const int per_cta = (r + 7) / 8 * 8 * kConsumerThreads;
  const int k = d.regs_per_sm / per_cta;
  return k < 8 ? k : 8;
}

// The launch of `rows` rows: the instance (*choice) and its shape.
int shape_for(const DeviceInfo& d, int64_t rows, int64_t hidden, int n, int sm_budget,
              Choice* choice, LaunchShape* shape) {
  int grid = grid_for(d, rows, sm_budget);
  if (sm_budget == 0 && rows > grid && rows <= 8 * static_cast<int64_t>(d.sms)) {
    // On the whole GPU with more rows than SMs: one direct-form CTA per row
    // while the rows fit in one wave of co-resident direct CTAs (k per SM, by
    // registers), instead of a ring CTA per SM that owns several rows.
    // Interleaved against the ring: at T = 160-304 (k >= 2) per launch never
    // slower, from one CUDA graph 1-30% faster and back to back 1-22% faster
    // at H = 4096 (N = 2, 4, 8) and H = 8192 (N = 2, 4); at T = 400-760
    // (k = 3-5: H = 4096, N = 2, 4; H = 8192, N = 2) back to back 10-27%
    // faster. At H = 8192, N = 8 (144 registers: k = 1, so two waves) it was
    // 6-17% slower back to back, which the register count excludes.
    const Choice w = select_kernel(static_cast<int>(hidden / 8), n, rows, static_cast<int>(rows),
                                   d.sms);
    if (w.direct && rows <= static_cast<int64_t>(direct_ctas_per_sm(d, w)) * d.sms)
      grid = static_cast<int>(rows);
  }
  const Choice c = select_kernel(static_cast<int>(hidden / 8), n, rows, grid, d.sms);
  if (c.direct) {
    Choice cc = c;
    cc.stages1 = 0;
    cc.split_num = 1;
    cc.split_den = 2;
    shape->grid = grid;
    shape->threads = kConsumerThreads;
    shape->smem_bytes = 0;
    shape->stages = 0;
    shape->kmax = c.kmax;
    *choice = cc;
    return TW_OK;
  }
  // one stage: a source's row (row ring) or a chunk of every source (chunk ring)
  const int stage_bytes = c.rowring ? c.kmax * kSlotBytes : (n + 1) * kSlotBytes * c.vpt;
  int stages = (d.smem_optin - kStaticSmemReserve) / (c.groups * stage_bytes);
  if (stages > kMaxStages / c.groups) stages = kMaxStages / c.groups;
  if (stages < 2) return TW_ERR_UNSUPPORTED;
  Choice cc = c;
  cc.stages1 = c.groups == 2 ? stages : 0;
  cc.split_num = 1;
  cc.split_den = 2;
  const int whole = (d.smem_optin - kStaticSmemReserve) / stage_bytes;  // stages of one ring
  if (c.groups == 2 && !c.rowring && stages == 2 && whole >= 5 && 2 * grid <= d.sms) {
    // Two chunk-ring pipelines of 2 stages each (N = 4 at 40 KiB a stage)
    // leave a fifth stage unused. Under an SM budget pipeline 0 takes it and
    // 13/20 of the rows: 107-110 -> 115-117 GB/s per SM at 2-16 SMs (shares
    // of 11/20, 3/5 and 7/10 measured 110-111, 113-116, 114-117). On the
    // whole GPU the even split was 1-2% faster.
    stages = 3;
    cc.stages1 = 2;
    cc.split_num = 13;
    cc.split_den = 20;
  }
  if (rows <= grid && !c.rowring && c.groups == 1) {
    // One row per CTA: a ring of the row's chunks holds the whole row. Where
    // that is under half an SM's shared memory (H <= 4096; H = 8192 with
    // N <= 4), the next launch's CTAs can become resident beside this one's
    // and prefetch their rows while it runs: -5 to -9% back to back at
    // T = 128-152, H = 2048-4096, N = 8; unchanged elsewhere within 1%.
    const int vpr = static_cast<int>(hidden / 8);
    const int row_chunks = (vpr + kSlotVec * c.vpt - 1) / (kSlotVec * c.vpt);
    if (stages > row_chunks) stages = row_chunks;
  }
  shape->grid = grid;
  shape->threads = c.groups * kConsumerThreads + 32;
  shape->smem_bytes = (stages + cc.stages1) * stage_bytes;
  shape->stages = stages;
  shape->kmax = c.kmax;
  *choice = cc;
  return TW_OK;
}

}  // namespace

int plan_launch(int64_t rows, int64_t hidden, int n, int sm_budget, LaunchShape* shape) {
  DeviceInfo* d = nullptr;
  int st = device_info(&d);
  if (st != TW_OK) return st;
  Choice c;
  return shape_for(*d, rows, hidden, n, sm_budget, &c, shape);
}

int launch_fused(const FusedArgs& a, cudaStream_t stream, int sm_budget, int* smid_out) {
  DeviceInfo* d = nullptr;
  int st = device_info(&d);
  if (st != TW_OK) return st;
  Choice choice;
  LaunchShape shape;
  st = shape_for(*d, a.rows, a.hidden, a.n, sm_budget, &choice, &shape);
  if (st != TW_OK) return st;
  if (shape.grid <= 0) return TW_OK;

  Params p;
  for (int r = 0; r < TW_MAX_PARTIALS; ++r)
    p.partials[r] = r < a.n ? static_cast<const uint4*>(a.partials[r]) : nullptr;
  p.gamma = static_cast<const uint4*>(a.gamma);
  p.residual = static_cast<uint4*>(a.residual);
  p.out = static_cast<uint4*>(a.out);
  p.smid_out = smid_out;
  // L2 policy per call, measured back to back, interleaved, on three GB300s.
  // With the prefetch below in place (some CTA owns more than one row),
  // normal loads win for N = 3..8 at every size (+1-6% at T = 384-4096,
  // H = 4096-16384). Evict-first loads with a streaming output win for
  // N <= 2 and N >= 9 while the output is at most an eighth of the L2 (+1-6%
  // at T <= 1024, H = 8192), and for N <= 2 again once the output reaches
  // 7/16 of the L2 (+1-3.5% at T = 4096-8192); in between, normal loads win
  // by 2-5%. With one row per CTA and no prefetch (a row over 144 KiB)
  // evict-first wins for N = 4 and 8 at every shape measured (+2-10% at
  // T = 32-152, H = 4096-16384); with the whole-row prefetch below, normal
  // loads win for N = 3-8 (+1-6% at T = 32-128, H = 8192), and N <= 2 keeps
  // evict-first through its small-output clause.
  const int64_t out_bytes = a.rows * a.hidden * 2;
  const int64_t l2 = static_cast<int64_t>(d->l2_bytes);
  const bool small_out = out_bytes * 8 <= l2;
  const bool large_out = out_bytes * 16 >= l2 * 7;
  const bool one_row_per_cta = a.rows <= shape.grid;
  const bool row_fits = static_cast<int64_t>(a.n + 1) * a.hidden * 2 <=
                        static_cast<int64_t>(kPrefetchPerCta);
  p.l2_stream = ((one_row_per_cta && !row_fits) || (a.n <= 2 && (small_out || large_out)) ||
                 (a.n >= 9 && small_out))
                    ? 1
                    : 0;
  // About 144 KiB per CTA, shared among the N + 1 sources. With one row per
  // CTA only when that covers the whole row ((N + 1) * H * 2 <= 144 KiB): the
  // next launch's CTAs land on SMs as this launch's one-row CTAs leave them,
  // and a whole-row prefetch took 7-17% off back-to-back launches at
  // T = 16-152 (H = 2048-8192 at every N; H = 16384 at N = 2), while a
  // partial one (H = 16384, N = 8; H = 32768) measured up to 12% slower.
  p.prefetch_bytes = (!one_row_per_cta || row_fits)
                         ? (kPrefetchPerCta / static_cast<uint32_t>(a.n + 1)) & ~15u
                         : 0u;
  p.rows = a.rows;
  p.vec_per_row = static_cast<int>(a.hidden / 8);
  p.n_partials = a.n;
  const int chunk_vec = kSlotVec * (choice.rowring ? 1 : choice.vpt);  // row ring: unused
  p.chunks = (p.vec_per_row + chunk_vec - 1) / chunk_vec;
  p.stages = shape.stages;
  p.stages1 = choice.stages1;
  p.split_num = choice.split_num;
  p.split_den = choice.split_den;
  p.eps = a.eps;
  p.hidden = static_cast<float>(a.hidden);

  const KernelFn fn = choice.fn;
  const int index = choice.index;
  if (!choice.direct && !d->attr_done[index].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d->attr_done[index].load(std::memory_order_relaxed)) {
      const int max_dyn = d->smem_optin - kStaticSmemReserve;
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, max_dyn) !=
          cudaSuccess)
        return TW_ERR_CUDA;
      d->attr_done[index].store(true, std::memory_order_release);
    }
  }
  // Launched with programmatic stream serialization: the CTAs may start while
  // the previous kernel in the stream drains (the kernel waits on
  // griddepcontrol.wait before any global-memory load or store; only the L2
  // prefetch hint goes out before it).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(shape.grid));
  cfg.blockDim = dim3(static_cast<unsigned>(shape.threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(shape.smem_bytes);
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

int launch_wait_probe(long long limit_ns, cudaStream_t stream) {
  wait_timeout_probe<<<1, 32, 0, stream>>>(static_cast<unsigned long long>(limit_ns));
  return cudaGetLastError() == cudaSuccess ? TW_OK : TW_ERR_CUDA;
}

int read_device_error(int reset, int* code) {
  if (cudaDeviceSynchronize() != cudaSuccess) return TW_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return TW_ERR_CUDA;
  if (reset) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return TW_ERR_CUDA;
  }
  if (code) *code = static_cast<int>(v);
  return TW_OK;
}

}  // namespace tw
