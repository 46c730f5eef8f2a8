/*
 * libtw -- fused reduce + residual + RMSNorm and wave-aware token splitting
 * on one GPU (sm_103a).
 *
 * Pages cited (by title and section):
 *   [W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
 *       Arithmetic, Not Finer Tiles"
 *   [G] "TokenWeave Guide: Compute-Communication Overlap for LLMs"
 *
 * Conventions shared by every call:
 *   - Tensors are bf16, row-major and contiguous: a [T, H] tensor is T token
 *     rows of H hidden values, row stride H elements. A shard or half of a
 *     tensor is passed by offsetting its pointers by row0 * H elements.
 *   - The caller owns every buffer. libtw allocates no device memory; it keeps
 *     only per-device launch attributes (SM count, shared-memory limit, L2
 *     size, which sets the per-call L2 policy).
 *   - Launches are asynchronous on the stream(s) given; a device fault shows
 *     at the caller's next synchronisation, as usual in CUDA. Work runs on the
 *     device that is current on the calling thread, and every pointer and
 *     stream must belong to that device. libtw does not check this (a query
 *     per pointer would cost more host time than a small step's launch); the
 *     Python binding refuses tensors and streams on other devices.
 *   - Every launch uses programmatic dependent launch: its thread blocks may
 *     become resident while the previous kernel on the stream is still
 *     running. The fused step's blocks then ask L2 to prefetch the first bytes
 *     of their input rows, a hint that reads nothing into the step. Every
 *     load and store of a launch happens after that kernel has completed, so
 *     stream order holds as for an ordinary launch.
 *   - Arguments are validated before any CUDA call. Every call returns a
 *     tw_status; no C++ exception crosses this boundary.
 *   - A stream argument is a cudaStream_t; NULL is the legacy default stream.
 */
#ifndef TW_H
#define TW_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are the library's only exported symbols. */
#if defined(__GNUC__)
#define TW_API __attribute__((visibility("default")))
#else
#define TW_API
#endif

struct CUstream_st;
typedef struct CUstream_st* tw_stream_t; /* == cudaStream_t */
struct CUevent_st;
typedef struct CUevent_st* tw_event_t; /* == cudaEvent_t */

/* Largest number of partial buffers (tensor-parallel ranks) one call sums. */
#define TW_MAX_PARTIALS 16
/* Largest hidden size: the kernel keeps a whole token row in registers. */
#define TW_MAX_HIDDEN 32768

typedef enum {
  TW_OK = 0,
  TW_ERR_INVALID_ARG = 1, /* null pointer, count or size out of range, overlap */
  TW_ERR_ALIGN = 2,       /* H % 8 != 0 or a pointer not 16-byte aligned */
  TW_ERR_UNSUPPORTED = 3, /* H > TW_MAX_HIDDEN */
  TW_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  TW_ERR_DEVICE = 5       /* a kernel gave up on a bounded wait (see tw_device_status) */
} tw_status;

/*
 * tw_fused_reduce_residual_rmsnorm -- the fused step.
 *
 * Defined by [W] "Fix two: RMSNorm was never insignificant" (the per-CTA
 * sketch and its four numbered steps) and [G] "Fused AllReduce-RMSNorm:
 * Bypassing Global Memory" / "The Standard RMSNorm Memory Round-Trip" (the
 * RMSNorm formula). On one GPU the N tensor-parallel ranks' contributions are
 * N buffers in this GPU's memory. For every token row t:
 *
 *     z       = ((P_0[t] + P_1[t]) + ... + P_{N-1}[t]) + R[t]   fp32, rank order
 *     R[t]    = bf16_rne(z)                                       in place
 *     r       = rsqrt( (sum_j z_j^2) / H + eps )                  fp32
 *     out[t]  = bf16_rne( (z * r) * gamma )                       fp32, one rounding
 *
 * The sum of squares is taken on the unrounded fp32 z ([W] step 2). Rows are
 * independent: any token-contiguous shard gives bitwise the same rows as the
 * whole batch, and so does every sm_budget (the per-row arithmetic does not
 * depend on the launch shape).
 *
 *   partials   host array of N device pointers, each bf16 [T, H], read only.
 *              The array is read during the call only; partials may alias
 *              one another.
 *   N          1 .. TW_MAX_PARTIALS.
 *   residual   device bf16 [T, H], read then overwritten with bf16(z).
 *   gamma      device bf16 [H], read only.
 *   eps        >= 0 and finite (1e-5 for the Llama workloads). With eps = 0
 *              a row whose z is all zero has no scale (0 * rsqrt(0)): its
 *              out row is NaN, as the formula gives; with eps > 0 it is 0.
 *   T          token rows, >= 0; T == 0 is a no-op returning TW_OK.
 *   H          hidden size, 8 .. TW_MAX_HIDDEN, a multiple of 8.
 *   out        device bf16 [T, H], written. It may be exactly the buffer of
 *              one partial (out == partials[r]) to write Y over that rank's
 *              partial; no other overlap with an input is allowed.
 *   stream     the stream to launch on.
 *   sm_budget  0: use the whole GPU (one CTA per SM; with more rows than SMs,
 *              one CTA per row while all of them fit on the GPU at once, which
 *              the register-loading form allows for small rows and small N).
 *              k > 0: launch at most k
 *              CTAs, each owning a contiguous range of about T / k rows, so
 *              the step occupies at most k SMs and co-runs with work on the
 *              other SMs ([W] "What it buys": 2 to 8 SMs). A CTA that owns
 *              more than one row requests enough shared memory that no second
 *              CTA of this kernel fits on its SM; with one row per CTA (T <= k
 *              or T <= the SM count) it stages at most that row (for N <= 8
 *              and H <= 16384 it loads the row into registers, with no
 *              staging), so such CTAs may share an SM with the next launch's
 *              CTAs. k above the SM count is clamped. Negative is invalid.
 *
 * Errors: TW_ERR_INVALID_ARG (N, T, H <= 0, eps, sm_budget, a null pointer,
 * residual/out overlapping each other or any input other than out ==
 * partials[r], T*H too large),
 * TW_ERR_ALIGN (H % 8 or any pointer not 16-byte aligned), TW_ERR_UNSUPPORTED
 * (H > TW_MAX_HIDDEN), TW_ERR_CUDA (device query or launch failure).
 */
TW_API int tw_fused_reduce_residual_rmsnorm(const void* const* partials, int N, void* residual,
                                     const void* gamma, float eps, int64_t T, int64_t H,
                                     void* out, tw_stream_t stream, int sm_budget);

/*
 * Offsets and threshold for tw_wave_split. Pass NULL for the pages' values:
 * offsets {0, 64, 128, 192, 256, 512} and a 1024-token threshold ([W] "Fix
 * one": the offline sweep's offsets and the dense-model threshold).
 *   offsets          NULL (with n_offsets == 0): every integer 0 .. half-1.
 *                    Otherwise n_offsets values >= 0 (both signs are tried).
 *   min_split_tokens below this token count no split is made.
 */
typedef struct {
  const int* offsets;
  int n_offsets;
  int min_split_tokens;
} tw_split_opts;

/*
 * tw_wave_split -- wave-aware prefix/suffix split of a token batch.
 *
 * Defined by [W] "The overlap trap" (a kernel of c CTAs on S SMs runs in
 * ceil(c / S) waves) and "Fix one: split at wave boundaries, unequally": the
 * batch is split exactly twice, prefix = half + offset and suffix = half -
 * offset with half = T / 2, and a split is admissible only if the waves of the
 * two pieces do not exceed the waves of the unsplit kernel. The worked example
 * (300 CTAs, 132 SMs: 132 / 168 in 3 waves, not 150 / 150 in 4) puts the
 * smaller piece first, so each offset is tried with both signs.
 *
 * Reading of the rule (the pages give it in CTAs, the call works in tokens):
 *   c(t)   = ceil(t * ctas_unsplit / num_tokens)   CTAs of a t-token piece
 *   W      = ceil(ctas_unsplit / num_sms)          unsplit waves
 *   admissible p: 0 < p < T and ceil(c(p)/S) + ceil(c(T-p)/S) <= W
 *   choice: the smallest |offset|, ties to the smaller prefix.
 *   no split, (T, 0), when T < min_split_tokens, W <= 1 (the single-wave
 *   rule of "Fix one") or no candidate is admissible; (0, 0) for T == 0.
 *
 *   num_tokens      T >= 0.
 *   ctas_unsplit    C >= 0, the unsplit kernel's CTA count for T tokens.
 *   num_sms         S > 0.
 *   opts            NULL or see tw_split_opts.
 *   prefix_tokens   out: p.   suffix_tokens   out: T - p.   (host pointers)
 *
 * Pure host integer code: no CUDA call, no GPU needed.
 * Errors: TW_ERR_INVALID_ARG (T < 0, C < 0, S <= 0, null output pointer,
 * n_offsets < 0, offsets NULL with n_offsets > 0, a negative offset).
 */
TW_API int tw_wave_split(int64_t num_tokens, int64_t ctas_unsplit, int num_sms, const tw_split_opts* opts,
                  int64_t* prefix_tokens, int64_t* suffix_tokens);

/*
 * tw_split_lookup -- the split plan from a lookup table of measured splits,
 * falling back to tw_wave_split.
 *
 * [W] "Fix one": because the GEMM kernels are closed, the split offset is
 * chosen offline by timing a forward pass for each offset and storing the
 * winner per token count in a lookup table, consulted every iteration. The
 * table here is n_entries pairs (table_tokens[i], table_prefix[i]), e.g. as
 * written by `bench.py --offset-sweep`. If num_tokens equals table_tokens[i]
 * for some i, the plan is (table_prefix[i], num_tokens - table_prefix[i]);
 * otherwise it is tw_wave_split(num_tokens, ctas_unsplit, num_sms, opts).
 * The first matching entry wins. Host-only integer code.
 *
 * Errors: TW_ERR_INVALID_ARG (n_entries < 0, a NULL table with n_entries >
 * 0, a matching entry whose prefix is outside [0, num_tokens], or any error
 * of tw_wave_split).
 */
TW_API int tw_split_lookup(const int64_t* table_tokens, const int64_t* table_prefix, int n_entries,
                    int64_t num_tokens, int64_t ctas_unsplit, int num_sms,
                    const tw_split_opts* opts, int64_t* prefix_tokens, int64_t* suffix_tokens);

/*
 * tw_run_split -- the fused step over a token batch split in two, on two
 * streams ([G] "Architectural Foundations of TokenWeave": the first chunk's
 * fused step runs on a second stream while the first stream goes on; [W]
 * "Fix one": prefix ops before suffix ops).
 *
 * Rows [0, prefix_tokens) run on stream_a and rows [prefix_tokens, T) on
 * stream_b, each as tw_fused_reduce_residual_rmsnorm with the same sm_budget
 * (so up to 2 * sm_budget SMs while both run). stream_b first waits for the
 * work already queued on stream_a; on return stream_a is ordered after both
 * halves. An empty half is not launched. The result is bitwise the same as
 * the unsplit call. The fork and join use two CUDA events per device that
 * each calling host thread takes on first use from a process-wide pool
 * (created there when the pool is empty) and hands back to it when the
 * thread exits; pooled events last until the process ends, so their number
 * stays bounded by the most threads that called at once. The call never
 * creates or destroys streams. stream_a == stream_b is allowed (the halves
 * then run in order, with no events). The call can be captured into a CUDA
 * graph (the two streams become a fork and a join in the graph) once an
 * eager call of the same shape has run on the thread, so that the kernel's
 * attributes and the events already exist.
 *
 * Arguments as for the fused call, plus prefix_tokens in [0, T].
 */
TW_API int tw_run_split(int64_t prefix_tokens, const void* const* partials, int N, void* residual,
                 const void* gamma, float eps, int64_t T, int64_t H, void* out,
                 tw_stream_t stream_a, tw_stream_t stream_b, int sm_budget);

/*
 * tw_run_wave_split -- plan and run in one call: the wave-aware split
 * tw_wave_split(T, ctas_unsplit, num_sms, opts), computed on every call
 * ([W] "Fix one": the split is decided each iteration), then tw_run_split
 * with that prefix. prefix_tokens and suffix_tokens (host pointers, each may
 * be NULL) receive the plan. The fused arguments are validated first, then
 * the planner's; both before any CUDA call. Arguments, ordering and errors
 * otherwise as for tw_wave_split and tw_run_split.
 */
TW_API int tw_run_wave_split(int64_t ctas_unsplit, int num_sms, const tw_split_opts* opts,
                      const void* const* partials, int N, void* residual, const void* gamma,
                      float eps, int64_t T, int64_t H, void* out, tw_stream_t stream_a,
                      tw_stream_t stream_b, int sm_budget, int64_t* prefix_tokens,
                      int64_t* suffix_tokens);

/*
 * tw_run_split_after -- the split step as the pages pipeline it against the
 * projection that produces the partials ([G] "Architectural Foundations of
 * TokenWeave" and "The Mathematics of Token-Splitting and Overlap": stream A
 * computes GEMM(T1) then GEMM(T2); stream B runs the fused step of T1 as soon
 * as GEMM(T1) is done, overlapping GEMM(T2), then the fused step of T2).
 *
 * On `stream`, in order: wait for `prefix_ready` (if not NULL), run the
 * fused step on rows [0, prefix_tokens); wait for `suffix_ready` (if not
 * NULL), run it on rows [prefix_tokens, T). The caller records the events on
 * the stream that produces the prefix's and the suffix's partials. Give
 * `stream` a high priority so its CTAs are placed ahead of the compute
 * kernel's as SMs free up, and an sm_budget so the compute keeps the rest.
 * The result is bitwise that of the unsplit call. Empty halves are skipped.
 * Arguments and errors as for tw_run_split; events are cudaEvent_t handles
 * owned by the caller.
 */
TW_API int tw_run_split_after(int64_t prefix_tokens, const void* const* partials, int N, void* residual,
                       const void* gamma, float eps, int64_t T, int64_t H, void* out,
                       tw_stream_t stream, tw_event_t prefix_ready, tw_event_t suffix_ready,
                       int sm_budget);

/*
 * tw_shard_rows -- the token-boundary shard of one rank, for the multi-GPU
 * form of the step ([W] "Fix two: RMSNorm was never insignificant": the
 * all-reduce is taken apart into a reduce-scatter and an all-gather at token
 * boundaries, so that each rank normalises only its own whole token rows).
 *
 * With s = ceil(num_tokens / world), rank r owns rows
 * [min(r * s, T), min((r + 1) * s, T)): shards are contiguous, disjoint, in
 * rank order and cover every row exactly once; every shard has s rows except
 * the last non-empty one, which may be shorter, and trailing ranks may own
 * none (T = 5 over 4 ranks gives 2, 2, 1 and 0 rows). A shard padded to s
 * rows is what an all-gather of equal-sized pieces moves.
 *
 *   num_tokens  T >= 0.
 *   world       number of ranks, >= 1.
 *   rank        0 .. world - 1.
 *   row0, rows  out (host pointers): first row and row count of the shard.
 *
 * Pure host integer code: no CUDA call, no GPU needed.
 * Errors: TW_ERR_INVALID_ARG (T < 0, world <= 0, rank out of range, a NULL
 * output pointer).
 */
TW_API int tw_shard_rows(int64_t num_tokens, int world, int rank, int64_t* row0, int64_t* rows);

/* Text of a tw_status value (static storage; never NULL). */
TW_API const char* tw_strerror(int status);

/*
 * tw_launch_shape -- the launch the fused call would make on the current
 * device: grid (CTAs, = SMs used), threads per CTA, dynamic shared memory
 * bytes and pipeline stages (0 stages and 0 bytes for a launch that loads
 * its one row per CTA straight into registers). Any output pointer may be
 * NULL. Queries device attributes (TW_ERR_CUDA without a GPU). Validation as
 * for the fused call.
 */
TW_API int tw_launch_shape(int64_t T, int64_t H, int N, int sm_budget, int* grid, int* threads,
                    int* smem_bytes, int* stages);

/*
 * tw_device_status -- read, and optionally clear, the device-side error word
 * that kernels set when a bounded wait gives up (a code other than 0 means
 * the outputs of some call since the last reset are not valid). Synchronises
 * the current device first. *code: 0 none; bit 0 a consumer gave up waiting
 * for staged data; bit 1 the producer gave up waiting for a free stage; bit 2
 * a final drain of in-flight copies gave up.
 */
TW_API int tw_device_status(int reset, int* code);

/*
 * tw_debug_wait_timeout -- a diagnostic of the kernels' bounded waits: one
 * CTA waits, with the same bounded-wait routine the fused kernel uses, on a
 * barrier phase that nothing completes. The wait gives up after limit_ns
 * (1 us .. 2 s) and sets bit 0 of the device error word, which
 * tw_device_status then reports. The GPU stays usable. For testing the
 * failure path without faulting or hanging a GPU.
 */
TW_API int tw_debug_wait_timeout(int64_t limit_ns, tw_stream_t stream);

/*
 * tw_fused_debug_smid -- the fused call, additionally writing the %smid of
 * each CTA to smid_out[blockIdx] (device int32 array with at least the
 * grid's length, see tw_launch_shape). For checking that an sm_budget of k
 * occupies at most k SMs.
 */
TW_API int tw_fused_debug_smid(const void* const* partials, int N, void* residual, const void* gamma,
                        float eps, int64_t T, int64_t H, void* out, tw_stream_t stream,
                        int sm_budget, int* smid_out);

/*
 * Unfused baseline: the two kernels the fused step replaces, for measuring
 * what the fusion saves on one GPU ([W] "Fix two": vLLM normalises after the
 * all-reduce has written its result; [G] "The Standard RMSNorm Memory
 * Round-Trip": the reduced tensor goes to HBM and a separate kernel reads it
 * back). Together they compute the same step with two extra bf16 roundings
 * and (N+5)*T*H*2 bytes of HBM traffic instead of (N+3)*T*H*2.
 *
 * tw_reduce_partials: sum_out[t] = bf16_rne(((P_0[t] + P_1[t]) + ...) + P_{N-1}[t]),
 * fp32 adds in rank order.
 *   partials   host array of N device pointers, bf16 [T, H], read only.
 *   sum_out    device bf16 [T, H], written; must not overlap a partial.
 *   Other arguments and errors as for the fused call (N 1..16, H % 8 == 0,
 *   16-byte aligned pointers, T == 0 a no-op).
 */
TW_API int tw_reduce_partials(const void* const* partials, int N, int64_t T, int64_t H, void* sum_out,
                       tw_stream_t stream);

/*
 * tw_add_rmsnorm: a standalone residual add + RMSNorm over the stored sum:
 *     x = fp32(sum[t]) + fp32(residual[t]);  residual[t] = bf16_rne(x);
 *     r = rsqrt(sum_j residual[t]_j^2 / H + eps)   (on the stored bf16 values)
 *     out[t] = bf16_rne((residual[t] * r) * gamma)
 *   sum        device bf16 [T, H], read only; may be the same pointer as out
 *              (each row is read before it is written), otherwise must not
 *              overlap out.
 *   residual   device bf16 [T, H], in/out; must not overlap sum, out or gamma.
 *   Other arguments and errors as for the fused call.
 */
TW_API int tw_add_rmsnorm(const void* sum, void* residual, const void* gamma, float eps, int64_t T,
                   int64_t H, void* out, tw_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* TW_H */
