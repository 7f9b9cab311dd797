/*
 * dopt.h -- C ABI of the sharded mixed-precision Adam step on one GPU.
 *
 * The operation is the data-parallel hot path of a Megatron-style
 * DistributedOptimizer (ZeRO-1) step over a contiguous param-and-grad buffer,
 * as described by the "Megatron-LM distrib_optimizer.py close reading" page
 * (xiaolong-dev.me, megatron-docs/optimizer/distrib_optimizer), the "ZeRO
 * memory ledger and Megatron DistributedOptimizer" page (llm-infra-atlas,
 * parallel/01_dp/02_zero_and_distributed_optimizer) and the "Megatron-LM
 * distributed package" page (2kiu.com).  Citations below name the page and
 * its section.
 *
 * Conventions (every entry point):
 *  - Return value: DOPT_OK (0) or a negative dopt_status.  Nothing aborts and
 *    no C++ exception crosses this boundary.  dopt_last_error() returns a
 *    thread-local message describing the last failure.
 *  - Device memory: every device pointer is allocated and owned by the
 *    caller, must be 16-byte aligned unless its description says otherwise,
 *    and stays owned by the caller.  The library allocates no device memory.
 *    The library-owned objects are the opaque shard map (host memory), freed
 *    by dopt_shard_map_free(), and the side stream and event that
 *    dopt_step and dopt_step_from_host create once per thread and device.
 *  - Streams: a dopt_stream is a cudaStream_t passed as a plain pointer
 *    (NULL = the legacy default stream).  Device entry points only enqueue
 *    work on it and return; dopt_step() and dopt_step_noalloc() wait until
 *    the step's results (found_inf, the grad norm) are known -- the AdamW
 *    pass may still be running on the stream when they return -- and
 *    dopt_step_from_host() waits for the whole step.  Work queued later on
 *    the same stream sees the updated state; a reader on the host or on
 *    another stream synchronises with the step's stream first.
 *  - Element counts are int64; dtypes are dopt_dtype codes.
 *  - Rank selection: rank in [0, DP) steps that rank's shard; DOPT_ALL_RANKS
 *    emulates every rank of the instance on this GPU, their shard arrays laid
 *    out rank-major (rank r's slot begins at r * shard_numel).
 *  - Flat shard layout: a rank's shard of a buffer is the concatenation, in
 *    bucket order, of its slice of every bucket (dopt_bucket_info.shard_base
 *    is where bucket b's slice starts).  main_grad, master, exp_avg and
 *    exp_avg_sq use this layout.  Only elements of parameters are read or
 *    written; padding positions of these arrays are never touched.
 */
#ifndef DOPT_H
#define DOPT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* dopt_stream; /* a cudaStream_t */

typedef enum { DOPT_F32 = 0, DOPT_BF16 = 1, DOPT_F16 = 2 } dopt_dtype;

typedef enum {
  DOPT_OK = 0,
  DOPT_E_INVALID = -1, /* bad argument (null, out of range, inconsistent)   */
  DOPT_E_ALIGN = -2,   /* a device pointer is not 16-byte aligned            */
  DOPT_E_SIZE = -3,    /* workspace too small, or a size exceeds a limit     */
  DOPT_E_CUDA = -4,    /* a CUDA runtime call or kernel launch failed        */
  DOPT_E_NOMEM = -5    /* host allocation failed                             */
} dopt_status;

/* Shard group of a buffer (distrib_optimizer page, "five groups"; ledger
 * page, section 3): bf16/fp16 params get an fp32 master copy of their shard
 * (shard_fp32_from_float16); fp32 params are stepped in place in the param
 * buffer (shard_fp32). */
typedef enum { DOPT_GROUP_FP32_FROM_FLOAT16 = 0, DOPT_GROUP_FP32 = 1 } dopt_group;

/* Layout of the emulated replica gradient buffers. */
typedef enum {
  DOPT_LAYOUT_FULL_BUFFER = 0, /* each replica is a whole grad buffer (numel)   */
  DOPT_LAYOUT_SHARD_ONLY = 1,  /* each replica holds only the selected rank's
                                  flat shard (shard_numel); one rank only      */
  DOPT_LAYOUT_BUCKET = 2       /* ZeRO-2 streaming: each replica holds only the
                                  bucket group being reduced, as laid out in
                                  the grad buffer from the group's first bucket
                                  on; dopt_step_reduce_buckets only (see there) */
} dopt_layout;

#define DOPT_ALL_RANKS (-1)
#define DOPT_MAX_REPLICAS 64

/* Range: [start, end) -- distrib_optimizer page, "Range class". */
typedef struct {
  int64_t start, end;
} dopt_range;

/* One model parameter, in model (registration) order. */
typedef struct {
  int64_t numel;      /* >= 0                                                */
  int32_t dtype;      /* dopt_dtype of the param                             */
  int32_t new_bucket; /* nonzero: this param must start a bucket of its own
                         (the page's _does_param_require_new_bucket)         */
  double wd_mult;     /* weight-decay multiplier of this param (1.0 usual)   */
} dopt_param_desc;

typedef struct {
  int32_t param_dtype, grad_dtype, group, n_buckets;
  int32_t n_params, reserved;
  int64_t numel;          /* padded buffer size, a multiple of DP            */
  int64_t numel_unpadded; /* sum of the buckets' unpadded sizes              */
  int64_t shard_numel;    /* numel / DP: one rank's flat shard               */
} dopt_buffer_info;

typedef struct {
  int64_t offset;         /* bucket start in the buffer                      */
  int64_t numel;          /* padded size, a multiple of lcm(DP,128)          */
  int64_t numel_unpadded;
  int64_t shard_numel;    /* numel / DP                                      */
  int64_t shard_base;     /* start of this bucket's slice in a flat shard    */
} dopt_bucket_info;

/* The four views of one param piece owned by one rank (distrib_optimizer
 * page, "Range class: four views", _build_model_gbuf_param_range_map), plus
 * where the piece sits in the rank's flat shard. */
typedef struct {
  int32_t param, buffer, bucket, rank;
  dopt_range gbuf_world;           /* in the whole buffer                    */
  dopt_range gbuf_world_in_bucket; /* relative to the bucket's offset        */
  dopt_range gbuf_local;           /* relative to the rank's bucket slice    */
  dopt_range param_range;          /* inside the param's own flat tensor     */
  int64_t shard_offset;            /* = bucket shard_base + gbuf_local.start */
} dopt_param_shard;

/* AdamW hyper-parameters, given like torch's Python floats (double).  step
 * is the step number t used for bias correction when the step is applied
 * (the count of applied steps so far plus one). */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
  int64_t step;
} dopt_adamw_hparams;

typedef struct dopt_shard_map dopt_shard_map; /* opaque, library-owned */

/* ---------------------------------------------------------------------------
 * Shard map (host only; no GPU needed).
 */

/*
 * Builds the buffers, buckets and per-rank shards of a param list.
 * distrib_optimizer page: "Buffer layout", "Bucket partition: reverse walk +
 * size trigger", "Two levels of padding", "Final memory size assertions",
 * "Bucket-level equal split"; distributed-package page, section 2.2 (2)-(3)
 * (default bucket size, one buffer per (param dtype, grad dtype)).
 *
 *  params, n_params : model params in registration order (n_params >= 1).
 *  dp_size          : data-parallel ranks sharing one optimizer instance.
 *  bucket_size      : 0 = the default max(40000000, 1000000 * dp_size);
 *                     < 0 = no size trigger (one bucket per buffer unless a
 *                     param asks for a new one); > 0 = elements.
 *  grad_reduce_in_fp32 : nonzero: every grad buffer is fp32; else the grad
 *                     dtype is the param dtype.
 *  pad_for_high_busbw  : nonzero: bucket ends are padded to
 *                     lcm(DP, 128, 2^16) instead of lcm(DP, 128).
 *  out              : receives the map; free it with dopt_shard_map_free.
 * Errors: DOPT_E_INVALID (null, n_params < 1, dp_size < 1, negative numel,
 * unknown dtype), DOPT_E_NOMEM.
 */
int dopt_build_shard_map(const dopt_param_desc* params, int32_t n_params, int32_t dp_size,
                         int64_t bucket_size, int32_t grad_reduce_in_fp32,
                         int32_t pad_for_high_busbw, dopt_shard_map** out);
void dopt_shard_map_free(dopt_shard_map* map);

int32_t dopt_num_buffers(const dopt_shard_map* map); /* < 0 on null map */
int32_t dopt_dp_size(const dopt_shard_map* map);
int dopt_buffer_info_get(const dopt_shard_map* map, int32_t buffer, dopt_buffer_info* out);
int dopt_bucket_info_get(const dopt_shard_map* map, int32_t buffer, int32_t bucket,
                         dopt_bucket_info* out);
/* param_index_map[param] = (start, end, bucket) inside its buffer. */
int dopt_param_index(const dopt_shard_map* map, int32_t param, int32_t* buffer,
                     int64_t* start, int64_t* end, int32_t* bucket);
/*
 * The pieces of params that rank `rank` owns in `buffer`, in flat-shard
 * order.  Writes at most `cap` entries to `out` (out may be NULL when cap is
 * 0) and the total count to *count.
 */
int dopt_rank_shards(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                     dopt_param_shard* out, int32_t cap, int32_t* count);
/* The number of buckets over all buffers (< 0 on a null map), and the
 * number of bucket `bucket` of `buffer` in that count (buffers in order,
 * buckets in order within a buffer; < 0 when out of range).  These index
 * the grad check table of dopt_step_args.grad_amax. */
int32_t dopt_total_buckets(const dopt_shard_map* map);
int32_t dopt_bucket_number(const dopt_shard_map* map, int32_t buffer, int32_t bucket);

/* ---------------------------------------------------------------------------
 * Device entry points.  `rank` is a rank or DOPT_ALL_RANKS; the workspace
 * must be at least dopt_workspace_bytes(map, rank) bytes of device memory
 * and is scratch owned by the caller (no initialisation needed).  A
 * workspace may serve only one step at a time.
 */
size_t dopt_workspace_bytes(const dopt_shard_map* map, int32_t rank);

/*
 * Emulated reduce-scatter (step A2): for every element of the selected
 * shard(s) of `buffer`, main_grad = fp32(round_grad_dtype(reduced sum)).
 * distrib_optimizer page section 7.1 (start_grad_sync: reduce-scatter of
 * each bucket's grad_data, output = this rank's shard); distributed-package
 * page section 2.2 (4) (average_in_collective: prescale 1/dp_size and SUM,
 * or AVG); ledger page section 5 (n_instances > 1: reduce-scatter inside
 * each instance, all-reduce of the shards between instances).
 *
 *  replicas     : host array of n_replicas device pointers, replica k being
 *                 rank k's grad buffer in the buffer's grad dtype; replica k
 *                 belongs to instance k / DP.  n_replicas = DP * n_instances.
 *  layout       : dopt_layout; DOPT_LAYOUT_SHARD_ONLY needs rank >= 0.
 *  main_grad    : fp32 output, n_ranks * shard_numel (flat-shard layout).
 * The replicas are summed in replica order, starting from the first term,
 * each pre-scaled by 1/(DP*n_instances) (or summed and then averaged), and
 * the sum is rounded once to the grad dtype (again after the inter-instance
 * sum when n_instances > 1).
 */
int dopt_grad_reduce_shard(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                           const void* const* replicas, int32_t n_replicas,
                           int32_t n_instances, int32_t layout, int32_t average_in_collective,
                           float* main_grad, void* workspace, size_t workspace_bytes,
                           dopt_stream stream);

/*
 * prepare_grads (step A3): main_grad *= inv_loss_scale in place, and records
 * per-CTA partials (fp64 sum of squares, non-finite flag) of this buffer in
 * the workspace for dopt_grad_norm.  distrib_optimizer page, the
 * MixedPrecisionOptimizer step skeleton (copy to fp32 main grads, unscale,
 * inf/NaN check).  Call it for every buffer before dopt_grad_norm.
 */
int dopt_prepare_grads(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                       float inv_loss_scale, float* main_grad, void* workspace,
                       size_t workspace_bytes, dopt_stream stream);

/*
 * Global grad norm and clip coefficient (step A4): sums the partials of every
 * buffer in a fixed order (deterministic), adds remote_sumsq / ORs
 * remote_found_inf (the contribution of ranks not emulated here), and
 * writes device scalars:
 *   *d_norm      = sqrt(sumsq) as fp32, NaN when found_inf;
 *   *d_clip_coef = max_norm / (norm + 1e-6) when max_norm > 0 and that is
 *                  < 1, else 1 (computed in fp64, rounded once to fp32);
 *   *d_found_inf = 1 if any main grad or the remote flag is non-finite.
 * Any of the three pointers may be NULL.  distrib_optimizer page,
 * MegatronOptimizer utilities (clip_grad_norm, get_grad_norm) and
 * get_grad_stats_parallel_group (the norm spans the whole instance).
 */
int dopt_grad_norm(const dopt_shard_map* map, int32_t rank, void* workspace,
                   size_t workspace_bytes, double remote_sumsq, int32_t remote_found_inf,
                   double max_norm, float* d_norm, float* d_clip_coef, int32_t* d_found_inf,
                   dopt_stream stream);

/*
 * AdamW on the fp32 shard and the write-back into the param buffer (steps A5
 * and A6).  Per element, with g = main_grad * (*d_clip_coef):
 *   p = p * (1 - lr*wd*wd_mult);  m = b1*m + (1-b1)*g;
 *   v = b2*v + ((1-b2)*g)*g;      p = p - lr/(1-b1^t) * m/(sqrt(v)/sqrt(1-b2^t) + eps)
 * then param_buffer[gbuf_world] = RNE cast of p (bf16/fp16 buffers).  For an
 * fp32 buffer the master IS the param buffer (updated in place at the
 * gbuf_world offsets) and `master` must be NULL.  If *d_found_inf is nonzero
 * nothing is written (the step is skipped on the device).
 * distrib_optimizer page: "Why a distributed optimizer" (fp32 master, m, v),
 * the optimizer-type assertion (torch AdamW), step_with_ready_grads, and the
 * _copy_main_params_to_model_params listing (fp32 -> bf16 copy into
 * param_data at gbuf_world_in_bucket).
 *  master, exp_avg, exp_avg_sq : fp32, n_ranks * shard_numel, flat layout.
 *  param_buffer : the whole param buffer (numel) in the param dtype.
 */
int dopt_adam_step(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                   const float* main_grad, float* master, float* exp_avg, float* exp_avg_sq,
                   void* param_buffer, const dopt_adamw_hparams* hp, const float* d_clip_coef,
                   const int32_t* d_found_inf, dopt_stream stream);

/* Everything one fused step needs; per-buffer arrays are host arrays indexed
 * by buffer (length dopt_num_buffers). */
typedef struct {
  const dopt_shard_map* map;
  int32_t rank;                   /* a rank or DOPT_ALL_RANKS                  */
  int32_t n_instances;            /* >= 1; replicas = DP * n_instances         */
  int32_t layout;                 /* dopt_layout of the replica grads          */
  int32_t average_in_collective;
  const void* const* const* replica_grads; /* [buffer][replica] device ptrs    */
  float* const* main_grad;        /* [buffer] step temporary, 4 B x shard
                                     numel (x ranks for DOPT_ALL_RANKS); see
                                     below                                   */
  float* const* master;           /* [buffer]; NULL for fp32 buffers           */
  float* const* exp_avg;          /* [buffer]                                  */
  float* const* exp_avg_sq;       /* [buffer]                                  */
  void* const* param_buffer;      /* [buffer] whole param buffer               */
  float inv_loss_scale;           /* 1 / loss scale (1 for bf16)               */
  int32_t remote_found_inf;
  double max_norm;                /* <= 0 disables clipping                    */
  double remote_sumsq;
  dopt_adamw_hparams hp;          /* hp.step = t of this step if applied       */
  void* workspace;
  size_t workspace_bytes;
  dopt_stream stream;
  /* Optional tracing: NULL, or 4 cudaEvent_t handles (as plain pointers)
   * recorded on `stream` before the reduce/prepare pass, after it, after
   * the norm finalize and after the AdamW pass, so a caller can time each
   * stage of the step with cudaEventElapsedTime.  In the fused step the
   * finalize runs inside the last reduce launch, so the second and third
   * events are recorded back to back.  Any entry may be NULL (not
   * recorded).  A timing event between the passes makes the AdamW pass
   * wait for the reduce grid to drain before it launches (about 5 us per
   * step, which only short steps notice); events 0 and 3 alone time the
   * whole step without that cost. */
  void* const* stage_events;
  /* scale_gradients factor (per-token loss normalization, 1/num_tokens):
   * multiplies the reduced grads in the grad dtype (one rounding) before
   * prepare_grads; Megatron distributed-package page section 4.6.  0 or 1
   * means no scaling. */
  float grad_scale;
  int32_t reserved;
  /* Optional device-resident step state, for steps replayed from a CUDA
   * graph (whose launch parameters cannot change between replays):
   *   d_step -- device int64: the count of applied steps.  When set, hp.step
   *             is ignored; the finalize pass uses *d_step + 1 for the bias
   *             corrections and writes it back only if the step is applied
   *             (a skipped step does not count).
   *   d_lr   -- device double: the learning rate, read by the finalize pass
   *             (only with d_step); NULL uses hp.lr.
   * Both 8-byte aligned.  With d_step, dopt_step_async, the bucket-staged
   * entry points and dopt_step_noalloc issue only kernel launches and
   * memsets on the stream once each kernel has run once on the device (its
   * shared-memory attribute is set on first use), so a step can be
   * captured in a graph after a warm-up step. */
  int64_t* d_step;
  const double* d_lr;
  /* Optional check of every replica's gradients before their reduction
   * (check_for_nan_in_grad / check_for_large_grads: the check_grads method
   * of the bucket groups, distributed-package page sections 2.4 and 3.2,
   * which looks at each bucket's gradients for NaN, Inf and unusually large
   * values before the communication).  NULL: no check.  Else a device array
   * of n_replicas x dopt_total_buckets(map) floats, replica-major, 4-byte
   * aligned: the reduce pass of the step sets grad_amax[k * total + j] to
   * the largest |g| among the elements of replica k in bucket j (buckets
   * numbered across buffers in buffer order, dopt_bucket_number) that the
   * step reads -- the selected rank's shard of each bucket, or every rank's
   * with DOPT_ALL_RANKS -- taken as stored in the grad dtype, before any
   * prescale, unscale or scale_gradients.  The value is NaN when one of
   * those grads is NaN, +inf when one is infinite (and none is NaN), and 0
   * for a bucket the step reads nothing of.  The step clears the slots it
   * sets first (dopt_step_reduce_buckets clears only its buckets' slots).
   * The check changes nothing else: the caller compares the values with its
   * own threshold for "unusually large" (the pages give none), and a
   * non-finite grad already skips the step through found_inf.  Costs no
   * extra memory traffic (the replica grads are read once either way). */
  float* grad_amax;
  /* Optional global norm terms in device memory, for a multi-rank step
   * whose ranks combine their local statistics on the device (the
   * all-reduce of get_grad_stats_parallel_group, distrib_optimizer page,
   * MegatronOptimizer utilities): NULL, or an 8-byte aligned double holding
   * the sum of squares over every rank of the optimizer instance, and a
   * 4-byte aligned int32 that is nonzero when any rank found a non-finite
   * grad -- typically the sum and the max, over the ranks, of what
   * dopt_step_local_stats wrote.  When d_global_sumsq is set, the finalize
   * reads both when it runs (in stream order) and uses them in place of its
   * own partial sums plus remote_sumsq / remote_found_inf; this rank's own
   * non-finite grads still skip the step.  Both must be set together.  Only
   * dopt_step_finalize uses them: the fused steps and dopt_step_from_host,
   * whose finalize follows the reduce inside one call, refuse them
   * (DOPT_E_INVALID). */
  const double* d_global_sumsq;
  const int32_t* d_global_found_inf;
} dopt_step_args;

/* The main-grad buffers of dopt_step_args are scratch between the reduce
 * pass and the AdamW pass of a fused or bucket-staged step.  For a buffer
 * with fp32 grads they receive the fp32 main grads (the reduced grads times
 * inv_loss_scale).  For a buffer with bf16/fp16 grads the reduced grads are
 * values of the grad dtype, so the reduce pass stores them in that dtype, in
 * the first half of the buffer (element i at 16-bit index i), and the AdamW
 * pass forms the fp32 main grad fp32(g) * inv_loss_scale from them -- the
 * same value, from half the bytes (the distrib_optimizer page's fp32 main
 * grad copy, kept as its exact 16-bit source between the passes).  The
 * separate entry points (dopt_grad_reduce_shard, dopt_prepare_grads,
 * dopt_adam_step) always use fp32 main grads. */

/* Statistics of the last step, kept at the start of its workspace:
 * the fp64 sum of squares (with the remote term), the reported norm (NaN
 * when skipped), the clip coefficient applied (1 when not clipping),
 * found_inf, whether the grads were clipped, and the number of main grads
 * equal to zero (MegatronOptimizer's count_zeros). */
typedef struct {
  double sumsq;
  float grad_norm;
  float clip_coef;
  int32_t found_inf;
  int32_t clipped;
  int64_t num_zeros;
  int32_t kernel_error; /* nonzero: a kernel gave up waiting for its own data
                           copies; the step was skipped (found_inf set) */
  int32_t reserved;
} dopt_step_stats;

/* Copies the statistics of the last step run with `workspace` (fused or
 * bucket-staged layout) to the host; waits for `stream`.  dopt_step,
 * dopt_step_noalloc and dopt_step_from_host return DOPT_E_CUDA when
 * kernel_error is set. */
int dopt_read_step_stats(const void* workspace, dopt_step_stats* out, dopt_stream stream);

/*
 * One fused optimizer step (steps A2..A6): for every buffer, reduce the
 * replicas, unscale, check inf/NaN and accumulate the sum of squares in one
 * pass; then the global norm, clip coefficient and skip decision on the
 * device (by the last CTA to finish the last reduce launch, without a
 * launch of its own); then AdamW and the write-back, skipped on the device
 * when found_inf.  Waits until the finalize has run (the AdamW pass is
 * already queued and may still be running), then returns *found_inf_out
 * (0/1) and *grad_norm_out (NaN when skipped) -- like the pages' optimizer,
 * whose step reads the norm back and leaves the update running.  The
 * caller advances its step count only when *found_inf_out is 0.  The
 * results are copied on a side stream (the one dopt_step_from_host uses),
 * so the AdamW pass does not wait for the copy.  MixedPrecisionOptimizer.step
 * skeleton of the distrib_optimizer page: prepare_grads -> (return on inf)
 * -> clip_grad_norm -> step_with_ready_grads.
 */
int dopt_step(const dopt_step_args* args, int32_t* found_inf_out, float* grad_norm_out);

/*
 * The same step without waiting: the results stay on the device, in
 * d_found_inf / d_norm (either may be NULL).  The caller decides when to
 * read them.
 */
int dopt_step_async(const dopt_step_args* args, int32_t* d_found_inf, float* d_norm);

/*
 * Bucket-staged step: the same arithmetic as dopt_step, split so the
 * reduce/prepare pass can run bucket by bucket as each bucket's grads become
 * ready, and the AdamW/write-back pass bucket by bucket in the order the next
 * forward pass needs the params.  distrib_optimizer page section 7.1
 * (overlap_grad_reduce: a bucket's reduce-scatter starts as soon as all its
 * grads are ready) and 7.2 (overlap_param_gather: the param all-gather of a
 * bucket is waited on by the forward pre-hook, which then launches the next
 * bucket's).
 *
 * Sequence for one step, all with the same args (args->stream may change
 * between calls; the caller orders the streams with events):
 *   1. dopt_step_reduce_buckets for every bucket of every buffer, exactly
 *      once (any grouping, any order);
 *   2. dopt_step_finalize (norm, clip coefficient, skip decision);
 *   3. dopt_step_update_buckets for every bucket of every buffer (skipped on
 *      the device when found_inf).
 * The workspace must hold dopt_workspace_bytes_bucketed(map, rank) bytes (one
 * partial-sum region per bucket); args->stage_events is not used.  A bucket
 * left out of step 1 leaves stale partials behind, and the norm is wrong.
 * dopt_step_reduce_buckets reduces a group of buckets in as few launches as
 * the kernels' run tables allow (one, for groups of up to 960 runs); with
 * d_step set it issues only launches and memsets, like the fused step.
 *
 * ZeRO-2 streaming (DeepSpeed page, ZeRO stage 2: each rank keeps only its
 * partition of the reduced grads, and the full grads of a bucket are given
 * up once the bucket's reduce-scatter is done; ZeRO ledger page, section 2:
 * 2P + 14P/N per card).  With args->layout = DOPT_LAYOUT_BUCKET, replica k
 * of buffer `buffer` (args->replica_grads[buffer][k]) holds only the grads
 * of buckets [bucket_first, bucket_first + bucket_count): element i of the
 * group, i.e. element offset(bucket_first) + i of the grad buffer, at index
 * i.  The replicas then need only the group's size, not the buffer's, and
 * may be refilled with another group's grads as soon as this call's work on
 * args->stream has run (record an event after it); a ring of two such
 * staging buffers per replica streams every bucket of a step.  The rank's
 * own grads beyond the group are never held.  The selected rank's
 * (or every rank's) slice of each bucket is read, as with the whole buffer.
 * dopt_step_finalize, dopt_step_local_stats and dopt_step_update_buckets
 * accept this layout and read no replica; every other entry point refuses
 * it (DOPT_E_INVALID).  For 16-bit grads the main grads between the passes
 * take 2 bytes per shard element (see the main-grad note above), the
 * ledger's 2P/N grad term.
 */
size_t dopt_workspace_bytes_bucketed(const dopt_shard_map* map, int32_t rank);
int dopt_step_reduce_buckets(const dopt_step_args* args, int32_t buffer, int32_t bucket_first,
                             int32_t bucket_count);
int dopt_step_finalize(const dopt_step_args* args, int32_t* d_found_inf, float* d_norm);
/* Between steps 1 and 2 of the bucket-staged sequence, for multi-rank
 * steps: writes this rank's local statistics to device memory on
 * args->stream -- *d_local_sumsq (8-byte aligned) = the fixed-order fp64 sum
 * of squares of the rank's main grads, *d_local_found_inf (4-byte aligned)
 * = 1 when one of them is non-finite (or a reduce launch gave up waiting),
 * else 0 -- and finalizes nothing.  The caller combines them across ranks
 * on the device and passes the results as args->d_global_sumsq and
 * args->d_global_found_inf to dopt_step_finalize. */
int dopt_step_local_stats(const dopt_step_args* args, double* d_local_sumsq, int32_t* d_local_found_inf);
int dopt_step_update_buckets(const dopt_step_args* args, int32_t buffer, int32_t bucket_first,
                             int32_t bucket_count);

/*
 * One step whose replica gradients start in host memory (no counterpart in
 * the pages, which start from grads already on the GPU: this is the front
 * end for grads that arrive from the host, and the path the end-to-end
 * benchmark times).  For every bucket of every buffer, in order, the
 * library copies the part of each replica the step reads -- the selected
 * rank's slice of the bucket (every rank's with DOPT_ALL_RANKS) in the full
 * layout, the bucket's part of the flat shard in the shard-only layout --
 * from host_replica_grads into the device replica buffers of args on
 * copy_stream, and reduces the bucket on args->stream as soon as its copies
 * have landed (dopt_step_reduce_buckets), so the reduce pass runs under the
 * transfer; then it finalizes, updates every bucket, waits for args->stream
 * and returns *found_inf_out and *grad_norm_out like dopt_step.
 *   host_replica_grads -- [buffer][replica] host pointers, same layout and
 *                   dtype as args->replica_grads; page-locked (pinned)
 *                   memory for asynchronous copies (pageable memory works,
 *                   with copies that do not overlap).
 *   copy_stream   -- a stream other than args->stream (NULL: the library's
 *                   own non-blocking stream for the current device).  It
 *                   first waits for the work already on args->stream.
 * The workspace must be the bucket-staged one (dopt_workspace_bytes_bucketed).
 * The device replica buffers are overwritten; the call returns only after
 * the step has finished, so the next call may reuse every buffer.
 * Errors: as dopt_step; DOPT_E_INVALID for NULL host pointers.
 */
int dopt_step_from_host(const dopt_step_args* args, const void* const* const* host_replica_grads,
                        dopt_stream copy_stream, int32_t* found_inf_out, float* grad_norm_out);

/*
 * dopt_step_noalloc -- the fused step of dopt_step for callers that cannot
 * allocate device memory.  No page describes this entry point; it exists for
 * the library's users, not for the method.
 *
 * Some callers have no way to obtain a workspace buffer: a host program whose
 * device memory is owned by another allocator (a framework's caching
 * allocator, or a pool that reserved the GPU at start-up) and that exposes no
 * raw allocation; a latency-bound loop that forbids device allocation after
 * start-up because cudaMalloc may synchronize the device and stall other
 * streams; a plugin interface that hands an operation only its inputs and
 * outputs.  This entry point needs no workspace: its scratch (step scalars
 * and per-CTA partial sums) is a static device array of
 * DOPT_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library holds until the process exits.
 *
 *  - args: as for dopt_step, except that args->workspace and
 *    args->workspace_bytes are ignored.  The caller still passes every input
 *    and output (replica grads, main grad, master, m, v, param buffers).
 *  - The first call on a device looks up the device address of the scratch
 *    array (with that device current); make that first call before any
 *    stream capture.  Later calls on the device reuse the address.  The
 *    address is kept for the life of the process: after cudaDeviceReset
 *    the library's module is loaded afresh, and this entry point must not
 *    be called again in that process.
 *  - The first call on each host thread and device also creates the side
 *    stream and event that dopt_step reads its results back on (no device
 *    memory).  A caller that allows no resource creation after start-up
 *    makes one call per thread and device during start-up.
 *  - Returns DOPT_E_SIZE when the map and rank selection need more scratch
 *    than the array holds (dopt_workspace_bytes(map, rank) >
 *    DOPT_NOALLOC_SCRATCH_BYTES): no work is enqueued then.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 *  - Every call uses the same array, which keeps the last call's contents;
 *    nothing in it needs to start at zero (each step writes every slot it
 *    reads).  Calls that overlap on the GPU -- on two streams, or from two
 *    threads without ordering -- race on the array and give wrong results:
 *    order them.
 * Returns found_inf and the grad norm like dopt_step, and like dopt_step it
 * waits only until those two are known: the AdamW pass may still be running
 * on args->stream when it returns, and it still reads the step scalars in
 * the shared array.  Queue the next call of this entry point behind
 * args->stream -- on the same stream, or after an event recorded on it or a
 * synchronize -- never on another stream that is not ordered after it.
 */
#define DOPT_NOALLOC_SCRATCH_BYTES (1u << 20)
int dopt_step_noalloc(const dopt_step_args* args, int32_t* found_inf_out, float* grad_norm_out);

/* ---------------------------------------------------------------------------
 * Host arithmetic of the pages (no GPU).
 */

/*
 * Per-card memory ledger with Adam and 16-bit params/grads, in bytes: ZeRO
 * ledger page, section 2 table (DDP 16P, ZeRO-1 4P + 12P/N, ZeRO-2 2P +
 * 14P/N, ZeRO-3 16P/N).  stage: 0 = DDP, 1..3 = ZeRO stage.  A sharded part
 * holds ceil(P/N) elements per card.  parts_out (may be NULL) receives 5
 * values: param, grad, master, exp_avg, exp_avg_sq bytes.  Returns the total,
 * or a negative dopt_status.
 */
int64_t dopt_memory_ledger(int64_t P, int32_t N, int32_t stage, int64_t* parts_out);

/*
 * Bytes one rank sends in a ring collective over N ranks on a buffer of P
 * elements of elem_bytes each, P padded up to a multiple of N: reduce-scatter
 * and all-gather (N-1) * (P/N) * b, all-reduce twice that.  ZeRO ledger page,
 * section 4 (reduce-scatter + all-gather = 2P = one all-reduce);
 * distrib_optimizer page section 8.2.  kind: 0 = RS, 1 = AG, 2 = AR.
 */
int64_t dopt_comm_bytes(int64_t P, int32_t N, int32_t elem_bytes, int32_t kind);

/* Dynamic loss scaler for fp16 (host state).  The pages give only the
 * initial scale (2^16, the DeepSpeed config of the ipipp.com page); the
 * policy is: on found_inf, count a hysteresis strike and, once `hysteresis`
 * strikes are used up, multiply by backoff; after growth_interval clean
 * steps in a row, multiply by growth and restore the hysteresis budget. */
typedef struct {
  double scale, growth_factor, backoff_factor, min_scale;
  int32_t growth_interval, hysteresis;
  int32_t growth_tracker, hysteresis_tracker;
} dopt_loss_scaler;

int dopt_loss_scaler_init(dopt_loss_scaler* s, double initial_scale, double growth_factor,
                          double backoff_factor, int32_t growth_interval, int32_t hysteresis,
                          double min_scale);
int dopt_loss_scaler_update(dopt_loss_scaler* s, int32_t found_inf);

/* ---------------------------------------------------------------------------
 * Reshardable optimizer state.  The distrib_optimizer page lists "fully
 * reshardable" checkpoint formats, which do not depend on the internal
 * buffer layout (no layout is printed).  Reading: state in model space.  The
 * model space of a buffer holds its params in the order they were given to
 * dopt_build_shard_map, each as one contiguous range of numel elements;
 * it does not depend on the DP size, the bucket size or the padding.  A
 * state saved in model space at one DP size loads at any other.
 */
typedef enum {
  DOPT_STATE_FLAT_SHARD = 0,   /* fp32 master / exp_avg / exp_avg_sq of the
                                  step: the rank's flat shard (all ranks'
                                  slots, rank-major, for DOPT_ALL_RANKS) */
  DOPT_STATE_PARAM_BUFFER = 1  /* the whole param buffer, in the param dtype
                                  (for an fp32 buffer: its master) */
} dopt_state_layout;

/* Elements of `buffer`'s model space: the sum of its params' numel (< 0 on
 * a bad map or buffer). */
int64_t dopt_model_numel(const dopt_shard_map* map, int32_t buffer);

/*
 * Copies the elements that `rank` owns (every rank's with DOPT_ALL_RANKS)
 * of one state tensor of `buffer` between its step layout and model space:
 * to_model writes model[model index] = state[layout index], from_model the
 * reverse; other elements of the destination are not touched (padding, and
 * params or pieces of other ranks).  Elements are fp32 for
 * DOPT_STATE_FLAT_SHARD and the param dtype for DOPT_STATE_PARAM_BUFFER.
 * Either pointer may be device or host memory (one cudaMemcpyAsync per
 * param piece, cudaMemcpyDefault, on `stream`; pageable host memory makes
 * the copies synchronous).  A checkpoint gathers all ranks' pieces; a
 * restore scatters each rank's own.  Errors: DOPT_E_INVALID (bad map,
 * buffer, rank or layout, NULL pointer), DOPT_E_CUDA.
 */
int dopt_state_to_model(const dopt_shard_map* map, int32_t buffer, int32_t rank, int32_t layout,
                        const void* state, void* model, dopt_stream stream);
int dopt_state_from_model(const dopt_shard_map* map, int32_t buffer, int32_t rank, int32_t layout,
                          const void* model, void* state, dopt_stream stream);

#if defined(DOPT_BOUNDS_CHECK) && DOPT_BOUNDS_CHECK
/* Debug builds only (DOPT_BOUNDS_CHECK=1): the release library neither
 * exports this hook nor tests for it in its kernels.  Test hook for the
 * bounded waits of the TMA-staged reduce pass: while set to tile >= 0, CTA 0
 * of every such launch announces its tile of that (CTA-local) index but
 * never copies it, so its wait runs out after about a second; the step then
 * reports kernel_error, returns DOPT_E_CUDA from dopt_step and is skipped,
 * and the CUDA context stays usable.  -1 turns the hook off (the default). */
int dopt_debug_starve_copy(int32_t tile);
#endif

/* Debug builds only (compiled with DOPT_BOUNDS_CHECK=1; the default build
 * returns DOPT_E_INVALID).  Every kernel of such a build checks each tile's
 * element ranges against the extents of the buffers it reads and writes
 * (each replica, the main grad, master/m/v, the param buffer, the grad-check
 * slots) and skips a tile that falls outside them instead of touching it.
 * This call copies the record of such tiles on the current device to out[4]
 * -- the number of failed checks, the first failure's check site, first
 * element and extent -- clears it, and waits for the device.  A count of 0
 * means every access stayed inside its buffer. */
int dopt_debug_bounds_record(int64_t* out);

/* Number of kernels this library has launched in this process (all
 * devices, all threads); a caller can difference it around a region. */
uint64_t dopt_kernel_launches(void);

const char* dopt_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* DOPT_H */
