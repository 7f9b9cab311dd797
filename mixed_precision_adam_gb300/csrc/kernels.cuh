// kernels.cuh -- what the device kernels of the sharded mixed-precision Adam
// step share: launch constants, the run table passed to every kernel, the
// kernel-parameter blocks, the workspace layout, and the host-side launch
// helpers.  Included by every CUDA translation unit of the library:
//   k1_f32.cu, k1_bf16.cu, k1_f16.cu -- K1 reduce/prepare, one grad dtype each
//   k3.cu                             -- K3 AdamW + cast back
//   dopt_cuda.cu                      -- K2 finalize and the C entry points
//
// The step is three HBM-bound passes over the selected shard(s):
//   K1 reduce_prepare : reads the N replica grads of every element, sums
//                       them (emulated reduce-scatter), rounds to the grad
//                       dtype, unscales, writes the fp32 main grad and keeps
//                       per-CTA partials of the sum of squares and of the
//                       non-finite flag.
//   K2 finalize       : one CTA sums the partials in a fixed order and decides
//                       norm, clip coefficient and skip on the device.
//   K3 adamw          : reads main grad, master, m, v once, writes master, m,
//                       v and the 16-bit param at its buffer offset once.
// No tensor cores: nothing here is a contraction.  The work is described to
// the kernels by a table of runs (contiguous in both the flat shard and the
// buffer) passed by value as a __grid_constant__ kernel parameter, so a step
// needs no host-to-device copy and no library-owned device memory.  Each run
// is cut into tiles; CTAs take tiles round-robin.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <string>

#include "dopt_internal.h"

#ifndef DOPT_K1_UNROLL
#define DOPT_K1_UNROLL 2
#endif
#ifndef DOPT_K3_UNROLL
#define DOPT_K3_UNROLL 1
#endif
#ifndef DOPT_K1_TMA
#define DOPT_K1_TMA 1  // 1: single-instance reduce stages replica tiles through shared memory with TMA
#endif
#ifndef DOPT_TMA_STAGES
#define DOPT_TMA_STAGES 2
#endif
#ifndef DOPT_TMA_TILE
#define DOPT_TMA_TILE 2048
#endif
#ifndef DOPT_TMA_EVICT_FIRST
#define DOPT_TMA_EVICT_FIRST 1  // 1: the replica tiles are marked first to leave L2
#endif
#ifndef DOPT_K1_MIN_BLOCKS
#define DOPT_K1_MIN_BLOCKS 2
#endif
#ifndef DOPT_K1_SHORT_PIPE
#define DOPT_K1_SHORT_PIPE 1  // 1: short fp32 single-instance reduces take the pipelined register kernel
#endif
#ifndef DOPT_K1N_FP32_MIN_BLOCKS
#define DOPT_K1N_FP32_MIN_BLOCKS 4  // register-staged K1, up to 4 fp32 replicas of one instance
#endif
#ifndef DOPT_KEEP_MAIN_L2_DIV
#define DOPT_KEEP_MAIN_L2_DIV 4  // fp32 main grads of a step at most L2 / this are kept in L2 (0: never)
#endif
#ifndef DOPT_K3_MIN_BLOCKS
#define DOPT_K3_MIN_BLOCKS 4
#endif
#ifndef DOPT_K3_PDL
#define DOPT_K3_PDL 1  // 1: the AdamW pass is launched as a programmatic dependent of the reduce pass
#endif
#ifndef DOPT_K3_STORE_HINT
#define DOPT_K3_STORE_HINT 0  // the AdamW pass's stores: 0 streaming, 1 L2 only, 2 write-back
#endif
#ifndef DOPT_BOUNDS_CHECK
#define DOPT_BOUNDS_CHECK 0  // 1: debug build; every tile is checked against the extents of its buffers
#endif

namespace dopt {

constexpr int kThreads = 256;              // threads per CTA
constexpr int kVec = 4;                    // contiguous elements per thread access
constexpr int kUnroll1 = DOPT_K1_UNROLL;   // K1 accesses per thread per tile
constexpr int kUnroll3 = DOPT_K3_UNROLL;   // K3 accesses per thread per tile
constexpr int kTile1 = kThreads * kVec * kUnroll1;  // K1 elements per tile
constexpr int kTile3 = kThreads * kVec * kUnroll3;  // K3 elements per tile
constexpr int kTmaTile = DOPT_TMA_TILE;    // elements per tile of the TMA-staged K1
constexpr int kTmaMinTilesPerSm = 16;      // shorter launches take the register-staged K1
constexpr int kShortTile = kThreads * kVec;  // elements per tile of K1 for short fp32 launches
static_assert(kTmaTile % (kThreads * kVec) == 0, "TMA tile");
constexpr int kMaxSeg = 960;               // runs per launch (kernel-parameter table)
constexpr int kMaxGrid = 1024;             // partial slots per launch region (CTAs per launch at most)
constexpr int kBatch = 8;                  // replicas loaded together
constexpr size_t kScalarBytes = 256;

// A run whose flat-shard and buffer starts are both multiples of 8 elements
// takes the vector paths.
__host__ __device__ __forceinline__ bool seg_aligned(int64_t local, int64_t world) {
  return ((local | world) & 7) == 0;
}

struct Seg {
  int64_t local;   // first element in the flat shard arrays (rank slot included)
  int64_t world;   // first element in the buffer
  int32_t len;     // elements
  int32_t tile0;   // first tile of this run in the launch
  union {
    double wd_mult;  // K3 tables: weight-decay multiplier of the run's param
    int32_t bucket;  // K1 tables: the run's bucket, numbered across all buffers
  };
};
static_assert(sizeof(Seg) == 32, "Seg layout");

// A launch's run table, held in the kernel's parameter block.  The GPU
// copies the whole block at every launch, so a launch whose runs fit in
// kSmallSeg entries takes a kernel compiled for that table (about 2 KB of
// parameters instead of about 31 KB): about a microsecond less per launch,
// which short steps notice.
template <int CAP>
struct SegTableT {
  int32_t n_seg;
  int32_t n_tiles;
  Seg seg[CAP];
};
using SegTable = SegTableT<kMaxSeg>;
constexpr int kSmallSeg = 32;

struct Partial {
  double sumsq;
  int32_t nonfinite;
  int32_t zeros;  // main grads equal to zero
};
static_assert(sizeof(Partial) == 16, "Partial layout");

// Device scalars of one step, at the start of the workspace: the public
// dopt_step_stats layout.
using Scalars = dopt_step_stats;
static_assert(sizeof(Scalars) == 40, "dopt_step_stats layout");
// Byte offset, inside the workspace's scalar area, of the word a reduce
// kernel sets when it gives up waiting for its own copies; the finalize
// pass reports it as dopt_step_stats.kernel_error and clears it.
constexpr size_t kErrorFlagOffset = 128;
// Byte offset of the step scalars the finalize pass computes when the step
// number (and learning rate) live in device memory.
constexpr size_t kDevStepOffset = 64;
struct DevStep {
  float step_size;  // (float)(lr / (1 - beta1^t))
  float bc2_sqrt;   // (float)sqrt(1 - beta2^t)
  double lr_wd;     // lr * weight_decay
};
constexpr int32_t kErrorMagic = 0x4B31544D;  // the flag's "set" value
// Byte offset of the ticket counter of the in-kernel finalize: the CTAs of a
// step's last reduce launch take tickets, and the last one finalizes.
constexpr size_t kFinCounterOffset = 160;

// The step number and learning rate of a step whose counter lives in device
// memory: the finalize reads them, computes the step scalars for the next
// step number and advances the counter only when the step is applied.
struct K2Step {
  int64_t* d_step;      // NULL: the host supplied the step scalars
  const double* d_lr;   // NULL: lr below
  double lr, wd, beta1, beta2;
  DevStep* out;
};

// Everything the finalize (norm, clip coefficient, skip decision, step
// statistics) reads and writes.
struct FinalizeArgs {
  const Partial* parts;  // every partial slot of the step, regions in order
  int32_t n_slots;
  int32_t remote_found;
  double remote_sumsq, max_norm;
  Scalars* sc;
  float* d_norm;
  float* d_coef;
  int32_t* d_found;
  int32_t* err_flag;
  K2Step step;
  // global terms in device memory (a multi-rank step): when set, they
  // replace the partial sum plus remote_sumsq / remote_found
  const double* d_global_sumsq;
  const int32_t* d_global_found;
  // local-only pass: when set, the block writes this rank's sum of squares
  // and non-finite flag here and finalizes nothing
  double* local_sumsq;
  int32_t* local_found;
};

// Debug builds (DOPT_BOUNDS_CHECK=1): the extents, in elements, of the
// buffers a launch touches, and a device record of the first tile whose
// range falls outside one of them: [count, site, first element, extent].
// Such a tile is skipped, not accessed.
struct Extents {
  int64_t rep;      // each replica (K1)
  int64_t main;     // the main-grad array (K1 writes, K3 reads)
  int64_t state;    // master, exp_avg, exp_avg_sq (K3)
  int64_t param;    // the param buffer (K3)
  int64_t buckets;  // grad-check slots per replica (K1 with the check)
  unsigned long long* record;
};

// Where a range is checked, as recorded.
enum BoundsSite : int {
  kSiteK1Rep = 1, kSiteK1Main = 2, kSiteK1Bucket = 3, kSiteTmaCopy = 4,
  kSiteK3Main = 5, kSiteK3State = 6, kSiteK3Master = 7, kSiteK3Param = 8
};

#if DOPT_BOUNDS_CHECK
__device__ __forceinline__ bool range_ok(const Extents& x, int site, int64_t lo, int64_t n, int64_t extent) {
  if (lo >= 0 && n >= 0 && lo + n <= extent) return true;
  if (atomicAdd(x.record, 1ull) == 0ull) {
    x.record[1] = (unsigned long long)site;
    x.record[2] = (unsigned long long)lo;
    x.record[3] = (unsigned long long)extent;
  }
  return false;
}
#define DOPT_RANGE_OK(params, site, lo, n, field) ::dopt::range_ok((params).ext, (site), (lo), (n), (params).ext.field)
#else
#define DOPT_RANGE_OK(params, site, lo, n, field) true
#endif

// A reduce launch's parameters: K1Head, then its run table.
struct K1Head {
  const void* rep[DOPT_MAX_REPLICAS];
  float* main_grad;
  Partial* partials;  // this launch's region of kMaxGrid slots (STATS only)
  int32_t n_rep, n_inst;
  float pre;        // (float)(1 / n_rep): prescale of average_in_collective = 0
  float inv_dpi;    // (float)(1 / (n_rep / n_inst))
  float inv_ninst;  // (float)(1 / n_inst)
  float inv_scale;  // 1 / loss scale
  int32_t average;
  float post_scale; // scale_gradients factor on the reduced grad (1 = none)
  int32_t* error_flag;  // set by a kernel that gave up waiting (TMA path)
#if DOPT_BOUNDS_CHECK
  int32_t starve_tile;  // test hook: CTA 0 never copies its tile of this index (-1: off)
#endif
  int32_t compact;      // 16-bit grads, statistics pass: store the reduced grads in the
                        // grad dtype instead of the fp32 main grads (see finish_store4)
  int32_t keep_main;    // fp32 main grads stored without the evict-first hint, to be
                        // read back from L2 (steps whose main grads fit L2 easily)
  // grad check (CHECK kernels only): amax[k * amax_stride + bucket] gathers
  // the fp32 bits of replica k's largest |g| in that bucket (atomic max)
  uint32_t* amax;
  int64_t amax_stride;
  // in-kernel finalize (the last reduce launch of a fused step): the last
  // CTA to take a ticket from *fin_counter runs it; NULL: none
  uint32_t* fin_counter;
  FinalizeArgs fin;
#if DOPT_BOUNDS_CHECK
  Extents ext;
#endif
};
template <int CAP>
struct K1ParamsT : K1Head {
  SegTableT<CAP> tab;
};
using K1Params = K1ParamsT<kMaxSeg>;

// An AdamW launch's parameters: K3Head, then its run table.
struct K3Head {
  const float* main_grad;
  float* master;      // flat shard, or NULL when the param buffer is the master
  float* exp_avg;
  float* exp_avg_sq;
  void* param;        // the whole param buffer
  const float* coef;  // device scalar
  const int32_t* found_inf;
  const DevStep* dev;  // step scalars from the finalize pass, or NULL: use the fields below
  double lr_wd;        // lr * weight_decay (host step)
  float b1, b2, omb1, omb2, eps, step_size, bc2_sqrt;
  float inv_scale;     // compact main grads: main = widen(stored) * inv_scale
  // 1: the launch before this one in the stream is a kernel of the same
  // step that writes none of master, m and v here (the step's reduce pass,
  // its finalize, or the AdamW pass of another buffer or bucket), so a CTA
  // may load its first tile's master, m and v before waiting for it
  int32_t early_state;
#if DOPT_BOUNDS_CHECK
  Extents ext;
#endif
};
template <int CAP>
struct K3ParamsT : K3Head {
  SegTableT<CAP> tab;
};
using K3Params = K3ParamsT<kMaxSeg>;

static_assert(sizeof(K1Params) <= 32764 && sizeof(K3Params) <= 32764, "kernel parameter limit");
static_assert(sizeof(K1ParamsT<kSmallSeg>) <= 4096 && sizeof(K3ParamsT<kSmallSeg>) <= 4096, "compact parameters");

// The same launch parameters with a run table of CAP entries; the table's
// runs must fit (n_seg <= CAP).
template <int CAP, typename Head, template <int> class ParamsT>
ParamsT<CAP> with_table_of(const ParamsT<kMaxSeg>& big) {
  ParamsT<CAP> out{};
  static_cast<Head&>(out) = static_cast<const Head&>(big);
  out.tab.n_seg = big.tab.n_seg;
  out.tab.n_tiles = big.tab.n_tiles;
  for (int i = 0; i < big.tab.n_seg; ++i) out.tab.seg[i] = big.tab.seg[i];
  return out;
}

// Programmatic dependent launch.  A reduce kernel lets the kernel after it
// in the stream start its CTAs once every reduce CTA has finished its tiles
// (the AdamW pass is launched with programmatic stream serialization), and
// that kernel waits for the whole reduce grid -- the finalize included --
// to complete and its writes to be visible before it reads anything.  For a
// kernel launched without the attribute, or after one that never signals,
// the wait returns at once.
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void wait_for_prior_grids() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Advances the run cursor of a CTA to the run holding tile t (tiles visited
// in increasing order, so the cursor only moves forward).
template <typename Tab>
__device__ __forceinline__ int seek(const Tab& tab, int si, int t) {
  while (si + 1 < tab.n_seg && tab.seg[si + 1].tile0 <= t) ++si;
  return si;
}

// beta^t by binary powering in fp64 (host and device compute it the same way).
__host__ __device__ __forceinline__ double pow_int(double b, int64_t t) {
  double r = 1.0, x = b;
  while (t > 0) {
    if (t & 1) r *= x;
    x *= x;
    t >>= 1;
  }
  return r;
}

// The finalize, run by one CTA of NT threads: sums the partial slots in a
// fixed order (each thread its slots at stride NT in four independent
// chains, then chains and threads in a fixed tree), adds the remote terms,
// and decides norm, clip coefficient and skip; writes the step statistics,
// the optional device results and the device step scalars.  Partials are
// read past L1 (they may have been written by other SMs moments before).
template <int NT>
__device__ __forceinline__ void finalize_block(const FinalizeArgs& f) {
  static_assert(NT % 32 == 0 && NT <= 1024, "whole warps");
  constexpr int NW = NT / 32;
  __shared__ double s_sum[NW];
  __shared__ int s_bad[NW];
  __shared__ long long s_zero[NW];
  double v[4] = {0.0, 0.0, 0.0, 0.0};
  int b = 0;
  long long z = 0;
  int i = threadIdx.x;
  // one 16-byte load per slot (the fp64 sum, then the flag and zero count
  // as the low and high words of the second half), eight slots in flight
  const double2* slot = reinterpret_cast<const double2*>(f.parts);
  auto take = [&](int j, int q) {
    const double2 d = __ldcg(slot + j);
    const long long fz = __double_as_longlong(d.y);
    v[q] += d.x;
    b |= (int)(fz & 0xFFFFFFFFll);
    z += (int)(fz >> 32);
  };
  // the error flag, read with the slots rather than after the sum
  const int err_early = (threadIdx.x == 0 && !f.local_sumsq) ? __ldcg(f.err_flag) : 0;
  // every slot's load issued before any is summed (up to eight per thread
  // per round; a short tail predicated rather than looped)
  for (; i < f.n_slots; i += 8 * NT) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = i + q * NT;
      if (j < f.n_slots) take(j, q & 3);
    }
  }
  // a fixed tree: lanes by xor shuffles within each warp, then the warps'
  // totals in warp order by thread 0 (one barrier instead of one per level)
  double sum = (v[0] + v[1]) + (v[2] + v[3]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    b |= __shfl_xor_sync(0xFFFFFFFFu, b, o);
    z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  }
  if (threadIdx.x % 32 == 0) {
    s_sum[threadIdx.x / 32] = sum;
    s_bad[threadIdx.x / 32] = b;
    s_zero[threadIdx.x / 32] = z;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < NW; ++w) {
      s_sum[0] += s_sum[w];
      s_bad[0] |= s_bad[w];
      s_zero[0] += s_zero[w];
    }
  }
  if (f.local_sumsq) {  // local statistics only; the finalize comes later
    if (threadIdx.x == 0) {
      *f.local_sumsq = s_sum[0];
      *f.local_found = (s_bad[0] || __ldcg(f.err_flag) == kErrorMagic) ? 1 : 0;
    }
    return;
  }
  if (threadIdx.x == 0) {
    const int kernel_error = err_early == kErrorMagic ? 1 : 0;
    *f.err_flag = 0;
    const double sumsq = f.d_global_sumsq ? __ldcg(f.d_global_sumsq) : s_sum[0] + f.remote_sumsq;
    const int remote_bad = f.d_global_sumsq ? (__ldcg(f.d_global_found) != 0) : (f.remote_found != 0);
    const int found = (s_bad[0] || remote_bad || kernel_error) ? 1 : 0;
    const double norm = sqrt(sumsq);
    double coef = 1.0;
    int clip = 0;
    if (f.max_norm > 0.0) {
      coef = f.max_norm / (norm + 1.0e-6);
      clip = coef < 1.0;
    }
    const float coef_f = clip ? (float)coef : 1.0f;
    const float norm_f = found ? __int_as_float(0x7FC00000) : (float)norm;
    Scalars* sc = f.sc;
    sc->sumsq = sumsq;
    sc->grad_norm = norm_f;
    sc->clip_coef = coef_f;
    sc->found_inf = found;
    sc->clipped = clip;
    sc->num_zeros = s_zero[0];
    sc->kernel_error = kernel_error;
    sc->reserved = 0;
    if (f.d_norm) *f.d_norm = norm_f;
    if (f.d_coef) *f.d_coef = coef_f;
    if (f.d_found) *f.d_found = found;
    const K2Step& st = f.step;
    if (st.d_step) {
      const int64_t t = *st.d_step + 1;
      const double lr = st.d_lr ? *st.d_lr : st.lr;
      st.out->step_size = (float)(lr / (1.0 - pow_int(st.beta1, t)));
      st.out->bc2_sqrt = (float)sqrt(1.0 - pow_int(st.beta2, t));
      st.out->lr_wd = lr * st.wd;
      if (!found) *st.d_step = t;  // a skipped step does not count
    }
  }
}

// The finalize of a reduce launch's last CTA, out of line: inlined, its
// fp64 scalar work would set the register count of every reduce kernel
// (88 where the streaming loop needs 48 to 62), costing occupancy on a path
// that runs once per step in one CTA.
static __device__ __noinline__ void finalize_call(const FinalizeArgs& f) { finalize_block<kThreads>(f); }

// Called by every thread of every CTA of a reduce launch after its partial
// is written (by thread 0): with a ticket counter set, the last CTA to take
// a ticket runs the finalize and returns the counter to zero for the next
// step.  No CTA waits for another.
__device__ __forceinline__ void finalize_if_last(const K1Head& p) {
  if (!p.fin_counter) return;
  __shared__ int s_last;
  if (threadIdx.x == 0) {
    __threadfence();  // this CTA's partial (and error flag) before its ticket
    s_last = atomicAdd(p.fin_counter, 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  finalize_call(p.fin);
  if (threadIdx.x == 0) *p.fin_counter = 0u;
}

// ------------------------------------------------------- host-side launch --

// SM count (and, when l2_bytes is given, the L2 size in bytes) of the
// current device, cached per thread and device.
int device_sms(int* sms, int* l2_bytes = nullptr);
// Counts a launch and turns a launch error into a status.
int check_launch(const char* what);

// Grid of a tile-striding kernel: as many CTAs as fit on the GPU at once
// (occupancy x SMs), at most one per tile and at most kMaxGrid.
template <typename K>
int grid_for(K kernel, int n_tiles, int* grid, size_t smem = 0) {
  int sms = 0;
  int st = device_sms(&sms);
  if (st) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, smem);
  if (e != cudaSuccess)
    return fail(DOPT_E_CUDA, std::string("occupancy query: ") + cudaGetErrorString(e));
  if (per_sm < 1) return fail(DOPT_E_CUDA, "occupancy query: the kernel does not fit on an SM");
  *grid = std::max(1, std::min({per_sm * sms, kMaxGrid, std::max(1, n_tiles)}));
  return DOPT_OK;
}

// Fills a launch's run table with runs[0, count) cut into tiles of
// tile_elems; bucket_base >= 0 makes it a K1 table (each run records its
// bucket as bucket_base + Run::bucket), otherwise a K3 table (each run
// records its weight-decay multiplier).
void fill_table(SegTable& tab, const Run* runs, int count, int tile_elems, int32_t bucket_base);

// One K1 launch: a chunk of at most kMaxSeg runs and how to treat them.
struct K1Launch {
  const Run* runs;
  int count;
  int32_t bucket_base;  // number of the first bucket of the runs' buffer
  bool full;            // replicas are whole grad buffers (else the flat shard)
  bool stats;           // write the norm partials
  bool check;           // gather the per-replica max |g| (needs stats)
};

// K1 over one launch, for one grad dtype (one translation unit each): picks
// the kernel, fills kp.tab for that kernel's tile and launches it.  The
// other fields of kp are filled by the caller.
int launch_k1_f32(K1Params& kp, const K1Launch& l, cudaStream_t s);
int launch_k1_bf16(K1Params& kp, const K1Launch& l, cudaStream_t s);
int launch_k1_f16(K1Params& kp, const K1Launch& l, cudaStream_t s);
// K3 over a chunk of runs for a param dtype; fills kp.tab.  main_dtype is
// DOPT_F32 for fp32 main grads, or the grad dtype (bf16/fp16) when K1 left
// the reduced grads in their compact form.
int launch_k3(int32_t param_dtype, int32_t main_dtype, K3Params& kp, const Run* runs, int count,
              cudaStream_t s);

}  // namespace dopt
