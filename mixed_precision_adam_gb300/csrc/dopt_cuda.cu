// dopt_cuda.cu -- device kernels and device entry points of the sharded
// mixed-precision Adam step, for sm_103a.
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
// is cut into tiles (kTile1 / kTile3 elements); CTAs take tiles round-robin.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "dopt_internal.h"

// Scratch of dopt_step_noalloc: the step scalars and partial-sum regions
// that dopt_step keeps in the caller's workspace.  Host code must not use
// this name as an address (it is a host-side stand-in): the device address
// comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DOPT_NOALLOC_SCRATCH_BYTES];

namespace {

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
#ifndef DOPT_K1_MIN_BLOCKS
#define DOPT_K1_MIN_BLOCKS 2
#endif
#ifndef DOPT_K3_MIN_BLOCKS
#define DOPT_K3_MIN_BLOCKS 4
#endif

constexpr int kThreads = 256;              // threads per CTA
constexpr int kVec = 4;                    // contiguous elements per thread access
constexpr int kUnroll1 = DOPT_K1_UNROLL;   // K1 accesses per thread per tile
constexpr int kUnroll3 = DOPT_K3_UNROLL;   // K3 accesses per thread per tile
constexpr int kTile1 = kThreads * kVec * kUnroll1;  // K1 elements per tile
constexpr int kTile3 = kThreads * kVec * kUnroll3;  // K3 elements per tile
constexpr int kMaxSeg = 960;               // runs per launch (kernel-parameter table)
constexpr int kMaxGrid = 2048;             // partial slots per launch region
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
  double wd_mult;  // weight-decay multiplier of the run's param (K3)
};
static_assert(sizeof(Seg) == 32, "Seg layout");

struct SegTable {
  int32_t n_seg;
  int32_t n_tiles;
  Seg seg[kMaxSeg];
};

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

struct K1Params {
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
  int32_t use_tma;      // host's choice: launch the TMA-staged kernel
  int32_t starve_tile;  // test hook: CTA 0 never copies its tile of this index (-1: off)
  SegTable tab;
};

struct K3Params {
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
  int32_t pad;
  SegTable tab;
};

static_assert(sizeof(K1Params) <= 32764 && sizeof(K3Params) <= 32764, "kernel parameter limit");

// ---------------------------------------------------------------- helpers --

// Loads of kVec grad elements are held in their raw encoding (float4 for
// fp32, two packed 16-bit pairs for bf16/fp16) until the reduction widens
// them, so a 16-bit grad keeps half the registers of an fp32 one and a
// thread can keep twice as many 16-bit accesses in flight.
template <typename T>
struct GradT;
template <>
struct GradT<float> {
  using Raw = float4;
  static constexpr int kUnroll = 1;  // multiplier of kUnroll1 for this type
  static __device__ __forceinline__ Raw load4(const void* p, int64_t i) {
    return __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
  }
  static __device__ __forceinline__ float at(const Raw& r, int j) {
    return j == 0 ? r.x : j == 1 ? r.y : j == 2 ? r.z : r.w;
  }
  static __device__ __forceinline__ float widen1(const void* p, int64_t i) {
    return __ldcs(static_cast<const float*>(p) + i);
  }
  static __device__ __forceinline__ void widen4(const void* p, int64_t i, float* x) {
    float4 v = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(p) + i));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  static __device__ __forceinline__ float round_to(float s) { return s; }
};
template <>
struct GradT<__nv_bfloat16> {
  using Raw = uint2;
  static constexpr int kUnroll = 2;
  static __device__ __forceinline__ Raw load4(const void* p, int64_t i) {
    return __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ float at(const Raw& r, int j) {
    const unsigned w = j < 2 ? r.x : r.y;
    return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  static __device__ __forceinline__ float widen1(const void* p, int64_t i) {
    unsigned short b = __ldcs(static_cast<const unsigned short*>(p) + i);
    return __uint_as_float((unsigned)b << 16);
  }
  static __device__ __forceinline__ void widen4(const void* p, int64_t i, float* x) {
    uint2 v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(p) + i));
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xFFFF0000u);
  }
  static __device__ __forceinline__ float round_to(float s) {
    return __bfloat162float(__float2bfloat16_rn(s));
  }
};
template <>
struct GradT<__half> {
  using Raw = uint2;
  static constexpr int kUnroll = 2;
  static __device__ __forceinline__ Raw load4(const void* p, int64_t i) {
    return __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ float at(const Raw& r, int j) {
    const unsigned w = j < 2 ? r.x : r.y;
    return __half2float(__ushort_as_half((unsigned short)((j & 1) ? (w >> 16) : (w & 0xFFFFu))));
  }
  static __device__ __forceinline__ float widen1(const void* p, int64_t i) {
    unsigned short b = __ldcs(static_cast<const unsigned short*>(p) + i);
    return __half2float(__ushort_as_half(b));
  }
  static __device__ __forceinline__ void widen4(const void* p, int64_t i, float* x) {
    uint2 v = __ldcs(reinterpret_cast<const uint2*>(static_cast<const unsigned short*>(p) + i));
    x[0] = __half2float(__ushort_as_half((unsigned short)(v.x & 0xFFFFu)));
    x[1] = __half2float(__ushort_as_half((unsigned short)(v.x >> 16)));
    x[2] = __half2float(__ushort_as_half((unsigned short)(v.y & 0xFFFFu)));
    x[3] = __half2float(__ushort_as_half((unsigned short)(v.y >> 16)));
  }
  static __device__ __forceinline__ float round_to(float s) {
    return __half2float(__float2half_rn(s));
  }
};

// Advances the run cursor of a CTA to the run holding tile t (tiles visited
// in increasing order, so the cursor only moves forward).
__device__ __forceinline__ int seek(const SegTable& tab, int si, int t) {
  while (si + 1 < tab.n_seg && tab.seg[si + 1].tile0 <= t) ++si;
  return si;
}

// Reduction of one element over the replicas, in replica order, starting
// from the first term; rounded to the grad dtype after each instance's sum
// and again after the inter-instance sum.
struct ReduceState {
  float s, total;
};

// Where replica k sits in the reduction: its index inside its instance,
// whether it opens / closes the instance's sum and whether its instance is
// the first one.  The same for every element, so computed once per replica.
struct ReplicaPos {
  bool opens, closes, first_inst;
};

__device__ __forceinline__ ReplicaPos replica_pos(int k, int dpi) {
  const int q = k % dpi;
  return ReplicaPos{q == 0, q == dpi - 1, k < dpi};
}

template <typename GT>
__device__ __forceinline__ void reduce_term(ReduceState& st, float x, ReplicaPos rp,
                                            const K1Params& p) {
  float term = p.average ? x : __fmul_rn(x, p.pre);
  st.s = rp.opens ? term : __fadd_rn(st.s, term);
  if (rp.closes) {
    float s = p.average ? __fmul_rn(st.s, p.inv_dpi) : st.s;
    s = GradT<GT>::round_to(s);
    st.total = rp.first_inst ? s : __fadd_rn(st.total, s);
  }
}

// The reduced grad in the grad dtype, times the scale_gradients factor
// (rounded to the grad dtype again; skipped for a factor of 1).
template <typename GT>
__device__ __forceinline__ float post_scaled(float red, float post_scale) {
  return post_scale == 1.0f ? red : GradT<GT>::round_to(__fmul_rn(red, post_scale));
}

template <typename GT>
__device__ __forceinline__ float reduce_finish(const ReduceState& st, const K1Params& p) {
  float total = st.total;
  if (p.n_inst > 1) {
    if (p.average) total = __fmul_rn(total, p.inv_ninst);
    total = GradT<GT>::round_to(total);
  }
  return __fmul_rn(post_scaled<GT>(total, p.post_scale), p.inv_scale);
}

// Sum of squares of a thread's main grads, accurate to about fp64 while
// computing in fp32: each square is split exactly into p + pe (FMA) and added
// with the error-free TwoSum, the errors gathered in c (the Dot2 scheme of
// Ogita, Rump & Oishi, "Accurate sum and dot product", SIAM J. Sci. Comput.
// 2005).  Squares of |x| >= 2^62 would overflow fp32 and go to an fp64
// accumulator instead, and the fp32 pair moves to fp64 before it could
// overflow; both rare paths are out-of-line calls, so no fp64 instruction
// is issued per element (GB300's fp64 rate is a small fraction of fp32's).
// A non-finite main grad makes the sum non-finite, and finite main grads
// cannot overflow it, so the non-finite check of prepare_grads is read off
// the sum.
__device__ __noinline__ double sumsq_wide(double d, float a, float b, float c, float e) {
  return d + (double)a * (double)a + (double)b * (double)b + (double)c * (double)c +
         (double)e * (double)e;
}
__device__ __noinline__ double sumsq_flush(double d, float s, float c) {
  return d + ((double)s + (double)c);
}

struct SumSq {
  float s = 0.f, c = 0.f;
  double d = 0.0;
  int zeros = 0;  // main grads equal to zero (count_zeros)
  __device__ __forceinline__ void dot2(float x) {
    float p = __fmul_rn(x, x);
    float pe = fmaf(x, x, -p);
    float t = __fadd_rn(s, p);
    float bp = __fsub_rn(t, s);
    float e = __fadd_rn(__fsub_rn(s, __fsub_rn(t, bp)), __fsub_rn(p, bp));
    s = t;
    c = __fadd_rn(c, __fadd_rn(e, pe));
  }
  __device__ __forceinline__ void add4(const float* x) {
    zeros += (x[0] == 0.f) + (x[1] == 0.f) + (x[2] == 0.f) + (x[3] == 0.f);
    float mx = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    if (mx >= 0x1p62f) {
      d = sumsq_wide(d, x[0], x[1], x[2], x[3]);
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j) dot2(x[j]);
    }
  }
  __device__ __forceinline__ void add1(float x) {
    zeros += (x == 0.f);
    if (fabsf(x) >= 0x1p62f) d = sumsq_wide(d, x, 0.f, 0.f, 0.f);
    else dot2(x);
  }
  // once per tile: keeps |s| below 2^100 (NaN also takes this path)
  __device__ __forceinline__ void maybe_flush() {
    if (!(fabsf(s) <= 0x1p100f)) {
      d = sumsq_flush(d, s, c);
      s = c = 0.f;
    }
  }
  __device__ __forceinline__ double value() const { return d + ((double)s + (double)c); }
};

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Writes this CTA's partial (sum of squares, non-finite flag) and zeroes the
// slots of its region that this launch leaves unused, so the finalize pass
// can always sum whole regions.
__device__ __forceinline__ void write_partial(const SumSq& acc, Partial* partials) {
  __shared__ double s_sum[kThreads / 32];
  __shared__ int s_zero[kThreads / 32];
  double v = warp_sum(acc.value());
  int z = acc.zeros;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xFFFFFFFFu, z, o);
  if (threadIdx.x % 32 == 0) {
    s_sum[threadIdx.x / 32] = v;
    s_zero[threadIdx.x / 32] = z;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    int zt = 0;
    for (int i = 0; i < kThreads / 32; ++i) {
      tot += s_sum[i];
      zt += s_zero[i];
    }
    partials[blockIdx.x] = Partial{tot, isfinite(tot) ? 0 : 1, zt};
    for (int i = gridDim.x + blockIdx.x; i < kMaxGrid; i += gridDim.x)
      partials[i] = Partial{0.0, 0, 0};
  }
}

// ------------------------------------------------------------------- K1 --

// General reduction: any replica count, instances, average_in_collective.
template <typename GT, bool FULL, bool STATS>
__global__ void __launch_bounds__(kThreads, DOPT_K1_MIN_BLOCKS)
k1_reduce_prepare(const __grid_constant__ K1Params p) {
  const int dpi = p.n_rep / p.n_inst;
  SumSq acc;
  int si = 0;
  for (int t = blockIdx.x; t < p.tab.n_tiles; t += gridDim.x) {
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    const int64_t off = (int64_t)(t - sg.tile0) * kTile1;
    const int n = (int)min((int64_t)kTile1, (int64_t)sg.len - off);
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const bool aligned = seg_aligned(sg.local, sg.world);

    ReduceState st[kUnroll1][kVec];
    bool vec_ok[kUnroll1];
#pragma unroll
    for (int u = 0; u < kUnroll1; ++u) vec_ok[u] = aligned && ((u * kThreads + threadIdx.x) * kVec + kVec <= n);

    // kBatch replicas x kUnroll1 accesses of kVec elements in flight
    for (int k0 = 0; k0 < p.n_rep; k0 += kBatch) {
      float x[kBatch][kUnroll1][kVec];
#pragma unroll
      for (int kk = 0; kk < kBatch; ++kk) {
        if (k0 + kk < p.n_rep) {
#pragma unroll
          for (int u = 0; u < kUnroll1; ++u) {
            const int e = (u * kThreads + threadIdx.x) * kVec;
            if (vec_ok[u]) GradT<GT>::widen4(p.rep[k0 + kk], r0 + e, x[kk][u]);
          }
        }
      }
#pragma unroll
      for (int kk = 0; kk < kBatch; ++kk) {
        if (k0 + kk < p.n_rep) {
          const ReplicaPos rp = replica_pos(k0 + kk, dpi);
#pragma unroll
          for (int u = 0; u < kUnroll1; ++u) {
            if (vec_ok[u]) {
#pragma unroll
              for (int j = 0; j < kVec; ++j) reduce_term<GT>(st[u][j], x[kk][u][j], rp, p);
            }
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll1; ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (vec_ok[u]) {
        float m[kVec];
#pragma unroll
        for (int j = 0; j < kVec; ++j) m[j] = reduce_finish<GT>(st[u][j], p);
        __stcs(reinterpret_cast<float4*>(p.main_grad + l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        if (STATS) acc.add4(m);
      } else if (e < n) {
        // scalar path: the ragged end of a run, or a run whose starts are
        // not 8-element aligned
        const int cnt = min(kVec, n - e);
        for (int j = 0; j < cnt; ++j) {
          ReduceState s1;
          s1.s = 0.f;
          s1.total = 0.f;
          for (int k = 0; k < p.n_rep; ++k)
            reduce_term<GT>(s1, GradT<GT>::widen1(p.rep[k], r0 + e + j), replica_pos(k, dpi), p);
          float m = reduce_finish<GT>(s1, p);
          p.main_grad[l0 + e + j] = m;
          if (STATS) acc.add1(m);
        }
      }
    }
    if (STATS) acc.maybe_flush();
  }
  if (STATS) write_partial(acc, p.partials);
}

// The common reductions: prescale by 1/N and sum (average_in_collective =
// false), NINST instances of DPI replicas each, both known at compile time.
// Same arithmetic as the general kernel, in the same order (each instance's
// replicas summed in order and rounded to the grad dtype, then the instance
// sums in order, rounded again when there is more than one), without its
// per-element selects.  Loads of one instance are in flight together.
template <typename GT, bool FULL, bool STATS, int DPI, int NINST>
__global__ void __launch_bounds__(kThreads, DOPT_K1_MIN_BLOCKS)
k1_reduce_prepare_n(const __grid_constant__ K1Params p) {
  constexpr int U = kUnroll1 * GradT<GT>::kUnroll;  // accesses per thread per tile
  constexpr int TILE = kThreads * kVec * U;
  SumSq acc;
  int si = 0;
  const float pre = p.pre, inv_scale = p.inv_scale;
  for (int t = blockIdx.x; t < p.tab.n_tiles; t += gridDim.x) {
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    const int64_t off = (int64_t)(t - sg.tile0) * TILE;
    const int n = (int)min((int64_t)TILE, (int64_t)sg.len - off);
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const bool aligned = seg_aligned(sg.local, sg.world);

    bool vec_ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) vec_ok[u] = aligned && (u * kThreads + threadIdx.x) * kVec + kVec <= n;
    float total[U][kVec];
#pragma unroll 1
    for (int j = 0; j < NINST; ++j) {  // one instance's loads live at a time
      typename GradT<GT>::Raw x[DPI][U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int e = (u * kThreads + threadIdx.x) * kVec;
        if (vec_ok[u]) {
#pragma unroll
          for (int k = 0; k < DPI; ++k) x[k][u] = GradT<GT>::load4(p.rep[j * DPI + k], r0 + e);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float sum = __fmul_rn(GradT<GT>::at(x[0][u], q), pre);
#pragma unroll
          for (int k = 1; k < DPI; ++k) sum = __fadd_rn(sum, __fmul_rn(GradT<GT>::at(x[k][u], q), pre));
          sum = GradT<GT>::round_to(sum);
          total[u][q] = (j == 0) ? sum : __fadd_rn(total[u][q], sum);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (vec_ok[u]) {
        float m[kVec];
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float tt = NINST > 1 ? GradT<GT>::round_to(total[u][q]) : total[u][q];
          m[q] = __fmul_rn(post_scaled<GT>(tt, p.post_scale), inv_scale);
        }
        __stcs(reinterpret_cast<float4*>(p.main_grad + l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        if (STATS) acc.add4(m);
      } else if (e < n) {
        const int cnt = min(kVec, n - e);
        for (int q = 0; q < cnt; ++q) {
          float tt = 0.f;
          for (int j = 0; j < NINST; ++j) {
            float sum = __fmul_rn(GradT<GT>::widen1(p.rep[j * DPI], r0 + e + q), pre);
            for (int k = 1; k < DPI; ++k)
              sum = __fadd_rn(sum, __fmul_rn(GradT<GT>::widen1(p.rep[j * DPI + k], r0 + e + q), pre));
            sum = GradT<GT>::round_to(sum);
            tt = (j == 0) ? sum : __fadd_rn(tt, sum);
          }
          if (NINST > 1) tt = GradT<GT>::round_to(tt);
          float m = __fmul_rn(post_scaled<GT>(tt, p.post_scale), inv_scale);
          p.main_grad[l0 + e + q] = m;
          if (STATS) acc.add1(m);
        }
      }
    }
    if (STATS) acc.maybe_flush();
  }
  if (STATS) write_partial(acc, p.partials);
}

// ---------------------------------------------------------- K1 with TMA --
//
// The single-instance reduction with every replica tile staged through
// shared memory by the bulk-copy engine (cp.async.bulk, one 1-D copy per
// replica per tile, completion counted in bytes on a per-stage mbarrier).
// A ring of DOPT_TMA_STAGES stages keeps up to stages x replicas x tile bytes
// in flight per SM independently of registers; thread 0 issues, every thread
// consumes.  Every wait is bounded: a CTA that gives up (decided uniformly)
// sets the error flag, marks its partial non-finite so the step is skipped,
// waits (bounded) for its copies still in flight and leaves.  Used for
// fp32 replicas when every run of the launch is 8-element aligned.

#ifndef DOPT_TMA_TILE
#define DOPT_TMA_TILE 2048
#endif
constexpr int kTmaTile = DOPT_TMA_TILE;     // elements per tile (a multiple of kThreads * kVec)
static_assert(kTmaTile % (kThreads * kVec) == 0, "TMA tile");
constexpr unsigned long long kWaitNs = 1000000000ull;  // give up a wait after 1 s

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Polls an mbarrier phase for at most kWaitNs nanoseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > kWaitNs) return false;
  }
}
#ifndef DOPT_TMA_EVICT_FIRST
#define DOPT_TMA_EVICT_FIRST 1  // 1: the replica tiles are marked first to leave L2
#endif
__device__ __forceinline__ void bulk_load(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
#if DOPT_TMA_EVICT_FIRST
  uint64_t policy;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"((unsigned long long)__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
#else
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"((unsigned long long)__cvta_generic_to_global(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
#endif
}

template <typename GT>
struct GradBits {
  using T = typename std::conditional<std::is_same<GT, float>::value, float, unsigned short>::type;
};

template <typename GT, int DPI>
__host__ __device__ constexpr size_t tma_smem_bytes() {
  return (size_t)DOPT_TMA_STAGES * DPI * kTmaTile * sizeof(typename GradBits<GT>::T) +
         DOPT_TMA_STAGES * sizeof(uint64_t);
}

template <typename GT, bool FULL, bool STATS, int DPI>
__global__ void __launch_bounds__(kThreads, 1) k1_reduce_prepare_tma(const __grid_constant__ K1Params p) {
  using E = typename GradBits<GT>::T;
  constexpr int S = DOPT_TMA_STAGES;
  constexpr int VALIGN = 16 / sizeof(E);  // elements per 16 bytes: bulk sizes are multiples of it
  extern __shared__ __align__(128) unsigned char smem[];
  E* tiles = reinterpret_cast<E*>(smem);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * DPI * kTmaTile * sizeof(E));
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int G = gridDim.x;
  const int my = p.tab.n_tiles > (int)blockIdx.x ? (p.tab.n_tiles - (int)blockIdx.x + G - 1) / G : 0;
  int si_issue = 0;
  // thread 0: start the copies of this CTA's i-th tile into stage i % S
  auto issue = [&](int i) {
    const int t = blockIdx.x + i * G;
    si_issue = seek(p.tab, si_issue, t);
    const Seg& sg = p.tab.seg[si_issue];
    const int64_t off = (int64_t)(t - sg.tile0) * kTmaTile;
    const int n = (int)min((int64_t)kTmaTile, (int64_t)sg.len - off);
    const int nv = n & ~(VALIGN - 1);
    const int64_t r0 = FULL ? sg.world + off : sg.local + off;
    const int stage = i % S;
    mbar_arrive_expect_tx(&bars[stage], (unsigned)(nv * sizeof(E)) * DPI);
    if (nv > 0 && !(blockIdx.x == 0 && i == p.starve_tile)) {
#pragma unroll
      for (int k = 0; k < DPI; ++k)
        bulk_load(tiles + ((size_t)stage * DPI + k) * kTmaTile, static_cast<const E*>(p.rep[k]) + r0,
                  (unsigned)(nv * sizeof(E)), &bars[stage]);
    }
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(S, my); ++i) issue(i);

  SumSq acc;
  int si = 0;
  bool failed = false;
  const float pre = p.pre, inv_scale = p.inv_scale;
  int i = 0;
  for (; i < my; ++i) {
    const int stage = i % S;
    const bool ok = mbar_wait_bounded(&bars[stage], (unsigned)((i / S) & 1));
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int t = blockIdx.x + i * G;
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    const int64_t off = (int64_t)(t - sg.tile0) * kTmaTile;
    const int n = (int)min((int64_t)kTmaTile, (int64_t)sg.len - off);
    const int nv = n & ~(VALIGN - 1);
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const E* st = tiles + (size_t)stage * DPI * kTmaTile;
#pragma unroll
    for (int u = 0; u < kTmaTile / (kThreads * kVec); ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (e + kVec <= nv) {
        float m[kVec];
        typename GradT<GT>::Raw x[DPI];
#pragma unroll
        for (int k = 0; k < DPI; ++k)
          x[k] = *reinterpret_cast<const typename GradT<GT>::Raw*>(st + (size_t)k * kTmaTile + e);
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float sum = __fmul_rn(GradT<GT>::at(x[0], q), pre);
#pragma unroll
          for (int k = 1; k < DPI; ++k) sum = __fadd_rn(sum, __fmul_rn(GradT<GT>::at(x[k], q), pre));
          m[q] = __fmul_rn(post_scaled<GT>(GradT<GT>::round_to(sum), p.post_scale), inv_scale);
        }
        __stcs(reinterpret_cast<float4*>(p.main_grad + l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        if (STATS) acc.add4(m);
      } else if (e < n) {
        // the last few elements of a run: not in the staged copy
        const int cnt = min(kVec, n - e);
        for (int q = 0; q < cnt; ++q) {
          float sum = __fmul_rn(GradT<GT>::widen1(p.rep[0], r0 + e + q), pre);
          for (int k = 1; k < DPI; ++k)
            sum = __fadd_rn(sum, __fmul_rn(GradT<GT>::widen1(p.rep[k], r0 + e + q), pre));
          float m = __fmul_rn(post_scaled<GT>(GradT<GT>::round_to(sum), p.post_scale), inv_scale);
          p.main_grad[l0 + e + q] = m;
          if (STATS) acc.add1(m);
        }
      }
    }
    if (STATS) acc.maybe_flush();
    __syncthreads();  // every thread is done with this stage
    if (threadIdx.x == 0 && i + S < my) issue(i + S);
  }
  if (failed) {
    if (threadIdx.x == 0) {
      *p.error_flag = kErrorMagic;
      // let the copies already issued land before the shared memory goes away
      for (int j = i; j < min(i + S, my); ++j) mbar_wait_bounded(&bars[j % S], (unsigned)((j / S) & 1));
    }
    __syncthreads();
    acc.s = __int_as_float(0x7FC00000);  // a NaN partial skips the step
  }
  if (STATS) write_partial(acc, p.partials);
}

// ------------------------------------------------------------------- K2 --

// The step number and learning rate of a step whose counter lives in device
// memory: the finalize pass reads them, computes the step scalars for the
// next step number and advances the counter only when the step is applied.
struct K2Step {
  int64_t* d_step;      // NULL: the host supplied the step scalars
  const double* d_lr;   // NULL: lr below
  double lr, wd, beta1, beta2;
  DevStep* out;
};

// beta^t by binary powering in fp64 (the host computes it the same way).
__host__ __device__ __forceinline__ double pow_int(double b, int64_t t) {
  double r = 1.0, x = b;
  while (t > 0) {
    if (t & 1) r *= x;
    x *= x;
    t >>= 1;
  }
  return r;
}

__global__ void __launch_bounds__(kThreads)
k2_finalize(const Partial* __restrict__ parts, int n_slots, double remote_sumsq,
            int remote_found_inf, double max_norm, Scalars* __restrict__ sc,
            float* d_norm, float* d_coef, int32_t* d_found, int32_t* err_flag, K2Step step) {
  __shared__ double s_sum[kThreads];
  __shared__ int s_bad[kThreads];
  __shared__ long long s_zero[kThreads];
  double v = 0.0;
  int b = 0;
  long long z = 0;
  for (int i = threadIdx.x; i < n_slots; i += kThreads) {
    v += parts[i].sumsq;
    b |= parts[i].nonfinite;
    z += parts[i].zeros;
  }
  s_sum[threadIdx.x] = v;
  s_bad[threadIdx.x] = b;
  s_zero[threadIdx.x] = z;
  __syncthreads();
  for (int w = kThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) {
      s_sum[threadIdx.x] += s_sum[threadIdx.x + w];
      s_bad[threadIdx.x] |= s_bad[threadIdx.x + w];
      s_zero[threadIdx.x] += s_zero[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int kernel_error = *err_flag == kErrorMagic ? 1 : 0;
    *err_flag = 0;
    const double sumsq = s_sum[0] + remote_sumsq;
    const int found = (s_bad[0] || remote_found_inf || kernel_error) ? 1 : 0;
    const double norm = sqrt(sumsq);
    double coef = 1.0;
    int clip = 0;
    if (max_norm > 0.0) {
      coef = max_norm / (norm + 1.0e-6);
      clip = coef < 1.0;
    }
    const float coef_f = clip ? (float)coef : 1.0f;
    const float norm_f = found ? __int_as_float(0x7FC00000) : (float)norm;
    sc->sumsq = sumsq;
    sc->grad_norm = norm_f;
    sc->clip_coef = coef_f;
    sc->found_inf = found;
    sc->clipped = clip;
    sc->num_zeros = s_zero[0];
    sc->kernel_error = kernel_error;
    sc->reserved = 0;
    if (d_norm) *d_norm = norm_f;
    if (d_coef) *d_coef = coef_f;
    if (d_found) *d_found = found;
    if (step.d_step) {
      const int64_t t = *step.d_step + 1;
      const double lr = step.d_lr ? *step.d_lr : step.lr;
      step.out->step_size = (float)(lr / (1.0 - pow_int(step.beta1, t)));
      step.out->bc2_sqrt = (float)sqrt(1.0 - pow_int(step.beta2, t));
      step.out->lr_wd = lr * step.wd;
      if (!found) *step.d_step = t;  // a skipped step does not count
    }
  }
}

// ------------------------------------------------------------------- K3 --

template <typename PT>
struct ParamT;
template <>
struct ParamT<__nv_bfloat16> {
  static constexpr bool kInPlace = false;
  static __device__ __forceinline__ void store4(void* p, int64_t i, const float* x) {
    unsigned short h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __bfloat16_as_ushort(__float2bfloat16_rn(x[j]));
    __stcs(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i),
           make_uint2((unsigned)h[0] | ((unsigned)h[1] << 16), (unsigned)h[2] | ((unsigned)h[3] << 16)));
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<unsigned short*>(p)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};
template <>
struct ParamT<__half> {
  static constexpr bool kInPlace = false;
  static __device__ __forceinline__ void store4(void* p, int64_t i, const float* x) {
    unsigned short h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __half_as_ushort(__float2half_rn(x[j]));
    __stcs(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i),
           make_uint2((unsigned)h[0] | ((unsigned)h[1] << 16), (unsigned)h[2] | ((unsigned)h[3] << 16)));
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<unsigned short*>(p)[i] = __half_as_ushort(__float2half_rn(x));
  }
};
template <>
struct ParamT<float> {
  static constexpr bool kInPlace = true;  // the fp32 param buffer is the master
  static __device__ __forceinline__ void store4(void*, int64_t, const float*) {}
  static __device__ __forceinline__ void store1(void*, int64_t, float) {}
};

// The decoupled weight-decay factor (float)(1 - lr*wd*wd_mult), formed in
// fp64; out of line so no fp64 instruction is issued per element -- it runs
// once per run change.
__device__ __noinline__ float decay_of(double lr_wd, double wd_mult) {
  return (float)(1.0 - lr_wd * wd_mult);
}

struct StepScalars {
  float step_size, bc2_sqrt;
  double lr_wd;
};

__device__ __forceinline__ StepScalars step_scalars(const K3Params& p) {
  if (p.dev) return StepScalars{p.dev->step_size, p.dev->bc2_sqrt, p.dev->lr_wd};
  return StepScalars{p.step_size, p.bc2_sqrt, p.lr_wd};
}

// One element of AdamW (torch semantics: decay the weight, update m and v,
// divide the bias-corrected sqrt(v) + eps into m, step), each operation
// rounded once in fp32.
__device__ __forceinline__ void adamw1(float g, float decay, const K3Params& p, const StepScalars& ss,
                                       float& w, float& m, float& v) {
  float pp = __fmul_rn(w, decay);
  float mm = __fadd_rn(__fmul_rn(p.b1, m), __fmul_rn(p.omb1, g));
  float vv = __fadd_rn(__fmul_rn(p.b2, v), __fmul_rn(__fmul_rn(p.omb2, g), g));
  float denom = __fadd_rn(__fdiv_rn(__fsqrt_rn(vv), ss.bc2_sqrt), p.eps);
  pp = __fsub_rn(pp, __fmul_rn(ss.step_size, __fdiv_rn(mm, denom)));
  w = pp;
  m = mm;
  v = vv;
}

// The AdamW pass with the loads of a thread's next tile issued before the
// current tile is computed and stored, so the memory pipe stays busy while
// the thread does arithmetic (software pipelining across tiles).
struct K3Tile {
  float4 g[kUnroll3], w[kUnroll3], m[kUnroll3], v[kUnroll3];
  int64_t l0, w0, m0;
  int n;
  float decay;
  bool aligned;
};

template <typename PT>
__device__ __forceinline__ void k3_load(const K3Params& p, float* wbase, int t, int& si, K3Tile& T,
                                        int& decay_si, float& decay, double lr_wd) {
  si = seek(p.tab, si, t);
  const Seg& sg = p.tab.seg[si];
  if (si != decay_si) {
    decay = decay_of(lr_wd, sg.wd_mult);
    decay_si = si;
  }
  const int64_t off = (int64_t)(t - sg.tile0) * kTile3;
  T.n = (int)min((int64_t)kTile3, (int64_t)sg.len - off);
  T.l0 = sg.local + off;
  T.w0 = sg.world + off;
  T.m0 = ParamT<PT>::kInPlace ? T.w0 : T.l0;
  T.aligned = seg_aligned(sg.local, sg.world);
  T.decay = decay;
#pragma unroll
  for (int u = 0; u < kUnroll3; ++u) {
    const int e = (u * kThreads + threadIdx.x) * kVec;
    if (T.aligned && e + kVec <= T.n) {
      T.g[u] = __ldcs(reinterpret_cast<const float4*>(p.main_grad + T.l0 + e));
      T.w[u] = __ldcs(reinterpret_cast<const float4*>(wbase + T.m0 + e));
      T.m[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg + T.l0 + e));
      T.v[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg_sq + T.l0 + e));
    }
  }
}

template <typename PT>
__global__ void __launch_bounds__(kThreads, DOPT_K3_MIN_BLOCKS) k3_adamw_pipe(const __grid_constant__ K3Params p) {
  if (*p.found_inf) return;  // skipped step: nothing is written
  const float c = *p.coef;
  const StepScalars ss = step_scalars(p);
  float* const wbase = ParamT<PT>::kInPlace ? static_cast<float*>(p.param) : p.master;
  int si = 0, decay_si = -1;
  float decay = 1.f;
  int t = blockIdx.x;
  if (t >= p.tab.n_tiles) return;
  K3Tile cur;
  k3_load<PT>(p, wbase, t, si, cur, decay_si, decay, ss.lr_wd);
  for (; t < p.tab.n_tiles; t += gridDim.x) {
    K3Tile nxt;
    const bool more = t + (int)gridDim.x < p.tab.n_tiles;
    if (more) k3_load<PT>(p, wbase, t + gridDim.x, si, nxt, decay_si, decay, ss.lr_wd);
#pragma unroll
    for (int u = 0; u < kUnroll3; ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (cur.aligned && e + kVec <= cur.n) {
        float g[kVec] = {cur.g[u].x, cur.g[u].y, cur.g[u].z, cur.g[u].w};
        float w[kVec] = {cur.w[u].x, cur.w[u].y, cur.w[u].z, cur.w[u].w};
        float m[kVec] = {cur.m[u].x, cur.m[u].y, cur.m[u].z, cur.m[u].w};
        float v[kVec] = {cur.v[u].x, cur.v[u].y, cur.v[u].z, cur.v[u].w};
#pragma unroll
        for (int j = 0; j < kVec; ++j) adamw1(__fmul_rn(g[j], c), cur.decay, p, ss, w[j], m[j], v[j]);
        __stcs(reinterpret_cast<float4*>(wbase + cur.m0 + e), make_float4(w[0], w[1], w[2], w[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg + cur.l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg_sq + cur.l0 + e), make_float4(v[0], v[1], v[2], v[3]));
        ParamT<PT>::store4(p.param, cur.w0 + e, w);
      } else if (e < cur.n) {
        const int cnt = min(kVec, cur.n - e);
        for (int j = 0; j < cnt; ++j) {
          float ww = wbase[cur.m0 + e + j], mm = p.exp_avg[cur.l0 + e + j], vv = p.exp_avg_sq[cur.l0 + e + j];
          adamw1(__fmul_rn(p.main_grad[cur.l0 + e + j], c), cur.decay, p, ss, ww, mm, vv);
          wbase[cur.m0 + e + j] = ww;
          p.exp_avg[cur.l0 + e + j] = mm;
          p.exp_avg_sq[cur.l0 + e + j] = vv;
          ParamT<PT>::store1(p.param, cur.w0 + e + j, ww);
        }
      }
    }
    if (more) cur = nxt;
  }
}

// ------------------------------------------------------------ host side --

thread_local std::vector<char> t_param_scratch;  // kernel-parameter staging
std::atomic<uint64_t> g_launches{0};             // kernels launched by this library
std::atomic<int32_t> g_starve_tile{-1};           // test hook, see dopt_debug_starve_copy

// The run table of one launch: runs [first, first + count) of a rank
// selection, with per-run decay for K3.
struct Chunk {
  int first, count, n_tiles;
};

std::vector<Chunk> chunks_of(const std::vector<dopt::Run>& runs) {
  std::vector<Chunk> out;
  int i = 0;
  do {
    Chunk c{i, 0, 0};
    while (i < (int)runs.size() && c.count < kMaxSeg) {
      ++c.count;
      ++i;
    }
    out.push_back(c);
  } while (i < (int)runs.size());
  return out;  // at least one (possibly empty) chunk
}

// Fills the kernel-parameter table of one chunk for tiles of `tile`
// elements.
void fill_table(SegTable& tab, const std::vector<dopt::Run>& runs, const Chunk& c, int tile_elems) {
  tab.n_seg = c.count;
  int tile = 0;
  for (int k = 0; k < c.count; ++k) {
    const dopt::Run& r = runs[c.first + k];
    Seg& s = tab.seg[k];
    s.local = r.local;
    s.world = r.world;
    s.len = (int32_t)r.len;
    s.tile0 = tile;
    s.wd_mult = r.wd_mult;
    tile += (int)((r.len + tile_elems - 1) / tile_elems);
  }
  tab.n_tiles = tile;
}

struct DeviceInfo {
  int device = -1, sms = 0;
};

int device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  static thread_local DeviceInfo cache;
  if (cache.device != dev) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return dopt::fail(DOPT_E_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    cache.device = dev;
    cache.sms = n;
  }
  *sms = cache.sms;
  return DOPT_OK;
}

template <typename K>
int grid_for(K kernel, int n_tiles, int* grid) {
  int sms = 0;
  int st = device_sms(&sms);
  if (st) return st;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
  if (e != cudaSuccess)
    return dopt::fail(DOPT_E_CUDA, std::string("occupancy query: ") + cudaGetErrorString(e));
  int g = std::max(1, per_sm) * sms;
  g = std::min(g, kMaxGrid);
  g = std::min(g, std::max(1, n_tiles));
  *grid = g;
  return DOPT_OK;
}

int check_launch(const char* what) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return DOPT_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_map_buffer_rank(const dopt_shard_map* m, int32_t buffer, int32_t rank, const char* fn) {
  if (!m) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL map");
  if (buffer < 0 || buffer >= (int32_t)m->buffers.size())
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": buffer out of range");
  if (rank != DOPT_ALL_RANKS && (rank < 0 || rank >= m->dp))
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": rank out of range");
  return DOPT_OK;
}

// Workspace layout: [Scalars | pad to 256] then, per buffer, per launch chunk
// of its run table, a region of kMaxGrid Partial slots.
int regions_before(dopt_shard_map* m, int32_t buffer, int32_t rank) {
  int n = 0;
  for (int32_t b = 0; b < buffer; ++b) n += (int)chunks_of(dopt::runs_for(m, b, rank)).size();
  return n;
}

int total_regions(dopt_shard_map* m, int32_t rank) {
  return regions_before(m, (int32_t)m->buffers.size(), rank);
}

size_t workspace_bytes(dopt_shard_map* m, int32_t rank) {
  return kScalarBytes + (size_t)total_regions(m, rank) * kMaxGrid * sizeof(Partial);
}

int check_workspace(dopt_shard_map* m, int32_t rank, void* ws, size_t bytes, const char* fn) {
  if (!ws) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL workspace");
  if (!aligned16(ws)) return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": workspace not 16-byte aligned");
  size_t need = workspace_bytes(m, rank);
  if (bytes < need)
    return dopt::fail(DOPT_E_SIZE, std::string(fn) + ": workspace needs " + std::to_string(need) +
                                       " bytes, got " + std::to_string(bytes));
  return DOPT_OK;
}

Partial* region_ptr(void* ws, int region) {
  return reinterpret_cast<Partial*>(static_cast<char*>(ws) + kScalarBytes) + (size_t)region * kMaxGrid;
}
Scalars* scalars_ptr(void* ws) { return static_cast<Scalars*>(ws); }

K1Params& k1_scratch() {
  t_param_scratch.resize(std::max(sizeof(K1Params), sizeof(K3Params)));
  return *reinterpret_cast<K1Params*>(t_param_scratch.data());
}
K3Params& k3_scratch() {
  t_param_scratch.resize(std::max(sizeof(K1Params), sizeof(K3Params)));
  return *reinterpret_cast<K3Params*>(t_param_scratch.data());
}

template <typename GT, bool FULL, bool STATS>
int launch_k1_t(K1Params& kp, int n_tiles, cudaStream_t s) {
  auto kern = k1_reduce_prepare<GT, FULL, STATS>;
  int grid = 0;
  int st = grid_for(kern, n_tiles, &grid);
  if (st) return st;
  kern<<<grid, kThreads, 0, s>>>(kp);
  return check_launch("k1_reduce_prepare launch");
}

template <typename GT, bool FULL, bool STATS, int DPI>
int launch_k1_tma(K1Params& kp, int n_tiles, cudaStream_t s) {
  auto kern = k1_reduce_prepare_tma<GT, FULL, STATS, DPI>;
  const size_t smem = tma_smem_bytes<GT, DPI>();
  // the dynamic shared-memory limit is raised once per device (a later call,
  // e.g. inside a stream capture, then issues nothing but the launch)
  static std::atomic<uint64_t> attr_set{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
  if (!bit || !(attr_set.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
      return dopt::fail(DOPT_E_CUDA, std::string("k1 tma smem attribute: ") + cudaGetErrorString(e));
    attr_set.fetch_or(bit);
  }
  int sms = 0, per_sm = 0;
  int st = device_sms(&sms);
  if (st) return st;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
  if (e != cudaSuccess || per_sm < 1)
    return dopt::fail(DOPT_E_CUDA, "k1 tma occupancy query failed");
  const int grid = std::max(1, std::min({per_sm * sms, kMaxGrid, std::max(1, n_tiles)}));
  kern<<<grid, kThreads, smem, s>>>(kp);
  return check_launch("k1_reduce_prepare_tma launch");
}

template <typename GT, bool FULL, bool STATS, int DPI, int NINST>
int launch_k1_n(K1Params& kp, int n_tiles, cudaStream_t s) {
  if (STATS && NINST == 1 && kp.use_tma) return launch_k1_tma<GT, FULL, STATS, DPI>(kp, n_tiles, s);
  auto kern = k1_reduce_prepare_n<GT, FULL, STATS, DPI, NINST>;
  int grid = 0;
  int st = grid_for(kern, n_tiles, &grid);
  if (st) return st;
  kern<<<grid, kThreads, 0, s>>>(kp);
  return check_launch("k1_reduce_prepare_n launch");
}

// The specialised kernel covers prescale-and-sum with one instance of 1, 2,
// 4 or 8 replicas, or two instances of 4 or 8; everything else runs the
// general kernel.
template <typename GT, bool FULL, bool STATS>
int launch_k1_g(K1Params& kp, int n_tiles, cudaStream_t s) {
  if (!kp.average) {
    const int dpi = kp.n_rep / kp.n_inst;
    if (kp.n_inst == 1) {
      switch (dpi) {
        case 1: return launch_k1_n<GT, FULL, STATS, 1, 1>(kp, n_tiles, s);
        case 2: return launch_k1_n<GT, FULL, STATS, 2, 1>(kp, n_tiles, s);
        case 4: return launch_k1_n<GT, FULL, STATS, 4, 1>(kp, n_tiles, s);
        case 8: return launch_k1_n<GT, FULL, STATS, 8, 1>(kp, n_tiles, s);
        default: break;
      }
    } else if (kp.n_inst == 2) {
      switch (dpi) {
        case 4: return launch_k1_n<GT, FULL, STATS, 4, 2>(kp, n_tiles, s);
        case 8: return launch_k1_n<GT, FULL, STATS, 8, 2>(kp, n_tiles, s);
        default: break;
      }
    }
  }
  return launch_k1_t<GT, FULL, STATS>(kp, n_tiles, s);
}

template <bool FULL, bool STATS>
int launch_k1_dt(int32_t gdt, K1Params& kp, int n_tiles, cudaStream_t s) {
  switch (gdt) {
    case DOPT_F32: return launch_k1_g<float, FULL, STATS>(kp, n_tiles, s);
    case DOPT_BF16: return launch_k1_g<__nv_bfloat16, FULL, STATS>(kp, n_tiles, s);
    case DOPT_F16: return launch_k1_g<__half, FULL, STATS>(kp, n_tiles, s);
  }
  return dopt::fail(DOPT_E_INVALID, "unknown grad dtype");
}

// Tile size (elements) of the K1 kernel that runs for these arguments: the
// specialised kernels give 16-bit grads twice the accesses per thread.
int k1_tile(int32_t gdt, int32_t n_rep, int32_t n_inst, int32_t average) {
  if (average) return kTile1;
  const int dpi = n_rep / n_inst;
  const bool special = (n_inst == 1 && (dpi == 1 || dpi == 2 || dpi == 4 || dpi == 8)) ||
                       (n_inst == 2 && (dpi == 4 || dpi == 8));
  if (!special) return kTile1;
  return gdt == DOPT_F32 ? kTile1 : 2 * kTile1;
}

// Launches K1 over every chunk of a run list; with stats, chunk i writes its
// partials to workspace region region_first + i.
int run_k1_runs(const std::vector<dopt::Run>& runs, int region_first, const void* const* replicas,
                int32_t n_rep, int32_t n_inst, int32_t full_layout, int32_t average, float inv_scale,
                int32_t gdt, float* main_grad, bool stats, void* ws, cudaStream_t s,
                float post_scale = 1.0f) {
  std::vector<Chunk> chunks = chunks_of(runs);
  int region = region_first;
  for (const Chunk& c : chunks) {
    K1Params& kp = k1_scratch();
    for (int k = 0; k < n_rep; ++k) kp.rep[k] = replicas[k];
    for (int k = n_rep; k < DOPT_MAX_REPLICAS; ++k) kp.rep[k] = nullptr;
    kp.main_grad = main_grad;
    kp.partials = stats ? region_ptr(ws, region++) : nullptr;
    kp.n_rep = n_rep;
    kp.n_inst = n_inst;
    kp.pre = (float)(1.0 / (double)n_rep);
    kp.inv_dpi = (float)(1.0 / (double)(n_rep / n_inst));
    kp.inv_ninst = (float)(1.0 / (double)n_inst);
    kp.inv_scale = inv_scale;
    kp.average = average ? 1 : 0;
    kp.post_scale = post_scale;
    kp.error_flag = ws ? reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kErrorFlagOffset) : nullptr;
    bool all_aligned = true;
    for (int k = 0; k < c.count; ++k) {
      const dopt::Run& r = runs[c.first + k];
      all_aligned &= (r.local % 8) == 0 && (r.world % 8) == 0;
    }
    const int dpi = n_rep / n_inst;
    // fp32 replicas only: 16-bit replicas stream faster through registers
    // (packed loads, four accesses per thread)
    kp.use_tma = (DOPT_K1_TMA && stats && ws && all_aligned && n_inst == 1 && !average &&
                  gdt == DOPT_F32 && (dpi == 1 || dpi == 2 || dpi == 4 || dpi == 8)) ? 1 : 0;
    kp.starve_tile = g_starve_tile.load(std::memory_order_relaxed);
    fill_table(kp.tab, runs, c, kp.use_tma ? kTmaTile : k1_tile(gdt, n_rep, n_inst, average));
    const int n_tiles = kp.tab.n_tiles;
    int st;
    if (stats)
      st = full_layout ? launch_k1_dt<true, true>(gdt, kp, n_tiles, s)
                       : launch_k1_dt<false, true>(gdt, kp, n_tiles, s);
    else
      st = full_layout ? launch_k1_dt<true, false>(gdt, kp, n_tiles, s)
                       : launch_k1_dt<false, false>(gdt, kp, n_tiles, s);
    if (st) return st;
  }
  return DOPT_OK;
}

// K1 over every run of (buffer, rank); partials go to the buffer's regions
// of the fused-step workspace layout.
int run_k1(dopt_shard_map* m, int32_t buffer, int32_t rank, const void* const* replicas,
           int32_t n_rep, int32_t n_inst, int32_t full_layout, int32_t average, float inv_scale,
           int32_t gdt, float* main_grad, bool stats, void* ws, cudaStream_t s,
           float post_scale = 1.0f) {
  return run_k1_runs(dopt::runs_for(m, buffer, rank), stats ? regions_before(m, buffer, rank) : 0,
                     replicas, n_rep, n_inst, full_layout, average, inv_scale, gdt, main_grad, stats,
                     ws, s, post_scale);
}

// scale_gradients factor of a step: 0 (unset) means 1.
float grad_scale_of(const dopt_step_args* a) { return a->grad_scale == 0.0f ? 1.0f : a->grad_scale; }

DevStep* dev_step_ptr(void* ws) {
  return reinterpret_cast<DevStep*>(static_cast<char*>(ws) + kDevStepOffset);
}

int run_k2_slots(int n_slots, void* ws, double remote_sumsq, int32_t remote_found, double max_norm,
                 float* d_norm, float* d_coef, int32_t* d_found, cudaStream_t s,
                 const dopt_step_args* a = nullptr) {
  K2Step step{nullptr, nullptr, 0.0, 0.0, 0.0, 0.0, dev_step_ptr(ws)};
  if (a && a->d_step) {
    step.d_step = a->d_step;
    step.d_lr = a->d_lr;
    step.lr = a->hp.lr;
    step.wd = a->hp.weight_decay;
    step.beta1 = a->hp.beta1;
    step.beta2 = a->hp.beta2;
  }
  k2_finalize<<<1, kThreads, 0, s>>>(region_ptr(ws, 0), n_slots, remote_sumsq, remote_found ? 1 : 0,
                                     max_norm, scalars_ptr(ws), d_norm, d_coef, d_found,
                                     reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kErrorFlagOffset),
                                     step);
  return check_launch("k2_finalize launch");
}

int run_k2(dopt_shard_map* m, int32_t rank, void* ws, double remote_sumsq, int32_t remote_found,
           double max_norm, float* d_norm, float* d_coef, int32_t* d_found, cudaStream_t s,
           const dopt_step_args* a = nullptr) {
  return run_k2_slots(total_regions(m, rank) * kMaxGrid, ws, remote_sumsq, remote_found, max_norm,
                      d_norm, d_coef, d_found, s, a);
}

int check_hparams(const dopt_adamw_hparams* hp, const char* fn) {
  if (!hp) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL hparams");
  bool ok = hp->step >= 1 && std::isfinite(hp->lr) && hp->lr >= 0 && hp->beta1 >= 0 &&
            hp->beta1 < 1 && hp->beta2 >= 0 && hp->beta2 < 1 && std::isfinite(hp->eps) &&
            hp->eps > 0 && std::isfinite(hp->weight_decay);
  if (!ok) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": bad AdamW hyper-parameters");
  return DOPT_OK;
}


template <typename PT>
int launch_k3_t(K3Params& kp, int n_tiles, cudaStream_t s) {
  auto kern = k3_adamw_pipe<PT>;
  int grid = 0;
  int st = grid_for(kern, n_tiles, &grid);
  if (st) return st;
  kern<<<grid, kThreads, 0, s>>>(kp);
  return check_launch("k3_adamw launch");
}

int run_k3_runs(const std::vector<dopt::Run>& runs, int32_t pdt, const float* main_grad, float* master,
                float* exp_avg, float* exp_avg_sq, void* param, const dopt_adamw_hparams* hp,
                const float* d_coef, const int32_t* d_found, cudaStream_t s,
                const DevStep* dev = nullptr) {
  std::vector<Chunk> chunks = chunks_of(runs);
  for (const Chunk& c : chunks) {
    K3Params& kp = k3_scratch();
    kp.main_grad = main_grad;
    kp.master = master;
    kp.exp_avg = exp_avg;
    kp.exp_avg_sq = exp_avg_sq;
    kp.param = param;
    kp.coef = d_coef;
    kp.found_inf = d_found;
    kp.dev = dev;
    kp.lr_wd = hp->lr * hp->weight_decay;
    kp.b1 = (float)hp->beta1;
    kp.b2 = (float)hp->beta2;
    kp.omb1 = (float)(1.0 - hp->beta1);
    kp.omb2 = (float)(1.0 - hp->beta2);
    kp.eps = (float)hp->eps;
    kp.step_size = (float)(hp->lr / (1.0 - pow_int(hp->beta1, hp->step)));
    kp.bc2_sqrt = (float)std::sqrt(1.0 - pow_int(hp->beta2, hp->step));
    kp.pad = 0;
    fill_table(kp.tab, runs, c, kTile3);
    const int n_tiles = kp.tab.n_tiles;
    int st;
    switch (pdt) {
      case DOPT_BF16: st = launch_k3_t<__nv_bfloat16>(kp, n_tiles, s); break;
      case DOPT_F16: st = launch_k3_t<__half>(kp, n_tiles, s); break;
      default: st = launch_k3_t<float>(kp, n_tiles, s); break;
    }
    if (st) return st;
  }
  return DOPT_OK;
}

int run_k3(dopt_shard_map* m, int32_t buffer, int32_t rank, const float* main_grad, float* master,
           float* exp_avg, float* exp_avg_sq, void* param, const dopt_adamw_hparams* hp,
           const float* d_coef, const int32_t* d_found, cudaStream_t s, const DevStep* dev = nullptr) {
  return run_k3_runs(dopt::runs_for(m, buffer, rank), m->buffers[buffer].param_dtype, main_grad, master,
                     exp_avg, exp_avg_sq, param, hp, d_coef, d_found, s, dev);
}

// ---- bucket-staged step: one partial region per (buffer, bucket, chunk) --

std::vector<std::vector<dopt::Run>> runs_by_bucket(dopt_shard_map* m, int32_t buffer, int32_t rank) {
  std::vector<std::vector<dopt::Run>> out(m->buffers[buffer].buckets.size());
  for (const dopt::Run& r : dopt::runs_for(m, buffer, rank)) out[r.bucket].push_back(r);
  return out;
}

// Region index of (buffer, bucket)'s first chunk; (nbuffers, 0) gives the total.
int bucketed_region(dopt_shard_map* m, int32_t rank, int32_t buffer, int32_t bucket) {
  int n = 0;
  for (int32_t b = 0; b < (int32_t)m->buffers.size(); ++b) {
    std::vector<std::vector<dopt::Run>> by = runs_by_bucket(m, b, rank);
    for (int32_t k = 0; k < (int32_t)by.size(); ++k) {
      if (b == buffer && k == bucket) return n;
      n += (int)chunks_of(by[k]).size();
    }
  }
  return n;
}

size_t bucketed_workspace_bytes(dopt_shard_map* m, int32_t rank) {
  return kScalarBytes +
         (size_t)bucketed_region(m, rank, (int32_t)m->buffers.size(), 0) * kMaxGrid * sizeof(Partial);
}

int check_state_ptrs(const dopt_shard_map* m, int32_t buffer, const float* master,
                     const float* exp_avg, const float* exp_avg_sq, const void* param,
                     const char* fn) {
  const bool fp32 = m->buffers[buffer].param_dtype == DOPT_F32;
  if (!exp_avg || !exp_avg_sq || !param || (!fp32 && !master))
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL state or param pointer");
  if (fp32 && master)
    return dopt::fail(DOPT_E_INVALID,
                      std::string(fn) + ": master must be NULL for an fp32 buffer (the param buffer is the master)");
  if (!aligned16(exp_avg) || !aligned16(exp_avg_sq) || !aligned16(param) || (master && !aligned16(master)))
    return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": state or param pointer not 16-byte aligned");
  return DOPT_OK;
}

int check_replicas(const dopt_shard_map* m, int32_t rank, const void* const* replicas,
                   int32_t n_rep, int32_t n_inst, int32_t layout, const char* fn) {
  if (n_inst < 1 || n_rep != m->dp * n_inst || n_rep > DOPT_MAX_REPLICAS)
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": n_replicas must be DP * n_instances (at most " +
                                          std::to_string(DOPT_MAX_REPLICAS) + ")");
  if (layout != DOPT_LAYOUT_FULL_BUFFER && layout != DOPT_LAYOUT_SHARD_ONLY)
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": unknown layout");
  if (layout == DOPT_LAYOUT_SHARD_ONLY && rank == DOPT_ALL_RANKS)
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": SHARD_ONLY layout needs a single rank");
  if (!replicas) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL replica array");
  for (int k = 0; k < n_rep; ++k) {
    if (!replicas[k]) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL replica pointer");
    if (!aligned16(replicas[k]))
      return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": replica pointer not 16-byte aligned");
  }
  return DOPT_OK;
}

// Checks a dopt_step_args for the fused step (bucketed = false) or the
// bucket-staged step (bucketed = true: the workspace uses that layout).
int check_step_args(const dopt_step_args* a, bool bucketed, const char* fn) {
  if (!a) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL args");
  int st = check_map_buffer_rank(a->map, 0, a->rank, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int32_t nb = (int32_t)m->buffers.size();
  const int32_t n_rep = m->dp * a->n_instances;
  if (bucketed) {
    if (!a->workspace) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL workspace");
    if (!aligned16(a->workspace))
      return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": workspace not 16-byte aligned");
    size_t need = bucketed_workspace_bytes(m, a->rank);
    if (a->workspace_bytes < need)
      return dopt::fail(DOPT_E_SIZE, std::string(fn) + ": workspace needs " + std::to_string(need) +
                                         " bytes (dopt_workspace_bytes_bucketed), got " +
                                         std::to_string(a->workspace_bytes));
  } else if ((st = check_workspace(m, a->rank, a->workspace, a->workspace_bytes, fn))) {
    return st;
  }
  if ((st = check_hparams(&a->hp, fn))) return st;
  if ((a->d_step && (reinterpret_cast<uintptr_t>(a->d_step) & 7)) ||
      (a->d_lr && (reinterpret_cast<uintptr_t>(a->d_lr) & 7)))
    return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": d_step / d_lr not 8-byte aligned");
  if (!a->replica_grads || !a->main_grad || !a->master || !a->exp_avg || !a->exp_avg_sq || !a->param_buffer)
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL per-buffer array");
  if (!std::isfinite(a->inv_loss_scale) || !(a->remote_sumsq >= 0) || std::isnan(a->max_norm) ||
      !std::isfinite(a->grad_scale))
    return dopt::fail(DOPT_E_INVALID,
                      std::string(fn) + ": bad inv_loss_scale, grad_scale, remote_sumsq or max_norm");
  for (int32_t b = 0; b < nb; ++b) {
    if ((st = check_replicas(m, a->rank, a->replica_grads[b], n_rep, a->n_instances, a->layout, fn))) return st;
    if ((st = check_state_ptrs(m, b, a->master[b], a->exp_avg[b], a->exp_avg_sq[b], a->param_buffer[b], fn)))
      return st;
    if (!a->main_grad[b]) return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": NULL main_grad");
    if (!aligned16(a->main_grad[b])) return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": main_grad not aligned");
  }
  return DOPT_OK;
}

int check_bucket_range(const dopt_shard_map* m, int32_t buffer, int32_t first, int32_t count,
                       const char* fn) {
  if (buffer < 0 || buffer >= (int32_t)m->buffers.size())
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": buffer out of range");
  const int32_t nbk = (int32_t)m->buffers[buffer].buckets.size();
  if (first < 0 || count < 1 || first > nbk - count)
    return dopt::fail(DOPT_E_INVALID, std::string(fn) + ": bucket range out of range");
  return DOPT_OK;
}

int record_stage(const dopt_step_args* a, int i, cudaStream_t s) {
  if (!a->stage_events || !a->stage_events[i]) return DOPT_OK;
  cudaError_t e = cudaEventRecord((cudaEvent_t)a->stage_events[i], s);
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string("stage event: ") + cudaGetErrorString(e));
  return DOPT_OK;
}

}  // namespace

extern "C" {

uint64_t dopt_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int dopt_debug_starve_copy(int32_t tile) {
  if (tile < -1) return dopt::fail(DOPT_E_INVALID, "dopt_debug_starve_copy: tile < -1");
  g_starve_tile.store(tile, std::memory_order_relaxed);
  return DOPT_OK;
}

int dopt_read_step_stats(const void* workspace, dopt_step_stats* out, dopt_stream stream) {
  if (!workspace || !out) return dopt::fail(DOPT_E_INVALID, "dopt_read_step_stats: NULL workspace or out");
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(out, workspace, sizeof(dopt_step_stats), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess)
    return dopt::fail(DOPT_E_CUDA, std::string("dopt_read_step_stats: ") + cudaGetErrorString(e));
  return DOPT_OK;
}

size_t dopt_workspace_bytes(const dopt_shard_map* map, int32_t rank) {
  if (!map || (rank != DOPT_ALL_RANKS && (rank < 0 || rank >= map->dp))) {
    dopt::fail(DOPT_E_INVALID, "dopt_workspace_bytes: bad map or rank");
    return 0;
  }
  return workspace_bytes(const_cast<dopt_shard_map*>(map), rank);
}

int dopt_grad_reduce_shard(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                           const void* const* replicas, int32_t n_replicas, int32_t n_instances,
                           int32_t layout, int32_t average_in_collective, float* main_grad,
                           void* workspace, size_t workspace_bytes_, dopt_stream stream) {
  const char* fn = "dopt_grad_reduce_shard";
  int st = check_map_buffer_rank(map, buffer, rank, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(map);
  if ((st = check_replicas(m, rank, replicas, n_replicas, n_instances, layout, fn))) return st;
  if (!main_grad) return dopt::fail(DOPT_E_INVALID, "dopt_grad_reduce_shard: NULL main_grad");
  if (!aligned16(main_grad)) return dopt::fail(DOPT_E_ALIGN, "dopt_grad_reduce_shard: main_grad not aligned");
  (void)workspace;
  (void)workspace_bytes_;
  return run_k1(m, buffer, rank, replicas, n_replicas, n_instances,
                layout == DOPT_LAYOUT_FULL_BUFFER, average_in_collective, 1.0f,
                m->buffers[buffer].grad_dtype, main_grad, false, nullptr, (cudaStream_t)stream);
}

int dopt_prepare_grads(const dopt_shard_map* map, int32_t buffer, int32_t rank,
                       float inv_loss_scale, float* main_grad, void* workspace,
                       size_t workspace_bytes_, dopt_stream stream) {
  const char* fn = "dopt_prepare_grads";
  int st = check_map_buffer_rank(map, buffer, rank, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(map);
  if ((st = check_workspace(m, rank, workspace, workspace_bytes_, fn))) return st;
  if (!main_grad) return dopt::fail(DOPT_E_INVALID, "dopt_prepare_grads: NULL main_grad");
  if (!aligned16(main_grad)) return dopt::fail(DOPT_E_ALIGN, "dopt_prepare_grads: main_grad not aligned");
  if (!std::isfinite(inv_loss_scale)) return dopt::fail(DOPT_E_INVALID, "dopt_prepare_grads: bad inv_loss_scale");
  // the main grad itself is the single input, read at its own (flat) index
  const void* one[1] = {main_grad};
  return run_k1(m, buffer, rank, one, 1, 1, 0, 0, inv_loss_scale, DOPT_F32, main_grad, true,
                workspace, (cudaStream_t)stream);
}

int dopt_grad_norm(const dopt_shard_map* map, int32_t rank, void* workspace, size_t workspace_bytes_,
                   double remote_sumsq, int32_t remote_found_inf, double max_norm, float* d_norm,
                   float* d_clip_coef, int32_t* d_found_inf, dopt_stream stream) {
  const char* fn = "dopt_grad_norm";
  int st = check_map_buffer_rank(map, 0, rank, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(map);
  if ((st = check_workspace(m, rank, workspace, workspace_bytes_, fn))) return st;
  if (!(remote_sumsq >= 0) || std::isnan(max_norm))
    return dopt::fail(DOPT_E_INVALID, "dopt_grad_norm: bad remote_sumsq or max_norm");
  return run_k2(m, rank, workspace, remote_sumsq, remote_found_inf, max_norm, d_norm, d_clip_coef,
                d_found_inf, (cudaStream_t)stream);
}

int dopt_adam_step(const dopt_shard_map* map, int32_t buffer, int32_t rank, const float* main_grad,
                   float* master, float* exp_avg, float* exp_avg_sq, void* param_buffer,
                   const dopt_adamw_hparams* hp, const float* d_clip_coef,
                   const int32_t* d_found_inf, dopt_stream stream) {
  const char* fn = "dopt_adam_step";
  int st = check_map_buffer_rank(map, buffer, rank, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(map);
  if ((st = check_hparams(hp, fn))) return st;
  if ((st = check_state_ptrs(m, buffer, master, exp_avg, exp_avg_sq, param_buffer, fn))) return st;
  if (!main_grad || !d_clip_coef || !d_found_inf)
    return dopt::fail(DOPT_E_INVALID, "dopt_adam_step: NULL main_grad, clip coef or found_inf");
  if (!aligned16(main_grad)) return dopt::fail(DOPT_E_ALIGN, "dopt_adam_step: main_grad not aligned");
  return run_k3(m, buffer, rank, main_grad, master, exp_avg, exp_avg_sq, param_buffer, hp, d_clip_coef,
                d_found_inf, (cudaStream_t)stream);
}

int dopt_step_async(const dopt_step_args* a, int32_t* d_found_inf, float* d_norm) {
  int st = check_step_args(a, false, "dopt_step");
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int32_t nb = (int32_t)m->buffers.size();
  const int32_t n_rep = m->dp * a->n_instances;
  cudaStream_t s = (cudaStream_t)a->stream;
  if ((st = record_stage(a, 0, s))) return st;
  for (int32_t b = 0; b < nb; ++b) {
    st = run_k1(m, b, a->rank, a->replica_grads[b], n_rep, a->n_instances,
                a->layout == DOPT_LAYOUT_FULL_BUFFER, a->average_in_collective, a->inv_loss_scale,
                m->buffers[b].grad_dtype, a->main_grad[b], true, a->workspace, s, grad_scale_of(a));
    if (st) return st;
  }
  if ((st = record_stage(a, 1, s))) return st;
  Scalars* sc = scalars_ptr(a->workspace);
  if ((st = run_k2(m, a->rank, a->workspace, a->remote_sumsq, a->remote_found_inf, a->max_norm, d_norm,
                   nullptr, d_found_inf, s, a)))
    return st;
  if ((st = record_stage(a, 2, s))) return st;
  const DevStep* dev = a->d_step ? dev_step_ptr(a->workspace) : nullptr;
  for (int32_t b = 0; b < nb; ++b) {
    st = run_k3(m, b, a->rank, a->main_grad[b], a->master[b], a->exp_avg[b], a->exp_avg_sq[b],
                a->param_buffer[b], &a->hp, &sc->clip_coef, &sc->found_inf, s, dev);
    if (st) return st;
  }
  return record_stage(a, 3, s);
}

size_t dopt_workspace_bytes_bucketed(const dopt_shard_map* map, int32_t rank) {
  if (!map || (rank != DOPT_ALL_RANKS && (rank < 0 || rank >= map->dp))) {
    dopt::fail(DOPT_E_INVALID, "dopt_workspace_bytes_bucketed: bad map or rank");
    return 0;
  }
  return bucketed_workspace_bytes(const_cast<dopt_shard_map*>(map), rank);
}

int dopt_step_reduce_buckets(const dopt_step_args* a, int32_t buffer, int32_t bucket_first,
                             int32_t bucket_count) {
  const char* fn = "dopt_step_reduce_buckets";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  if ((st = check_bucket_range(m, buffer, bucket_first, bucket_count, fn))) return st;
  std::vector<std::vector<dopt::Run>> by = runs_by_bucket(m, buffer, a->rank);
  const int32_t n_rep = m->dp * a->n_instances;
  for (int32_t k = bucket_first; k < bucket_first + bucket_count; ++k) {
    st = run_k1_runs(by[k], bucketed_region(m, a->rank, buffer, k), a->replica_grads[buffer], n_rep,
                     a->n_instances, a->layout == DOPT_LAYOUT_FULL_BUFFER, a->average_in_collective,
                     a->inv_loss_scale, m->buffers[buffer].grad_dtype, a->main_grad[buffer], true,
                     a->workspace, (cudaStream_t)a->stream, grad_scale_of(a));
    if (st) return st;
  }
  return DOPT_OK;
}

int dopt_step_finalize(const dopt_step_args* a, int32_t* d_found_inf, float* d_norm) {
  const char* fn = "dopt_step_finalize";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int n_slots = bucketed_region(m, a->rank, (int32_t)m->buffers.size(), 0) * kMaxGrid;
  return run_k2_slots(n_slots, a->workspace, a->remote_sumsq, a->remote_found_inf, a->max_norm, d_norm,
                      nullptr, d_found_inf, (cudaStream_t)a->stream, a);
}

int dopt_step_update_buckets(const dopt_step_args* a, int32_t buffer, int32_t bucket_first,
                             int32_t bucket_count) {
  const char* fn = "dopt_step_update_buckets";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  if ((st = check_bucket_range(m, buffer, bucket_first, bucket_count, fn))) return st;
  std::vector<std::vector<dopt::Run>> by = runs_by_bucket(m, buffer, a->rank);
  std::vector<dopt::Run> runs;
  for (int32_t k = bucket_first; k < bucket_first + bucket_count; ++k)
    runs.insert(runs.end(), by[k].begin(), by[k].end());
  Scalars* sc = scalars_ptr(a->workspace);
  return run_k3_runs(runs, m->buffers[buffer].param_dtype, a->main_grad[buffer], a->master[buffer],
                     a->exp_avg[buffer], a->exp_avg_sq[buffer], a->param_buffer[buffer], &a->hp, &sc->clip_coef,
                     &sc->found_inf, (cudaStream_t)a->stream,
                     a->d_step ? dev_step_ptr(a->workspace) : nullptr);
}

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static scratch on the current device, looked up on
// the first call per device.
int noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string("dopt_step_noalloc: cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return dopt::fail(DOPT_E_INVALID, "dopt_step_noalloc: device index out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return dopt::fail(DOPT_E_CUDA, std::string("dopt_step_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DOPT_OK;
}
}  // namespace

int dopt_step_noalloc(const dopt_step_args* a, int32_t* found_inf_out, float* grad_norm_out) {
  if (!a) return dopt::fail(DOPT_E_INVALID, "dopt_step_noalloc: NULL args");
  int st = check_map_buffer_rank(a->map, 0, a->rank, "dopt_step_noalloc");
  if (st) return st;
  size_t need = workspace_bytes(const_cast<dopt_shard_map*>(a->map), a->rank);
  if (need > DOPT_NOALLOC_SCRATCH_BYTES)
    return dopt::fail(DOPT_E_SIZE, "dopt_step_noalloc: this map and rank selection need " + std::to_string(need) +
                                       " bytes of scratch; the static scratch holds " +
                                       std::to_string((size_t)DOPT_NOALLOC_SCRATCH_BYTES) + " (use dopt_step with a workspace)");
  void* scratch = nullptr;
  if ((st = noalloc_scratch(&scratch))) return st;
  dopt_step_args with_scratch = *a;
  with_scratch.workspace = scratch;
  with_scratch.workspace_bytes = DOPT_NOALLOC_SCRATCH_BYTES;
  return dopt_step(&with_scratch, found_inf_out, grad_norm_out);
}

int dopt_step(const dopt_step_args* a, int32_t* found_inf_out, float* grad_norm_out) {
  int st = dopt_step_async(a, nullptr, nullptr);
  if (st) return st;
  Scalars host{};
  cudaStream_t s = (cudaStream_t)a->stream;
  cudaError_t e = cudaMemcpyAsync(&host, a->workspace, sizeof(Scalars), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return dopt::fail(DOPT_E_CUDA, std::string("dopt_step: ") + cudaGetErrorString(e));
  if (found_inf_out) *found_inf_out = host.found_inf;
  if (grad_norm_out) *grad_norm_out = host.grad_norm;
  if (host.kernel_error)
    return dopt::fail(DOPT_E_CUDA,
                      "dopt_step: a kernel gave up waiting for its own data copies; the step was skipped");
  return DOPT_OK;
}

}  // extern "C"
