// k1.cuh -- K1, the reduce/prepare pass: the emulated reduce-scatter of N
// replica grads into the fp32 main grad, fused with prepare_grads (unscale,
// non-finite detection, zero count), the partial sums of squares of the
// grad norm and, optionally, the check of every replica's grads before the
// reduction.  Included once per grad dtype (k1_f32.cu, k1_bf16.cu,
// k1_f16.cu), each instantiating launch_k1_for<its dtype>.
//
// Three kernels, chosen per launch:
//   k1_reduce_prepare      any replica and instance count (run time)
//   k1_reduce_prepare_n    1, 2, 4 or 8 replicas per instance, one or two
//                          instances, summing or averaging (compile time)
//   k1_reduce_prepare_tma  the same with one instance, fp32 replicas, the
//                          replica tiles staged in shared memory by bulk copies
// All three compute the same values in the same order.  With 16-bit grads
// the statistics pass may keep the reduced grads in the grad dtype instead
// of the fp32 main grads (K1Params::compact).  Debug builds
// (DOPT_BOUNDS_CHECK=1) check each tile's ranges against the extents of the
// replicas, the main grad and the grad-check slots, and skip a tile outside
// them (DOPT_RANGE_OK); the default build compiles the checks out.
#pragma once

#include <type_traits>

#include "kernels.cuh"
#include "tma.cuh"

namespace dopt {

// ------------------------------------------------------- grad encodings --

// Loads of kVec grad elements are held in their raw encoding (float4 for
// fp32, two packed 16-bit pairs for bf16/fp16) until the reduction widens
// them, so a 16-bit grad keeps half the registers of an fp32 one and a
// thread can keep twice as many 16-bit accesses in flight.
//
// The grad check keeps a running maximum of |g| as integer bits: for a
// non-negative float the order of its bit pattern is the order of its
// value, +inf lies above every finite value and NaN above +inf, so the
// maximum of the bits of |g| is the largest magnitude, or +inf when there
// is an infinity, or a NaN when there is a NaN.  A thread's running maximum
// is one 32-bit word: the fp32 bits for fp32 grads, two 16-bit halves for
// bf16/fp16 (maximised half by half, as the packed loads hold them).
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
  static constexpr bool kCompact = false;  // the reduced grad is the fp32 main grad itself
  static __device__ __forceinline__ void store4c(void*, int64_t, const float*) {}
  static __device__ __forceinline__ void store1c(void*, int64_t, float) {}
  // grad check
  static __device__ __forceinline__ uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }
  static __device__ __forceinline__ uint32_t abs4(const Raw& r) {
    return max(max(abs_bits(r.x), abs_bits(r.y)), max(abs_bits(r.z), abs_bits(r.w)));
  }
  static __device__ __forceinline__ uint32_t abs1(const void* p, int64_t i) {
    return abs_bits(static_cast<const float*>(p)[i]);
  }
  static __device__ __forceinline__ uint32_t amax(uint32_t a, uint32_t b) { return max(a, b); }
  static __device__ __forceinline__ uint32_t f32_bits(uint32_t a) { return a; }
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
  // compact store of reduced grads that are bf16 values already (exact)
  static constexpr bool kCompact = true;
  static __device__ __forceinline__ void store4c(void* p, int64_t i, const float* r) {
    __stcs(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i),
           make_uint2((__float_as_uint(r[0]) >> 16) | (__float_as_uint(r[1]) & 0xFFFF0000u),
                      (__float_as_uint(r[2]) >> 16) | (__float_as_uint(r[3]) & 0xFFFF0000u)));
  }
  static __device__ __forceinline__ void store1c(void* p, int64_t i, float r) {
    static_cast<unsigned short*>(p)[i] = (unsigned short)(__float_as_uint(r) >> 16);
  }
  // grad check: halves of |g| bits; bf16 is the top half of the same fp32
  static __device__ __forceinline__ uint32_t abs4(const Raw& r) {
    return __vmaxu2(r.x & 0x7FFF7FFFu, r.y & 0x7FFF7FFFu);
  }
  static __device__ __forceinline__ uint32_t abs1(const void* p, int64_t i) {
    return static_cast<const unsigned short*>(p)[i] & 0x7FFFu;
  }
  static __device__ __forceinline__ uint32_t amax(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
  static __device__ __forceinline__ uint32_t f32_bits(uint32_t a) {
    return max(a & 0xFFFFu, a >> 16) << 16;
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
  // compact store of reduced grads that are fp16 values already (exact)
  static constexpr bool kCompact = true;
  static __device__ __forceinline__ void store4c(void* p, int64_t i, const float* r) {
    const unsigned a = __half_as_ushort(__float2half_rn(r[0])), b = __half_as_ushort(__float2half_rn(r[1]));
    const unsigned c = __half_as_ushort(__float2half_rn(r[2])), d = __half_as_ushort(__float2half_rn(r[3]));
    __stcs(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i), make_uint2(a | (b << 16), c | (d << 16)));
  }
  static __device__ __forceinline__ void store1c(void* p, int64_t i, float r) {
    static_cast<unsigned short*>(p)[i] = __half_as_ushort(__float2half_rn(r));
  }
  // grad check: halves of |g| bits, widened to fp32 bits once at the end
  // (the widening keeps the order, +inf and NaN)
  static __device__ __forceinline__ uint32_t abs4(const Raw& r) {
    return __vmaxu2(r.x & 0x7FFF7FFFu, r.y & 0x7FFF7FFFu);
  }
  static __device__ __forceinline__ uint32_t abs1(const void* p, int64_t i) {
    return static_cast<const unsigned short*>(p)[i] & 0x7FFFu;
  }
  static __device__ __forceinline__ uint32_t amax(uint32_t a, uint32_t b) { return __vmaxu2(a, b); }
  static __device__ __forceinline__ uint32_t f32_bits(uint32_t a) {
    const unsigned short h = (unsigned short)max(a & 0xFFFFu, a >> 16);
    return __float_as_uint(__half2float(__ushort_as_half(h)));
  }
};

// Merges a warp's per-lane maxima of replica k in one bucket into
// amax[k * stride + bucket] (fp32 bits of |g|; an atomic max, so the
// result does not depend on the order of the CTAs).  Called by whole warps.
template <typename GT>
__device__ __forceinline__ void amax_flush(uint32_t bits, const K1Head& p, int k, int bucket) {
  const uint32_t v = __reduce_max_sync(0xFFFFFFFFu, GradT<GT>::f32_bits(bits));
  if ((threadIdx.x & 31) == 0 && v != 0u) atomicMax(p.amax + (size_t)k * p.amax_stride + bucket, v);
}

// ------------------------------------------------------------ reduction --

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
                                            const K1Head& p) {
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

// The same arithmetic with the averaging choice known at compile time (the
// specialised kernels): a replica's term is prescaled by 1/N when the
// collective sums, taken as is when it averages; an instance's sum is
// averaged over its ranks (when averaging) and rounded to the grad dtype;
// with several instances their sum is averaged (when averaging) and
// rounded again.
template <bool AVG>
__device__ __forceinline__ float term_of(float x, float pre) {
  return AVG ? x : __fmul_rn(x, pre);
}
template <typename GT, bool AVG>
__device__ __forceinline__ float instance_value(float s, float inv_dpi) {
  return GradT<GT>::round_to(AVG ? __fmul_rn(s, inv_dpi) : s);
}
template <typename GT, bool AVG, int NINST>
__device__ __forceinline__ float across_instances(float t, float inv_ninst) {
  if (NINST == 1) return t;
  return GradT<GT>::round_to(AVG ? __fmul_rn(t, inv_ninst) : t);
}

// The reduced grad of an element in the grad dtype, after scale_gradients
// (before the unscale that makes it the fp32 main grad).
template <typename GT>
__device__ __forceinline__ float reduce_value(const ReduceState& st, const K1Head& p) {
  float total = st.total;
  if (p.n_inst > 1) {
    if (p.average) total = __fmul_rn(total, p.inv_ninst);
    total = GradT<GT>::round_to(total);
  }
  return post_scaled<GT>(total, p.post_scale);
}

// Turns kVec reduced grads v (grad-dtype values) of main-grad index i into
// fp32 main grads in place (v * inv_scale) and stores them, or, in the
// compact form, stores the reduced grads themselves in the grad dtype first
// (half the bytes; the AdamW pass forms the same main grads from them).
template <typename GT, bool STATS>
__device__ __forceinline__ void finish_store4(const K1Head& p, int64_t i, float* v) {
  if constexpr (STATS && GradT<GT>::kCompact) {
    if (p.compact) {
      GradT<GT>::store4c(p.main_grad, i, v);
#pragma unroll
      for (int j = 0; j < kVec; ++j) v[j] = __fmul_rn(v[j], p.inv_scale);
      return;
    }
  }
#pragma unroll
  for (int j = 0; j < kVec; ++j) v[j] = __fmul_rn(v[j], p.inv_scale);
  if (p.keep_main)  // a short step: the AdamW pass will find the main grads in L2
    __stcg(reinterpret_cast<float4*>(p.main_grad + i), make_float4(v[0], v[1], v[2], v[3]));
  else
    __stcs(reinterpret_cast<float4*>(p.main_grad + i), make_float4(v[0], v[1], v[2], v[3]));
}
template <typename GT, bool STATS>
__device__ __forceinline__ float finish_store1(const K1Head& p, int64_t i, float r) {
  const float m = __fmul_rn(r, p.inv_scale);
  if constexpr (STATS && GradT<GT>::kCompact) {
    if (p.compact) {
      GradT<GT>::store1c(p.main_grad, i, r);
      return m;
    }
  }
  p.main_grad[i] = m;
  return m;
}

// ---------------------------------------------------------- norm partials --

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
static __device__ __noinline__ double sumsq_wide(double d, float a, float b, float c, float e) {
  return d + (double)a * (double)a + (double)b * (double)b + (double)c * (double)c +
         (double)e * (double)e;
}
static __device__ __noinline__ double sumsq_flush(double d, float s, float c) {
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
// With CHECK, each warp folds its per-replica maxima of a tile into shared
// memory (the replica count is known only at run time), and the CTA merges
// them into the global table whenever its tiles move to another bucket.
template <typename GT, bool FULL, bool STATS, bool CHECK>
__global__ void __launch_bounds__(kThreads, DOPT_K1_MIN_BLOCKS)
k1_reduce_prepare(const __grid_constant__ K1Params p) {
  __shared__ uint32_t s_amax[DOPT_MAX_REPLICAS];
  const int dpi = p.n_rep / p.n_inst;
  SumSq acc;
  int si = 0, cur_bucket = -1;
  if constexpr (CHECK) {
    for (int k = threadIdx.x; k < DOPT_MAX_REPLICAS; k += kThreads) s_amax[k] = 0u;
    __syncthreads();
  }
  // CTA-wide: merge the shared maxima into the bucket's slots and clear them
  auto flush_bucket = [&](int bucket) {
    __syncthreads();
    if (threadIdx.x < p.n_rep) {
      const uint32_t v = s_amax[threadIdx.x];
      if (v) atomicMax(p.amax + (size_t)threadIdx.x * p.amax_stride + bucket, v);
      s_amax[threadIdx.x] = 0u;
    }
    __syncthreads();
  };
  for (int t = blockIdx.x; t < p.tab.n_tiles; t += gridDim.x) {
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    const int64_t off = (int64_t)(t - sg.tile0) * kTile1;
    const int n = (int)min((int64_t)kTile1, (int64_t)sg.len - off);
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const bool aligned = seg_aligned(sg.local, sg.world);
    if (!(DOPT_RANGE_OK(p, kSiteK1Rep, r0, n, rep) && DOPT_RANGE_OK(p, kSiteK1Main, l0, n, main) &&
          (!CHECK || DOPT_RANGE_OK(p, kSiteK1Bucket, sg.bucket, 1, buckets))))
      continue;  // debug builds only: a tile outside its buffers is skipped (CTA-uniform)
    if constexpr (CHECK) {
      if (sg.bucket != cur_bucket) {
        if (cur_bucket >= 0) flush_bucket(cur_bucket);
        cur_bucket = sg.bucket;
      }
    }

    ReduceState st[kUnroll1][kVec];
    bool vec_ok[kUnroll1];
#pragma unroll
    for (int u = 0; u < kUnroll1; ++u) vec_ok[u] = aligned && ((u * kThreads + threadIdx.x) * kVec + kVec <= n);

    // B replicas x kUnroll1 accesses of kVec elements in flight (half as
    // many with the check, whose maxima take registers too)
    constexpr int B = CHECK ? kBatch / 2 : kBatch;
    for (int k0 = 0; k0 < p.n_rep; k0 += B) {
      float x[B][kUnroll1][kVec];
#pragma unroll
      for (int kk = 0; kk < B; ++kk) {
        if (k0 + kk < p.n_rep) {
#pragma unroll
          for (int u = 0; u < kUnroll1; ++u) {
            const int e = (u * kThreads + threadIdx.x) * kVec;
            if (vec_ok[u]) GradT<GT>::widen4(p.rep[k0 + kk], r0 + e, x[kk][u]);
          }
        }
      }
#pragma unroll
      for (int kk = 0; kk < B; ++kk) {
        if (k0 + kk < p.n_rep) {
          const ReplicaPos rp = replica_pos(k0 + kk, dpi);
          uint32_t mx = 0u;
#pragma unroll
          for (int u = 0; u < kUnroll1; ++u) {
            if (vec_ok[u]) {
#pragma unroll
              for (int j = 0; j < kVec; ++j) {
                reduce_term<GT>(st[u][j], x[kk][u][j], rp, p);
                if (CHECK) mx = max(mx, GradT<float>::abs_bits(x[kk][u][j]));
              }
            }
          }
          if (CHECK) {
            mx = __reduce_max_sync(0xFFFFFFFFu, mx);
            if ((threadIdx.x & 31) == 0 && mx) atomicMax(&s_amax[k0 + kk], mx);
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
        for (int j = 0; j < kVec; ++j) m[j] = reduce_value<GT>(st[u][j], p);
        finish_store4<GT, STATS>(p, l0 + e, m);
        if (STATS) acc.add4(m);
      } else if (e < n) {
        // scalar path: the ragged end of a run, or a run whose starts are
        // not 8-element aligned
        const int cnt = min(kVec, n - e);
        for (int j = 0; j < cnt; ++j) {
          ReduceState s1;
          s1.s = 0.f;
          s1.total = 0.f;
          for (int k = 0; k < p.n_rep; ++k) {
            const float xk = GradT<GT>::widen1(p.rep[k], r0 + e + j);
            reduce_term<GT>(s1, xk, replica_pos(k, dpi), p);
            if (CHECK) {
              const uint32_t b = GradT<float>::abs_bits(xk);
              if (b) atomicMax(&s_amax[k], b);
            }
          }
          const float m = finish_store1<GT, STATS>(p, l0 + e + j, reduce_value<GT>(s1, p));
          if (STATS) acc.add1(m);
        }
      }
    }
    if (STATS) acc.maybe_flush();
  }
  allow_dependent_launch();
  if constexpr (CHECK) {
    if (cur_bucket >= 0) flush_bucket(cur_bucket);
  }
  if (STATS) {
    write_partial(acc, p.partials);
    finalize_if_last(p);
  }
}

// The common reductions: NINST instances of DPI replicas each and the
// averaging choice (AVG: average_in_collective) known at compile time.
// Same arithmetic as the general kernel, in the same order (each instance's
// replicas summed in order and rounded to the grad dtype, then the instance
// sums in order, rounded again when there is more than one), without its
// per-element selects.  Loads of one instance are in flight together.  With
// CHECK every thread keeps a running maximum per replica in registers and
// each warp merges it into the global table when its tiles move to another
// bucket.
// Up to four fp32 replicas of one instance fit in 64 registers, so four
// CTAs share an SM: twice the loads in flight of the two-CTA bound.
template <typename GT, int DPI, int NINST>
constexpr int k1n_min_blocks() {
  return (sizeof(GT) == 4 && DPI <= 4 && NINST == 1) ? DOPT_K1N_FP32_MIN_BLOCKS : DOPT_K1_MIN_BLOCKS;
}

template <typename GT, bool FULL, bool STATS, bool CHECK, bool AVG, int DPI, int NINST>
__global__ void __launch_bounds__(kThreads, (k1n_min_blocks<GT, DPI, NINST>()))
k1_reduce_prepare_n(const __grid_constant__ K1Params p) {
  constexpr int U = kUnroll1 * GradT<GT>::kUnroll;  // accesses per thread per tile
  constexpr int TILE = kThreads * kVec * U;
  SumSq acc;
  int si = 0, cur_bucket = -1;
  uint32_t amx[NINST][DPI];  // unused (and dropped by the compiler) without CHECK
#pragma unroll
  for (int j = 0; j < NINST; ++j)
#pragma unroll
    for (int k = 0; k < DPI; ++k) amx[j][k] = 0u;
  auto flush_bucket = [&](int bucket) {
#pragma unroll
    for (int j = 0; j < NINST; ++j)
#pragma unroll
      for (int k = 0; k < DPI; ++k) {
        amax_flush<GT>(amx[j][k], p, j * DPI + k, bucket);
        amx[j][k] = 0u;
      }
  };
  const float pre = p.pre;
  for (int t = blockIdx.x; t < p.tab.n_tiles; t += gridDim.x) {
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    const int64_t off = (int64_t)(t - sg.tile0) * TILE;
    const int n = (int)min((int64_t)TILE, (int64_t)sg.len - off);
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const bool aligned = seg_aligned(sg.local, sg.world);
    if (!(DOPT_RANGE_OK(p, kSiteK1Rep, r0, n, rep) && DOPT_RANGE_OK(p, kSiteK1Main, l0, n, main) &&
          (!CHECK || DOPT_RANGE_OK(p, kSiteK1Bucket, sg.bucket, 1, buckets))))
      continue;  // debug builds only: a tile outside its buffers is skipped (CTA-uniform)
    if constexpr (CHECK) {
      if (sg.bucket != cur_bucket) {
        if (cur_bucket >= 0) flush_bucket(cur_bucket);
        cur_bucket = sg.bucket;
      }
    }

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
      if (CHECK) {
        // j is a run-time index: select the instance's registers by compare
#pragma unroll
        for (int jj = 0; jj < NINST; ++jj) {
          if (jj == j) {
#pragma unroll
            for (int u = 0; u < U; ++u) {
              if (vec_ok[u]) {
#pragma unroll
                for (int k = 0; k < DPI; ++k) amx[jj][k] = GradT<GT>::amax(amx[jj][k], GradT<GT>::abs4(x[k][u]));
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float sum = term_of<AVG>(GradT<GT>::at(x[0][u], q), pre);
#pragma unroll
          for (int k = 1; k < DPI; ++k) sum = __fadd_rn(sum, term_of<AVG>(GradT<GT>::at(x[k][u], q), pre));
          sum = instance_value<GT, AVG>(sum, p.inv_dpi);
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
          float tt = across_instances<GT, AVG, NINST>(total[u][q], p.inv_ninst);
          m[q] = post_scaled<GT>(tt, p.post_scale);
        }
        finish_store4<GT, STATS>(p, l0 + e, m);
        if (STATS) acc.add4(m);
      } else if (e < n) {
        const int cnt = min(kVec, n - e);
        for (int q = 0; q < cnt; ++q) {
          float tt = 0.f;
#pragma unroll
          for (int j = 0; j < NINST; ++j) {
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < DPI; ++k) {
              const int64_t i = r0 + e + q;
              const float term = term_of<AVG>(GradT<GT>::widen1(p.rep[j * DPI + k], i), pre);
              sum = k == 0 ? term : __fadd_rn(sum, term);
              if (CHECK) amx[j][k] = GradT<GT>::amax(amx[j][k], GradT<GT>::abs1(p.rep[j * DPI + k], i));
            }
            sum = instance_value<GT, AVG>(sum, p.inv_dpi);
            tt = (j == 0) ? sum : __fadd_rn(tt, sum);
          }
          tt = across_instances<GT, AVG, NINST>(tt, p.inv_ninst);
          const float m = finish_store1<GT, STATS>(p, l0 + e + q, post_scaled<GT>(tt, p.post_scale));
          if (STATS) acc.add1(m);
        }
      }
    }
    if (STATS) acc.maybe_flush();
  }
  allow_dependent_launch();
  if constexpr (CHECK) {
    if (cur_bucket >= 0) flush_bucket(cur_bucket);
  }
  if (STATS) {
    write_partial(acc, p.partials);
    finalize_if_last(p);
  }
}

// ------------------------------------------------- K1 for short launches --
//
// fp32 replicas of one instance in a launch too short for the bulk-copy
// pipeline: one access of kVec elements per thread per tile (kShortTile
// elements), with the loads of a CTA's next tile issued before the current
// tile's arithmetic (software pipelining across tiles, as in the AdamW
// pass), so every CTA keeps two tiles of replica reads in flight and the
// last round of tiles is short.  Same arithmetic, in the same order, as
// the other kernels.

template <int DPI>
struct ShortTile {
  float4 x[DPI];
  int64_t l0, r0;
  int n;
  bool aligned;
};

template <bool FULL, int DPI, typename P>
__device__ __forceinline__ void short_load(const P& p, int& si, int t, ShortTile<DPI>& T) {
  si = seek(p.tab, si, t);
  const Seg& sg = p.tab.seg[si];
  const int64_t off = (int64_t)(t - sg.tile0) * kShortTile;
  T.n = (int)min((int64_t)kShortTile, (int64_t)sg.len - off);
  T.l0 = sg.local + off;
  T.r0 = FULL ? sg.world + off : T.l0;
  T.aligned = seg_aligned(sg.local, sg.world);
  if (!(DOPT_RANGE_OK(p, kSiteK1Rep, T.r0, T.n, rep) && DOPT_RANGE_OK(p, kSiteK1Main, T.l0, T.n, main)))
    T.n = 0;  // debug builds only: a tile outside its buffers is skipped
  const int e = threadIdx.x * kVec;
  if (T.aligned && e + kVec <= T.n) {
#pragma unroll
    for (int k = 0; k < DPI; ++k) T.x[k] = GradT<float>::load4(p.rep[k], T.r0 + e);
  }
}

template <int DPI>
constexpr int k1s_min_blocks() {
  return DPI <= 4 ? 4 : 2;
}

template <bool FULL, bool STATS, bool AVG, int DPI, int CAP = kMaxSeg>
__global__ void __launch_bounds__(kThreads, (k1s_min_blocks<DPI>()))
k1_reduce_prepare_short(const __grid_constant__ K1ParamsT<CAP> p) {
  SumSq acc;
  const float pre = p.pre;
  int si = 0;
  int t = blockIdx.x;
  if (t < p.tab.n_tiles) {
    ShortTile<DPI> cur;
    short_load<FULL, DPI>(p, si, t, cur);
    for (; t < p.tab.n_tiles; t += gridDim.x) {
      const bool more = t + (int)gridDim.x < p.tab.n_tiles;
      ShortTile<DPI> nxt;
      if (more) short_load<FULL, DPI>(p, si, t + gridDim.x, nxt);
      const int e = threadIdx.x * kVec;
      if (cur.aligned && e + kVec <= cur.n) {
        float m[kVec];
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float sum = term_of<AVG>(GradT<float>::at(cur.x[0], q), pre);
#pragma unroll
          for (int k = 1; k < DPI; ++k) sum = __fadd_rn(sum, term_of<AVG>(GradT<float>::at(cur.x[k], q), pre));
          m[q] = post_scaled<float>(instance_value<float, AVG>(sum, p.inv_dpi), p.post_scale);
        }
        finish_store4<float, STATS>(p, cur.l0 + e, m);
        if (STATS) acc.add4(m);
      } else if (e < cur.n) {
        // the ragged end of a run, or a run whose starts are not 8-element aligned
        const int cnt = min(kVec, cur.n - e);
        for (int q = 0; q < cnt; ++q) {
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < DPI; ++k) {
            const float term = term_of<AVG>(GradT<float>::widen1(p.rep[k], cur.r0 + e + q), pre);
            sum = k == 0 ? term : __fadd_rn(sum, term);
          }
          const float m = finish_store1<float, STATS>(p, cur.l0 + e + q,
                                                      post_scaled<float>(instance_value<float, AVG>(sum, p.inv_dpi),
                                                                         p.post_scale));
          if (STATS) acc.add1(m);
        }
      }
      if (STATS) acc.maybe_flush();
      if (more) cur = nxt;
    }
  }
  allow_dependent_launch();
  if (STATS) {
    write_partial(acc, p.partials);
    finalize_if_last(p);
  }
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

template <typename GT>
struct GradBits {
  using T = typename std::conditional<std::is_same<GT, float>::value, float, unsigned short>::type;
};

template <typename GT, int DPI>
__host__ __device__ constexpr size_t tma_smem_bytes() {
  return (size_t)DOPT_TMA_STAGES * DPI * kTmaTile * sizeof(typename GradBits<GT>::T) +
         DOPT_TMA_STAGES * sizeof(uint64_t);
}

template <typename GT, bool FULL, bool STATS, bool CHECK, bool AVG, int DPI>
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
    // debug builds: a tile outside the replicas is not copied, and its stage
    // completes on the arrival alone
    const bool copy_ok = DOPT_RANGE_OK(p, kSiteTmaCopy, r0, n, rep);
    mbar_arrive_expect_tx(&bars[stage], copy_ok ? (unsigned)(nv * sizeof(E)) * DPI : 0u);
#if DOPT_BOUNDS_CHECK
    const bool starved = blockIdx.x == 0 && i == p.starve_tile;  // test hook of the debug build
#else
    constexpr bool starved = false;
#endif
    if (copy_ok && nv > 0 && !starved) {
#pragma unroll
      for (int k = 0; k < DPI; ++k)
        bulk_load(tiles + ((size_t)stage * DPI + k) * kTmaTile, static_cast<const E*>(p.rep[k]) + r0,
                  (unsigned)(nv * sizeof(E)), &bars[stage]);
    }
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(S, my); ++i) issue(i);

  SumSq acc;
  int si = 0, cur_bucket = -1;
  uint32_t amx[DPI];  // unused (and dropped by the compiler) without CHECK
#pragma unroll
  for (int k = 0; k < DPI; ++k) amx[k] = 0u;
  auto flush_bucket = [&](int bucket) {
#pragma unroll
    for (int k = 0; k < DPI; ++k) {
      amax_flush<GT>(amx[k], p, k, bucket);
      amx[k] = 0u;
    }
  };
  bool failed = false;
  const float pre = p.pre;
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
    const int64_t l0 = sg.local + off;
    const int64_t r0 = FULL ? sg.world + off : l0;
    const int n_run = (int)min((int64_t)kTmaTile, (int64_t)sg.len - off);
    // debug builds: a tile outside its buffers gets no elements (no access)
    const int n = (DOPT_RANGE_OK(p, kSiteK1Rep, r0, n_run, rep) && DOPT_RANGE_OK(p, kSiteK1Main, l0, n_run, main) &&
                   (!CHECK || DOPT_RANGE_OK(p, kSiteK1Bucket, sg.bucket, 1, buckets)))
                      ? n_run
                      : 0;
    const int nv = n & ~(VALIGN - 1);
    const E* st = tiles + (size_t)stage * DPI * kTmaTile;
    if constexpr (CHECK) {
      if (sg.bucket != cur_bucket) {
        if (cur_bucket >= 0) flush_bucket(cur_bucket);
        cur_bucket = sg.bucket;
      }
    }
#pragma unroll
    for (int u = 0; u < kTmaTile / (kThreads * kVec); ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (e + kVec <= nv) {
        float m[kVec];
        typename GradT<GT>::Raw x[DPI];
#pragma unroll
        for (int k = 0; k < DPI; ++k)
          x[k] = *reinterpret_cast<const typename GradT<GT>::Raw*>(st + (size_t)k * kTmaTile + e);
        if (CHECK) {
#pragma unroll
          for (int k = 0; k < DPI; ++k) amx[k] = GradT<GT>::amax(amx[k], GradT<GT>::abs4(x[k]));
        }
#pragma unroll
        for (int q = 0; q < kVec; ++q) {
          float sum = term_of<AVG>(GradT<GT>::at(x[0], q), pre);
#pragma unroll
          for (int k = 1; k < DPI; ++k) sum = __fadd_rn(sum, term_of<AVG>(GradT<GT>::at(x[k], q), pre));
          m[q] = post_scaled<GT>(instance_value<GT, AVG>(sum, p.inv_dpi), p.post_scale);
        }
        finish_store4<GT, STATS>(p, l0 + e, m);
        if (STATS) acc.add4(m);
      } else if (e < n) {
        // the last few elements of a run: not in the staged copy
        const int cnt = min(kVec, n - e);
        for (int q = 0; q < cnt; ++q) {
          float sum = 0.f;
#pragma unroll
          for (int k = 0; k < DPI; ++k) {
            const float term = term_of<AVG>(GradT<GT>::widen1(p.rep[k], r0 + e + q), pre);
            sum = k == 0 ? term : __fadd_rn(sum, term);
            if (CHECK) amx[k] = GradT<GT>::amax(amx[k], GradT<GT>::abs1(p.rep[k], r0 + e + q));
          }
          const float m =
              finish_store1<GT, STATS>(p, l0 + e + q, post_scaled<GT>(instance_value<GT, AVG>(sum, p.inv_dpi), p.post_scale));
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
  allow_dependent_launch();
  if constexpr (CHECK) {
    if (cur_bucket >= 0) flush_bucket(cur_bucket);
  }
  if (STATS) {
    write_partial(acc, p.partials);
    finalize_if_last(p);
  }
}

// ------------------------------------------------------------ launchers --

template <typename K, typename P>
int launch_plain(K kern, const P& kp, cudaStream_t s, const char* what) {
  int grid = 0;
  int st = grid_for(kern, kp.tab.n_tiles, &grid);
  if (st) return st;
  kern<<<grid, kThreads, 0, s>>>(kp);
  return check_launch(what);
}

template <typename GT, bool FULL, bool STATS, bool CHECK, bool AVG, int DPI>
int launch_tma(K1Params& kp, cudaStream_t s) {
  auto kern = k1_reduce_prepare_tma<GT, FULL, STATS, CHECK, AVG, DPI>;
  const size_t smem = tma_smem_bytes<GT, DPI>();
  static std::atomic<uint64_t> attr_set{0};
  int st = allow_dynamic_smem(kern, smem, attr_set, "k1 tma");
  if (st) return st;
  int grid = 0;
  st = grid_for(kern, kp.tab.n_tiles, &grid, smem);
  if (st) return st;
  kern<<<grid, kThreads, smem, s>>>(kp);
  return check_launch("k1_reduce_prepare_tma launch");
}

// The specialised kernels cover one instance of 1, 2, 4 or 8 replicas, or
// two instances of 4 or 8, summing or averaging (AVG must match the
// launch's average_in_collective); fp32 replicas in a single instance whose
// runs are all 8-element aligned are staged by TMA (16-bit replicas stream
// faster through registers: packed loads, four accesses per thread).
// Everything else runs the general kernel.
template <typename GT, bool FULL, bool STATS, bool CHECK, bool AVG>
int launch_k1_sel(K1Params& kp, const K1Launch& l, cudaStream_t s) {
  const int dpi = kp.n_rep / kp.n_inst;
  const bool special = (kp.average != 0) == AVG &&
                       ((kp.n_inst == 1 && (dpi == 1 || dpi == 2 || dpi == 4 || dpi == 8)) ||
                        (kp.n_inst == 2 && (dpi == 4 || dpi == 8)));
  bool all_aligned = true;
  for (int k = 0; k < l.count; ++k) all_aligned &= seg_aligned(l.runs[k].local, l.runs[k].world);
  constexpr bool kTmaKind = DOPT_K1_TMA && STATS && std::is_same<GT, float>::value;
  // fp32 replicas of one instance in a launch too short to give every CTA
  // several bulk-copied tiles stream through registers instead: there the
  // copy pipeline's fill and drain and the uneven last round of tiles cost
  // more than the staging saves
  constexpr bool kF32 = std::is_same<GT, float>::value;
  bool shrt = false;
  if (kF32 && special && kp.n_inst == 1) {
    fill_table(kp.tab, l.runs, l.count, kTmaTile, l.bucket_base);
    int sms = 0;
    if (int st = device_sms(&sms)) return st;
    shrt = kp.tab.n_tiles < kTmaMinTilesPerSm * sms;
  }
  const bool tma = kTmaKind && kp.error_flag && special && kp.n_inst == 1 && all_aligned && !shrt;
  if constexpr (kF32 && !CHECK) {
    if (shrt && DOPT_K1_SHORT_PIPE) {
      fill_table(kp.tab, l.runs, l.count, kShortTile, l.bucket_base);
      const char* w = "k1_reduce_prepare_short launch";
      if constexpr (STATS) {  // the steps' statistics pass: the compact parameter block when it fits
        if (kp.tab.n_seg <= kSmallSeg) {
          const K1ParamsT<kSmallSeg> sp = with_table_of<kSmallSeg, K1Head>(kp);
          switch (dpi) {
            case 1: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 1, kSmallSeg>, sp, s, w);
            case 2: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 2, kSmallSeg>, sp, s, w);
            case 4: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 4, kSmallSeg>, sp, s, w);
            default: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 8, kSmallSeg>, sp, s, w);
          }
        }
      }
      switch (dpi) {
        case 1: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 1>, kp, s, w);
        case 2: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 2>, kp, s, w);
        case 4: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 4>, kp, s, w);
        default: return launch_plain(k1_reduce_prepare_short<FULL, STATS, AVG, 8>, kp, s, w);
      }
    }
  }
  const int tile = tma ? kTmaTile : special ? kThreads * kVec * kUnroll1 * GradT<GT>::kUnroll : kTile1;
  fill_table(kp.tab, l.runs, l.count, tile, l.bucket_base);
  if constexpr (kTmaKind) {
    if (tma) {
      switch (dpi) {
        case 1: return launch_tma<GT, FULL, STATS, CHECK, AVG, 1>(kp, s);
        case 2: return launch_tma<GT, FULL, STATS, CHECK, AVG, 2>(kp, s);
        case 4: return launch_tma<GT, FULL, STATS, CHECK, AVG, 4>(kp, s);
        default: return launch_tma<GT, FULL, STATS, CHECK, AVG, 8>(kp, s);
      }
    }
  }
  const char* what = "k1_reduce_prepare_n launch";
  if (special && kp.n_inst == 1) {
    switch (dpi) {
      case 1: return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 1, 1>, kp, s, what);
      case 2: return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 2, 1>, kp, s, what);
      case 4: return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 4, 1>, kp, s, what);
      default: return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 8, 1>, kp, s, what);
    }
  }
  if (special) {
    if (dpi == 4) return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 4, 2>, kp, s, what);
    return launch_plain(k1_reduce_prepare_n<GT, FULL, STATS, CHECK, AVG, 8, 2>, kp, s, what);
  }
  return launch_plain(k1_reduce_prepare<GT, FULL, STATS, CHECK>, kp, s, "k1_reduce_prepare launch");
}

template <typename GT, bool STATS, bool CHECK, bool AVG>
int launch_k1_layout(K1Params& kp, const K1Launch& l, cudaStream_t s) {
  return l.full ? launch_k1_sel<GT, true, STATS, CHECK, AVG>(kp, l, s)
                : launch_k1_sel<GT, false, STATS, CHECK, AVG>(kp, l, s);
}

// The grad check rides on the statistics pass only (the fused and
// bucket-staged steps); the plain reduction has no check, and averaging in
// it takes the general kernel.
template <typename GT>
int launch_k1_for(K1Params& kp, const K1Launch& l, cudaStream_t s) {
  if (l.check && !l.stats) return fail(DOPT_E_INVALID, "the grad check needs the statistics pass");
  if (!l.stats) return launch_k1_layout<GT, false, false, false>(kp, l, s);
  if (kp.average)
    return l.check ? launch_k1_layout<GT, true, true, true>(kp, l, s) : launch_k1_layout<GT, true, false, true>(kp, l, s);
  return l.check ? launch_k1_layout<GT, true, true, false>(kp, l, s) : launch_k1_layout<GT, true, false, false>(kp, l, s);
}

}  // namespace dopt
