// k3.cu -- K3, the AdamW pass: reads the fp32 main grad, master weight, m
// and v of every shard element once, applies the clip coefficient and the
// AdamW update (torch semantics, fp32), writes master, m and v back and
// casts the new master into the bf16/fp16 param buffer at the element's
// buffer offset (the stand-in for the param all-gather).  An fp32 param
// buffer is its own master and is stepped in place.  A step the finalize
// pass marked as skipped writes nothing.  Debug builds (DOPT_BOUNDS_CHECK=1)
// check each tile against the extents of the main grad, master/m/v and the
// param buffer and skip a tile outside them.
#include "kernels.cuh"

namespace dopt {

// The AdamW pass's result stores: streaming (evict-first) by default;
// DOPT_K3_STORE_HINT 1 caches them in L2 only, 2 uses plain write-back stores.
template <typename T>
__device__ __forceinline__ void st_out(T* p, const T& v) {
#if DOPT_K3_STORE_HINT == 1
  __stcg(p, v);
#elif DOPT_K3_STORE_HINT == 2
  *p = v;
#else
  __stcs(p, v);
#endif
}

template <typename PT>
struct ParamT;
template <>
struct ParamT<__nv_bfloat16> {
  static constexpr bool kInPlace = false;
  static __device__ __forceinline__ uint2 pack4(const float* x) {
    unsigned short h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __bfloat16_as_ushort(__float2bfloat16_rn(x[j]));
    return make_uint2((unsigned)h[0] | ((unsigned)h[1] << 16), (unsigned)h[2] | ((unsigned)h[3] << 16));
  }
  static __device__ __forceinline__ void store4(void* p, int64_t i, const float* x) {
    st_out(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i), pack4(x));
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<unsigned short*>(p)[i] = __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
};
template <>
struct ParamT<__half> {
  static constexpr bool kInPlace = false;
  static __device__ __forceinline__ uint2 pack4(const float* x) {
    unsigned short h[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) h[j] = __half_as_ushort(__float2half_rn(x[j]));
    return make_uint2((unsigned)h[0] | ((unsigned)h[1] << 16), (unsigned)h[2] | ((unsigned)h[3] << 16));
  }
  static __device__ __forceinline__ void store4(void* p, int64_t i, const float* x) {
    st_out(reinterpret_cast<uint2*>(static_cast<unsigned short*>(p) + i), pack4(x));
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<unsigned short*>(p)[i] = __half_as_ushort(__float2half_rn(x));
  }
};
template <>
struct ParamT<float> {
  static constexpr bool kInPlace = true;  // the fp32 param buffer is the master
  static __device__ __forceinline__ uint2 pack4(const float*) { return make_uint2(0u, 0u); }
  static __device__ __forceinline__ void store4(void*, int64_t, const float*) {}
  static __device__ __forceinline__ void store1(void*, int64_t, float) {}
};

// How the main grads reach K3: fp32 main grads, or (16-bit grad buffers in
// the fused and bucket-staged steps) the reduced grads in the grad dtype,
// from which main = fp32(stored) * inv_scale is formed exactly as K1 formed
// it -- the same fp32 value, from half the bytes.
template <typename MG>
struct MainT;
template <>
struct MainT<float> {
  using Raw = float4;
  static __device__ __forceinline__ Raw load4(const float* p, int64_t i) {
    return __ldcs(reinterpret_cast<const float4*>(p + i));
  }
  static __device__ __forceinline__ void widen4(const Raw& r, float, float* g) {
    g[0] = r.x; g[1] = r.y; g[2] = r.z; g[3] = r.w;
  }
  static __device__ __forceinline__ float load1(const float* p, int64_t i, float) { return p[i]; }
};
template <>
struct MainT<__nv_bfloat16> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw load4(const float* p, int64_t i) {
    return __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ void widen4(const Raw& r, float inv_scale, float* g) {
    g[0] = __fmul_rn(__uint_as_float(r.x << 16), inv_scale);
    g[1] = __fmul_rn(__uint_as_float(r.x & 0xFFFF0000u), inv_scale);
    g[2] = __fmul_rn(__uint_as_float(r.y << 16), inv_scale);
    g[3] = __fmul_rn(__uint_as_float(r.y & 0xFFFF0000u), inv_scale);
  }
  static __device__ __forceinline__ float load1(const float* p, int64_t i, float inv_scale) {
    const unsigned short b = reinterpret_cast<const unsigned short*>(p)[i];
    return __fmul_rn(__uint_as_float((unsigned)b << 16), inv_scale);
  }
};
template <>
struct MainT<__half> {
  using Raw = uint2;
  static __device__ __forceinline__ Raw load4(const float* p, int64_t i) {
    return __ldcs(reinterpret_cast<const uint2*>(reinterpret_cast<const unsigned short*>(p) + i));
  }
  static __device__ __forceinline__ float h(unsigned bits) {
    return __half2float(__ushort_as_half((unsigned short)bits));
  }
  static __device__ __forceinline__ void widen4(const Raw& r, float inv_scale, float* g) {
    g[0] = __fmul_rn(h(r.x & 0xFFFFu), inv_scale);
    g[1] = __fmul_rn(h(r.x >> 16), inv_scale);
    g[2] = __fmul_rn(h(r.y & 0xFFFFu), inv_scale);
    g[3] = __fmul_rn(h(r.y >> 16), inv_scale);
  }
  static __device__ __forceinline__ float load1(const float* p, int64_t i, float inv_scale) {
    return __fmul_rn(h(reinterpret_cast<const unsigned short*>(p)[i]), inv_scale);
  }
};

// The decoupled weight-decay factor (float)(1 - lr*wd*wd_mult), formed in
// fp64; out of line so no fp64 instruction is issued per element -- it runs
// once per run change.
static __device__ __noinline__ float decay_of(double lr_wd, double wd_mult) {
  return (float)(1.0 - lr_wd * wd_mult);
}

struct StepScalars {
  float step_size, bc2_sqrt;
  double lr_wd;
};

__device__ __forceinline__ StepScalars step_scalars(const K3Head& p) {
  if (p.dev) return StepScalars{p.dev->step_size, p.dev->bc2_sqrt, p.dev->lr_wd};
  return StepScalars{p.step_size, p.bc2_sqrt, p.lr_wd};
}

// One element of AdamW (torch semantics: decay the weight, update m and v,
// divide the bias-corrected sqrt(v) + eps into m, step), each operation
// rounded once in fp32.
__device__ __forceinline__ void adamw1(float g, float decay, const K3Head& p, const StepScalars& ss,
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
template <typename MG>
struct K3Tile {
  typename MainT<MG>::Raw g[kUnroll3];
  float4 w[kUnroll3], m[kUnroll3], v[kUnroll3];
  int64_t l0, w0, m0;
  int n;
  float decay;
  bool aligned;
};

// Where tile t lies: its run, its element count and its first element in
// the flat shard (l0), in the param buffer (w0) and in the master array (m0:
// the param buffer itself for fp32 params).  No loads.
template <typename PT, typename MG, typename P>
__device__ __forceinline__ void k3_place(const P& p, int t, int& si, K3Tile<MG>& T) {
  si = seek(p.tab, si, t);
  const Seg& sg = p.tab.seg[si];
  const int64_t off = (int64_t)(t - sg.tile0) * kTile3;
  T.n = (int)min((int64_t)kTile3, (int64_t)sg.len - off);
  T.l0 = sg.local + off;
  T.w0 = sg.world + off;
  T.m0 = ParamT<PT>::kInPlace ? T.w0 : T.l0;
  // debug builds: a tile outside its buffers gets no elements (no access)
  if (!(DOPT_RANGE_OK(p, kSiteK3Main, T.l0, T.n, main) && DOPT_RANGE_OK(p, kSiteK3State, T.l0, T.n, state) &&
        (ParamT<PT>::kInPlace ? DOPT_RANGE_OK(p, kSiteK3Master, T.m0, T.n, param)
                              : DOPT_RANGE_OK(p, kSiteK3Master, T.m0, T.n, state) &&
                                    DOPT_RANGE_OK(p, kSiteK3Param, T.w0, T.n, param))))
    T.n = 0;
  T.aligned = seg_aligned(sg.local, sg.world);
}

// The weight-decay factor of the tile's run (recomputed only when the run
// changes).
template <typename MG, typename P>
__device__ __forceinline__ void k3_decay(const P& p, int si, K3Tile<MG>& T, int& decay_si, float& decay,
                                         double lr_wd) {
  if (si != decay_si) {
    decay = decay_of(lr_wd, p.tab.seg[si].wd_mult);
    decay_si = si;
  }
  T.decay = decay;
}

// The tile's master weights (or fp32 params), m and v.
template <typename MG>
__device__ __forceinline__ void k3_load_state(const K3Head& p, const float* wbase, K3Tile<MG>& T) {
#pragma unroll
  for (int u = 0; u < kUnroll3; ++u) {
    const int e = (u * kThreads + threadIdx.x) * kVec;
    if (T.aligned && e + kVec <= T.n) {
      T.w[u] = __ldcs(reinterpret_cast<const float4*>(wbase + T.m0 + e));
      T.m[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg + T.l0 + e));
      T.v[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg_sq + T.l0 + e));
    }
  }
}

// The tile's main grads.
template <typename MG>
__device__ __forceinline__ void k3_load_grad(const K3Head& p, K3Tile<MG>& T) {
#pragma unroll
  for (int u = 0; u < kUnroll3; ++u) {
    const int e = (u * kThreads + threadIdx.x) * kVec;
    if (T.aligned && e + kVec <= T.n) T.g[u] = MainT<MG>::load4(p.main_grad, T.l0 + e);
  }
}

template <typename PT, typename MG, typename P>
__device__ __forceinline__ void k3_load(const P& p, const float* wbase, int t, int& si, K3Tile<MG>& T,
                                        int& decay_si, float& decay, double lr_wd) {
  k3_place<PT, MG>(p, t, si, T);
  k3_decay<MG>(p, si, T, decay_si, decay, lr_wd);
  k3_load_grad<MG>(p, T);
  k3_load_state<MG>(p, wbase, T);
}

template <typename PT, typename MG, int CAP>
__global__ void __launch_bounds__(kThreads, DOPT_K3_MIN_BLOCKS) k3_adamw_pipe(const __grid_constant__ K3ParamsT<CAP> p) {
  float* const wbase = ParamT<PT>::kInPlace ? static_cast<float*>(p.param) : p.master;
  int si = 0;
  int t = blockIdx.x;
  K3Tile<MG> cur;
  // the first tile's master, m and v, which the launch before this one does
  // not write, are loaded while that launch ends (its last CTA finalizes)
  const bool early = p.early_state && t < p.tab.n_tiles;
  if (early) {
    k3_place<PT, MG>(p, t, si, cur);
    k3_load_state<MG>(p, wbase, cur);
  }
  wait_for_prior_grids();    // the reduce pass and its finalize are done
  if (*p.found_inf) return;  // skipped step: nothing is written
  const float c = *p.coef;
  const StepScalars ss = step_scalars(p);
  int decay_si = -1;
  float decay = 1.f;
  if (t >= p.tab.n_tiles) return;
  if (early) {
    k3_decay<MG>(p, si, cur, decay_si, decay, ss.lr_wd);
    k3_load_grad<MG>(p, cur);
  } else {
    k3_load<PT, MG>(p, wbase, t, si, cur, decay_si, decay, ss.lr_wd);
  }
  for (; t < p.tab.n_tiles; t += gridDim.x) {
    K3Tile<MG> nxt;
    const bool more = t + (int)gridDim.x < p.tab.n_tiles;
    if (more) k3_load<PT, MG>(p, wbase, t + gridDim.x, si, nxt, decay_si, decay, ss.lr_wd);
#pragma unroll
    for (int u = 0; u < kUnroll3; ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (cur.aligned && e + kVec <= cur.n) {
        float g[kVec];
        MainT<MG>::widen4(cur.g[u], p.inv_scale, g);
        float w[kVec] = {cur.w[u].x, cur.w[u].y, cur.w[u].z, cur.w[u].w};
        float m[kVec] = {cur.m[u].x, cur.m[u].y, cur.m[u].z, cur.m[u].w};
        float v[kVec] = {cur.v[u].x, cur.v[u].y, cur.v[u].z, cur.v[u].w};
#pragma unroll
        for (int j = 0; j < kVec; ++j) adamw1(__fmul_rn(g[j], c), cur.decay, p, ss, w[j], m[j], v[j]);
        st_out(reinterpret_cast<float4*>(wbase + cur.m0 + e), make_float4(w[0], w[1], w[2], w[3]));
        st_out(reinterpret_cast<float4*>(p.exp_avg + cur.l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        st_out(reinterpret_cast<float4*>(p.exp_avg_sq + cur.l0 + e), make_float4(v[0], v[1], v[2], v[3]));
        ParamT<PT>::store4(p.param, cur.w0 + e, w);
      } else if (e < cur.n) {
        const int cnt = min(kVec, cur.n - e);
        for (int j = 0; j < cnt; ++j) {
          float ww = wbase[cur.m0 + e + j], mm = p.exp_avg[cur.l0 + e + j], vv = p.exp_avg_sq[cur.l0 + e + j];
          adamw1(__fmul_rn(MainT<MG>::load1(p.main_grad, cur.l0 + e + j, p.inv_scale), c), cur.decay, p, ss,
                 ww, mm, vv);
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


template <typename PT, typename MG, int CAP>
int launch_k3_cap(const K3ParamsT<CAP>& kp, cudaStream_t s) {
  auto kern = k3_adamw_pipe<PT, MG, CAP>;
  int grid = 0;
  int st = grid_for(kern, kp.tab.n_tiles, &grid);
  if (st) return st;
  // programmatic stream serialization: the CTAs may start while the reduce
  // pass before it finishes (each waits in wait_for_prior_grids)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = DOPT_K3_PDL;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, kp);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // reported here, not left for the next call to find
    return fail(DOPT_E_CUDA, std::string("k3_adamw launch: ") + cudaGetErrorString(e));
  }
  return check_launch("k3_adamw launch");
}

// With the compact parameter block when the launch's runs fit in it.
template <typename PT, typename MG>
int launch_k3_t(const K3Params& kp, cudaStream_t s) {
  if (kp.tab.n_seg <= kSmallSeg) return launch_k3_cap<PT, MG, kSmallSeg>(with_table_of<kSmallSeg, K3Head>(kp), s);
  return launch_k3_cap<PT, MG, kMaxSeg>(kp, s);
}

// Param and grad dtypes pair up as the buffers allow: a 16-bit param buffer
// has grads in its own dtype or in fp32, an fp32 param buffer fp32 grads.
int launch_k3(int32_t param_dtype, int32_t main_dtype, K3Params& kp, const Run* runs, int count,
              cudaStream_t s) {
  const bool compact = main_dtype != DOPT_F32;
  if (compact && main_dtype != param_dtype)
    return fail(DOPT_E_INVALID, "compact main grads need the grad dtype of the param buffer");
  fill_table(kp.tab, runs, count, kTile3, -1);
  switch (param_dtype) {
    case DOPT_BF16:
      return compact ? launch_k3_t<__nv_bfloat16, __nv_bfloat16>(kp, s) : launch_k3_t<__nv_bfloat16, float>(kp, s);
    case DOPT_F16:
      return compact ? launch_k3_t<__half, __half>(kp, s) : launch_k3_t<__half, float>(kp, s);
    default:
      return launch_k3_t<float, float>(kp, s);
  }
}

}  // namespace dopt
