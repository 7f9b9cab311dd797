// k3.cu -- K3, the AdamW pass: reads the fp32 main grad, master weight, m
// and v of every shard element once, applies the clip coefficient and the
// AdamW update (torch semantics, fp32), writes master, m and v back and
// casts the new master into the bf16/fp16 param buffer at the element's
// buffer offset (the stand-in for the param all-gather).  An fp32 param
// buffer is its own master and is stepped in place.  A step the finalize
// pass marked as skipped writes nothing.
#include "kernels.cuh"
#include "tma.cuh"

namespace dopt {

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

// How the main grads reach K3: fp32 main grads, or (16-bit grad buffers in
// the fused and bucket-staged steps) the reduced grads in the grad dtype,
// from which main = fp32(stored) * inv_scale is formed exactly as K1 formed
// it -- the same fp32 value, from half the bytes.
template <typename MG>
struct MainT;
template <>
struct MainT<float> {
  using Elem = float;
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
  using Elem = unsigned short;
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
  using Elem = unsigned short;
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
template <typename MG>
struct K3Tile {
  typename MainT<MG>::Raw g[kUnroll3];
  float4 w[kUnroll3], m[kUnroll3], v[kUnroll3];
  int64_t l0, w0, m0;
  int n;
  float decay;
  bool aligned;
};

template <typename PT, typename MG>
__device__ __forceinline__ void k3_load(const K3Params& p, float* wbase, int t, int& si, K3Tile<MG>& T,
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
      T.g[u] = MainT<MG>::load4(p.main_grad, T.l0 + e);
      T.w[u] = __ldcs(reinterpret_cast<const float4*>(wbase + T.m0 + e));
      T.m[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg + T.l0 + e));
      T.v[u] = __ldcs(reinterpret_cast<const float4*>(p.exp_avg_sq + T.l0 + e));
    }
  }
}

template <typename PT, typename MG>
__global__ void __launch_bounds__(kThreads, DOPT_K3_MIN_BLOCKS) k3_adamw_pipe(const __grid_constant__ K3Params p) {
  if (*p.found_inf) return;  // skipped step: nothing is written
  const float c = *p.coef;
  const StepScalars ss = step_scalars(p);
  float* const wbase = ParamT<PT>::kInPlace ? static_cast<float*>(p.param) : p.master;
  int si = 0, decay_si = -1;
  float decay = 1.f;
  int t = blockIdx.x;
  if (t >= p.tab.n_tiles) return;
  K3Tile<MG> cur;
  k3_load<PT, MG>(p, wbase, t, si, cur, decay_si, decay, ss.lr_wd);
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
        __stcs(reinterpret_cast<float4*>(wbase + cur.m0 + e), make_float4(w[0], w[1], w[2], w[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg + cur.l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg_sq + cur.l0 + e), make_float4(v[0], v[1], v[2], v[3]));
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

// ---------------------------------------------------------- K3 with TMA --
//
// The same pass with the four input streams of a tile (main grad, master,
// m, v) staged in shared memory by the bulk-copy engine: thread 0 issues one
// 1-D copy per stream per tile onto the stage's mbarrier, a ring of
// DOPT_K3_TMA_STAGES stages keeps them in flight, every thread computes from
// shared memory and stores its results straight to global memory.  Used when
// every run of the launch is 8-element aligned (copies start on 16 bytes)
// and the step has a workspace to report a failed wait in.  Every wait is
// bounded: a CTA that gives up (decided uniformly) sets *error = 2, waits
// (bounded) for its copies still in flight and leaves; the step is then
// applied only in part, and the entry point reports it.
constexpr int kK3TmaTile = DOPT_K3_TMA_TILE;
static_assert(kK3TmaTile % (kThreads * kVec) == 0, "K3 TMA tile");

template <typename MG>
__host__ __device__ constexpr size_t k3_stage_bytes() {
  return (size_t)kK3TmaTile * (sizeof(typename MainT<MG>::Elem) + 12);
}
template <typename MG>
__host__ __device__ constexpr size_t k3_tma_smem_bytes() {
  return (size_t)DOPT_K3_TMA_STAGES * k3_stage_bytes<MG>() + DOPT_K3_TMA_STAGES * sizeof(uint64_t);
}

template <typename PT, typename MG>
__global__ void __launch_bounds__(kThreads, 2) k3_adamw_tma(const __grid_constant__ K3Params p) {
  if (*p.found_inf) return;  // skipped step: nothing is written
  using ME = typename MainT<MG>::Elem;
  constexpr int S = DOPT_K3_TMA_STAGES;
  constexpr int T = kK3TmaTile;
  constexpr size_t kMainBytes = (size_t)T * sizeof(ME);
  constexpr size_t kStage = k3_stage_bytes<MG>();
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S * kStage);
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const float c = *p.coef;
  const StepScalars ss = step_scalars(p);
  float* const wbase = ParamT<PT>::kInPlace ? static_cast<float*>(p.param) : p.master;
  const int G = gridDim.x;
  const int my = p.tab.n_tiles > (int)blockIdx.x ? (p.tab.n_tiles - (int)blockIdx.x + G - 1) / G : 0;
  int si_issue = 0;
  // thread 0: start the copies of this CTA's i-th tile into stage i % S
  auto issue = [&](int i) {
    const int t = blockIdx.x + i * G;
    si_issue = seek(p.tab, si_issue, t);
    const Seg& sg = p.tab.seg[si_issue];
    const int64_t off = (int64_t)(t - sg.tile0) * T;
    const int n = (int)min((int64_t)T, (int64_t)sg.len - off);
    const int nv = n & ~7;  // whole 16-byte pieces of every stream
    const int64_t l0 = sg.local + off;
    const int64_t m0 = ParamT<PT>::kInPlace ? sg.world + off : l0;
    unsigned char* st = smem + (size_t)(i % S) * kStage;
    uint64_t* bar = &bars[i % S];
    mbar_arrive_expect_tx(bar, (unsigned)nv * (unsigned)(sizeof(ME) + 12));
    if (nv > 0 && !(blockIdx.x == 0 && i == p.starve_tile)) {
      bulk_load(st, reinterpret_cast<const ME*>(p.main_grad) + l0, (unsigned)(nv * sizeof(ME)), bar);
      bulk_load(st + kMainBytes, wbase + m0, (unsigned)nv * 4u, bar);
      bulk_load(st + kMainBytes + (size_t)T * 4, p.exp_avg + l0, (unsigned)nv * 4u, bar);
      bulk_load(st + kMainBytes + (size_t)T * 8, p.exp_avg_sq + l0, (unsigned)nv * 4u, bar);
    }
  };
  if (threadIdx.x == 0)
    for (int i = 0; i < min(S, my); ++i) issue(i);

  int si = 0, decay_si = -1;
  float decay = 1.f;
  bool failed = false;
  int i = 0;
  for (; i < my; ++i) {
    const bool ok = mbar_wait_bounded(&bars[i % S], (unsigned)((i / S) & 1));
    if (__syncthreads_or(!ok)) {
      failed = true;
      break;
    }
    const int t = blockIdx.x + i * G;
    si = seek(p.tab, si, t);
    const Seg& sg = p.tab.seg[si];
    if (si != decay_si) {
      decay = decay_of(ss.lr_wd, sg.wd_mult);
      decay_si = si;
    }
    const int64_t off = (int64_t)(t - sg.tile0) * T;
    const int n = (int)min((int64_t)T, (int64_t)sg.len - off);
    const int nv = n & ~7;
    const int64_t l0 = sg.local + off, w0 = sg.world + off;
    const int64_t m0 = ParamT<PT>::kInPlace ? w0 : l0;
    const unsigned char* st = smem + (size_t)(i % S) * kStage;
    const ME* s_main = reinterpret_cast<const ME*>(st);
    const float* s_w = reinterpret_cast<const float*>(st + kMainBytes);
    const float* s_m = s_w + T;
    const float* s_v = s_m + T;
#pragma unroll
    for (int u = 0; u < T / (kThreads * kVec); ++u) {
      const int e = (u * kThreads + threadIdx.x) * kVec;
      if (e + kVec <= nv) {
        float g[kVec];
        MainT<MG>::widen4(*reinterpret_cast<const typename MainT<MG>::Raw*>(s_main + e), p.inv_scale, g);
        const float4 w4 = *reinterpret_cast<const float4*>(s_w + e);
        const float4 m4 = *reinterpret_cast<const float4*>(s_m + e);
        const float4 v4 = *reinterpret_cast<const float4*>(s_v + e);
        float w[kVec] = {w4.x, w4.y, w4.z, w4.w};
        float m[kVec] = {m4.x, m4.y, m4.z, m4.w};
        float v[kVec] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int j = 0; j < kVec; ++j) adamw1(__fmul_rn(g[j], c), decay, p, ss, w[j], m[j], v[j]);
        __stcs(reinterpret_cast<float4*>(wbase + m0 + e), make_float4(w[0], w[1], w[2], w[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg + l0 + e), make_float4(m[0], m[1], m[2], m[3]));
        __stcs(reinterpret_cast<float4*>(p.exp_avg_sq + l0 + e), make_float4(v[0], v[1], v[2], v[3]));
        ParamT<PT>::store4(p.param, w0 + e, w);
      } else if (e < n) {
        // the last few elements of a run: not in the staged copies
        const int cnt = min(kVec, n - e);
        for (int j = 0; j < cnt; ++j) {
          float ww = wbase[m0 + e + j], mm = p.exp_avg[l0 + e + j], vv = p.exp_avg_sq[l0 + e + j];
          adamw1(__fmul_rn(MainT<MG>::load1(p.main_grad, l0 + e + j, p.inv_scale), c), decay, p, ss, ww, mm,
                 vv);
          wbase[m0 + e + j] = ww;
          p.exp_avg[l0 + e + j] = mm;
          p.exp_avg_sq[l0 + e + j] = vv;
          ParamT<PT>::store1(p.param, w0 + e + j, ww);
        }
      }
    }
    __syncthreads();  // every thread is done with this stage
    if (threadIdx.x == 0 && i + S < my) issue(i + S);
  }
  if (failed && threadIdx.x == 0) {
    *p.error = 2;
    // let the copies already issued land before the shared memory goes away
    for (int j = i; j < min(i + S, my); ++j) mbar_wait_bounded(&bars[j % S], (unsigned)((j / S) & 1));
  }
}

template <typename PT, typename MG>
int launch_k3_t(K3Params& kp, cudaStream_t s, bool tma) {
  if (tma) {
    auto kern = k3_adamw_tma<PT, MG>;
    const size_t smem = k3_tma_smem_bytes<MG>();
    static std::atomic<uint64_t> attr_set{0};
    int st = allow_dynamic_smem(kern, smem, attr_set, "k3 tma");
    if (st) return st;
    int grid = 0;
    st = grid_for(kern, kp.tab.n_tiles, &grid, smem);
    if (st) return st;
    kern<<<grid, kThreads, smem, s>>>(kp);
    return check_launch("k3_adamw_tma launch");
  }
  auto kern = k3_adamw_pipe<PT, MG>;
  int grid = 0;
  int st = grid_for(kern, kp.tab.n_tiles, &grid);
  if (st) return st;
  kern<<<grid, kThreads, 0, s>>>(kp);
  return check_launch("k3_adamw launch");
}

// Param and grad dtypes pair up as the buffers allow: a 16-bit param buffer
// has grads in its own dtype or in fp32, an fp32 param buffer fp32 grads.
int launch_k3(int32_t param_dtype, int32_t main_dtype, K3Params& kp, const Run* runs, int count,
              cudaStream_t s) {
  const bool compact = main_dtype != DOPT_F32;
  if (compact && main_dtype != param_dtype)
    return fail(DOPT_E_INVALID, "compact main grads need the grad dtype of the param buffer");
  bool all_aligned = true;
  for (int k = 0; k < count; ++k) all_aligned &= seg_aligned(runs[k].local, runs[k].world);
  const bool tma = DOPT_K3_TMA && kp.error && all_aligned;
  fill_table(kp.tab, runs, count, tma ? kK3TmaTile : kTile3, -1);
  switch (param_dtype) {
    case DOPT_BF16:
      return compact ? launch_k3_t<__nv_bfloat16, __nv_bfloat16>(kp, s, tma)
                     : launch_k3_t<__nv_bfloat16, float>(kp, s, tma);
    case DOPT_F16:
      return compact ? launch_k3_t<__half, __half>(kp, s, tma) : launch_k3_t<__half, float>(kp, s, tma);
    default:
      return launch_k3_t<float, float>(kp, s, tma);
  }
}

}  // namespace dopt
