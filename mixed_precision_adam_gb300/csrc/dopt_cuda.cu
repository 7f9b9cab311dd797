// dopt_cuda.cu -- K2 (the finalize pass) and the C entry points of the
// device step: argument checks, the workspace layout, cutting the run lists
// into launch chunks and issuing K1 -> K2 -> K3 on the caller's stream.
// The K1 kernels live in k1.cuh (one translation unit per grad dtype), K3 in
// k3.cu; kernels.cuh holds what they share.
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "kernels.cuh"

// Scratch of dopt_step_noalloc: the step scalars and partial-sum regions
// that dopt_step keeps in the caller's workspace.  Host code must not use
// this name as an address (it is a host-side stand-in): the device address
// comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DOPT_NOALLOC_SCRATCH_BYTES];

#if DOPT_BOUNDS_CHECK
// Debug builds: the record of the first tile found outside its buffers
// ([count, site, first element, extent]), read by dopt_debug_bounds_record.
static __device__ unsigned long long g_bounds_record[4];
#endif

namespace {
std::atomic<uint64_t> g_launches{0};  // kernels launched by this library

// A named range on the host timeline of a profiler (NVTX; no cost without
// one attached) around a step and its passes.
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};
}  // namespace

namespace dopt {

// ------------------------------------------------------------------- K2 --

constexpr int kFinThreads = 512;  // the finalize pass is one CTA

__global__ void __launch_bounds__(kFinThreads)
k2_finalize(const FinalizeArgs f) {
  finalize_block<kFinThreads>(f);
}

// ------------------------------------------- launch helpers (kernels.cuh) --

struct DeviceInfo {
  int device = -1, sms = 0, l2_bytes = 0;
};

int device_sms(int* sms, int* l2_bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  static thread_local DeviceInfo cache;
  if (cache.device != dev) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess)
      return fail(DOPT_E_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    int l2 = 0;
    e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
    if (e != cudaSuccess)
      return fail(DOPT_E_CUDA, std::string("cudaDeviceGetAttribute: ") + cudaGetErrorString(e));
    cache.device = dev;
    cache.sms = n;
    cache.l2_bytes = l2;
  }
  *sms = cache.sms;
  if (l2_bytes) *l2_bytes = cache.l2_bytes;
  return DOPT_OK;
}

int check_launch(const char* what) {
  g_launches.fetch_add(1, std::memory_order_relaxed);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return DOPT_OK;
}

void fill_table(SegTable& tab, const Run* runs, int count, int tile_elems, int32_t bucket_base) {
  tab.n_seg = count;
  int tile = 0;
  for (int k = 0; k < count; ++k) {
    const Run& r = runs[k];
    Seg& s = tab.seg[k];
    s.local = r.local;
    s.world = r.world;
    s.len = (int32_t)r.len;
    s.tile0 = tile;
    if (bucket_base >= 0) {
      s.wd_mult = 0.0;  // clears the whole field before the bucket takes part of it
      s.bucket = bucket_base + r.bucket;
    } else {
      s.wd_mult = r.wd_mult;
    }
    tile += (int)((r.len + tile_elems - 1) / tile_elems);
  }
  tab.n_tiles = tile;
}

}  // namespace dopt

namespace {
using namespace dopt;

thread_local std::vector<char> t_param_scratch;  // kernel-parameter staging
#if DOPT_BOUNDS_CHECK
std::atomic<int32_t> g_starve_tile{-1};           // test hook, see dopt_debug_starve_copy
#endif

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

// What a K1 pass does, apart from the runs it covers.
struct K1Job {
  const void* const* replicas;
  int32_t n_rep = 0, n_inst = 1;
  bool full = true;          // replicas are whole grad buffers
  int32_t average = 0;       // average_in_collective
  float inv_scale = 1.0f;    // 1 / loss scale
  float post_scale = 1.0f;   // scale_gradients factor
  int32_t gdt = DOPT_F32;    // grad dtype
  float* main_grad = nullptr;
  bool stats = false;        // write norm partials to the workspace
  void* ws = nullptr;
  uint32_t* amax = nullptr;  // grad check table, or NULL
  int64_t amax_stride = 0;   // buckets of all buffers
  int32_t bucket_base = 0;   // number of the buffer's first bucket
  bool compact = false;      // 16-bit grads: keep the reduced grads in the grad dtype
  bool keep_main = false;    // fp32 main grads stored to stay in L2 for the AdamW pass
  const FinalizeArgs* fin = nullptr;  // finalize in the last launch's last CTA (fused step)
  uint32_t* fin_counter = nullptr;
  int64_t ext_rep = 0, ext_main = 0;  // element extents of each replica and of main_grad
};

// Element extents of a rank selection's flat-shard arrays and of one
// replica in the given layout (whole buffer, or the selection's shard).
int64_t shard_extent(const dopt_shard_map* m, int32_t buffer, int32_t rank) {
  return (int64_t)n_rank_slots(m, rank) * shard_numel(m, buffer);
}
int64_t replica_extent(const dopt_shard_map* m, int32_t buffer, int32_t rank, bool full) {
  return full ? m->buffers[buffer].numel : shard_extent(m, buffer, rank);
}

#if DOPT_BOUNDS_CHECK
// Device address of g_bounds_record on the current device.
int bounds_record(unsigned long long** out) {
  static std::mutex mu;
  static unsigned long long* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) return fail(DOPT_E_CUDA, "bounds record: cudaGetDevice");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_bounds_record);
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("bounds record: ") + cudaGetErrorString(e));
    addr[dev] = static_cast<unsigned long long*>(a);
  }
  *out = addr[dev];
  return DOPT_OK;
}
#endif

// Launches K1 over every chunk of a run list; with stats, chunk i writes its
// partials to workspace region region_first + i.
int run_k1_runs(const std::vector<Run>& runs, int region_first, const K1Job& j, cudaStream_t s) {
  std::vector<Chunk> chunks = chunks_of(runs);
  int region = region_first;
  for (const Chunk& c : chunks) {
    K1Params& kp = k1_scratch();
    for (int k = 0; k < j.n_rep; ++k) kp.rep[k] = j.replicas[k];
    for (int k = j.n_rep; k < DOPT_MAX_REPLICAS; ++k) kp.rep[k] = nullptr;
    kp.main_grad = j.main_grad;
    kp.partials = j.stats ? region_ptr(j.ws, region++) : nullptr;
    kp.n_rep = j.n_rep;
    kp.n_inst = j.n_inst;
    kp.pre = (float)(1.0 / (double)j.n_rep);
    kp.inv_dpi = (float)(1.0 / (double)(j.n_rep / j.n_inst));
    kp.inv_ninst = (float)(1.0 / (double)j.n_inst);
    kp.inv_scale = j.inv_scale;
    kp.average = j.average ? 1 : 0;
    kp.post_scale = j.post_scale;
    kp.error_flag = j.ws ? reinterpret_cast<int32_t*>(static_cast<char*>(j.ws) + kErrorFlagOffset) : nullptr;
#if DOPT_BOUNDS_CHECK
    kp.starve_tile = g_starve_tile.load(std::memory_order_relaxed);
#endif
    kp.compact = j.compact && j.stats ? 1 : 0;
    kp.keep_main = j.keep_main ? 1 : 0;
    kp.amax = j.amax;
    kp.amax_stride = j.amax_stride;
    const bool last = &c == &chunks.back();
    kp.fin_counter = (j.fin && last) ? j.fin_counter : nullptr;
    if (kp.fin_counter) kp.fin = *j.fin;
#if DOPT_BOUNDS_CHECK
    kp.ext = Extents{j.ext_rep, j.ext_main, 0, 0, j.amax_stride, nullptr};
    if (int st = bounds_record(&kp.ext.record)) return st;
#endif
    const K1Launch l{runs.data() + c.first, c.count, j.bucket_base, j.full, j.stats, j.amax != nullptr};
    int st;
    switch (j.gdt) {
      case DOPT_F32: st = launch_k1_f32(kp, l, s); break;
      case DOPT_BF16: st = launch_k1_bf16(kp, l, s); break;
      case DOPT_F16: st = launch_k1_f16(kp, l, s); break;
      default: st = fail(DOPT_E_INVALID, "unknown grad dtype");
    }
    if (st) return st;
  }
  return DOPT_OK;
}

// Number of bucket `bucket` of `buffer` among the buckets of all buffers
// (buffer order); (n_buffers, 0) gives the total.
int32_t bucket_number(const dopt_shard_map* m, int32_t buffer, int32_t bucket) {
  int32_t n = 0;
  for (int32_t b = 0; b < buffer; ++b) n += (int32_t)m->buffers[b].buckets.size();
  return n + bucket;
}

// Whether a step's main grads (every buffer of the rank selection) are
// small enough next to L2 to be stored for the AdamW pass to read back
// from L2 rather than from DRAM.
bool keep_main_in_l2(const dopt_shard_map* m, int32_t rank) {
  if (DOPT_KEEP_MAIN_L2_DIV <= 0) return false;
  int sms = 0, l2 = 0;
  if (device_sms(&sms, &l2) != DOPT_OK) return false;
  size_t bytes = 0;
  for (int32_t b = 0; b < (int32_t)m->buffers.size(); ++b)
    bytes += (size_t)shard_extent(m, b, rank) * (m->buffers[b].grad_dtype == DOPT_F32 ? 4 : 2);
  return bytes <= (size_t)l2 / DOPT_KEEP_MAIN_L2_DIV;
}

// The K1 job of buffer b of a step.
K1Job step_job(const dopt_step_args* a, int32_t b) {
  const dopt_shard_map* m = a->map;
  K1Job j;
  j.replicas = a->replica_grads[b];
  j.n_rep = m->dp * a->n_instances;
  j.n_inst = a->n_instances;
  j.full = a->layout != DOPT_LAYOUT_SHARD_ONLY;  // whole buffers and bucket groups: buffer indices
  j.average = a->average_in_collective;
  j.inv_scale = a->inv_loss_scale;
  j.post_scale = a->grad_scale == 0.0f ? 1.0f : a->grad_scale;  // 0 (unset) means 1
  j.gdt = m->buffers[b].grad_dtype;
  j.main_grad = a->main_grad[b];
  j.stats = true;
  j.ws = a->workspace;
  j.amax = reinterpret_cast<uint32_t*>(a->grad_amax);
  j.amax_stride = bucket_number(m, (int32_t)m->buffers.size(), 0);
  j.bucket_base = bucket_number(m, b, 0);
  j.compact = j.gdt != DOPT_F32;
  j.ext_rep = replica_extent(m, b, a->rank, j.full);
  j.ext_main = shard_extent(m, b, a->rank);
  j.keep_main = keep_main_in_l2(m, a->rank);
  return j;
}

// Clears the grad-check slots of buckets [first, first + count) (numbered
// across buffers) for every replica.
int clear_amax(const dopt_step_args* a, int32_t first, int32_t count, cudaStream_t s) {
  if (!a->grad_amax || count <= 0) return DOPT_OK;
  const dopt_shard_map* m = a->map;
  const size_t total = (size_t)bucket_number(m, (int32_t)m->buffers.size(), 0);
  const size_t n_rep = (size_t)m->dp * a->n_instances;
  cudaError_t e = cudaMemset2DAsync(a->grad_amax + first, total * sizeof(float), 0, (size_t)count * sizeof(float),
                                    n_rep, s);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("grad check clear: ") + cudaGetErrorString(e));
  return DOPT_OK;
}

// K1 over every run of (buffer, rank) for the separate entry points;
// partials go to the buffer's regions of the fused-step workspace layout.
int run_k1(dopt_shard_map* m, int32_t buffer, int32_t rank, const K1Job& j, cudaStream_t s) {
  return run_k1_runs(runs_for(m, buffer, rank), j.stats ? regions_before(m, buffer, rank) : 0, j, s);
}

DevStep* dev_step_ptr(void* ws) {
  return reinterpret_cast<DevStep*>(static_cast<char*>(ws) + kDevStepOffset);
}

// The finalize arguments of a step whose partial regions fill n_slots
// slots of workspace ws (device step state from a when it has some).
FinalizeArgs finalize_args(int n_slots, void* ws, double remote_sumsq, int32_t remote_found, double max_norm,
                           float* d_norm, float* d_coef, int32_t* d_found, const dopt_step_args* a) {
  FinalizeArgs f{};
  f.parts = region_ptr(ws, 0);
  f.n_slots = n_slots;
  f.remote_found = remote_found ? 1 : 0;
  f.remote_sumsq = remote_sumsq;
  f.max_norm = max_norm;
  f.sc = scalars_ptr(ws);
  f.d_norm = d_norm;
  f.d_coef = d_coef;
  f.d_found = d_found;
  f.err_flag = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + kErrorFlagOffset);
  f.step = K2Step{nullptr, nullptr, 0.0, 0.0, 0.0, 0.0, dev_step_ptr(ws)};
  if (a) {
    f.d_global_sumsq = a->d_global_sumsq;
    f.d_global_found = a->d_global_found_inf;
  }
  if (a && a->d_step) {
    f.step.d_step = a->d_step;
    f.step.d_lr = a->d_lr;
    f.step.lr = a->hp.lr;
    f.step.wd = a->hp.weight_decay;
    f.step.beta1 = a->hp.beta1;
    f.step.beta2 = a->hp.beta2;
  }
  return f;
}

int run_k2_slots(int n_slots, void* ws, double remote_sumsq, int32_t remote_found, double max_norm,
                 float* d_norm, float* d_coef, int32_t* d_found, cudaStream_t s,
                 const dopt_step_args* a = nullptr) {
  k2_finalize<<<1, kFinThreads, 0, s>>>(
      finalize_args(n_slots, ws, remote_sumsq, remote_found, max_norm, d_norm, d_coef, d_found, a));
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


// What a K3 pass does, apart from the runs it covers.
struct K3Job {
  int32_t param_dtype = DOPT_F32;
  int32_t main_dtype = DOPT_F32;  // DOPT_F32, or the grad dtype for compact main grads
  float inv_scale = 1.0f;         // compact main grads: main = widen(stored) * inv_scale
  const float* main_grad = nullptr;
  float* master = nullptr;
  float* exp_avg = nullptr;
  float* exp_avg_sq = nullptr;
  void* param = nullptr;
  const dopt_adamw_hparams* hp = nullptr;
  const float* d_coef = nullptr;
  const int32_t* d_found = nullptr;
  const DevStep* dev = nullptr;   // device step scalars, or NULL: from hp
  // the launch before this pass is a kernel of the same step that writes
  // none of its master, m and v (K3Head::early_state)
  bool early_state = false;
  int64_t ext_main = 0, ext_state = 0, ext_param = 0;  // element extents (debug builds check them)
};

int run_k3_runs(const std::vector<Run>& runs, const K3Job& j, cudaStream_t s) {
  const dopt_adamw_hparams* hp = j.hp;
  std::vector<Chunk> chunks = chunks_of(runs);
  for (const Chunk& c : chunks) {
    K3Params& kp = k3_scratch();
    kp.main_grad = j.main_grad;
    kp.master = j.master;
    kp.exp_avg = j.exp_avg;
    kp.exp_avg_sq = j.exp_avg_sq;
    kp.param = j.param;
    kp.coef = j.d_coef;
    kp.found_inf = j.d_found;
    kp.dev = j.dev;
    kp.lr_wd = hp->lr * hp->weight_decay;
    kp.b1 = (float)hp->beta1;
    kp.b2 = (float)hp->beta2;
    kp.omb1 = (float)(1.0 - hp->beta1);
    kp.omb2 = (float)(1.0 - hp->beta2);
    kp.eps = (float)hp->eps;
    kp.step_size = (float)(hp->lr / (1.0 - pow_int(hp->beta1, hp->step)));
    kp.bc2_sqrt = (float)std::sqrt(1.0 - pow_int(hp->beta2, hp->step));
    kp.inv_scale = j.inv_scale;
    kp.early_state = j.early_state ? 1 : 0;
#if DOPT_BOUNDS_CHECK
    kp.ext = Extents{0, j.ext_main, j.ext_state, j.ext_param, 0, nullptr};
    if (int st = bounds_record(&kp.ext.record)) return st;
#endif
    int st = launch_k3(j.param_dtype, j.main_dtype, kp, runs.data() + c.first, c.count, s);
    if (st) return st;
  }
  return DOPT_OK;
}

// The K3 job of buffer b of a fused or bucket-staged step: a 16-bit grad
// buffer's main grads arrive in their compact form (see step_job).
K3Job step_job3(const dopt_step_args* a, int32_t b) {
  const dopt_shard_map* m = a->map;
  Scalars* sc = scalars_ptr(a->workspace);
  K3Job j;
  j.param_dtype = m->buffers[b].param_dtype;
  j.main_dtype = m->buffers[b].grad_dtype;
  j.inv_scale = a->inv_loss_scale;
  j.main_grad = a->main_grad[b];
  j.master = a->master[b];
  j.exp_avg = a->exp_avg[b];
  j.exp_avg_sq = a->exp_avg_sq[b];
  j.param = a->param_buffer[b];
  j.hp = &a->hp;
  j.d_coef = &sc->clip_coef;
  j.d_found = &sc->found_inf;
  j.dev = a->d_step ? dev_step_ptr(a->workspace) : nullptr;
  j.ext_main = j.ext_state = shard_extent(m, b, a->rank);
  j.ext_param = m->buffers[b].numel;
  return j;
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
  if (layout != DOPT_LAYOUT_FULL_BUFFER && layout != DOPT_LAYOUT_SHARD_ONLY && layout != DOPT_LAYOUT_BUCKET)
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
  if (!bucketed && a->layout == DOPT_LAYOUT_BUCKET)
    return fail(DOPT_E_INVALID, std::string(fn) + ": the bucket layout is for the bucket-staged step only");
  if ((st = check_hparams(&a->hp, fn))) return st;
  if ((a->d_step && (reinterpret_cast<uintptr_t>(a->d_step) & 7)) ||
      (a->d_lr && (reinterpret_cast<uintptr_t>(a->d_lr) & 7)))
    return dopt::fail(DOPT_E_ALIGN, std::string(fn) + ": d_step / d_lr not 8-byte aligned");
  if (a->grad_amax && (reinterpret_cast<uintptr_t>(a->grad_amax) & 3))
    return fail(DOPT_E_ALIGN, std::string(fn) + ": grad_amax not 4-byte aligned");
  if (!bucketed && a->d_global_sumsq)
    return fail(DOPT_E_INVALID, std::string(fn) +
                                    ": d_global_sumsq is for the bucket-staged finalize (dopt_step_finalize)");
  if (!a->d_global_sumsq != !a->d_global_found_inf)
    return fail(DOPT_E_INVALID, std::string(fn) + ": d_global_sumsq and d_global_found_inf go together");
  if ((a->d_global_sumsq && (reinterpret_cast<uintptr_t>(a->d_global_sumsq) & 7)) ||
      (a->d_global_found_inf && (reinterpret_cast<uintptr_t>(a->d_global_found_inf) & 3)))
    return fail(DOPT_E_ALIGN, std::string(fn) + ": d_global_sumsq / d_global_found_inf misaligned");
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

// The fused step, enqueued in two parts split where its results are known:
// the reduce launches with the finalize in the last one (stage events 0-2),
// then the AdamW launches (stage event 3).  Arguments already checked.
int enqueue_reduce(const dopt_step_args* a, int32_t* d_found_inf, float* d_norm) {
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int32_t nb = (int32_t)m->buffers.size();
  cudaStream_t s = (cudaStream_t)a->stream;
  int st = record_stage(a, 0, s);
  if (st) return st;
  if ((st = clear_amax(a, 0, bucket_number(m, nb, 0), s))) return st;
  // the finalize runs in the last CTA of the last reduce launch: its ticket
  // counter starts every step at zero
  uint32_t* counter = reinterpret_cast<uint32_t*>(static_cast<char*>(a->workspace) + kFinCounterOffset);
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("dopt_step: ") + cudaGetErrorString(e));
  const FinalizeArgs fin = finalize_args(total_regions(m, a->rank) * kMaxGrid, a->workspace, a->remote_sumsq,
                                         a->remote_found_inf, a->max_norm, d_norm, nullptr, d_found_inf, a);
  {
    Range r("reduce_prepare+finalize");
    // the largest buffer's launch goes last and carries the finalize, whose
    // tail then overlaps nothing but that launch's own last CTAs (the
    // partials' order in the sum is fixed by buffer, not by launch order)
    std::vector<int32_t> order(nb);
    for (int32_t b = 0; b < nb; ++b) order[b] = b;
    std::stable_sort(order.begin(), order.end(),
                     [&](int32_t x, int32_t y) { return shard_numel(m, x) < shard_numel(m, y); });
    for (int32_t i = 0; i < nb; ++i) {
      K1Job j = step_job(a, order[i]);
      if (i == nb - 1) {
        j.fin = &fin;
        j.fin_counter = counter;
      }
      if ((st = run_k1(m, order[i], a->rank, j, s))) return st;
    }
  }
  if ((st = record_stage(a, 1, s))) return st;
  return record_stage(a, 2, s);  // the finalize ran inside the last reduce launch
}

int enqueue_update(const dopt_step_args* a) {
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  cudaStream_t s = (cudaStream_t)a->stream;
  Range r("adamw");
  for (int32_t b = 0; b < (int32_t)m->buffers.size(); ++b) {
    // queued right behind the step's reduce pass or the previous buffer's
    // AdamW pass, all in this call
    K3Job j = step_job3(a, b);
    j.early_state = true;
    int st = run_k3_runs(runs_for(m, b, a->rank), j, s);
    if (st) return st;
  }
  return record_stage(a, 3, s);
}

}  // namespace

using namespace dopt;

extern "C" {

uint64_t dopt_kernel_launches(void) { return g_launches.load(std::memory_order_relaxed); }

int dopt_debug_bounds_record(int64_t* out) {
  if (!out) return fail(DOPT_E_INVALID, "dopt_debug_bounds_record: NULL out");
#if DOPT_BOUNDS_CHECK
  unsigned long long* rec = nullptr;
  if (int st = bounds_record(&rec)) return st;
  unsigned long long h[4] = {0, 0, 0, 0};
  cudaError_t e = cudaMemcpy(h, rec, sizeof(h), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess) e = cudaMemset(rec, 0, sizeof(h));
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("dopt_debug_bounds_record: ") + cudaGetErrorString(e));
  for (int k = 0; k < 4; ++k) out[k] = (int64_t)h[k];
  return DOPT_OK;
#else
  return fail(DOPT_E_INVALID, "dopt_debug_bounds_record: this library was built without DOPT_BOUNDS_CHECK");
#endif
}

#if DOPT_BOUNDS_CHECK
int dopt_debug_starve_copy(int32_t tile) {
  if (tile < -1) return fail(DOPT_E_INVALID, "dopt_debug_starve_copy: tile < -1");
  g_starve_tile.store(tile, std::memory_order_relaxed);
  return DOPT_OK;
}
#endif

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
  if (layout == DOPT_LAYOUT_BUCKET)
    return dopt::fail(DOPT_E_INVALID, "dopt_grad_reduce_shard: the bucket layout is for the bucket-staged step only");
  if (!main_grad) return dopt::fail(DOPT_E_INVALID, "dopt_grad_reduce_shard: NULL main_grad");
  if (!aligned16(main_grad)) return dopt::fail(DOPT_E_ALIGN, "dopt_grad_reduce_shard: main_grad not aligned");
  (void)workspace;
  (void)workspace_bytes_;
  K1Job j;
  j.replicas = replicas;
  j.n_rep = n_replicas;
  j.n_inst = n_instances;
  j.full = layout == DOPT_LAYOUT_FULL_BUFFER;
  j.average = average_in_collective;
  j.gdt = m->buffers[buffer].grad_dtype;
  j.main_grad = main_grad;
  j.ext_rep = replica_extent(m, buffer, rank, j.full);
  j.ext_main = shard_extent(m, buffer, rank);
  return run_k1(m, buffer, rank, j, (cudaStream_t)stream);
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
  K1Job j;
  j.replicas = one;
  j.n_rep = 1;
  j.full = false;
  j.inv_scale = inv_loss_scale;
  j.main_grad = main_grad;
  j.stats = true;
  j.ws = workspace;
  j.ext_rep = j.ext_main = shard_extent(m, buffer, rank);
  return run_k1(m, buffer, rank, j, (cudaStream_t)stream);
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
  K3Job j;
  j.param_dtype = m->buffers[buffer].param_dtype;
  j.main_grad = main_grad;
  j.master = master;
  j.exp_avg = exp_avg;
  j.exp_avg_sq = exp_avg_sq;
  j.param = param_buffer;
  j.hp = hp;
  j.d_coef = d_clip_coef;
  j.d_found = d_found_inf;
  j.ext_main = j.ext_state = shard_extent(m, buffer, rank);
  j.ext_param = m->buffers[buffer].numel;
  return run_k3_runs(runs_for(m, buffer, rank), j, (cudaStream_t)stream);
}

int dopt_step_async(const dopt_step_args* a, int32_t* d_found_inf, float* d_norm) {
  Range step_range("dopt_step");
  int st = check_step_args(a, false, "dopt_step");
  if (st) return st;
  if ((st = enqueue_reduce(a, d_found_inf, d_norm))) return st;
  return enqueue_update(a);
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
  Range range("dopt_step_reduce_buckets");
  const char* fn = "dopt_step_reduce_buckets";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  if ((st = check_bucket_range(m, buffer, bucket_first, bucket_count, fn))) return st;
  std::vector<std::vector<Run>> by = runs_by_bucket(m, buffer, a->rank);
  cudaStream_t s = (cudaStream_t)a->stream;
  if ((st = clear_amax(a, bucket_number(m, buffer, bucket_first), bucket_count, s))) return st;
  K1Job j = step_job(a, buffer);
  // the group's runs in as few launches as the run tables allow; their
  // partials fill the group's first regions, and the group's other regions
  // are zeroed so that no partial of an earlier step is left in them
  std::vector<Run> runs;
  int regions = 0;
  for (int32_t k = bucket_first; k < bucket_first + bucket_count; ++k) {
    runs.insert(runs.end(), by[k].begin(), by[k].end());
    regions += (int)chunks_of(by[k]).size();
  }
  if (a->layout == DOPT_LAYOUT_BUCKET) {
    // replicas hold the group only: buffer indices from the group's first
    // bucket on (bucket offsets are multiples of 64 elements, so the runs'
    // 8-element alignment is kept)
    const Buffer& buf = m->buffers[buffer];
    const Bucket& last = buf.buckets[bucket_first + bucket_count - 1];
    const int64_t base = buf.buckets[bucket_first].offset;
    for (Run& r : runs) r.world -= base;
    j.ext_rep = last.offset + last.numel - base;
  }
  const int first = bucketed_region(m, a->rank, buffer, bucket_first);
  if ((st = run_k1_runs(runs, first, j, s))) return st;
  const int used = (int)chunks_of(runs).size();
  if (used < regions) {
    cudaError_t e = cudaMemsetAsync(region_ptr(a->workspace, first + used), 0,
                                    (size_t)(regions - used) * kMaxGrid * sizeof(Partial), s);
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
  }
  return DOPT_OK;
}

int dopt_step_finalize(const dopt_step_args* a, int32_t* d_found_inf, float* d_norm) {
  Range range("dopt_step_finalize");
  const char* fn = "dopt_step_finalize";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int n_slots = bucketed_region(m, a->rank, (int32_t)m->buffers.size(), 0) * kMaxGrid;
  return run_k2_slots(n_slots, a->workspace, a->remote_sumsq, a->remote_found_inf, a->max_norm, d_norm,
                      nullptr, d_found_inf, (cudaStream_t)a->stream, a);
}

int dopt_step_local_stats(const dopt_step_args* a, double* d_local_sumsq, int32_t* d_local_found_inf) {
  Range range("dopt_step_local_stats");
  const char* fn = "dopt_step_local_stats";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  if (!d_local_sumsq || !d_local_found_inf)
    return fail(DOPT_E_INVALID, std::string(fn) + ": NULL d_local_sumsq or d_local_found_inf");
  if ((reinterpret_cast<uintptr_t>(d_local_sumsq) & 7) || (reinterpret_cast<uintptr_t>(d_local_found_inf) & 3))
    return fail(DOPT_E_ALIGN, std::string(fn) + ": d_local_sumsq / d_local_found_inf misaligned");
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int n_slots = bucketed_region(m, a->rank, (int32_t)m->buffers.size(), 0) * kMaxGrid;
  FinalizeArgs f = finalize_args(n_slots, a->workspace, 0.0, 0, a->max_norm, nullptr, nullptr, nullptr, nullptr);
  f.local_sumsq = d_local_sumsq;
  f.local_found = d_local_found_inf;
  k2_finalize<<<1, kFinThreads, 0, (cudaStream_t)a->stream>>>(f);
  return check_launch("k2_finalize (local statistics) launch");
}

int dopt_step_update_buckets(const dopt_step_args* a, int32_t buffer, int32_t bucket_first,
                             int32_t bucket_count) {
  Range range("dopt_step_update_buckets");
  const char* fn = "dopt_step_update_buckets";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  if ((st = check_bucket_range(m, buffer, bucket_first, bucket_count, fn))) return st;
  std::vector<std::vector<dopt::Run>> by = runs_by_bucket(m, buffer, a->rank);
  std::vector<dopt::Run> runs;
  for (int32_t k = bucket_first; k < bucket_first + bucket_count; ++k)
    runs.insert(runs.end(), by[k].begin(), by[k].end());
  return run_k3_runs(runs, step_job3(a, buffer), (cudaStream_t)a->stream);
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

namespace {
// Per thread and device: the copy stream of dopt_step_from_host when the
// caller gives none, and the event that orders its copies with the step.
struct HostCopyResources {
  cudaStream_t stream = nullptr;
  cudaEvent_t ready = nullptr;
  ~HostCopyResources() {  // at thread exit; errors (a runtime already shut down) are moot
    if (ready) cudaEventDestroy(ready);
    if (stream) cudaStreamDestroy(stream);
  }
};
thread_local HostCopyResources t_host_copy[kMaxDevices];

int host_copy_resources(HostCopyResources** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(DOPT_E_INVALID, "device index out of range");
  HostCopyResources& r = t_host_copy[dev];
  if (!r.stream) {
    e = cudaStreamCreateWithFlags(&r.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&r.ready, cudaEventDisableTiming);
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string("copy stream: ") + cudaGetErrorString(e));
  }
  *out = &r;
  return DOPT_OK;
}

// Reads the step scalars back and turns them into the results of a
// synchronous step.
int finish_sync_step(const dopt_step_args* a, int32_t* found_inf_out, float* grad_norm_out, const char* fn) {
  Scalars host{};
  cudaStream_t s = (cudaStream_t)a->stream;
  cudaError_t e = cudaMemcpyAsync(&host, a->workspace, sizeof(Scalars), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
  if (found_inf_out) *found_inf_out = host.found_inf;
  if (grad_norm_out) *grad_norm_out = host.grad_norm;
  if (host.kernel_error)
    return fail(DOPT_E_CUDA,
                std::string(fn) + ": a kernel gave up waiting for its own data copies; the step was skipped");
  return DOPT_OK;
}
}  // namespace

int dopt_step_from_host(const dopt_step_args* a, const void* const* const* host_replica_grads,
                        dopt_stream copy_stream, int32_t* found_inf_out, float* grad_norm_out) {
  Range range("dopt_step_from_host");
  const char* fn = "dopt_step_from_host";
  int st = check_step_args(a, true, fn);
  if (st) return st;
  if (a->d_global_sumsq)
    return fail(DOPT_E_INVALID, std::string(fn) + ": d_global_sumsq is for the bucket-staged finalize (dopt_step_finalize)");
  if (a->layout == DOPT_LAYOUT_BUCKET)
    return fail(DOPT_E_INVALID, std::string(fn) + ": the bucket layout is for dopt_step_reduce_buckets only");
  dopt_shard_map* m = const_cast<dopt_shard_map*>(a->map);
  const int32_t nb = (int32_t)m->buffers.size();
  const int32_t n_rep = m->dp * a->n_instances;
  if (!host_replica_grads) return fail(DOPT_E_INVALID, std::string(fn) + ": NULL host replica array");
  for (int32_t b = 0; b < nb; ++b) {
    if (!host_replica_grads[b]) return fail(DOPT_E_INVALID, std::string(fn) + ": NULL host replica array");
    for (int32_t k = 0; k < n_rep; ++k)
      if (!host_replica_grads[b][k]) return fail(DOPT_E_INVALID, std::string(fn) + ": NULL host replica pointer");
  }
  HostCopyResources* res = nullptr;
  if ((st = host_copy_resources(&res))) return st;
  cudaStream_t s = (cudaStream_t)a->stream;
  cudaStream_t cs = copy_stream ? (cudaStream_t)copy_stream : res->stream;
  if (cs == s) return fail(DOPT_E_INVALID, std::string(fn) + ": copy_stream must differ from args->stream");
  auto cuda_ok = [&](cudaError_t e, const char* what) {
    return e == cudaSuccess ? DOPT_OK : fail(DOPT_E_CUDA, std::string(fn) + ": " + what + ": " + cudaGetErrorString(e));
  };
  // the copies overwrite the device replicas: after the work already queued
  if ((st = cuda_ok(cudaEventRecord(res->ready, s), "event record"))) return st;
  if ((st = cuda_ok(cudaStreamWaitEvent(cs, res->ready, 0), "stream wait"))) return st;
  if ((st = clear_amax(a, 0, bucket_number(m, nb, 0), s))) return st;
  const bool full = a->layout == DOPT_LAYOUT_FULL_BUFFER;
  int region = 0;  // bucketed workspace: regions in (buffer, bucket, chunk) order
  for (int32_t b = 0; b < nb; ++b) {
    const Buffer& buf = m->buffers[b];
    const size_t esz = buf.grad_dtype == DOPT_F32 ? 4 : 2;
    const std::vector<std::vector<Run>> by = runs_by_bucket(m, b, a->rank);
    const K1Job j = step_job(a, b);
    for (int32_t k = 0; k < (int32_t)buf.buckets.size(); ++k) {
      const Bucket& bk = buf.buckets[k];
      const int64_t slice = bk.numel / m->dp;
      int64_t first, count;  // elements of every replica the bucket's reduce reads
      if (!full) {
        first = bk.shard_base;
        count = slice;
      } else if (a->rank == DOPT_ALL_RANKS) {
        first = bk.offset;
        count = bk.numel;
      } else {
        first = bk.offset + (int64_t)a->rank * slice;
        count = slice;
      }
      for (int32_t r = 0; r < n_rep && count > 0; ++r) {
        char* dst = static_cast<char*>(const_cast<void*>(a->replica_grads[b][r])) + first * esz;
        const char* src = static_cast<const char*>(host_replica_grads[b][r]) + first * esz;
        if ((st = cuda_ok(cudaMemcpyAsync(dst, src, (size_t)count * esz, cudaMemcpyHostToDevice, cs),
                          "host-to-device copy")))
          return st;
      }
      if ((st = cuda_ok(cudaEventRecord(res->ready, cs), "event record"))) return st;
      if ((st = cuda_ok(cudaStreamWaitEvent(s, res->ready, 0), "stream wait"))) return st;
      if ((st = run_k1_runs(by[k], region, j, s))) return st;
      region += (int)chunks_of(by[k]).size();
    }
  }
  if ((st = run_k2_slots(region * kMaxGrid, a->workspace, a->remote_sumsq, a->remote_found_inf, a->max_norm,
                         nullptr, nullptr, nullptr, s, a)))
    return st;
  for (int32_t b = 0; b < nb; ++b)
    if ((st = run_k3_runs(runs_for(m, b, a->rank), step_job3(a, b), s))) return st;
  return finish_sync_step(a, found_inf_out, grad_norm_out, fn);
}

namespace {
// One param piece of a rank's shard: where it sits in the state layout and
// in model space (elements), and its length.
struct StatePiece {
  int64_t state, model, len;
};

// The pieces of `rank` (every rank's for DOPT_ALL_RANKS) in `buffer`, with
// their model-space offsets (the buffer's params in model order).
std::vector<StatePiece> state_pieces(const dopt_shard_map* m, int32_t b, int32_t rank, int32_t layout) {
  const Buffer& buf = m->buffers[b];
  std::unordered_map<int32_t, int64_t> model_start;
  int64_t acc = 0;
  for (int32_t pid : buf.params) {
    model_start[pid] = acc;
    acc += m->params[pid].numel;
  }
  const int64_t S = buf.numel / m->dp;
  const int32_t first = rank == DOPT_ALL_RANKS ? 0 : rank;
  const int32_t last = rank == DOPT_ALL_RANKS ? m->dp - 1 : rank;
  std::vector<StatePiece> out;
  for (int32_t r = first; r <= last; ++r) {
    for (const Bucket& bk : buf.buckets) {
      const int64_t slice = bk.numel / m->dp;
      const int64_t w0 = bk.offset + (int64_t)r * slice, w1 = w0 + slice;
      for (int32_t pid : bk.params) {
        const Param& p = m->params[pid];
        const int64_t lo = std::max(p.start, w0), hi = std::min(p.end, w1);
        if (hi <= lo) continue;
        const int64_t state = layout == DOPT_STATE_FLAT_SHARD ? (int64_t)(r - first) * S + bk.shard_base + (lo - w0)
                                                               : lo;
        out.push_back(StatePiece{state, model_start[pid] + (lo - p.start), hi - lo});
      }
    }
  }
  return out;
}

int state_copy(const dopt_shard_map* map, int32_t b, int32_t rank, int32_t layout, const void* src, void* dst,
               dopt_stream stream, bool to_model, const char* fn) {
  int st = check_map_buffer_rank(map, b, rank, fn);
  if (st) return st;
  if (layout != DOPT_STATE_FLAT_SHARD && layout != DOPT_STATE_PARAM_BUFFER)
    return fail(DOPT_E_INVALID, std::string(fn) + ": unknown state layout");
  if (!src || !dst) return fail(DOPT_E_INVALID, std::string(fn) + ": NULL pointer");
  const int32_t pdt = map->buffers[b].param_dtype;
  const size_t es = layout == DOPT_STATE_FLAT_SHARD || pdt == DOPT_F32 ? 4 : 2;
  for (const StatePiece& pc : state_pieces(map, b, rank, layout)) {
    const int64_t from = to_model ? pc.state : pc.model, to = to_model ? pc.model : pc.state;
    cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst) + to * es, static_cast<const char*>(src) + from * es,
                                    (size_t)pc.len * es, cudaMemcpyDefault, (cudaStream_t)stream);
    if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
  }
  return DOPT_OK;
}
}  // namespace

int64_t dopt_model_numel(const dopt_shard_map* map, int32_t buffer) {
  if (!map || buffer < 0 || buffer >= (int32_t)map->buffers.size())
    return fail(DOPT_E_INVALID, "dopt_model_numel: bad map or buffer");
  int64_t n = 0;
  for (int32_t pid : map->buffers[buffer].params) n += map->params[pid].numel;
  return n;
}

int dopt_state_to_model(const dopt_shard_map* map, int32_t buffer, int32_t rank, int32_t layout,
                        const void* state, void* model, dopt_stream stream) {
  return state_copy(map, buffer, rank, layout, state, model, stream, true, "dopt_state_to_model");
}

int dopt_state_from_model(const dopt_shard_map* map, int32_t buffer, int32_t rank, int32_t layout,
                          const void* model, void* state, dopt_stream stream) {
  return state_copy(map, buffer, rank, layout, model, state, stream, false, "dopt_state_from_model");
}

int dopt_step(const dopt_step_args* a, int32_t* found_inf_out, float* grad_norm_out) {
  const char* fn = "dopt_step";
  Range step_range(fn);
  int st = check_step_args(a, false, fn);
  if (st) return st;
  HostCopyResources* res = nullptr;
  if ((st = host_copy_resources(&res))) return st;
  cudaStream_t s = (cudaStream_t)a->stream;
  if ((st = enqueue_reduce(a, nullptr, nullptr))) return st;
  // the results are known once the finalize has run: copy them on the side
  // stream while the AdamW pass runs on the step's stream
  cudaError_t e = cudaEventRecord(res->ready, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(res->stream, res->ready, 0);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
  if ((st = enqueue_update(a))) return st;
  Scalars host{};
  e = cudaMemcpyAsync(&host, a->workspace, sizeof(Scalars), cudaMemcpyDeviceToHost, res->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(res->stream);
  if (e != cudaSuccess) return fail(DOPT_E_CUDA, std::string(fn) + ": " + cudaGetErrorString(e));
  if (found_inf_out) *found_inf_out = host.found_inf;
  if (grad_norm_out) *grad_norm_out = host.grad_norm;
  if (host.kernel_error)
    return fail(DOPT_E_CUDA, std::string(fn) + ": a kernel gave up waiting for its own data copies; the step was skipped");
  return DOPT_OK;
}

}  // extern "C"
