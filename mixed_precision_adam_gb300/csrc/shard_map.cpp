// shard_map.cpp -- host side of the library: the shard map (buffers, buckets,
// per-rank views), the runs the kernels walk, the memory ledger, ring
// communication volumes and the dynamic loss scaler.
//
// Shard map: "Megatron-LM distrib_optimizer.py close reading" page
// (xiaolong-dev.me), sections "Buffer layout", "Bucket partition: reverse
// walk + size trigger", "Two levels of padding", "Final memory size
// assertions", "Bucket-level equal split" and "Range class: four views";
// Megatron distributed-package page (2kiu.com) section 2.2 (2)-(3).
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <numeric>

#include "dopt_internal.h"

namespace {
thread_local std::string g_last_error;

int64_t round_up(int64_t x, int64_t d) { return ((x + d - 1) / d) * d; }

int64_t lcm64(int64_t a, int64_t b) { return a / std::gcd(a, b) * b; }

bool valid_dtype(int32_t d) { return d == DOPT_F32 || d == DOPT_BF16 || d == DOPT_F16; }

// Lays out the params of one buffer: walks them from the last registered
// to the first (roughly the order backward produces their grads), starts
// each at a multiple of 64 elements, and closes a bucket once it reaches
// bucket_size (or when a param asks for a bucket of its own), padding the
// closed bucket's end to the bucket divisor so every bucket splits evenly
// over the DP ranks.
void lay_out_buffer(dopt_shard_map* m, int32_t b, int64_t bucket_size, int64_t divisor) {
  dopt::Buffer& buf = m->buffers[b];
  int64_t bucket_begin = 0;  // first element of the bucket being filled
  int64_t next = 0;          // first free element
  int64_t last_end = 0;
  std::vector<int32_t> members;

  auto close_bucket = [&](int64_t end_unpadded) -> int64_t {
    dopt::Bucket bk;
    bk.offset = bucket_begin;
    int64_t end = round_up(end_unpadded, divisor);
    bk.numel = end - bucket_begin;
    bk.numel_unpadded = end_unpadded - bucket_begin;
    bk.params = members;
    buf.buckets.push_back(std::move(bk));
    members.clear();
    bucket_begin = end;
    return end;
  };

  for (auto it = buf.params.rbegin(); it != buf.params.rend(); ++it) {
    dopt::Param& p = m->params[*it];
    int64_t start = round_up(next, 64);
    if (p.new_bucket && !members.empty()) start = close_bucket(start);
    p.start = start;
    p.end = start + p.numel;
    p.bucket = (int32_t)buf.buckets.size();
    members.push_back(*it);
    last_end = p.end;
    bool full = bucket_size > 0 && p.end - bucket_begin >= bucket_size;
    next = (full || p.new_bucket) ? close_bucket(p.end) : p.end;
  }
  if (!members.empty()) close_bucket(last_end);

  int64_t shard_base = 0;
  for (dopt::Bucket& bk : buf.buckets) {
    std::sort(bk.params.begin(), bk.params.end(),
              [&](int32_t x, int32_t y) { return m->params[x].start < m->params[y].start; });
    bk.shard_base = shard_base;
    shard_base += bk.numel / m->dp;
    buf.numel_unpadded += bk.numel_unpadded;
  }
  buf.numel = buf.buckets.empty() ? 0 : buf.buckets.back().offset + buf.buckets.back().numel;
}

int64_t cache_key(int32_t buffer, int32_t rank) {
  return (int64_t)buffer * 1000003 + (int64_t)(rank + 1);
}
}  // namespace

namespace dopt {

int fail(int status, const std::string& msg) {
  g_last_error = msg;
  return status;
}

const std::vector<Run>& runs_for(dopt_shard_map* m, int32_t buffer, int32_t rank) {
  std::lock_guard<std::mutex> lock(m->mu);
  auto key = cache_key(buffer, rank);
  auto found = m->runs_cache.find(key);
  if (found != m->runs_cache.end()) return found->second;

  const Buffer& buf = m->buffers[buffer];
  const int64_t S = buf.numel / m->dp;
  std::vector<Run> runs;
  int32_t first = rank == DOPT_ALL_RANKS ? 0 : rank;
  int32_t last = rank == DOPT_ALL_RANKS ? m->dp - 1 : rank;
  for (int32_t r = first; r <= last; ++r) {
    int64_t slot_base = (int64_t)(r - first) * S;
    for (int32_t k = 0; k < (int32_t)buf.buckets.size(); ++k) {
      const Bucket& bk = buf.buckets[k];
      int64_t s = bk.numel / m->dp;
      int64_t w0 = bk.offset + (int64_t)r * s, w1 = w0 + s;
      for (int32_t pid : bk.params) {
        const Param& p = m->params[pid];
        int64_t lo = std::max(p.start, w0), hi = std::min(p.end, w1);
        if (hi <= lo) continue;
        Run run{slot_base + bk.shard_base + (lo - w0), lo, hi - lo, p.wd_mult, k};
        if (!runs.empty()) {
          Run& prev = runs.back();
          if (prev.local + prev.len == run.local && prev.world + prev.len == run.world &&
              prev.wd_mult == run.wd_mult && prev.bucket == run.bucket) {
            prev.len += run.len;
            continue;
          }
        }
        runs.push_back(run);
      }
    }
  }
  // keep every run below kMaxRunLen elements (kernel tables hold 32-bit lengths)
  std::vector<Run> split;
  for (const Run& r : runs) {
    for (int64_t o = 0; o < r.len; o += kMaxRunLen)
      split.push_back(Run{r.local + o, r.world + o, std::min(kMaxRunLen, r.len - o), r.wd_mult, r.bucket});
  }
  return m->runs_cache.emplace(key, std::move(split)).first->second;
}

}  // namespace dopt

extern "C" {

const char* dopt_last_error(void) { return g_last_error.c_str(); }

int dopt_build_shard_map(const dopt_param_desc* params, int32_t n_params, int32_t dp_size,
                         int64_t bucket_size, int32_t grad_reduce_in_fp32,
                         int32_t pad_for_high_busbw, dopt_shard_map** out) {
  if (!out) return dopt::fail(DOPT_E_INVALID, "dopt_build_shard_map: out is NULL");
  *out = nullptr;
  if (!params || n_params < 1)
    return dopt::fail(DOPT_E_INVALID, "dopt_build_shard_map: need at least one param");
  if (dp_size < 1) return dopt::fail(DOPT_E_INVALID, "dopt_build_shard_map: dp_size < 1");
  for (int32_t i = 0; i < n_params; ++i) {
    if (params[i].numel < 0 || !valid_dtype(params[i].dtype) || !std::isfinite(params[i].wd_mult))
      return dopt::fail(DOPT_E_INVALID, "dopt_build_shard_map: bad param " + std::to_string(i));
  }
  dopt_shard_map* m = new (std::nothrow) dopt_shard_map();
  if (!m) return dopt::fail(DOPT_E_NOMEM, "dopt_build_shard_map: out of host memory");
  try {
    m->dp = dp_size;
    // bucket size: default max(40M, 1M * DP); negative = no size trigger
    int64_t bs = bucket_size;
    if (bs == 0) bs = std::max<int64_t>(40000000, (int64_t)1000000 * dp_size);
    if (bs < 0) bs = 0;
    int64_t divisor = lcm64(dp_size, 128);
    if (pad_for_high_busbw) divisor = lcm64(divisor, 65536);

    m->params.resize(n_params);
    for (int32_t i = 0; i < n_params; ++i) {
      dopt::Param& p = m->params[i];
      p.numel = params[i].numel;
      p.dtype = params[i].dtype;
      p.new_bucket = params[i].new_bucket != 0;
      p.wd_mult = params[i].wd_mult;
      int32_t gdt = grad_reduce_in_fp32 ? DOPT_F32 : p.dtype;
      int32_t b = -1;
      for (size_t k = 0; k < m->buffers.size(); ++k)
        if (m->buffers[k].param_dtype == p.dtype && m->buffers[k].grad_dtype == gdt) b = (int32_t)k;
      if (b < 0) {
        dopt::Buffer nb;
        nb.param_dtype = p.dtype;
        nb.grad_dtype = gdt;
        m->buffers.push_back(nb);
        b = (int32_t)m->buffers.size() - 1;
      }
      p.buffer = b;
      m->buffers[b].params.push_back(i);
    }
    for (int32_t b = 0; b < (int32_t)m->buffers.size(); ++b) {
      lay_out_buffer(m, b, bs, divisor);
      const dopt::Buffer& buf = m->buffers[b];
      if (buf.numel_unpadded > buf.numel || buf.numel % dp_size != 0) {
        delete m;
        return dopt::fail(DOPT_E_INVALID, "dopt_build_shard_map: inconsistent layout");
      }
    }
  } catch (const std::bad_alloc&) {
    delete m;
    return dopt::fail(DOPT_E_NOMEM, "dopt_build_shard_map: out of host memory");
  }
  *out = m;
  return DOPT_OK;
}

void dopt_shard_map_free(dopt_shard_map* map) { delete map; }

int32_t dopt_num_buffers(const dopt_shard_map* m) {
  if (!m) return dopt::fail(DOPT_E_INVALID, "dopt_num_buffers: NULL map");
  return (int32_t)m->buffers.size();
}

int32_t dopt_dp_size(const dopt_shard_map* m) {
  if (!m) return dopt::fail(DOPT_E_INVALID, "dopt_dp_size: NULL map");
  return m->dp;
}

int32_t dopt_total_buckets(const dopt_shard_map* m) {
  if (!m) return dopt::fail(DOPT_E_INVALID, "dopt_total_buckets: NULL map");
  int32_t n = 0;
  for (const dopt::Buffer& buf : m->buffers) n += (int32_t)buf.buckets.size();
  return n;
}

int32_t dopt_bucket_number(const dopt_shard_map* m, int32_t buffer, int32_t bucket) {
  if (!m || buffer < 0 || buffer >= (int32_t)m->buffers.size() || bucket < 0 ||
      bucket >= (int32_t)m->buffers[buffer].buckets.size())
    return dopt::fail(DOPT_E_INVALID, "dopt_bucket_number: bad map, buffer or bucket");
  int32_t n = 0;
  for (int32_t b = 0; b < buffer; ++b) n += (int32_t)m->buffers[b].buckets.size();
  return n + bucket;
}

int dopt_buffer_info_get(const dopt_shard_map* m, int32_t b, dopt_buffer_info* out) {
  if (!m || !out || b < 0 || b >= (int32_t)m->buffers.size())
    return dopt::fail(DOPT_E_INVALID, "dopt_buffer_info_get: bad map, buffer or out");
  const dopt::Buffer& buf = m->buffers[b];
  out->param_dtype = buf.param_dtype;
  out->grad_dtype = buf.grad_dtype;
  out->group = buf.param_dtype == DOPT_F32 ? DOPT_GROUP_FP32 : DOPT_GROUP_FP32_FROM_FLOAT16;
  out->n_buckets = (int32_t)buf.buckets.size();
  out->n_params = (int32_t)buf.params.size();
  out->reserved = 0;
  out->numel = buf.numel;
  out->numel_unpadded = buf.numel_unpadded;
  out->shard_numel = buf.numel / m->dp;
  return DOPT_OK;
}

int dopt_bucket_info_get(const dopt_shard_map* m, int32_t b, int32_t k, dopt_bucket_info* out) {
  if (!m || !out || b < 0 || b >= (int32_t)m->buffers.size() || k < 0 ||
      k >= (int32_t)m->buffers[b].buckets.size())
    return dopt::fail(DOPT_E_INVALID, "dopt_bucket_info_get: bad map, buffer, bucket or out");
  const dopt::Bucket& bk = m->buffers[b].buckets[k];
  out->offset = bk.offset;
  out->numel = bk.numel;
  out->numel_unpadded = bk.numel_unpadded;
  out->shard_numel = bk.numel / m->dp;
  out->shard_base = bk.shard_base;
  return DOPT_OK;
}

int dopt_param_index(const dopt_shard_map* m, int32_t param, int32_t* buffer, int64_t* start,
                     int64_t* end, int32_t* bucket) {
  if (!m || param < 0 || param >= (int32_t)m->params.size())
    return dopt::fail(DOPT_E_INVALID, "dopt_param_index: bad map or param");
  const dopt::Param& p = m->params[param];
  if (buffer) *buffer = p.buffer;
  if (start) *start = p.start;
  if (end) *end = p.end;
  if (bucket) *bucket = p.bucket;
  return DOPT_OK;
}

int dopt_rank_shards(const dopt_shard_map* m, int32_t b, int32_t rank, dopt_param_shard* out,
                     int32_t cap, int32_t* count) {
  if (!m || !count || b < 0 || b >= (int32_t)m->buffers.size() || rank < 0 || rank >= m->dp ||
      cap < 0 || (cap > 0 && !out))
    return dopt::fail(DOPT_E_INVALID, "dopt_rank_shards: bad argument");
  const dopt::Buffer& buf = m->buffers[b];
  int32_t n = 0;
  for (int32_t k = 0; k < (int32_t)buf.buckets.size(); ++k) {
    const dopt::Bucket& bk = buf.buckets[k];
    int64_t s = bk.numel / m->dp;
    int64_t w0 = bk.offset + (int64_t)rank * s, w1 = w0 + s;
    for (int32_t pid : bk.params) {
      const dopt::Param& p = m->params[pid];
      int64_t lo = std::max(p.start, w0), hi = std::min(p.end, w1);
      if (hi <= lo) continue;
      if (n < cap) {
        dopt_param_shard& o = out[n];
        o.param = pid;
        o.buffer = b;
        o.bucket = k;
        o.rank = rank;
        o.gbuf_world = {lo, hi};
        o.gbuf_world_in_bucket = {lo - bk.offset, hi - bk.offset};
        o.gbuf_local = {lo - w0, hi - w0};
        o.param_range = {lo - p.start, hi - p.start};
        o.shard_offset = bk.shard_base + (lo - w0);
      }
      ++n;
    }
  }
  *count = n;
  return DOPT_OK;
}

int64_t dopt_memory_ledger(int64_t P, int32_t N, int32_t stage, int64_t* parts_out) {
  if (P < 0 || N < 1 || stage < 0 || stage > 3)
    return dopt::fail(DOPT_E_INVALID, "dopt_memory_ledger: bad P, N or stage");
  const int64_t shard = (P + N - 1) / N;  // elements of a sharded part per card
  // bytes per param: 16-bit param 2, 16-bit grad 2, fp32 master 4, m 4, v 4
  const int64_t param = 2 * (stage >= 3 ? shard : P);
  const int64_t grad = 2 * (stage >= 2 ? shard : P);
  const int64_t state = 4 * (stage >= 1 ? shard : P);
  if (parts_out) {
    parts_out[0] = param;
    parts_out[1] = grad;
    parts_out[2] = state;
    parts_out[3] = state;
    parts_out[4] = state;
  }
  return param + grad + 3 * state;
}

int64_t dopt_comm_bytes(int64_t P, int32_t N, int32_t elem_bytes, int32_t kind) {
  if (P < 0 || N < 1 || elem_bytes < 1 || kind < 0 || kind > 2)
    return dopt::fail(DOPT_E_INVALID, "dopt_comm_bytes: bad argument");
  const int64_t chunk = (P + N - 1) / N;  // one rank's slice, P padded to N slices
  const int64_t one_pass = (int64_t)(N - 1) * chunk * elem_bytes;
  return kind == 2 ? 2 * one_pass : one_pass;
}

int dopt_loss_scaler_init(dopt_loss_scaler* s, double initial_scale, double growth_factor,
                          double backoff_factor, int32_t growth_interval, int32_t hysteresis,
                          double min_scale) {
  if (!s || !(initial_scale > 0) || !(growth_factor >= 1) || !(backoff_factor > 0) ||
      !(backoff_factor <= 1) || growth_interval < 1 || hysteresis < 1 || !(min_scale > 0))
    return dopt::fail(DOPT_E_INVALID, "dopt_loss_scaler_init: bad argument");
  s->scale = initial_scale;
  s->growth_factor = growth_factor;
  s->backoff_factor = backoff_factor;
  s->min_scale = min_scale;
  s->growth_interval = growth_interval;
  s->hysteresis = hysteresis;
  s->growth_tracker = 0;
  s->hysteresis_tracker = hysteresis;
  return DOPT_OK;
}

int dopt_loss_scaler_update(dopt_loss_scaler* s, int32_t found_inf) {
  if (!s) return dopt::fail(DOPT_E_INVALID, "dopt_loss_scaler_update: NULL scaler");
  if (found_inf) {
    s->growth_tracker = 0;
    s->hysteresis_tracker -= 1;
    if (s->hysteresis_tracker <= 0) s->scale = std::max(s->scale * s->backoff_factor, s->min_scale);
  } else {
    s->growth_tracker += 1;
    if (s->growth_tracker == s->growth_interval) {
      s->growth_tracker = 0;
      s->hysteresis_tracker = s->hysteresis;
      s->scale *= s->growth_factor;
    }
  }
  return DOPT_OK;
}

}  // extern "C"
