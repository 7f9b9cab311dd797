// dopt_internal.h -- host-side structures shared by the shard-map code and
// the CUDA entry points of the library.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/dopt.h"

namespace dopt {

struct Param {
  int64_t numel = 0;
  int32_t dtype = DOPT_F32;
  bool new_bucket = false;
  double wd_mult = 1.0;
  int32_t buffer = -1;
  int32_t bucket = -1;
  int64_t start = 0, end = 0;  // position in its buffer
};

struct Bucket {
  int64_t offset = 0, numel = 0, numel_unpadded = 0, shard_base = 0;
  std::vector<int32_t> params;  // sorted by start
};

struct Buffer {
  int32_t param_dtype = DOPT_F32, grad_dtype = DOPT_F32;
  std::vector<int32_t> params;  // model order
  std::vector<Bucket> buckets;
  int64_t numel = 0, numel_unpadded = 0;
};

// A maximal run of one rank's shard that is contiguous both in the flat
// shard (local) and in the buffer (world) and has one weight-decay
// multiplier.  Runs never cover padding.
struct Run {
  int64_t local = 0;  // includes the rank slot (slot * shard_numel) in all-ranks mode
  int64_t world = 0;
  int64_t len = 0;
  double wd_mult = 1.0;
  int32_t bucket = 0;  // runs never span two buckets
};

}  // namespace dopt

struct dopt_shard_map {
  int32_t dp = 1;
  std::vector<dopt::Param> params;
  std::vector<dopt::Buffer> buffers;
  // runs per (buffer, rank selection), built on first use
  std::mutex mu;
  std::unordered_map<int64_t, std::vector<dopt::Run>> runs_cache;
};

namespace dopt {

// Sets the thread-local error message and returns the status.
int fail(int status, const std::string& msg);

// Runs of `rank` (or every rank, rank-major, for DOPT_ALL_RANKS) in a buffer.
// Runs are at most kMaxRunLen elements long.
const std::vector<Run>& runs_for(dopt_shard_map* map, int32_t buffer, int32_t rank);

constexpr int64_t kMaxRunLen = int64_t(1) << 30;

inline int64_t shard_numel(const dopt_shard_map* m, int32_t buffer) {
  return m->buffers[buffer].numel / m->dp;
}
inline int32_t n_rank_slots(const dopt_shard_map* m, int32_t rank) {
  return rank == DOPT_ALL_RANKS ? m->dp : 1;
}

}  // namespace dopt
