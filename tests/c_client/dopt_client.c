/*
 * dopt_client.c -- a plain C11 client of the library's C ABI (include/dopt.h),
 * used by tests/test_c_client.py to show that the boundary works from C with
 * no Python and no torch in between.
 *
 *   dopt_client map          prints the shard map of a fixed param list as
 *                            text lines (host only, no GPU needed)
 *   dopt_client step OUTDIR  (built with -DDOPT_CLIENT_CUDA) runs one fused
 *                            step on cudaMalloc'd buffers and writes the
 *                            results to OUTDIR for the test to compare with
 *                            the CPU oracle
 *
 * The param list, the inputs and the hyper-parameters are fixed here and
 * restated by the test: every input is a small multiple of a power of two,
 * exact in fp32 and (for the params) in bf16.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "dopt.h"

#define N_PARAMS 4
static const dopt_param_desc PARAMS[N_PARAMS] = {
    {1000, DOPT_BF16, 0, 1.0}, {300, DOPT_F32, 0, 0.0}, {2500, DOPT_BF16, 0, 1.0}, {77, DOPT_BF16, 1, 0.5}};
#define DP 4
#define DP_MAX DP
static const int64_t BUCKET = 1500;

static int fail(const char* what, int st) {
  fprintf(stderr, "%s failed (%d): %s\n", what, st, dopt_last_error());
  return 1;
}

static int print_map(const dopt_shard_map* m) {
  int32_t nb = dopt_num_buffers(m);
  printf("buffers %d\n", nb);
  for (int32_t b = 0; b < nb; ++b) {
    dopt_buffer_info bi;
    int st = dopt_buffer_info_get(m, b, &bi);
    if (st) return fail("dopt_buffer_info_get", st);
    printf("buffer %d param_dtype %d grad_dtype %d numel %lld numel_unpadded %lld shard_numel %lld buckets %d\n", b,
           bi.param_dtype, bi.grad_dtype, (long long)bi.numel, (long long)bi.numel_unpadded, (long long)bi.shard_numel,
           bi.n_buckets);
    for (int32_t k = 0; k < bi.n_buckets; ++k) {
      dopt_bucket_info bk;
      if ((st = dopt_bucket_info_get(m, b, k, &bk))) return fail("dopt_bucket_info_get", st);
      printf("bucket %d %d offset %lld numel %lld numel_unpadded %lld\n", b, k, (long long)bk.offset,
             (long long)bk.numel, (long long)bk.numel_unpadded);
    }
    for (int32_t r = 0; r < DP; ++r) {
      int32_t count = 0;
      if ((st = dopt_rank_shards(m, b, r, NULL, 0, &count))) return fail("dopt_rank_shards", st);
      dopt_param_shard* ps = (dopt_param_shard*)calloc((size_t)(count > 0 ? count : 1), sizeof(dopt_param_shard));
      if ((st = dopt_rank_shards(m, b, r, ps, count, &count))) return fail("dopt_rank_shards", st);
      for (int32_t j = 0; j < count; ++j)
        printf("piece %d %d param %d bucket %d world %lld %lld param_range %lld %lld shard_offset %lld\n", b, r,
               ps[j].param, ps[j].bucket, (long long)ps[j].gbuf_world.start, (long long)ps[j].gbuf_world.end,
               (long long)ps[j].param_range.start, (long long)ps[j].param_range.end, (long long)ps[j].shard_offset);
      free(ps);
    }
  }
  return 0;
}

#ifdef DOPT_CLIENT_CUDA
#include <cuda_runtime_api.h>

#define MAX_BUF 4

/* Replica k's gradient at element i of buffer b. */
static float grad_value(int b, int k, int64_t i) { return (float)((i * 37 + k * 11 + b * 5) % 29 - 14) / 1024.0f; }
/* The param at element i of buffer b (exact in bf16). */
static float param_value(int b, int64_t i) { return (float)((i * 13 + b) % 41 - 20) / 256.0f; }

static uint16_t bf16_bits(float x) { /* exact for the values above */
  uint32_t u;
  memcpy(&u, &x, 4);
  return (uint16_t)(u >> 16);
}
static float bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, 4);
  return x;
}

#define CK(call)                                                            \
  do {                                                                      \
    cudaError_t e_ = (call);                                                \
    if (e_ != cudaSuccess) {                                                \
      fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));           \
      return 1;                                                             \
    }                                                                       \
  } while (0)

static int write_file(const char* dir, const char* name, int b, const void* data, size_t bytes) {
  char path[4096];
  snprintf(path, sizeof path, "%s/b%d_%s.bin", dir, b, name);
  FILE* f = fopen(path, "wb");
  if (!f || fwrite(data, 1, bytes, f) != bytes) return 1;
  fclose(f);
  return 0;
}

static int run_step(const dopt_shard_map* m, const char* outdir) {
  const int32_t nb = dopt_num_buffers(m);
  if (nb < 1 || nb > MAX_BUF) return fail("buffer count", nb);
  const void* reps[MAX_BUF][DP_MAX];
  const void* const* rep_rows[MAX_BUF];
  float *main_d[MAX_BUF], *master_d[MAX_BUF], *m_d[MAX_BUF], *v_d[MAX_BUF];
  void* param_d[MAX_BUF];
  dopt_buffer_info info[MAX_BUF];
  int st;
  for (int32_t b = 0; b < nb; ++b) {
    if ((st = dopt_buffer_info_get(m, b, &info[b]))) return fail("dopt_buffer_info_get", st);
    const int64_t n = info[b].numel, S = info[b].shard_numel, nl = DP * S;
    float* g = (float*)malloc((size_t)n * 4);
    for (int k = 0; k < DP; ++k) {
      for (int64_t i = 0; i < n; ++i) g[i] = grad_value(b, k, i);
      void* d = NULL;
      CK(cudaMalloc(&d, (size_t)n * 4));
      CK(cudaMemcpy(d, g, (size_t)n * 4, cudaMemcpyHostToDevice));
      reps[b][k] = d;
    }
    free(g);
    rep_rows[b] = reps[b];
    const int bf16 = info[b].param_dtype == DOPT_BF16;
    const size_t pbytes = (size_t)n * (bf16 ? 2 : 4);
    unsigned char* p = (unsigned char*)malloc(pbytes);
    for (int64_t i = 0; i < n; ++i) {
      if (bf16) ((uint16_t*)p)[i] = bf16_bits(param_value(b, i));
      else ((float*)p)[i] = param_value(b, i);
    }
    CK(cudaMalloc(&param_d[b], pbytes));
    CK(cudaMemcpy(param_d[b], p, pbytes, cudaMemcpyHostToDevice));
    float* zero = (float*)calloc((size_t)nl, 4);
    CK(cudaMalloc((void**)&main_d[b], (size_t)nl * 4));
    CK(cudaMalloc((void**)&m_d[b], (size_t)nl * 4));
    CK(cudaMalloc((void**)&v_d[b], (size_t)nl * 4));
    CK(cudaMemcpy(m_d[b], zero, (size_t)nl * 4, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(v_d[b], zero, (size_t)nl * 4, cudaMemcpyHostToDevice));
    master_d[b] = NULL;
    if (bf16) {  /* the fp32 master of every rank's shard, from the param buffer */
      float* master = zero;
      for (int32_t r = 0; r < DP; ++r) {
        int32_t count = 0;
        if ((st = dopt_rank_shards(m, b, r, NULL, 0, &count))) return fail("dopt_rank_shards", st);
        dopt_param_shard* ps = (dopt_param_shard*)calloc((size_t)(count > 0 ? count : 1), sizeof *ps);
        if ((st = dopt_rank_shards(m, b, r, ps, count, &count))) return fail("dopt_rank_shards", st);
        for (int32_t j = 0; j < count; ++j)
          for (int64_t e = 0; e < ps[j].gbuf_world.end - ps[j].gbuf_world.start; ++e)
            master[r * S + ps[j].shard_offset + e] = bf16_value(((uint16_t*)p)[ps[j].gbuf_world.start + e]);
        free(ps);
      }
      CK(cudaMalloc((void**)&master_d[b], (size_t)nl * 4));
      CK(cudaMemcpy(master_d[b], master, (size_t)nl * 4, cudaMemcpyHostToDevice));
    }
    free(zero);
    free(p);
  }
  const size_t ws_bytes = dopt_workspace_bytes(m, DOPT_ALL_RANKS);
  void* ws = NULL;
  CK(cudaMalloc(&ws, ws_bytes));

  dopt_step_args a;
  memset(&a, 0, sizeof a);
  a.map = m;
  a.rank = DOPT_ALL_RANKS;
  a.n_instances = 1;
  a.layout = DOPT_LAYOUT_FULL_BUFFER;
  a.replica_grads = rep_rows;
  a.main_grad = main_d;
  a.master = master_d;
  a.exp_avg = m_d;
  a.exp_avg_sq = v_d;
  a.param_buffer = param_d;
  a.inv_loss_scale = 1.0f;
  a.max_norm = 0.5;
  a.hp.lr = 1e-3;
  a.hp.beta1 = 0.9;
  a.hp.beta2 = 0.95;
  a.hp.eps = 1e-8;
  a.hp.weight_decay = 0.1;
  a.hp.step = 1;
  a.workspace = ws;
  a.workspace_bytes = ws_bytes;
  a.grad_scale = 1.0f;
  int32_t found = -1;
  float norm = 0.f;
  if ((st = dopt_step(&a, &found, &norm))) return fail("dopt_step", st);
  CK(cudaDeviceSynchronize());

  char path[4096];
  snprintf(path, sizeof path, "%s/result.txt", outdir);
  FILE* f = fopen(path, "w");
  if (!f) return 1;
  fprintf(f, "%d %.9g\n", found, norm);
  fclose(f);
  for (int32_t b = 0; b < nb; ++b) {
    const int64_t n = info[b].numel, nl = DP * info[b].shard_numel;
    const size_t pbytes = (size_t)n * (info[b].param_dtype == DOPT_BF16 ? 2 : 4);
    void* h = malloc(pbytes > (size_t)nl * 4 ? pbytes : (size_t)nl * 4);
    CK(cudaMemcpy(h, param_d[b], pbytes, cudaMemcpyDeviceToHost));
    if (write_file(outdir, "param", b, h, pbytes)) return 1;
    const struct { const char* name; float* d; } outs[3] = {{"master", master_d[b]}, {"exp_avg", m_d[b]},
                                                           {"exp_avg_sq", v_d[b]}};
    for (int o = 0; o < 3; ++o) {
      if (!outs[o].d) continue;
      CK(cudaMemcpy(h, outs[o].d, (size_t)nl * 4, cudaMemcpyDeviceToHost));
      if (write_file(outdir, outs[o].name, b, h, (size_t)nl * 4)) return 1;
    }
    free(h);
  }
  return 0;
}
#endif

int main(int argc, char** argv) {
  if (argc < 2) {
    fprintf(stderr, "usage: %s map | step OUTDIR\n", argv[0]);
    return 2;
  }
  dopt_shard_map* m = NULL;
  int st = dopt_build_shard_map(PARAMS, N_PARAMS, DP, BUCKET, 1, 0, &m);
  if (st) return fail("dopt_build_shard_map", st);
  int rc = 2;
  if (strcmp(argv[1], "map") == 0) rc = print_map(m);
#ifdef DOPT_CLIENT_CUDA
  else if (strcmp(argv[1], "step") == 0 && argc > 2) rc = run_step(m, argv[2]);
#endif
  dopt_shard_map_free(m);
  return rc;
}
