/*
 * oracle.c -- plain, slow, scalar CPU oracle of the numeric steps of the
 * sharded mixed-precision Adam step (Megatron DistributedOptimizer, ZeRO-1).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this code; the product path never
 * does.  It shares no code with the CUDA path; its only shared dependency is
 * the seeded input generator (synth/synth.h), used by the streaming checks.
 *
 * Compiled with -O2 -ffp-contract=off: every fp32 operation below rounds
 * once, in the order written.  The steps follow the pages in their order:
 *
 *   A2 reduce-scatter (emulated): "Distributed optimizer" page (xiaolong-dev,
 *      megatron-docs/optimizer/distrib_optimizer), section 7.1 start_grad_sync;
 *      the Megatron distributed-package page, section 2.2 (4) gradient scaling
 *      (prescale 1/dp_size and SUM, or AVG in the collective); the ZeRO ledger
 *      page (llm-infra-atlas 02_zero_and_distributed_optimizer), section 5
 *      (distributed-optimizer instances: reduce-scatter inside an instance,
 *      all-reduce between instances).
 *   A2' scale_gradients: the Megatron distributed-package page, section 4.6
 *      (per-token loss normalization: after the data-parallel grad sync, the
 *      reduced grads are multiplied by 1/num_tokens in the grad buffer; read
 *      as one multiply rounded to the grad dtype).  A factor of 1 is the
 *      identity and skips the step.
 *   A2 check (check_for_nan_in_grad / check_for_large_grads): the Megatron
 *      distributed-package page, sections 2.4 and 3.2 -- each bucket's grads
 *      looked at for NaN, Inf and large values before the communication
 *      (read as: the largest |g| per replica and bucket).
 *   A3 prepare_grads: distrib_optimizer page, "MixedPrecisionOptimizer" layer
 *      (copy to fp32 main grad, unscale, inf/NaN detection) and the grad copy
 *      listing (bf16 -> fp32 .float()).
 *   A4 norm and clip: distrib_optimizer page, MegatronOptimizer utilities
 *      (clip_grad_norm / get_grad_norm) and the step skeleton (prepare ->
 *      clip -> step_with_ready_grads).
 *   A5 AdamW on the fp32 shard: distrib_optimizer page, "Why a distributed
 *      optimizer" (fp32 master, m, v) and the optimizer-type assertion
 *      (torch.optim.AdamW).  No equation is printed on any page; the reading
 *      taken is torch AdamW: decoupled decay first, then bias-corrected
 *      m / (sqrt(v) + eps).
 *   A6 write-back: distrib_optimizer page, _copy_main_params_to_model_params
 *      listing (fp32 -> bf16 copy_, read as round-to-nearest-even).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#include "../synth/synth.h"

enum { OR_F32 = 0, OR_BF16 = 1, OR_F16 = 2 };

/* ------------------------------------------------------------------------ */
/* Exact widening of 16-bit floats to fp32, from the IEEE / bfloat16 formats. */

static float or_bits_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}
static uint32_t or_f32_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

float or_bf16_to_f32(uint16_t h) { return or_bits_f32((uint32_t)h << 16); }

float or_f16_to_f32(uint16_t h) {
  uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
  int32_t exp = (h >> 10) & 0x1F;
  uint32_t man = h & 0x3FFu;
  if (exp == 31) /* inf / NaN */
    return or_bits_f32(sign | 0x7F800000u | (man << 13));
  if (exp == 0) { /* zero / subnormal: man * 2^-24, exact */
    float v = ldexpf((float)man, -24);
    return sign ? -v : v;
  }
  {
    float v = ldexpf((float)(man | 0x400u), exp - 25);
    return sign ? -v : v;
  }
}

float or_widen(const void* p, int32_t dt, int64_t i) {
  if (dt == OR_F32) return ((const float*)p)[i];
  if (dt == OR_BF16) return or_bf16_to_f32(((const uint16_t*)p)[i]);
  return or_f16_to_f32(((const uint16_t*)p)[i]);
}

/* ------------------------------------------------------------------------ */
/* Round-to-nearest-even of fp32 to bfloat16 and to binary16, written from
 * the definition: keep the leading bits, look at the dropped remainder,
 * round up when it is above half an ulp, or exactly half with an odd kept
 * part.  NaN stays NaN; overflow goes to infinity. */

uint16_t or_round_bf16(float x) {
  uint32_t u = or_f32_bits(x);
  uint32_t kept = u >> 16, rem = u & 0xFFFFu;
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) /* NaN */
    return (uint16_t)(kept | 0x0040u);
  if (rem > 0x8000u || (rem == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

uint16_t or_round_f16(float x) {
  uint32_t u = or_f32_bits(x);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  uint32_t absu = u & 0x7FFFFFFFu;
  if (absu > 0x7F800000u) return (uint16_t)(sign | 0x7E00u); /* NaN */
  if (absu == 0x7F800000u) return (uint16_t)(sign | 0x7C00u);
  {
    float a = or_bits_f32(absu);
    if (a >= 65520.0f) return (uint16_t)(sign | 0x7C00u); /* rounds past 65504 */
    if (a < 6.103515625e-05f) {
      /* subnormal range: count units of 2^-24, round to an integer */
      float q = a * 16777216.0f; /* exact: scaling by 2^24 */
      uint32_t fl = (uint32_t)q;
      float frac = q - (float)fl; /* exact */
      if (frac > 0.5f || (frac == 0.5f && (fl & 1u))) fl += 1u;
      return (uint16_t)(sign | fl); /* fl == 0x400 encodes 2^-14 */
    }
    {
      int32_t e = (int32_t)(absu >> 23) - 127;            /* -14 .. 15 */
      uint32_t sig = (absu & 0x7FFFFFu) | 0x800000u;      /* 24 bits   */
      uint32_t kept = sig >> 13, rem = sig & 0x1FFFu;     /* 11 bits   */
      if (rem > 0x1000u || (rem == 0x1000u && (kept & 1u))) kept += 1u;
      if (kept == 0x800u) { kept = 0x400u; e += 1; }
      if (e + 15 >= 31) return (uint16_t)(sign | 0x7C00u);
      return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(kept & 0x3FFu));
    }
  }
}

float or_round_to(float x, int32_t dt) {
  if (dt == OR_BF16) return or_bf16_to_f32(or_round_bf16(x));
  if (dt == OR_F16) return or_f16_to_f32(or_round_f16(x));
  return x;
}

static int or_is_finite(float x) { return (or_f32_bits(x) & 0x7F800000u) != 0x7F800000u; }

/* ------------------------------------------------------------------------ */
/* A2: one element of the emulated reduce-scatter.
 *
 * g[k] holds replica k's gradient for the element, widened to fp32.  The
 * n_rep replicas form n_inst distributed-optimizer instances of
 * dpi = n_rep / n_inst ranks each (replica k belongs to instance k / dpi).
 *
 *   average_in_collective = 0: every replica is pre-scaled by 1/dp_size
 *     (dp_size = n_rep) and the collective sums.
 *   average_in_collective = 1: the collective averages: sum, then times
 *     1/dpi inside an instance and 1/n_inst between instances.
 *
 * A sum runs in replica order and starts from its first term.  The output of
 * the reduce-scatter inside an instance is in the grad buffer's dtype (one
 * rounding of the fp32 sum); with more than one instance, the all-reduce of
 * those outputs is summed in instance order and rounded to the grad dtype
 * again.
 */
static float or_reduce_element(const float* g, int32_t n_rep, int32_t n_inst,
                               int32_t gdt, int32_t average) {
  int32_t dpi = n_rep / n_inst;
  float pre = (float)(1.0 / (double)n_rep);
  float total = 0.0f;
  for (int32_t j = 0; j < n_inst; ++j) {
    float s = 0.0f;
    for (int32_t q = 0; q < dpi; ++q) {
      float x = g[j * dpi + q];
      float term = average ? x : x * pre;
      s = (q == 0) ? term : s + term;
    }
    if (average) s = s * (float)(1.0 / (double)dpi);
    s = or_round_to(s, gdt);
    total = (j == 0) ? s : total + s;
  }
  if (n_inst > 1) {
    if (average) total = total * (float)(1.0 / (double)n_inst);
    total = or_round_to(total, gdt);
  }
  return total;
}

/* A2': the reduced grad (in the grad dtype) times the scale_gradients
 * factor, rounded to the grad dtype; factor 1 leaves it unchanged. */
static float or_scale_gradients(float red, float factor, int32_t gdt) {
  if (factor == 1.0f) return red;
  return or_round_to(red * factor, gdt);
}

/*
 * A2 + A2' + A3 over a run of len elements.  rep[k] is replica k's array in
 * the grad dtype gdt; element j of the run sits at index rep_index0 + j in
 * every replica.  main_out[j] = fp32(scaled reduced grad) * inv_scale.
 * Returns the number of non-finite main-grad values written.
 */
int64_t or_reduce_prepare_run(const void* const* rep, int32_t n_rep, int32_t n_inst,
                              int32_t gdt, int32_t average, int64_t rep_index0,
                              int64_t len, float grad_scale, float inv_scale, float* main_out) {
  float g[256];
  int64_t bad = 0;
  if (n_rep <= 0 || n_rep > 256 || n_inst <= 0 || n_rep % n_inst) return -1;
  for (int64_t j = 0; j < len; ++j) {
    for (int32_t k = 0; k < n_rep; ++k) g[k] = or_widen(rep[k], gdt, rep_index0 + j);
    {
      float red = or_scale_gradients(or_reduce_element(g, n_rep, n_inst, gdt, average),
                                     grad_scale, gdt);
      float mg = red * inv_scale;
      main_out[j] = mg;
      if (!or_is_finite(mg)) ++bad;
    }
  }
  return bad;
}

/*
 * A2 check (check_for_nan_in_grad / check_for_large_grads): the Megatron
 * distributed-package page, section 2.4 (the bucket groups' check_grads
 * method looks at every bucket's gradients for NaN, Inf and unusually large
 * values before the communication) and the options table of section 3.2.
 * The pages give no threshold for "large"; the reading taken is the largest
 * magnitude, which a caller compares with its own threshold.  Over a run of
 * one replica's gradients as stored (grad dtype gdt, indices index0 ..
 * index0 + len - 1): returns NaN when the run holds a NaN, else the largest
 * |g| (+inf when it holds an infinity), 0 for an empty run.
 */
double or_grad_amax_run(const void* rep, int32_t gdt, int64_t index0, int64_t len) {
  double m = 0.0;
  for (int64_t j = 0; j < len; ++j) {
    double x = (double)or_widen(rep, gdt, index0 + j);
    if (x != x) return NAN;
    if (x < 0) x = -x;
    if (x > m) m = x;
  }
  return m;
}

/* A4: sum of squares of a run of main grads, in fp64, in index order. */
double or_sumsq_run(const float* main_grad, int64_t len) {
  double s = 0.0;
  for (int64_t j = 0; j < len; ++j) s += (double)main_grad[j] * (double)main_grad[j];
  return s;
}

/*
 * A4: from the global sum of squares to the reported norm and the clip
 * coefficient: norm = sqrt(sumsq); coef = max_norm / (norm + 1e-6), used
 * only when max_norm > 0 and coef < 1 (clip_grad_norm "if enabled").
 * Returns 1 when the gradients are to be scaled by *coef.
 */
int32_t or_clip_coef(double sumsq, double max_norm, double* norm_out, double* coef_out) {
  double norm = sqrt(sumsq);
  double coef = 1.0;
  int32_t clip = 0;
  if (max_norm > 0.0) {
    coef = max_norm / (norm + 1.0e-6);
    clip = coef < 1.0;
  }
  *norm_out = norm;
  *coef_out = clip ? coef : 1.0;
  return clip;
}

/* Hyper-parameters as the user gives them (double, like torch's Python floats). */
typedef struct {
  double lr, beta1, beta2, eps, weight_decay;
} or_hparams;

/* beta^t by the C library's pow, in double. */
static double or_pow(double b, int64_t t) { return pow(b, (double)t); }

/*
 * A5 + A6 over a run of len elements of one parameter's shard.
 *   g = main * (float)coef when clip, else main.
 *   Per element, in fp32, in this order (torch AdamW reading):
 *     p = p * decay                         decay = 1 - lr*wd*wd_mult
 *     m = beta1*m + (1-beta1)*g
 *     v = beta2*v + ((1-beta2)*g)*g
 *     denom = sqrt(v) / sqrt(1-beta2^t) + eps
 *     p = p - (lr / (1-beta1^t)) * (m / denom)
 *   The step-level scalars are computed in double and rounded once to fp32.
 *   param_out (may be NULL) receives the write-back of p in pdt: an RNE cast
 *   for bf16/fp16, the value itself for fp32.
 */
void or_adamw_run(const float* main_grad, int64_t len, double coef, int32_t clip,
                  float* master, float* exp_avg, float* exp_avg_sq,
                  const or_hparams* hp, double wd_mult, int64_t t,
                  void* param_out, int32_t pdt) {
  float b1 = (float)hp->beta1, b2 = (float)hp->beta2;
  float omb1 = (float)(1.0 - hp->beta1), omb2 = (float)(1.0 - hp->beta2);
  float eps = (float)hp->eps;
  float step_size = (float)(hp->lr / (1.0 - or_pow(hp->beta1, t)));
  float bc2_sqrt = (float)sqrt(1.0 - or_pow(hp->beta2, t));
  float decay = (float)(1.0 - hp->lr * hp->weight_decay * wd_mult);
  float c = (float)coef;
  for (int64_t j = 0; j < len; ++j) {
    float g = clip ? main_grad[j] * c : main_grad[j];
    float p = master[j] * decay;
    float m = b1 * exp_avg[j] + omb1 * g;
    float v = b2 * exp_avg_sq[j] + (omb2 * g) * g;
    float denom = sqrtf(v) / bc2_sqrt + eps;
    p = p - step_size * (m / denom);
    master[j] = p;
    exp_avg[j] = m;
    exp_avg_sq[j] = v;
    if (param_out) {
      if (pdt == OR_BF16) ((uint16_t*)param_out)[j] = or_round_bf16(p);
      else if (pdt == OR_F16) ((uint16_t*)param_out)[j] = or_round_f16(p);
      else ((float*)param_out)[j] = p;
    }
  }
}

/* ------------------------------------------------------------------------ */
/* Streaming form for full-size checks: the replica gradients of a run are
 * drawn from the seeded generator (synth.h) element by element instead of
 * being read from memory, so a shard of hundreds of millions of elements
 * can be checked without holding its replicas in host RAM.  Replica k of
 * the run is the generator stream keys[k]; element j is generator index
 * index0 + j, encoded in the grad dtype gdt by the generator's truncation.
 * Returns the fp64 sum of squares of the main grads; *n_bad receives the
 * count of non-finite main grads. */
double or_stream_sumsq(const uint64_t* keys, int32_t n_rep, int32_t n_inst,
                       int32_t gdt, int32_t average, float factor,
                       uint64_t index0, int64_t len, float grad_scale, float inv_scale,
                       int64_t* n_bad) {
  float g[256];
  double s = 0.0;
  int64_t bad = 0;
  if (n_rep <= 0 || n_rep > 256 || n_inst <= 0 || n_rep % n_inst) { *n_bad = -1; return 0.0; }
  for (int64_t j = 0; j < len; ++j) {
    for (int32_t k = 0; k < n_rep; ++k) {
      float x = synth_normal(keys[k], index0 + (uint64_t)j, factor);
      if (gdt == OR_BF16) g[k] = or_bf16_to_f32(synth_bf16_trunc_bits(x));
      else if (gdt == OR_F16) g[k] = or_f16_to_f32(synth_f16_trunc_bits(x));
      else g[k] = x;
    }
    {
      float mg = or_scale_gradients(or_reduce_element(g, n_rep, n_inst, gdt, average),
                                    grad_scale, gdt) * inv_scale;
      if (!or_is_finite(mg)) ++bad;
      s += (double)mg * (double)mg;
    }
  }
  *n_bad = bad;
  return s;
}

/* The same streaming draw as or_stream_sumsq, keeping the main grads: A2 +
 * A2' + A3 over a run whose replica k is generator stream keys[k] at
 * indices index0 .. index0 + len - 1.  main_out[j] receives the element's
 * main grad; returns the count of non-finite ones (-1 on bad counts).  Lets
 * a full-size check recompute every element of a window of whole buckets
 * without holding the replicas in host RAM. */
int64_t or_stream_reduce_prepare_run(const uint64_t* keys, int32_t n_rep, int32_t n_inst,
                                     int32_t gdt, int32_t average, float factor,
                                     uint64_t index0, int64_t len, float grad_scale,
                                     float inv_scale, float* main_out) {
  float g[256];
  int64_t bad = 0;
  if (n_rep <= 0 || n_rep > 256 || n_inst <= 0 || n_rep % n_inst) return -1;
  for (int64_t j = 0; j < len; ++j) {
    for (int32_t k = 0; k < n_rep; ++k) {
      float x = synth_normal(keys[k], index0 + (uint64_t)j, factor);
      if (gdt == OR_BF16) g[k] = or_bf16_to_f32(synth_bf16_trunc_bits(x));
      else if (gdt == OR_F16) g[k] = or_f16_to_f32(synth_f16_trunc_bits(x));
      else g[k] = x;
    }
    {
      float mg = or_scale_gradients(or_reduce_element(g, n_rep, n_inst, gdt, average),
                                    grad_scale, gdt) * inv_scale;
      main_out[j] = mg;
      if (!or_is_finite(mg)) ++bad;
    }
  }
  return bad;
}
