/*
 * synth_host.c -- host fills of the seeded synthetic input generator (synth.h).
 * Exported with a C ABI for the tests, the benchmark and the oracle's streaming
 * checks.  No optimizer arithmetic lives here.
 */
#include <stddef.h>
#include <stdint.h>
#include "synth.h"
#include "synth_kinds.h"

uint64_t synth_key_for(uint64_t seed, uint32_t stream, uint32_t step, uint32_t replica) {
  return synth_key(seed, stream, step, replica);
}

void synth_fill_normal(void* dst, int32_t kind, int64_t n, uint64_t key,
                       uint64_t index0, float factor) {
  for (int64_t i = 0; i < n; ++i) {
    float x = synth_normal(key, index0 + (uint64_t)i, factor);
    switch (kind) {
      case SYNTH_OUT_F32: ((float*)dst)[i] = x; break;
      case SYNTH_OUT_BF16: ((uint16_t*)dst)[i] = synth_bf16_trunc_bits(x); break;
      case SYNTH_OUT_F16: ((uint16_t*)dst)[i] = synth_f16_trunc_bits(x); break;
      case SYNTH_OUT_F32_OF_BF16: ((float*)dst)[i] = synth_bf16_trunc_value(x); break;
      case SYNTH_OUT_F32_OF_F16: ((float*)dst)[i] = synth_f16_trunc_value(x); break;
      default: return;
    }
  }
}

void synth_fill_uniform_f32(float* dst, int64_t n, uint64_t key, uint64_t index0,
                            float scale) {
  for (int64_t i = 0; i < n; ++i) dst[i] = synth_uniform(key, index0 + (uint64_t)i, scale);
}

/* Per-element bits, exposed so tests can check the definition itself. */
uint64_t synth_bits_at(uint64_t key, uint64_t index) { return synth_bits(key, index); }

/* Values of one stream at arbitrary indices (for sampled checks). */
void synth_gather_normal(void* dst, int32_t kind, const uint64_t* indices, int64_t n,
                         uint64_t key, float factor) {
  for (int64_t i = 0; i < n; ++i) synth_fill_normal((char*)dst + i * (kind == SYNTH_OUT_BF16 || kind == SYNTH_OUT_F16 ? 2 : 4),
                                                    kind, 1, key, indices[i], factor);
}
