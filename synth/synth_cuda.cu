/*
 * synth_cuda.cu -- device fills of the seeded synthetic input generator
 * (synth.h).  Bit-identical to the host fills in synth_host.c: the same
 * integer hash, one exact int->float conversion and one round-to-nearest fp32
 * multiply per value.  No optimizer arithmetic lives here.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "synth.h"
#include "synth_kinds.h"

template <int KIND>
__global__ void synth_normal_kernel(void* __restrict__ dst, int64_t n, uint64_t key,
                                    uint64_t index0, float factor) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    float x = synth_normal(key, index0 + (uint64_t)i, factor);
    if (KIND == SYNTH_OUT_F32) ((float*)dst)[i] = x;
    if (KIND == SYNTH_OUT_BF16) ((uint16_t*)dst)[i] = synth_bf16_trunc_bits(x);
    if (KIND == SYNTH_OUT_F16) ((uint16_t*)dst)[i] = synth_f16_trunc_bits(x);
    if (KIND == SYNTH_OUT_F32_OF_BF16) ((float*)dst)[i] = synth_bf16_trunc_value(x);
    if (KIND == SYNTH_OUT_F32_OF_F16) ((float*)dst)[i] = synth_f16_trunc_value(x);
  }
}

__global__ void synth_uniform_kernel(float* __restrict__ dst, int64_t n, uint64_t key,
                                     uint64_t index0, float scale) {
  int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
    dst[i] = synth_uniform(key, index0 + (uint64_t)i, scale);
}

static int synth_grid(int64_t n) {
  int64_t blocks = (n + 255) / 256;
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  return (int)blocks;
}

extern "C" int synth_cuda_fill_normal(void* dst, int32_t kind, int64_t n, uint64_t key,
                                      uint64_t index0, float factor, void* stream) {
  if (n <= 0) return 0;
  if (dst == nullptr) return (int)cudaErrorInvalidValue;
  cudaStream_t s = (cudaStream_t)stream;
  int g = synth_grid(n);
  switch (kind) {
    case SYNTH_OUT_F32: synth_normal_kernel<SYNTH_OUT_F32><<<g, 256, 0, s>>>(dst, n, key, index0, factor); break;
    case SYNTH_OUT_BF16: synth_normal_kernel<SYNTH_OUT_BF16><<<g, 256, 0, s>>>(dst, n, key, index0, factor); break;
    case SYNTH_OUT_F16: synth_normal_kernel<SYNTH_OUT_F16><<<g, 256, 0, s>>>(dst, n, key, index0, factor); break;
    case SYNTH_OUT_F32_OF_BF16: synth_normal_kernel<SYNTH_OUT_F32_OF_BF16><<<g, 256, 0, s>>>(dst, n, key, index0, factor); break;
    case SYNTH_OUT_F32_OF_F16: synth_normal_kernel<SYNTH_OUT_F32_OF_F16><<<g, 256, 0, s>>>(dst, n, key, index0, factor); break;
    default: return (int)cudaErrorInvalidValue;
  }
  return (int)cudaGetLastError();
}

extern "C" int synth_cuda_fill_uniform_f32(float* dst, int64_t n, uint64_t key,
                                           uint64_t index0, float scale, void* stream) {
  if (n <= 0) return 0;
  if (dst == nullptr) return (int)cudaErrorInvalidValue;
  synth_uniform_kernel<<<synth_grid(n), 256, 0, (cudaStream_t)stream>>>(dst, n, key, index0, scale);
  return (int)cudaGetLastError();
}
