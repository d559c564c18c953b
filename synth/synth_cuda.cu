// Device filler of the seeded input generator (definition in synth_hash.h):
// fills large tensors in HBM with the same bits the host filler produces.
// Test and benchmark inputs only; no fused GEMM + epilogue arithmetic here.
#include <cuda_runtime.h>
#include <stdint.h>

#include "synth_hash.h"

namespace {

__global__ void fill_normal_kernel(void* out, int dtype, uint64_t rows, uint64_t cols,
                                   uint64_t key, float scale) {
  const uint64_t total = rows * cols;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += stride) {
    // __fmul_rn: one rounded multiply, never contracted into anything else
    float v = __fmul_rn((float)synth_irwin_hall8(key, e), scale);
    if (dtype == SYNTH_F16)
      ((uint16_t*)out)[e] = synth_f32_to_f16_bits(v);
    else if (dtype == SYNTH_BF16)
      ((uint16_t*)out)[e] = synth_f32_to_bf16_bits(v);
    else
      ((float*)out)[e] = v;
  }
}

__global__ void fill_mask_kernel(uint32_t* out, uint64_t M, uint64_t N, uint64_t nw,
                                 uint64_t key) {
  const uint64_t total = nw * N;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    uint64_t w = i / N;
    int64_t valid = (int64_t)M - 32 * (int64_t)w;
    uint32_t keep = valid >= 32 ? 0xFFFFFFFFu : (valid <= 0 ? 0u : ((1u << valid) - 1u));
    out[i] = (uint32_t)synth_at(key, i) & keep;
  }
}

int grid_for(uint64_t total) {
  uint64_t blocks = (total + 255) / 256;
  if (blocks > 152ull * 32ull) blocks = 152ull * 32ull;
  if (blocks == 0) blocks = 1;
  return (int)blocks;
}

}  // namespace

extern "C" float synth_scale(double sigma);

// Fill a device [rows, cols] row-major tensor with N(0, sigma) draws.
// Returns a cudaError_t value (0 on success).
extern "C" int synth_dev_fill_normal(void* dptr, int dtype, int64_t rows, int64_t cols,
                                     uint64_t seed, uint32_t tensor_id, double sigma,
                                     void* stream) {
  if (rows < 0 || cols < 0 || (dtype != SYNTH_F16 && dtype != SYNTH_BF16 && dtype != SYNTH_F32))
    return (int)cudaErrorInvalidValue;
  uint64_t total = (uint64_t)rows * (uint64_t)cols;
  if (total == 0) return 0;
  fill_normal_kernel<<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(
      dptr, dtype, (uint64_t)rows, (uint64_t)cols, synth_key(seed, tensor_id), synth_scale(sigma));
  return (int)cudaGetLastError();
}

// Fill the device column-word Bernoulli(1/2) mask of logical shape [M, N]
// (ceil(M/32) word-rows of N uint32).
extern "C" int synth_dev_fill_mask_words(uint32_t* dptr, int64_t M, int64_t N, uint64_t seed,
                                         uint32_t tensor_id, void* stream) {
  if (M < 0 || N < 0) return (int)cudaErrorInvalidValue;
  uint64_t nw = ((uint64_t)M + 31) / 32;
  uint64_t total = nw * (uint64_t)N;
  if (total == 0) return 0;
  fill_mask_kernel<<<grid_for(total), 256, 0, (cudaStream_t)stream>>>(
      dptr, (uint64_t)M, (uint64_t)N, nw, synth_key(seed, tensor_id));
  return (int)cudaGetLastError();
}
