// Host-side view of the kernels: one launcher per epilog family, each
// dispatching on dtype, B storage and tile width to a template instance.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace gf {

struct LaunchArgs {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const CUtensorMap* tmB2;  // second B operand (SwiGLU up projection); else = tmB
  // CTA-pair kernel with 256 x 512 tiles: the 16-bit outputs out and aux_out
  // as TMA store targets (32 x 32 boxes, 64-byte swizzle); else = tmA
  const CUtensorMap* tmOut;
  const CUtensorMap* tmAux;
  const GemmParams* params;
  int grid;
  int bf16;     // 0: fp16, 1: bf16
  int b_mn;     // 1: B stored [K, N] (MN-major), 0: [N, K] (K-major)
  int tile_n;   // 128 or 256 (single-CTA kernel)
  int pair;     // 1: the CTA-pair kernel (256 x 256 tiles)
  int wide;     // with pair: 256 x 512 tiles (one accumulator in two halves)
  int split;    // with pair: split-k work units (256 x 256 tiles, EPILOG_NONE)
  int pdl;      // 1: programmatic dependent launch (set-up overlaps the previous kernel)
  cudaStream_t stream;
};

cudaError_t launch_none_bias(int epi, const LaunchArgs& a);   // EPI_NONE, EPI_BIAS
cudaError_t launch_relu(int epi, const LaunchArgs& a);        // EPI_RELU_BIAS, EPI_RELU_AUX_BIAS
cudaError_t launch_drelu(const LaunchArgs& a);                // EPI_DRELU_BGRAD
cudaError_t launch_gelu(int epi, const LaunchArgs& a);        // EPI_GELU_BIAS, _AUX_BIAS, EPI_DGELU_BGRAD
cudaError_t launch_swiglu(int epi, const LaunchArgs& a);      // EPI_SWIGLU, _SAVE, EPI_DSWIGLU
cudaError_t launch_bgrad_finalize(const float* partial, int num_m_blocks, int n, float* bgrad,
                                  cudaStream_t stream, int pdl);
// ring depth of the kernel the plan launches (pair with tile_n 512: wide tiles)
int stages_for(int tile_n, int pair, int epi);
// resident CTA pairs of the pair kernel (0 if it cannot launch)
int pair_max_clusters_any();

}  // namespace gf
