// Instances: DRELU_BGRAD, and the fixed-order bias-gradient finalize.
#include "dispatch.cuh"

namespace gf {

// bgrad[n] = sum over m blocks of partial[mb][n], in ascending mb order split
// over 8 fixed slices: the same bits on every run.
__global__ void __launch_bounds__(256) bgrad_finalize_kernel(const float* __restrict__ partial,
                                                             int num_m_blocks, int N,
                                                             float* __restrict__ bgrad) {
  __shared__ float red[8][33];
  grid_dep_wait();  // the partials of the GEMM kernel before it
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int slice = threadIdx.x >> 5;
  const int col = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (col < N)
    for (int mb = slice; mb < num_m_blocks; mb += 8) s += partial[(size_t)mb * N + col];
  red[slice][lane] = s;
  __syncthreads();
  if (slice == 0 && col < N) {
    float t = red[0][lane];
#pragma unroll
    for (int k = 1; k < 8; ++k) t += red[k][lane];
    bgrad[col] = t;
  }
}

cudaError_t launch_drelu(const LaunchArgs& a) { return launch_epi<EPI_DRELU_BGRAD>(a); }

cudaError_t launch_bgrad_finalize(const float* partial, int num_m_blocks, int n, float* bgrad,
                                  cudaStream_t stream, int pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n + 31) / 32, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bgrad_finalize_kernel, partial, num_m_blocks, n, bgrad);
}

}  // namespace gf
