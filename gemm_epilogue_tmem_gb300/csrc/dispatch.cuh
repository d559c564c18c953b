// Template instance selection: dtype x B storage x tile width.
#pragma once

#include "gemm_kernel.cuh"
#include "gemm_kernel_2sm.cuh"
#include "launch.h"

namespace gf {

template <int EPI, typename T, bool B_MN, int BN>
cudaError_t launch_instance(const LaunchArgs& a) {
  auto kernel = gemm_epilog_kernel<EPI, T, B_MN, BN>;
  constexpr int smem = TileCfg<BN, epi_dual(EPI) ? 2 : 1, epi_has_bgrad(EPI)>::kSmemBytes;
  static bool attr_set = false;  // once per instance and process
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, *a.tmA, *a.tmB, *a.tmB2, *a.params);
}

template <int EPI, typename T, bool B_MN, bool WIDE = false, bool SPLITK = false>
cudaError_t launch_pair_instance(const LaunchArgs& a) {
  auto kernel = gemm_epilog_pair_kernel<EPI, T, B_MN, WIDE, SPLITK>;
  using C = PairCfg<epi_dual(EPI) ? 2 : 1, epi_has_bgrad(EPI), WIDE, pair_epi8(EPI, WIDE),
                    pair_stg(EPI, WIDE), pair_side_ring(EPI, WIDE), pair_stg2(EPI, WIDE)>;
  constexpr int smem = C::kSmemBytes;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if constexpr (WIDE) {
      // the wide kernel hands registers from its control warpgroup to its
      // epilogue warpgroups (setmaxnreg); the split adds up only for this
      // launch register count, so refuse to launch a build that differs
      cudaFuncAttributes fa;
      e = cudaFuncGetAttributes(&fa, kernel);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != C::kLaunchRegs) return cudaErrorInvalidKernelImage;
    }
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.grid, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = a.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, *a.tmA, *a.tmB, *a.tmB2, *a.tmOut, *a.tmAux, *a.params);
}

// Largest number of CTA pairs of this instance that can be resident at once.
template <int EPI, typename T, bool B_MN>
int pair_max_clusters() {
  auto kernel = gemm_epilog_pair_kernel<EPI, T, B_MN>;
  using C = PairCfg<epi_dual(EPI) ? 2 : 1, epi_has_bgrad(EPI), false, pair_epi8(EPI, false),
                    pair_stg(EPI, false)>;
  constexpr int smem = C::kSmemBytes;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(C::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

// two-B-operand epilogs: B given [n, k] (K-major), 128-wide single-CTA tiles or CTA pairs
// (256 x 128 tiles, or 256 x 256 wide tiles)
template <int EPI>
cudaError_t launch_dual(const LaunchArgs& a) {
  if (a.b_mn) return cudaErrorInvalidValue;
  if (a.pair && a.wide)
    return a.bf16 ? launch_pair_instance<EPI, __nv_bfloat16, false, true>(a)
                  : launch_pair_instance<EPI, __half, false, true>(a);
  if (a.pair)
    return a.bf16 ? launch_pair_instance<EPI, __nv_bfloat16, false>(a)
                  : launch_pair_instance<EPI, __half, false>(a);
  return a.bf16 ? launch_instance<EPI, __nv_bfloat16, false, 128>(a)
                : launch_instance<EPI, __half, false, 128>(a);
}

template <int EPI>
cudaError_t launch_epi(const LaunchArgs& a) {
  if (a.pair && a.split) {  // split-k units: EPILOG_NONE only
    if constexpr (EPI == EPI_NONE) {
      if (a.wide) {
        if (a.bf16)
          return a.b_mn ? launch_pair_instance<EPI, __nv_bfloat16, true, true, true>(a)
                        : launch_pair_instance<EPI, __nv_bfloat16, false, true, true>(a);
        return a.b_mn ? launch_pair_instance<EPI, __half, true, true, true>(a)
                      : launch_pair_instance<EPI, __half, false, true, true>(a);
      }
      if (a.bf16)
        return a.b_mn ? launch_pair_instance<EPI, __nv_bfloat16, true, false, true>(a)
                      : launch_pair_instance<EPI, __nv_bfloat16, false, false, true>(a);
      return a.b_mn ? launch_pair_instance<EPI, __half, true, false, true>(a)
                    : launch_pair_instance<EPI, __half, false, false, true>(a);
    }
    return cudaErrorInvalidValue;
  }
  if (a.pair && a.wide) {
    if (a.bf16)
      return a.b_mn ? launch_pair_instance<EPI, __nv_bfloat16, true, true>(a)
                    : launch_pair_instance<EPI, __nv_bfloat16, false, true>(a);
    return a.b_mn ? launch_pair_instance<EPI, __half, true, true>(a)
                  : launch_pair_instance<EPI, __half, false, true>(a);
  }
  if (a.pair) {
    if (a.bf16)
      return a.b_mn ? launch_pair_instance<EPI, __nv_bfloat16, true>(a)
                    : launch_pair_instance<EPI, __nv_bfloat16, false>(a);
    return a.b_mn ? launch_pair_instance<EPI, __half, true>(a)
                  : launch_pair_instance<EPI, __half, false>(a);
  }
  if (a.tile_n == 256) {
    if (a.bf16)
      return a.b_mn ? launch_instance<EPI, __nv_bfloat16, true, 256>(a)
                    : launch_instance<EPI, __nv_bfloat16, false, 256>(a);
    return a.b_mn ? launch_instance<EPI, __half, true, 256>(a)
                  : launch_instance<EPI, __half, false, 256>(a);
  }
  if (a.bf16)
    return a.b_mn ? launch_instance<EPI, __nv_bfloat16, true, 128>(a)
                  : launch_instance<EPI, __nv_bfloat16, false, 128>(a);
  return a.b_mn ? launch_instance<EPI, __half, true, 128>(a)
                : launch_instance<EPI, __half, false, 128>(a);
}

}  // namespace gf
