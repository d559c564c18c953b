// Template instance selection: dtype x B storage x tile width.
#pragma once

#include "gemm_kernel.cuh"
#include "launch.h"

namespace gf {

template <int EPI, typename T, bool B_MN, int BN>
cudaError_t launch_instance(const LaunchArgs& a) {
  auto kernel = gemm_epilog_kernel<EPI, T, B_MN, BN>;
  constexpr int smem = TileCfg<BN>::kSmemBytes;
  static bool attr_set = false;  // once per instance and process
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kernel<<<a.grid, kThreads, smem, a.stream>>>(*a.tmA, *a.tmB, *a.params);
  return cudaGetLastError();
}

template <int EPI>
cudaError_t launch_epi(const LaunchArgs& a) {
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
