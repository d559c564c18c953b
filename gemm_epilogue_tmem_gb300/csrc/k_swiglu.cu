// Instances: the gate+up SwiGLU forward (two B operands, with or without
// saving g and u) and the dSwiGLU backward epilogue.
#include "dispatch.cuh"

namespace gf {

cudaError_t launch_swiglu(int epi, const LaunchArgs& a) {
  if (epi == EPI_SWIGLU) return launch_dual<EPI_SWIGLU>(a);
  if (epi == EPI_SWIGLU_SAVE) return launch_dual<EPI_SWIGLU_SAVE>(a);
  return launch_epi<EPI_DSWIGLU>(a);
}

}  // namespace gf
