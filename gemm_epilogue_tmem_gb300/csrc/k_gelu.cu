// Instances: GELU_BIAS, GELU_AUX_BIAS and DGELU_BGRAD.
#include "dispatch.cuh"

namespace gf {

cudaError_t launch_gelu(int epi, const LaunchArgs& a) {
  if (epi == EPI_GELU_AUX_BIAS) return launch_epi<EPI_GELU_AUX_BIAS>(a);
  if (epi == EPI_DGELU_BGRAD) return launch_epi<EPI_DGELU_BGRAD>(a);
  return launch_epi<EPI_GELU_BIAS>(a);
}

}  // namespace gf
