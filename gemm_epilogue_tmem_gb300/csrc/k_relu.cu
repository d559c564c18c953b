// Instances: RELU_BIAS and RELU_AUX_BIAS.
#include "dispatch.cuh"

namespace gf {

cudaError_t launch_relu(int epi, const LaunchArgs& a) {
  return epi == EPI_RELU_AUX_BIAS ? launch_epi<EPI_RELU_AUX_BIAS>(a)
                                  : launch_epi<EPI_RELU_BIAS>(a);
}

}  // namespace gf
