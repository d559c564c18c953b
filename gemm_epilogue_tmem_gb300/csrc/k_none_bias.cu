// Instances: EPILOG_NONE and BIAS.
#include "dispatch.cuh"

namespace gf {

cudaError_t launch_none_bias(int epi, const LaunchArgs& a) {
  return epi == EPI_BIAS ? launch_epi<EPI_BIAS>(a) : launch_epi<EPI_NONE>(a);
}

int smem_bytes_for(int tile_n) {
  return tile_n == 256 ? TileCfg<256>::kSmemBytes : TileCfg<128>::kSmemBytes;
}

int pair_stages() { return PairCfg<1>::kStages; }

int pair_max_clusters_any() { return pair_max_clusters<EPI_NONE, __half, false>(); }

int stages_for(int tile_n) {
  return tile_n == 256 ? TileCfg<256>::kStages : TileCfg<128>::kStages;
}

}  // namespace gf
