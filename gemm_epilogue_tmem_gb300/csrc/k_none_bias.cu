// Instances: EPILOG_NONE and BIAS; the ring depth of each kernel shape.
#include "dispatch.cuh"

namespace gf {

cudaError_t launch_none_bias(int epi, const LaunchArgs& a) {
  return epi == EPI_BIAS ? launch_epi<EPI_BIAS>(a) : launch_epi<EPI_NONE>(a);
}

int stages_for(int tile_n, int pair, int epi) {
  const bool red = epi_has_bgrad(epi);
  if (epi_dual(epi) && pair && tile_n == 256) return PairCfg<2, false, true>::kStages;
  if (epi_dual(epi) && pair)
    return pair_stg(epi, false) ? PairCfg<2, false, false, false, true>::kStages
                                : PairCfg<2, false>::kStages;
  if (pair && tile_n != 512 && pair_side_ring(epi, false) > 0)
    return PairCfg<1, false, false, false, true, pair_side_ring(EPI_DSWIGLU, false)>::kStages;
  if (pair && tile_n != 512 && pair_stg(epi, false))
    return red ? PairCfg<1, true, false, false, true>::kStages
               : PairCfg<1, false, false, false, true>::kStages;
  if (epi_dual(epi))
    return pair ? (red ? PairCfg<2, true>::kStages : PairCfg<2, false>::kStages)
                : (red ? TileCfg<128, 2, true>::kStages : TileCfg<128, 2, false>::kStages);
  if (pair && tile_n == 512)
    return red ? PairCfg<1, true, true>::kStages : PairCfg<1, false, true>::kStages;
  if (pair) return red ? PairCfg<1, true>::kStages : PairCfg<1, false>::kStages;
  if (tile_n == 256) return red ? TileCfg<256, 1, true>::kStages : TileCfg<256, 1, false>::kStages;
  return red ? TileCfg<128, 1, true>::kStages : TileCfg<128, 1, false>::kStages;
}

int pair_max_clusters_any() { return pair_max_clusters<EPI_NONE, __half, false>(); }

}  // namespace gf
