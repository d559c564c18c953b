// Kernel parameter block and codes shared by the kernels and the host runtime.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define GF_HD __host__ __device__
#else
#define GF_HD
#endif

namespace gf {

enum Epi : int {
  EPI_NONE = 0,
  EPI_RELU_BIAS = 1,
  EPI_RELU_AUX_BIAS = 2,
  EPI_DRELU_BGRAD = 3,
  EPI_BIAS = 4,
  EPI_GELU_BIAS = 5,
  EPI_GELU_AUX_BIAS = 6,
  EPI_DGELU_BGRAD = 7,
  EPI_SWIGLU = 8,       // h = silu(x Wg^T) * (x Wu^T): two B operands, two accumulators
  EPI_SWIGLU_SAVE = 9,  // ... and g, u saved for the backward
  EPI_DSWIGLU = 10,     // d_gate, d_up of h = silu(g) * u from dh = dout Wd
};

// Shared-memory budget of one CTA (227 KB) and the ring depth that fills it:
// 1 KB of alignment slack, 256 B of barriers, the bias-gradient scratch, then
// as many stages as fit (at most 8).
constexpr int kSmemPerCta = 227 * 1024;
constexpr int kSmemAlignSlack = 1024;
constexpr int kSmemCtrlBytes = 512;
GF_HD constexpr int ring_stages(int stage_bytes, int red_bytes) {
  return (kSmemPerCta - kSmemAlignSlack - kSmemCtrlBytes - red_bytes) / stage_bytes > 8
             ? 8
             : (kSmemPerCta - kSmemAlignSlack - kSmemCtrlBytes - red_bytes) / stage_bytes;
}

// epilogs with two B operands (and two accumulators per tile)
GF_HD constexpr bool epi_dual(int epi) { return epi == EPI_SWIGLU || epi == EPI_SWIGLU_SAVE; }

// epilogs that reduce a bias gradient over the rows of each tile
GF_HD constexpr bool epi_has_bgrad(int epi) { return epi == EPI_DRELU_BGRAD || epi == EPI_DGELU_BGRAD; }
// epilogs that add a bias
GF_HD constexpr bool epi_has_bias(int epi) {
  return epi == EPI_RELU_BIAS || epi == EPI_RELU_AUX_BIAS || epi == EPI_BIAS ||
         epi == EPI_GELU_BIAS || epi == EPI_GELU_AUX_BIAS;
}

// bits of the device status word
enum : int {
  ST_TIMEOUT_PRODUCER = 1,
  ST_TIMEOUT_MMA_SMEM = 2,
  ST_TIMEOUT_MMA_TMEM = 4,
  ST_TIMEOUT_EPILOGUE = 8,
  ST_TIMEOUT_DRAIN = 16,
};

struct GemmParams {
  int32_t M, N, K;
  int32_t num_m_blocks, num_n_blocks, num_k_blocks, num_tiles, group_m;
  int32_t raster_n;      // 0: groups of group_m row blocks; 1: groups of group_m column blocks
  int32_t bias_axis;     // 0: bias[N] per column, 1: bias[M] per row
  int32_t bgrad_atomic;  // DRELU_BGRAD: 1 = atomicAdd into bgrad[N], 0 = partials
  const void* bias;
  void* out;
  uint32_t* aux_out;
  const uint32_t* aux_in;
  void* aux_out2;        // SWIGLU_SAVE: u
  const void* aux_in2;   // DSWIGLU: saved u
  float* bgrad;  // atomic: bgrad[N] (zeroed first); two-pass: partials [num_m_blocks][N]
  int32_t* status;
  uint64_t wait_limit_ns;
  int32_t drop_load;  // test hook: 1-based index of a stage load to skip (0: none)
  int32_t l2_hint_a;  // L2 policy of the A loads: 0 none, 1 evict first, 2 evict last
  int32_t l2_hint_b;  // ... of the B loads
  // CTA-pair kernel, dynamic schedule (null: static): [0] the next tile to
  // take, [1] pairs that have run out of tiles; both zero between launches
  int* tile_counter;
  int32_t b_mn_3d;    // MN-major B through a 3-D map: one box per k-slice brings every
                      // 64-column chunk of the tile (0: one 2-D box per chunk)
  // single-CTA kernel, split k: each tile's k-blocks are shared by k_splits
  // CTAs, kb_per_split each (the last may have fewer); 0 or 1: no split
  int32_t k_splits;
  int32_t kb_per_split;
  float* splitk_ws;     // fp32 partial sums [num_tiles][k_splits][tile_n / 4][128] float4
  int32_t* splitk_cnt;  // [num_tiles] splits done per tile; zero between launches
  // CTA-pair kernel, split k: tiles [0, split_from) run whole, each later
  // tile as k_splits units of kb_per_split k-blocks; partials and counters
  // per (split tile, CTA rank): [(t - split_from) * 2 + rank]
  int32_t split_from;
};

}  // namespace gf
