// Host runtime behind include/gf.h: plan validation and tile choice, device
// workspace, TMA tensor maps and kernel launch.
//
// The plan / execute / free split follows the stateful Matmul of the pages
// ("Fusing Matmul Epilogs with nvmath-python", "Forward-pass capabilities in
// the source"; nvmath-python / cuBLASLt page, steps 2-3 and "plan reuse"):
// everything that can be decided once (checks, tile shape, workspace) is done
// by the plan, and execute only encodes the tensor maps of the caller's
// pointers and launches.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>
#include <new>

#include "gf.h"
#include "launch.h"
#include "params.h"
#include "runtime_internal.h"

struct gf_plan {
  int64_t m, n, k;
  gf_dtype dtype;
  int epi;               // gf::Epi code (the public gf_epilog values, plus SwiGLU forms)
  gf_bias_axis bias_axis;
  gf_b_layout b_layout;
  int device;
  int num_sms;
  int tile_n;
  int forced_tile_n;
  int forced_kernel;     // 0 auto, 1 single CTA, 2 CTA pair, 3 CTA pair with 256 x 512 tiles
  int forced_group_m;    // 0 auto, else row (or column) blocks per raster group
  int forced_raster;     // 0 auto, 1 groups of row blocks, 2 groups of column blocks
  int raster_n;          // 1: raster groups of column blocks (B panels stay in L2)
  int l2_hint_a, l2_hint_b;  // L2 eviction policy of the A / B loads (0 none, 1 first, 2 last)
  int one_tile_per_cta;  // 1: grid of one tile per CTA (pair); the hardware orders the tiles
  int static_schedule;   // 1: persistent CTA pairs walk every gridDim-th tile (default: counter)
  int pair;              // the plan uses the CTA-pair kernel
  int wide;              // ... with 256 x 512 tiles
  int max_pair_clusters; // resident CTA pairs (0: the pair kernel cannot run)
  int stages;
  int grid;
  int num_m_blocks, num_n_blocks, num_k_blocks, num_tiles, group_m;
  gf_bgrad_mode bgrad_mode;
  uint64_t wait_limit_ns;
  int drop_load;
  int32_t* d_status;     // device status word (bounded-wait time-outs)
  float* d_partials;     // [num_m_blocks][n] fp32, DRELU_BGRAD two-pass only
  size_t partial_bytes;
  int forced_split;      // 0 the plan's choice, 1 no split, else k-splits per tile
  int split_from;        // CTA-pair split k: the first tile split into k-split units
  int k_splits;          // single-CTA kernel: CTAs sharing the k-blocks of one tile
  int kb_per_split;
  void* d_splitk;        // split-k partial sums, then the per-tile counters
  size_t splitk_bytes;   // capacity of d_splitk
  size_t splitk_cnt_offset;
  int pdl;               // 1: launches overlap their set-up with the previous kernel
  // Tensor maps of the last execute, reused while the operand pointers and
  // the plan's tiling are unchanged (encoding them is host work on every
  // call otherwise). `gen` counts tiling changes; the cache is valid for
  // cache_gen == gen.
  uint64_t gen;
  uint64_t cache_gen;
  bool cache_valid;
  const void* cache_A;
  const void* cache_B;
  const void* cache_B2;
  const void* cache_out;
  const void* cache_aux;
  bool cache_b_mn_3d;
  CUtensorMap cache_tmA, cache_tmB, cache_tmB2, cache_tmOut, cache_tmAux;
  std::mutex cache_mu;
};

namespace {

thread_local gf_status g_last = GF_OK;

gf_status fail(gf_status s) {
  g_last = s;
  return s;
}

constexpr int kBM = 128;
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;
// largest split-k partial-sum workspace a plan takes
constexpr size_t kMaxSplitkBytes = size_t(256) << 20;

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetDevice_v2000 g_ctx_get_device = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_get_current = nullptr;
std::once_flag g_driver_once;

void load_driver_entry_points() {
  std::call_once(g_driver_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetDevice", &fn, 2000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_device = reinterpret_cast<PFN_cuCtxGetDevice_v2000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
  });
}

// The device of the calling thread's current driver context (the one a
// framework such as PyTorch made current), else this runtime's device.
gf_status current_device(int* dev) {
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    return GF_ERR_NO_DEVICE;
  }
  load_driver_entry_points();
  CUdevice d;
  if (g_ctx_get_device && g_ctx_get_device(&d) == CUDA_SUCCESS) {
    *dev = static_cast<int>(d);
    return GF_OK;
  }
  if (cudaGetDevice(dev) != cudaSuccess) return GF_ERR_CUDA;
  return GF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool needs_bias(int e) { return gf::epi_has_bias(e); }

// epilogs that reduce the bias gradient (per-column sums of the epilogue output)
bool has_bgrad(int e) { return gf::epi_has_bgrad(e); }
bool needs_aux_out(int e) {
  return e == gf::EPI_RELU_AUX_BIAS || e == gf::EPI_GELU_AUX_BIAS || e == gf::EPI_SWIGLU_SAVE ||
         e == gf::EPI_DSWIGLU;
}
bool needs_aux_in(int e) { return has_bgrad(e) || e == gf::EPI_DSWIGLU; }

// 3-D tensor map over a row-major [k, n] matrix of 16-bit elements seen as
// [n / 64][k][64]: a box of 64 x box_k x chunks brings `chunks` consecutive
// 64-column (128-byte) chunks of box_k rows, chunk after chunk, the layout of
// the MN-major operand in shared memory. n must be a multiple of 64.
bool encode_mn_3d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t n, uint64_t k,
                  uint32_t box_k, uint32_t chunks) {
  cuuint64_t dims[3] = {64, k, n / 64};
  cuuint64_t strides[2] = {n * 2, 128};
  cuuint32_t box[3] = {64, box_k, chunks};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, dt == GF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        3, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D tensor map over a row-major [outer, inner] matrix of 16-bit elements,
// boxes of box_inner x box_outer, 128-byte swizzle, zero fill out of bounds.
// Store target of the 256 x 512 tiles' epilogue: a row-major [rows, cols]
// matrix of 16-bit elements written in 32 x 32 boxes (64-byte rows) from a
// staging buffer laid out with the 64-byte swizzle.
bool encode_store_2d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t cols,
                     uint64_t rows) {
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {32, 32};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt == GF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_2d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t inner, uint64_t outer,
               uint32_t box_inner, uint32_t box_outer) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_inner, box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, dt == GF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                           : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                        2, const_cast<void*>(ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

void plan_tiles(gf_plan* p) {
  const bool dual = gf::epi_dual(p->epi);
  const int64_t mblocks = (p->m + kBM - 1) / kBM;
  p->num_m_blocks = static_cast<int>(mblocks);
  p->num_k_blocks = static_cast<int>((p->k + 63) / 64);
  p->raster_n = p->forced_raster == 2 ? 1 : 0;
  p->group_m = p->forced_group_m > 0 ? p->forced_group_m : 8;
  p->k_splits = 1;
  p->kb_per_split = p->num_k_blocks;
  // The CTA-pair kernel (256 x 256 tiles over two SMs; 256 x 128 per operand
  // with two B operands) moves 2/3 of the operand bytes per flop of the
  // single-CTA tile; take it when its tiles fill the resident pairs, else the
  // single-CTA kernel with the tile width that keeps the SMs busy.
  // Wide pair tiles (256 x 512) need 3/4 of the operand bytes per flop of
  // the 256 x 256 pair tile, whose mainloop the L2 side of the operand
  // stream holds to ~85 % of the tensor rate, and they release each
  // accumulator half as soon as it is in registers. The plan takes them
  // when a tile's mainloop is long enough to cover a drain (k >= 2048) and
  // their coarser waves, at the wide tile's higher efficiency, cost no more
  // than the 256 x 256 schedule (measured on the GELU and SwiGLU shapes:
  // 1.4-9 % faster, except where the wide waves quantise worse, e.g. 80
  // tiles on 76 pairs). With two B operands the tiles are half as wide
  // (256 x 128 and 256 x 256 outputs, each output column taking a column of
  // both operands).
  const int64_t m2 = (p->m + 255) / 256;
  const int pair_n_narrow = dual ? 128 : 256;
  const int pair_n_wide = dual ? 256 : 512;
  const int64_t tiles256 = m2 * ((p->n + pair_n_narrow - 1) / pair_n_narrow);
  const int64_t tiles512 = m2 * ((p->n + pair_n_wide - 1) / pair_n_wide);
  const int64_t cl = p->max_pair_clusters > 0 ? p->max_pair_clusters : 1;
  // The plan's split k of the CTA-pair tiles (EPILOG_NONE): when `tiles`
  // leave the last wave of the resident pairs at most half full, that
  // wave's tiles are shared by several pairs each (k-blocks in consecutive
  // runs), so that it ends after a fraction of a tile; the tiles before run
  // whole. Beyond three waves the tiles' own spread in time already fills
  // part of the last wave, and the split paid only on long tiles (k >= 8192:
  // measured on the SwiGLU down GEMM; at k = 4096 over 13 waves it gave
  // nothing). Returns the splits, or 0.
  auto last_wave_split = [&](int64_t tiles) -> int {
    if (dual || p->epi != gf::EPI_NONE || p->forced_split != 0 || p->max_pair_clusters <= 0)
      return 0;
    const int64_t rem = tiles % cl;
    if (rem == 0 || 2 * rem > cl || p->num_k_blocks < (tiles <= 3 * cl ? 32 : 128)) return 0;
    int64_t w = cl / rem;
    if (w > 8) w = 8;
    if (w > p->num_k_blocks / 8) w = p->num_k_blocks / 8;
    return w >= 2 ? static_cast<int>(w) : 0;
  };
  // the time of `tiles` in eighths of a tile's time per pair
  auto eighths = [&](int64_t tiles) -> int64_t {
    const int w = last_wave_split(tiles);
    const int64_t full = tiles / cl;
    return 8 * full + (tiles == full * cl ? 0 : w ? (8 + w - 1) / w : 8);
  };
  // (two B operands: the wide tile saves less -- 1-3 % at the power cap on
  // the SwiGLU gate+up, where the 256 x 128 tile was 1.2 % faster at
  // M = 2048, 8 against 15 waves)
  const bool wide_fits = p->max_pair_clusters > 0;
  const int64_t wide_gain = dual ? 104 : 112;
  const bool wide_pays =
      wide_fits && p->k >= 2048 && 100 * 2 * eighths(tiles512) <= wide_gain * eighths(tiles256);
  const bool wide = wide_fits && (p->forced_kernel == 3 || (p->forced_kernel == 0 && wide_pays));
  const int pair_n = wide ? pair_n_wide : pair_n_narrow;
  const int64_t pair_tiles = wide ? tiles512 : tiles256;
  bool pair = false;
  if (p->forced_kernel == 2 || p->forced_kernel == 3)
    pair = p->max_pair_clusters > 0;
  else if (p->forced_kernel == 0)
    pair = p->max_pair_clusters > 0 && p->forced_tile_n == 0 && p->m > 128 &&
           tiles256 >= p->max_pair_clusters;
  p->pair = pair ? 1 : 0;
  p->wide = pair && wide ? 1 : 0;
  // wide tiles: groups of 4 column blocks (4 B panels of 512 columns stay in
  // L2 while A streams) measured 0.3-0.7 % faster at the power cap than
  // groups of 8 row blocks on the large linear pair
  if (p->wide && p->forced_raster == 0) {
    p->raster_n = 1;
    if (p->forced_group_m == 0) p->group_m = 4;
  }
  p->split_from = 0;
  if (pair) {
    p->tile_n = pair_n;
    p->stages = gf::stages_for(pair_n, 1, p->epi);
    p->num_n_blocks = static_cast<int>((p->n + pair_n - 1) / pair_n);
    p->num_tiles = static_cast<int>(pair_tiles);
    // Split k (EPILOG_NONE, 256 x 256 or wide tiles): the plan's split of
    // a last wave (above); GF_OPT_SPLIT_K >= 2 splits every tile that many
    // ways.
    int want = 0;
    int64_t from = 0;
    if (!dual && p->epi == gf::EPI_NONE && p->num_k_blocks >= 2) {
      if (p->forced_split >= 2) {
        want = p->forced_split;
      } else {
        want = last_wave_split(pair_tiles);
        from = pair_tiles / cl * cl;
      }
    }
    if (want >= 2) {
      const int kps = (p->num_k_blocks + want - 1) / want;
      const int ks = (p->num_k_blocks + kps - 1) / kps;  // every split gets k-blocks
      const size_t ws = static_cast<size_t>(pair_tiles - from) * 2 * ks * kBM * pair_n * 4;
      if (ks >= 2 && ws <= kMaxSplitkBytes) {
        p->k_splits = ks;
        p->kb_per_split = kps;
        p->split_from = static_cast<int>(from);
      }
    }
    const int64_t units = p->split_from + (pair_tiles - p->split_from) * p->k_splits;
    const int64_t clusters = units < p->max_pair_clusters ? units : p->max_pair_clusters;
    p->grid = static_cast<int>(2 * (p->one_tile_per_cta ? units : clusters));
    return;
  }
  int tn = p->forced_tile_n;
  if (dual) {
    tn = 128;  // two 128-column accumulators per buffer fill the tensor memory
  } else if (tn == 0) {
    // 256-wide tiles halve the B traffic per flop; take 128 when the wide
    // tiles would leave SMs idle
    const int64_t wide = mblocks * ((p->n + 255) / 256);
    tn = wide >= p->num_sms ? 256 : 128;
  }
  p->tile_n = tn;
  p->stages = gf::stages_for(tn, 0, p->epi);
  p->num_n_blocks = static_cast<int>((p->n + tn - 1) / tn);
  const int64_t tiles = mblocks * p->num_n_blocks;
  p->num_tiles = static_cast<int>(tiles);
  // Split k: when the tiles leave most SMs idle, the k-blocks of each tile
  // are shared by several CTAs whose fp32 partial sums meet in the plan's
  // workspace; the last CTA of a tile to finish adds them and runs the
  // epilogue. The plan's choice: when k has at least 16 blocks and the tiles
  // fill at most half the SMs, as many splits as the idle SMs take, at most
  // 8 and at most sqrt(k-blocks / 2) (a split's mainloop then stays longer
  // than the partial-sum hand-over, which moves (splits + 1) x 64 KB).
  int want = 0;
  if (!dual && p->num_k_blocks >= 2 && tiles > 0) {
    if (p->forced_split >= 2) {
      want = p->forced_split;
    } else if (p->forced_split == 0 && p->num_k_blocks >= 16 && 2 * tiles <= p->num_sms) {
      int r = 1;
      while ((r + 1) * (r + 1) <= p->num_k_blocks / 2) ++r;
      const int64_t idle = p->num_sms / tiles;
      want = static_cast<int>(idle < r ? idle : r);
      if (want > 8) want = 8;
    }
  }
  if (want >= 2) {
    const int kps = (p->num_k_blocks + want - 1) / want;
    const int ks = (p->num_k_blocks + kps - 1) / kps;  // every split gets k-blocks
    const size_t ws = static_cast<size_t>(tiles) * ks * kBM * tn * 4;
    if (ks >= 2 && ws <= kMaxSplitkBytes) {
      p->k_splits = ks;
      p->kb_per_split = kps;
    }
  }
  const int64_t units = tiles * p->k_splits;
  p->grid = static_cast<int>(p->one_tile_per_cta || units < p->num_sms ? units : p->num_sms);
}

// The split-k workspace of the plan's current tiling: fp32 partial sums
// [tiles][splits][tile_n / 4][128] float4, then one zeroed counter per tile. Grown when
// too small; on failure the plan falls back to no split.
gf_status ensure_splitk(gf_plan* p) {
  if (p->k_splits < 2) return GF_OK;
  // partial sums per split tile, or per (split tile, CTA rank) for the pair kernel
  const size_t parts = p->pair ? 2 * static_cast<size_t>(p->num_tiles - p->split_from)
                               : static_cast<size_t>(p->num_tiles);
  const size_t ws = parts * p->k_splits * kBM * p->tile_n * 4;
  const size_t need = ws + parts * 4;
  gf_status st = GF_OK;
  if (need > p->splitk_bytes) {
    if (p->d_splitk) cudaFree(p->d_splitk);
    p->d_splitk = nullptr;
    p->splitk_bytes = 0;
    if (cudaMalloc(&p->d_splitk, need) == cudaSuccess)
      p->splitk_bytes = need;
    else
      st = GF_ERR_OUT_OF_MEMORY;
  }
  if (st == GF_OK) {
    p->splitk_cnt_offset = ws;
    if (cudaMemset(static_cast<char*>(p->d_splitk) + ws, 0, parts * 4) != cudaSuccess)
      st = GF_ERR_CUDA;
  }
  if (st != GF_OK) {
    cudaGetLastError();
    p->forced_split = 1;
    plan_tiles(p);
  }
  return st;
}

// plan_tiles, then the workspace the new tiling needs
gf_status replan(gf_plan* p) {
  ++p->gen;  // the tensor maps' boxes may change with the tiling
  plan_tiles(p);
  return ensure_splitk(p);
}

// Validation, device checks, tile choice and workspace: the plan step of
// every public plan constructor. epi is a gf::Epi code.
gf_plan* plan_create(int64_t m, int64_t n, int64_t k, gf_dtype dtype, int epi,
                     gf_bias_axis bias_axis, gf_b_layout b_layout) {
  g_last = GF_OK;
  // argument checks first: they need no device
  if (m < 0 || n < 0 || k < 0 || m > kMaxDim || n > kMaxDim || k > kMaxDim) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  if (dtype != GF_F16 && dtype != GF_BF16) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  if (bias_axis != GF_BIAS_COL && bias_axis != GF_BIAS_ROW) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  if (b_layout != GF_B_KN && b_layout != GF_B_NK) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  if (n % 8 != 0 || k % 8 != 0) {  // 16-byte row strides for the tensor maps
    fail(GF_ERR_UNSUPPORTED);
    return nullptr;
  }
  if (has_bgrad(epi) && bias_axis != GF_BIAS_COL) {
    fail(GF_ERR_UNSUPPORTED);
    return nullptr;
  }
  // ceil(m/128) * ceil(n/128) tiles must fit the int32 tile counter
  if (((m + 127) / 128) * ((n + 127) / 128) > kMaxDim) {
    fail(GF_ERR_UNSUPPORTED);
    return nullptr;
  }

  int dev = 0;
  gf_status st = current_device(&dev);
  if (st != GF_OK) {
    fail(st);
    return nullptr;
  }
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    fail(GF_ERR_CUDA);
    return nullptr;
  }
  if (prop.major != 10 || prop.minor != 3) {  // the kernels are built for sm_103a only
    fail(GF_ERR_UNSUPPORTED);
    return nullptr;
  }
  load_driver_entry_points();
  if (!g_encode) {
    fail(GF_ERR_CUDA);
    return nullptr;
  }
  if (cudaSetDevice(dev) != cudaSuccess) {
    fail(GF_ERR_CUDA);
    return nullptr;
  }

  gf_plan* p = new (std::nothrow) gf_plan();
  if (!p) {
    fail(GF_ERR_OUT_OF_MEMORY);
    return nullptr;
  }
  p->m = m;
  p->n = n;
  p->k = k;
  p->dtype = dtype;
  p->epi = epi;
  p->bias_axis = bias_axis;
  p->b_layout = b_layout;
  p->device = dev;
  p->num_sms = prop.multiProcessorCount;
  // defaults, and the environment overrides of experiments (an option set
  // on the plan afterwards wins)
  p->bgrad_mode = GF_BGRAD_TWO_PASS;
  p->pdl = 1;
  const char* env_bgrad = getenv("GF_BGRAD_MODE");
  if (env_bgrad && strcmp(env_bgrad, "atomic") == 0) p->bgrad_mode = GF_BGRAD_ATOMIC;
  p->wait_limit_ns = 2000000000ull;
  const char* env_wait = getenv("GF_WAIT_LIMIT_US");
  if (env_wait) {
    const long long us = atoll(env_wait);
    if (us >= 1000 && us <= 600000000) p->wait_limit_ns = static_cast<uint64_t>(us) * 1000ull;
  }
  const char* env_tile = getenv("GF_TILE_N");
  p->forced_tile_n = env_tile && (atoi(env_tile) == 128 || atoi(env_tile) == 256) ? atoi(env_tile) : 0;
  const char* env_kernel = getenv("GF_KERNEL");
  p->forced_kernel = env_kernel ? atoi(env_kernel) : 0;
  if (p->forced_kernel < 0 || p->forced_kernel > 3) p->forced_kernel = 0;
  p->max_pair_clusters = gf::pair_max_clusters_any();
  cudaGetLastError();
  plan_tiles(p);

  if (cudaMalloc(&p->d_status, 256) != cudaSuccess) {
    cudaGetLastError();
    delete p;
    fail(GF_ERR_OUT_OF_MEMORY);
    return nullptr;
  }
  if (cudaMemset(p->d_status, 0, 256) != cudaSuccess) {
    cudaFree(p->d_status);
    delete p;
    fail(GF_ERR_CUDA);
    return nullptr;
  }
  if (has_bgrad(epi) && m > 0 && n > 0) {
    // one fp32 partial per 128-row block and column, whatever the tile choice
    p->partial_bytes = static_cast<size_t>((m + kBM - 1) / kBM) * static_cast<size_t>(n) * 4;
    if (cudaMalloc(&p->d_partials, p->partial_bytes) != cudaSuccess) {
      cudaGetLastError();
      cudaFree(p->d_status);
      delete p;
      fail(GF_ERR_OUT_OF_MEMORY);
      return nullptr;
    }
  }
  if (ensure_splitk(p) != GF_OK) {
    if (p->d_partials) cudaFree(p->d_partials);
    cudaFree(p->d_status);
    delete p;
    fail(GF_ERR_OUT_OF_MEMORY);
    return nullptr;
  }
  return p;
}

struct ExecArgs {
  const void* A;
  const void* B;
  const void* B2;
  const void* bias;
  void* out;
  const void* aux_in;
  const void* aux_in2;
  void* aux_out;
  void* aux_out2;
  float* bgrad;
};

// Checks the pointers the plan's epilog needs, encodes the tensor maps and
// launches: the execute step of every public entry point.
gf_status execute_impl(const gf_plan* p, const ExecArgs& x, cudaStream_t st) {
  const bool empty = p->m == 0 || p->n == 0;
  const int e = p->epi;
  const bool dual = gf::epi_dual(e);
  // pointer checks: required pointers present and 16-byte aligned
  if (!empty) {
    if (!x.out || !aligned16(x.out)) return fail(GF_ERR_INVALID_VALUE);
    if (p->k > 0 && (!x.A || !x.B || !aligned16(x.A) || !aligned16(x.B)))
      return fail(GF_ERR_INVALID_VALUE);
    if (dual && p->k > 0 && (!x.B2 || !aligned16(x.B2))) return fail(GF_ERR_INVALID_VALUE);
    if (needs_bias(e) && (!x.bias || !aligned16(x.bias))) return fail(GF_ERR_INVALID_VALUE);
    if (needs_aux_out(e) && (!x.aux_out || !aligned16(x.aux_out)))
      return fail(GF_ERR_INVALID_VALUE);
    if (e == gf::EPI_SWIGLU_SAVE && (!x.aux_out2 || !aligned16(x.aux_out2)))
      return fail(GF_ERR_INVALID_VALUE);
    if (needs_aux_in(e) && (!x.aux_in || !aligned16(x.aux_in))) return fail(GF_ERR_INVALID_VALUE);
    if (e == gf::EPI_DSWIGLU && (!x.aux_in2 || !aligned16(x.aux_in2)))
      return fail(GF_ERR_INVALID_VALUE);
  }
  if (has_bgrad(e) && p->n > 0 && (!x.bgrad || !aligned16(x.bgrad)))
    return fail(GF_ERR_INVALID_VALUE);

  if (cudaSetDevice(p->device) != cudaSuccess) return fail(GF_ERR_CUDA);

  if (empty) {
    // nothing to multiply; the bias gradient of zero rows is zero
    if (has_bgrad(e) && p->n > 0 &&
        cudaMemsetAsync(x.bgrad, 0, static_cast<size_t>(p->n) * 4, st) != cudaSuccess)
      return fail(GF_ERR_CUDA);
    return GF_OK;
  }

  CUtensorMap tmA, tmB, tmB2, tmOut, tmAux;
  bool b_mn_3d = false;
  memset(&tmA, 0, sizeof tmA);
  memset(&tmB, 0, sizeof tmB);
  memset(&tmB2, 0, sizeof tmB2);
  memset(&tmOut, 0, sizeof tmOut);
  memset(&tmAux, 0, sizeof tmAux);
  // the 256 x 512 tiles store their 16-bit outputs by TMA
  const bool store_maps = p->pair && p->wide;
  const bool aux16 = e == gf::EPI_GELU_AUX_BIAS || e == gf::EPI_DSWIGLU;
  gf_plan* pm = const_cast<gf_plan*>(p);  // the map cache only
  std::unique_lock<std::mutex> cache_lock(pm->cache_mu);
  const bool cached = p->cache_valid && p->cache_gen == p->gen && p->cache_A == x.A &&
                      p->cache_B == x.B && (!dual || p->cache_B2 == x.B2) &&
                      (!store_maps ||
                       (p->cache_out == x.out && (!aux16 || p->cache_aux == x.aux_out)));
  if (cached) {
    tmA = p->cache_tmA;
    tmB = p->cache_tmB;
    tmB2 = p->cache_tmB2;
    tmOut = p->cache_tmOut;
    tmAux = p->cache_tmAux;
    b_mn_3d = p->cache_b_mn_3d;
  } else {
    if (p->k > 0) {
      if (!encode_2d(&tmA, x.A, p->dtype, p->k, p->m, 64, kBM)) return fail(GF_ERR_INVALID_VALUE);
      // K-major B boxes: a pair CTA loads half of the tile's columns, or with
      // two B operands all of the tile's columns of one operand; the wide
      // tiles load 128-row parts
      const uint32_t rows_nk =
          p->pair && (!dual || p->wide) ? 128u : static_cast<uint32_t>(p->tile_n);
      // MN-major B: one 3-D box per k-slice for all of this CTA's column
      // chunks when n is a multiple of 64, else one 2-D box per chunk
      b_mn_3d = p->b_layout == GF_B_KN && p->n % 64 == 0 &&
                encode_mn_3d(&tmB, x.B, p->dtype, p->n, p->k, 64, rows_nk / 64);
      const bool ok = b_mn_3d ||
                      (p->b_layout == GF_B_KN
                           ? encode_2d(&tmB, x.B, p->dtype, p->n, p->k, 64, 64)
                           : encode_2d(&tmB, x.B, p->dtype, p->k, p->n, 64, rows_nk));
      if (!ok) return fail(GF_ERR_INVALID_VALUE);
      if (dual && !encode_2d(&tmB2, x.B2, p->dtype, p->k, p->n, 64, rows_nk))
        return fail(GF_ERR_INVALID_VALUE);
    }
    if (store_maps) {
      if (!encode_store_2d(&tmOut, x.out, p->dtype, p->n, p->m)) return fail(GF_ERR_INVALID_VALUE);
      if (aux16 && !encode_store_2d(&tmAux, x.aux_out, p->dtype, p->n, p->m))
        return fail(GF_ERR_INVALID_VALUE);
    }
    pm->cache_tmA = tmA;
    pm->cache_tmB = tmB;
    pm->cache_tmB2 = tmB2;
    pm->cache_tmOut = tmOut;
    pm->cache_tmAux = tmAux;
    pm->cache_b_mn_3d = b_mn_3d;
    pm->cache_A = x.A;
    pm->cache_B = x.B;
    pm->cache_B2 = dual ? x.B2 : nullptr;
    pm->cache_out = x.out;
    pm->cache_aux = x.aux_out;
    pm->cache_gen = p->gen;
    pm->cache_valid = true;
  }
  cache_lock.unlock();

  gf::GemmParams prm;
  memset(&prm, 0, sizeof prm);
  prm.M = static_cast<int32_t>(p->m);
  prm.N = static_cast<int32_t>(p->n);
  prm.K = static_cast<int32_t>(p->k);
  prm.num_m_blocks = p->num_m_blocks;
  prm.num_n_blocks = p->num_n_blocks;
  prm.num_k_blocks = p->num_k_blocks;
  prm.num_tiles = p->num_tiles;
  prm.group_m = p->group_m;
  prm.raster_n = p->raster_n;
  prm.bias_axis = p->bias_axis == GF_BIAS_ROW ? 1 : 0;
  prm.bias = x.bias;
  prm.out = x.out;
  prm.aux_out = static_cast<uint32_t*>(x.aux_out);
  prm.aux_in = static_cast<const uint32_t*>(x.aux_in);
  prm.aux_out2 = x.aux_out2;
  prm.aux_in2 = x.aux_in2;
  prm.status = p->d_status;
  prm.wait_limit_ns = p->wait_limit_ns;
  prm.drop_load = p->drop_load;
  prm.l2_hint_a = p->l2_hint_a;
  prm.l2_hint_b = p->l2_hint_b;
  prm.b_mn_3d = b_mn_3d ? 1 : 0;
  if (p->k_splits > 1) {
    prm.split_from = p->split_from;
    prm.k_splits = p->k_splits;
    prm.kb_per_split = p->kb_per_split;
    prm.splitk_ws = static_cast<float*>(p->d_splitk);
    prm.splitk_cnt =
        reinterpret_cast<int32_t*>(static_cast<char*>(p->d_splitk) + p->splitk_cnt_offset);
  }
  if (p->pair && !p->static_schedule && !p->one_tile_per_cta) {
    // the tile counter and the count of pairs that have finished sit in the
    // plan's status block, 64 bytes past the status word; both are zero
    // between launches (the last pair of a launch resets them)
    prm.tile_counter = p->d_status + 16;
  }

  const bool atomic = has_bgrad(e) && p->bgrad_mode == GF_BGRAD_ATOMIC;
  if (has_bgrad(e)) {
    prm.bgrad_atomic = atomic ? 1 : 0;
    prm.bgrad = atomic ? x.bgrad : p->d_partials;
    if (atomic && cudaMemsetAsync(x.bgrad, 0, static_cast<size_t>(p->n) * 4, st) != cudaSuccess)
      return fail(GF_ERR_CUDA);
  }

  gf::LaunchArgs la;
  la.tmA = &tmA;
  la.tmB = &tmB;
  la.tmB2 = dual ? &tmB2 : &tmB;
  la.tmOut = &tmOut;
  la.tmAux = &tmAux;
  la.params = &prm;
  la.grid = p->grid;
  la.bf16 = p->dtype == GF_BF16 ? 1 : 0;
  la.b_mn = p->b_layout == GF_B_KN ? 1 : 0;
  la.tile_n = p->tile_n;
  la.pair = p->pair;
  la.wide = p->wide;
  la.split = p->pair && p->k_splits > 1 ? 1 : 0;
  la.pdl = p->pdl;
  la.stream = st;

  cudaError_t err;
  switch (e) {
    case gf::EPI_NONE:
    case gf::EPI_BIAS: err = gf::launch_none_bias(e, la); break;
    case gf::EPI_RELU_BIAS:
    case gf::EPI_RELU_AUX_BIAS: err = gf::launch_relu(e, la); break;
    case gf::EPI_DRELU_BGRAD: err = gf::launch_drelu(la); break;
    case gf::EPI_GELU_BIAS:
    case gf::EPI_GELU_AUX_BIAS:
    case gf::EPI_DGELU_BGRAD: err = gf::launch_gelu(e, la); break;
    case gf::EPI_SWIGLU:
    case gf::EPI_SWIGLU_SAVE:
    case gf::EPI_DSWIGLU: err = gf::launch_swiglu(e, la); break;
    default: return fail(GF_ERR_INVALID_VALUE);
  }
  if (err != cudaSuccess) return fail(GF_ERR_CUDA);
  if (has_bgrad(e) && !atomic) {
    err = gf::launch_bgrad_finalize(p->d_partials, p->num_m_blocks, static_cast<int>(p->n),
                                    x.bgrad, st, p->pdl);
    if (err != cudaSuccess) return fail(GF_ERR_CUDA);
  }
  return GF_OK;
}

}  // namespace

namespace gf {

// Shared with the other host entry points of the library (runtime_internal.h).
gf_status runtime_current_device(int* dev) { return current_device(dev); }

CUcontext runtime_current_context() {
  load_driver_entry_points();
  CUcontext c = nullptr;
  if (!g_ctx_get_current || g_ctx_get_current(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

gf_status runtime_fail(gf_status s) { return fail(s); }

bool runtime_encode_2d(CUtensorMap* map, const void* ptr, gf_dtype dt, uint64_t inner,
                       uint64_t outer, uint32_t box_inner, uint32_t box_outer) {
  load_driver_entry_points();
  return g_encode != nullptr && encode_2d(map, ptr, dt, inner, outer, box_inner, box_outer);
}

}  // namespace gf

extern "C" {

GF_API const char* gf_status_string(gf_status s) {
  switch (s) {
    case GF_OK: return "GF_OK";
    case GF_ERR_INVALID_VALUE: return "GF_ERR_INVALID_VALUE: invalid argument";
    case GF_ERR_UNSUPPORTED: return "GF_ERR_UNSUPPORTED: valid but not supported";
    case GF_ERR_NO_DEVICE: return "GF_ERR_NO_DEVICE: no CUDA device";
    case GF_ERR_CUDA: return "GF_ERR_CUDA: a CUDA call failed";
    case GF_ERR_OUT_OF_MEMORY: return "GF_ERR_OUT_OF_MEMORY: workspace allocation failed";
    case GF_ERR_DEVICE_TIMEOUT: return "GF_ERR_DEVICE_TIMEOUT: a bounded wait in a kernel gave up";
  }
  return "unknown gf_status";
}

GF_API gf_status gf_last_error(void) { return g_last; }

GF_API gf_plan* gf_matmul_plan_ex(int64_t m, int64_t n, int64_t k, gf_dtype dtype,
                                  gf_epilog epilog, gf_bias_axis bias_axis,
                                  gf_b_layout b_layout) {
  if (epilog < GF_EPILOG_NONE || epilog > GF_EPILOG_DGELU_BGRAD) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  // the public gf_epilog values are the kernels' epilog codes
  return plan_create(m, n, k, dtype, static_cast<int>(epilog), bias_axis, b_layout);
}

GF_API gf_plan* gf_swiglu_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype, int save_gu) {
  if (save_gu != 0 && save_gu != 1) {
    fail(GF_ERR_INVALID_VALUE);
    return nullptr;
  }
  return plan_create(m, n, k, dtype, save_gu ? gf::EPI_SWIGLU_SAVE : gf::EPI_SWIGLU, GF_BIAS_COL,
                     GF_B_NK);
}

GF_API gf_plan* gf_dswiglu_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype) {
  return plan_create(m, n, k, dtype, gf::EPI_DSWIGLU, GF_BIAS_COL, GF_B_KN);
}

GF_API gf_plan* gf_matmul_plan(int64_t m, int64_t n, int64_t k, gf_dtype dtype, gf_epilog epilog,
                               gf_bias_axis bias_axis) {
  return gf_matmul_plan_ex(m, n, k, dtype, epilog, bias_axis, GF_B_KN);
}

GF_API gf_status gf_plan_set_option(gf_plan* p, gf_option option, int64_t value) {
  if (!p) return fail(GF_ERR_INVALID_VALUE);
  switch (option) {
    case GF_OPT_BGRAD_MODE:
      if (value != GF_BGRAD_TWO_PASS && value != GF_BGRAD_ATOMIC) return fail(GF_ERR_INVALID_VALUE);
      p->bgrad_mode = static_cast<gf_bgrad_mode>(value);
      return GF_OK;
    case GF_OPT_WAIT_LIMIT_US:
      if (value < 1000 || value > 600000000) return fail(GF_ERR_INVALID_VALUE);
      p->wait_limit_ns = static_cast<uint64_t>(value) * 1000ull;
      return GF_OK;
    case GF_OPT_TILE_N:
      if (value != 0 && value != 128 && value != 256) return fail(GF_ERR_INVALID_VALUE);
      p->forced_tile_n = static_cast<int>(value);
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_KERNEL:
      if (value < 0 || value > 3) return fail(GF_ERR_INVALID_VALUE);
      if (value >= 2 && p->max_pair_clusters == 0) return fail(GF_ERR_UNSUPPORTED);
      p->forced_kernel = static_cast<int>(value);
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_L2_HINTS:
      if (value < 0 || value > 22 || value % 10 > 2 || value / 10 > 2)
        return fail(GF_ERR_INVALID_VALUE);
      p->l2_hint_a = static_cast<int>(value / 10);
      p->l2_hint_b = static_cast<int>(value % 10);
      ++p->gen;  // the B map's form depends on the hint
      return GF_OK;
    case GF_OPT_SCHEDULE:
      if (value < 0 || value > 3) return fail(GF_ERR_INVALID_VALUE);
      p->one_tile_per_cta = value == 1 ? 1 : 0;
      p->static_schedule = value == 3 ? 1 : 0;
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_GROUP_M:
      if (value < 0 || value > 4096) return fail(GF_ERR_INVALID_VALUE);
      p->forced_group_m = static_cast<int>(value);
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_RASTER:
      if (value < 0 || value > 2) return fail(GF_ERR_INVALID_VALUE);
      p->forced_raster = static_cast<int>(value);
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_PDL:
      if (value != 0 && value != 1) return fail(GF_ERR_INVALID_VALUE);
      p->pdl = static_cast<int>(value);
      return GF_OK;
    case GF_OPT_SPLIT_K:
      if (value < 0 || value > 64) return fail(GF_ERR_INVALID_VALUE);
      p->forced_split = static_cast<int>(value);
      return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
    case GF_OPT_FAULT_DROP_LOAD:
      if (value < 0 || value > kMaxDim) return fail(GF_ERR_INVALID_VALUE);
      p->drop_load = static_cast<int>(value);
      return GF_OK;
  }
  return fail(GF_ERR_INVALID_VALUE);
}

GF_API gf_status gf_matmul_autotune(gf_plan* p, const void* A, const void* B, const void* bias,
                                    void* out, const void* aux_in, void* aux_out, float* bgrad,
                                    struct CUstream_st* stream, int32_t reps) {
  if (!p || p->epi > gf::EPI_DGELU_BGRAD || reps < 1 || reps > 100)
    return fail(GF_ERR_INVALID_VALUE);
  if (p->m == 0 || p->n == 0) return GF_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  ExecArgs x = {A, B, nullptr, bias, out, aux_in, nullptr, aux_out, nullptr, bgrad};
  // candidates: {kernel (1 single, 2 pair, 3 pair with 256 x 512 tiles), tile_n, schedule,
  // group_m, k-split (0 the plan's choice, 1 none, else splits per tile)}
  struct Cand { int kernel, tile_n, schedule, group_m, split; };
  const Cand cands[] = {{2, 0, 2, 8, 0},   {2, 0, 2, 4, 0},   {2, 0, 2, 16, 0}, {2, 0, 3, 8, 0},
                        {3, 0, 2, 8, 0},   {3, 0, 2, 16, 0},  {3, 0, 2, 4, 0},  {1, 256, 0, 8, 0},
                        {1, 128, 0, 8, 0}, {1, 256, 0, 4, 0}, {1, 128, 0, 8, 1}, {1, 128, 0, 8, 2},
                        {1, 128, 0, 8, 4}, {1, 128, 0, 8, 8}};
  const int saved[6] = {p->forced_kernel, p->forced_tile_n, p->one_tile_per_cta,
                        p->static_schedule, p->forced_group_m, p->forced_split};
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
    return fail(GF_ERR_CUDA);
  float best_ms = -1.f;
  Cand best = cands[0];
  gf_status st_out = GF_OK;
  for (const Cand& c : cands) {
    if (c.kernel >= 2 && p->max_pair_clusters == 0) continue;
    if (c.kernel == 3 && gf::epi_dual(p->epi)) continue;
    p->forced_kernel = c.kernel;
    p->forced_tile_n = c.tile_n;
    p->one_tile_per_cta = 0;
    p->static_schedule = c.schedule == 3 ? 1 : 0;
    p->forced_group_m = c.group_m;
    p->forced_split = c.split;
    if (replan(p) != GF_OK) continue;
    // an explicit split the tiling does not take is the same run as split 1
    if (c.split >= 2 && p->k_splits != c.split) continue;
    gf_status s = execute_impl(p, x, st);  // warm-up, and the check of the arguments
    if (s != GF_OK) {
      st_out = s;
      break;
    }
    cudaEventRecord(e0, st);
    for (int r = 0; r < reps && s == GF_OK; ++r) s = execute_impl(p, x, st);
    cudaEventRecord(e1, st);
    if (s != GF_OK || cudaEventSynchronize(e1) != cudaSuccess) {
      st_out = s != GF_OK ? s : GF_ERR_CUDA;
      break;
    }
    float ms = 0.f;
    cudaEventElapsedTime(&ms, e0, e1);
    if (best_ms < 0.f || ms < best_ms) {
      best_ms = ms;
      best = c;
    }
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st_out != GF_OK || best_ms < 0.f) {
    p->forced_kernel = saved[0];
    p->forced_tile_n = saved[1];
    p->one_tile_per_cta = saved[2];
    p->static_schedule = saved[3];
    p->forced_group_m = saved[4];
    p->forced_split = saved[5];
    replan(p);
    return st_out != GF_OK ? fail(st_out) : fail(GF_ERR_UNSUPPORTED);
  }
  p->forced_kernel = best.kernel;
  p->forced_tile_n = best.tile_n;
  p->one_tile_per_cta = 0;
  p->static_schedule = best.schedule == 3 ? 1 : 0;
  p->forced_group_m = best.group_m;
  p->forced_split = best.split;
  return replan(p) == GF_OK ? GF_OK : fail(GF_ERR_OUT_OF_MEMORY);
}

GF_API gf_status gf_plan_describe(const gf_plan* p, int32_t* tile_m, int32_t* tile_n,
                                  int32_t* stages, int32_t* grid, int64_t* workspace_bytes) {
  if (!p) return fail(GF_ERR_INVALID_VALUE);
  if (tile_m) *tile_m = p->pair ? 2 * kBM : kBM;
  if (tile_n) *tile_n = p->tile_n;
  if (stages) *stages = p->stages;
  if (grid) *grid = p->grid;
  if (workspace_bytes)
    *workspace_bytes = static_cast<int64_t>(p->partial_bytes + p->splitk_bytes) + 256;
  return GF_OK;
}

GF_API gf_status gf_plan_launches(const gf_plan* p, int32_t* launches) {
  if (!p || !launches) return fail(GF_ERR_INVALID_VALUE);
  const bool finalize = has_bgrad(p->epi) && p->bgrad_mode != GF_BGRAD_ATOMIC;
  *launches = p->m == 0 || p->n == 0 ? 0 : 1 + (finalize ? 1 : 0);
  return GF_OK;
}

GF_API gf_status gf_plan_k_splits(const gf_plan* p, int32_t* k_splits) {
  if (!p || !k_splits) return fail(GF_ERR_INVALID_VALUE);
  *k_splits = p->k_splits;
  return GF_OK;
}

GF_API gf_status gf_matmul_execute(const gf_plan* p, const void* A, const void* B,
                                   const void* bias, void* out, const void* aux_in,
                                   void* aux_out, float* bgrad, struct CUstream_st* stream) {
  if (!p || p->epi > gf::EPI_DGELU_BGRAD) return fail(GF_ERR_INVALID_VALUE);
  ExecArgs x = {A, B, nullptr, bias, out, aux_in, nullptr, aux_out, nullptr, bgrad};
  return execute_impl(p, x, reinterpret_cast<cudaStream_t>(stream));
}

GF_API gf_status gf_swiglu_execute(const gf_plan* p, const void* x_in, const void* Wg,
                                   const void* Wu, void* h, void* g_out, void* u_out,
                                   struct CUstream_st* stream) {
  if (!p || !gf::epi_dual(p->epi)) return fail(GF_ERR_INVALID_VALUE);
  ExecArgs x = {x_in, Wg, Wu, nullptr, h, nullptr, nullptr, g_out, u_out, nullptr};
  return execute_impl(p, x, reinterpret_cast<cudaStream_t>(stream));
}

GF_API gf_status gf_dswiglu_execute(const gf_plan* p, const void* dout, const void* Wd,
                                    const void* g, const void* u, void* d_gate, void* d_up,
                                    struct CUstream_st* stream) {
  if (!p || p->epi != gf::EPI_DSWIGLU) return fail(GF_ERR_INVALID_VALUE);
  ExecArgs x = {dout, Wd, nullptr, nullptr, d_gate, g, u, d_up, nullptr, nullptr};
  return execute_impl(p, x, reinterpret_cast<cudaStream_t>(stream));
}

GF_API gf_status gf_plan_status(const gf_plan* p, struct CUstream_st* stream) {
  if (!p) return fail(GF_ERR_INVALID_VALUE);
  if (cudaSetDevice(p->device) != cudaSuccess) return fail(GF_ERR_CUDA);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return fail(GF_ERR_CUDA);
  int32_t word = 0;
  if (cudaMemcpy(&word, p->d_status, 4, cudaMemcpyDeviceToHost) != cudaSuccess)
    return fail(GF_ERR_CUDA);
  if (word != 0) {
    // which waits gave up: 1 producer, 2 MMA on a stage, 4 MMA on an
    // accumulator buffer, 8 epilogue, 16 teardown drain
    if (getenv("GF_DEBUG")) fprintf(stderr, "gf: device status word 0x%x\n", word);
    // the status word, and the dynamic schedule's tile counters that a launch
    // which gave up may leave part-way
    if (cudaMemset(p->d_status, 0, 256) != cudaSuccess) return fail(GF_ERR_CUDA);
    // a launch that gave up may leave split-k counters part-way
    const size_t counters = p->pair ? 2 * static_cast<size_t>(p->num_tiles - p->split_from)
                                    : static_cast<size_t>(p->num_tiles);
    if (p->k_splits > 1 &&
        cudaMemset(static_cast<char*>(p->d_splitk) + p->splitk_cnt_offset, 0, counters * 4) !=
            cudaSuccess)
      return fail(GF_ERR_CUDA);
    return fail(GF_ERR_DEVICE_TIMEOUT);
  }
  return GF_OK;
}

GF_API void gf_plan_free(gf_plan* p) {
  if (!p) return;
  cudaSetDevice(p->device);
  if (p->d_partials) cudaFree(p->d_partials);
  if (p->d_splitk) cudaFree(p->d_splitk);
  if (p->d_status) cudaFree(p->d_status);
  delete p;
}

}  // extern "C"
