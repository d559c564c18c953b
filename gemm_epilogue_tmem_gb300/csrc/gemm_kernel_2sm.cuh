// CTA-pair variant of the fused GEMM + epilogue kernel: a cluster of two
// CTAs on two SMs computes one 256 x 256 output tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16 per instruction).
//
//   - Each CTA loads its own 128 rows of A and its own half of the B columns
//     for every k-slice (TMA, 128-byte swizzle, no multicast): per SM the
//     operand traffic per flop is 2/3 of the single-CTA 128 x 256 tile's.
//   - Two B operands (gate+up SwiGLU): the pair's "halves" of B are the two
//     weights -- rank 0 loads 128 rows of the gate weight, rank 1 the same
//     rows of the up weight -- so one N = 256 MMA puts g in accumulator
//     columns 0..127 and u in 128..255 of every row: a 256 x 128 output tile
//     at the MMA rate of the single-operand kernel.
//   - The stage-full barrier lives in the leader CTA (rank 0): the leader's
//     producer expects the bytes of both CTAs, the peer's TMA loads signal
//     the leader's barrier (.cta_group::2).
//   - The leader's MMA thread issues the pair MMA; commits are multicast to
//     both CTAs (stage-empty, accumulator-full barriers).
//   - Each CTA drains its own 128 TMEM lanes (its 128 rows x BN columns)
//     with the same epilogue as the single-CTA kernel; both CTAs' epilogue
//     warps release the accumulator buffer on the leader's barrier.
//   - Tiles: static (pair c takes tiles c, c + pairs, ...) or dynamic: the
//     leader's producer takes the next tile from a global counter and hands
//     its index to every role of both CTAs through a 4-deep ring in shared
//     memory. The last pair to run out of tiles resets the counter (and the
//     count of finished pairs beside it), so no host-side reset is enqueued
//     between launches. Dynamic keeps the tiles in flight a contiguous run of the
//     raster order, so operand panels shared by neighbouring tiles are read
//     from HBM about once instead of once per drifting pair.
//   - Wide tiles (WIDE): 256 x 512 per pair, two N = 256 MMAs per k-step
//     into the two halves of one 512-column accumulator. A k-slice of A then
//     feeds twice the flops, so a stage brings 48 KB per 1024 MMA cycles per
//     SM instead of 32 KB per 512: 3/4 of the operand bytes per flop, for
//     SMs whose tensor-copy ingress, not the tensor pipe, sets the pace of
//     the 256-wide tile. The price is a single accumulator: the epilogue
//     drains half 0 and releases it, then half 1; the MMA thread starts the
//     next tile on half 0 over the stages already loaded and adds the half-1
//     products of those stages once half 1 is free, and runs a tile's last
//     ring of k-slices into half 0 first so that half 0's drain starts early.
//     Eight epilogue warps (two per TMEM lane quarter, each with half of the
//     columns) keep that exposed drain short.
//     With two B operands (gate+up SwiGLU) a wide tile is 256 x 256 outputs:
//     each CTA loads two 128-row parts of its own weight, so accumulator half
//     h holds g and u of output columns 128 h .. 128 h + 127 side by side.
//   - Teardown: drains, then a cluster barrier, then a pair TMEM dealloc.
#pragma once

#include "gemm_kernel.cuh"

namespace gf {

// Eight epilogue warps (two per TMEM lane quarter) for the wide tiles, whose
// drain is partly exposed. (The 256 x 256 tiles' drain runs under the next
// mainloop; their epilogues that read 16-bit side inputs per element ran
// slower with eight warps than with four.)
GF_HD constexpr bool pair_epi8(int epi, bool wide) { return wide && epi >= 0; }

// A 2 KB shared-memory staging buffer per epilogue warp: 64-byte row-segment
// output stores, and coalesced loads of saved 16-bit activations. The wide
// tiles, and on 256 x 256 tiles the epilogs that store two or three 16-bit
// outputs per element or read saved activations (one ring stage makes room
// for it where the bias-gradient scratch has not already).
GF_HD constexpr bool pair_stg(int epi, bool wide) {
  return wide || epi == EPI_GELU_AUX_BIAS || epi == EPI_SWIGLU_SAVE || epi == EPI_DSWIGLU ||
         epi == EPI_DGELU_BGRAD;
}

// Chunk slots of the dSwiGLU side-input ring per epilogue warp (256 x 256
// tiles): the saved g and u of three 32-column chunks in flight ahead of the
// drain, which is otherwise bound by the latency of those reads.
GF_HD constexpr int pair_side_ring(int epi, bool wide) {
  return !wide && epi == EPI_DSWIGLU ? 3 : 0;
}

// A second 2 KB staging buffer per epilogue warp (in place of the 1 KB
// side-input buffer, which the dSwiGLU epilog does not use): the wide tiles'
// dSwiGLU drain stores d_up from one buffer and d_gate from the other, so
// that its two TMA stores per chunk do not wait for each other.
GF_HD constexpr bool pair_stg2(int epi, bool wide) { return wide && epi == EPI_DSWIGLU; }

// NB = number of B operands: 1, or 2 for the gate+up SwiGLU (g and u side by
// side in one accumulator); RED = the epilog reduces a bias gradient and
// needs the [4][BN] scratch; WIDE = two N = 256 MMAs per k-step into one
// 512-column accumulator (256 x 512 tiles; 256 x 256 with two B operands); EPI8 =
// eight epilogue warps (pair_epi8); SRING = side-input ring slots per
// epilogue warp (pair_side_ring).
template <int NB = 1, bool RED = false, bool WIDE = false, bool EPI8 = WIDE, bool STG = WIDE,
          int SRING = 0, bool STG2 = false>
struct PairCfg {
  // output columns of a tile
  static constexpr int BN = WIDE ? (NB == 2 ? 256 : 512) : (NB == 2 ? 128 : 256);
  static constexpr int kABytes = kBM * kBK * 2;        // 16 KB: this CTA's 128 rows of A
  // one 16 KB B part: this CTA's 128 of an MMA's 256 B columns, or (two
  // operands) the tile's 128 columns of this CTA's operand; wide: two parts
  static constexpr int kBPartBytes = 128 * kBK * 2;
  static constexpr int kStageBBytes = (WIDE ? 2 : 1) * kBPartBytes;
  static constexpr int kAccCols = WIDE ? 512 : 256;    // TMEM columns of one accumulator
  static constexpr int kNumAcc = WIDE ? 1 : 2;         // accumulator buffers
  static constexpr int kTmemCols = kNumAcc * kAccCols; // 512 either way
  // epilogue warps: EPI8 drains with two warps per TMEM lane quarter (each
  // takes half of the columns)
  static constexpr int kEpiWarps = EPI8 ? 8 : 4;
  // warps before the epilogue warps: producer, MMA; wide: + two idle warps,
  // so that the control and the epilogue roles are whole warpgroups whose
  // registers can be redistributed (setmaxnreg): the epilogue warps of the
  // wide tiles hold a quarter's worth of the accumulator in registers
  static constexpr int kCtlWarps = WIDE ? 4 : 2;
  static constexpr int kThreads = 32 * (kCtlWarps + kEpiWarps);
  // wide: registers per thread at launch (65536 / 384, in steps of 8), and
  // after the redistribution: control warpgroup 56, epilogue warpgroups 224
  static constexpr int kLaunchRegs = WIDE ? 168 : 0;
  static constexpr int kCtlRegs = 56;
  static constexpr int kEpiRegs = 224;
  static_assert(!WIDE || (kCtlWarps == 4 && kEpiWarps == 8 &&
                          32 * (kCtlWarps * kCtlRegs + kEpiWarps * kEpiRegs) <=
                              kThreads * kLaunchRegs &&
                          kThreads * kLaunchRegs <= 65536),
                "register redistribution within the launch's registers");
  // consumers of a tile index: leader MMA + peer producer + both CTAs' epilogue warps
  static constexpr int kTileConsumers = 2 + 2 * kEpiWarps;
  static constexpr int kCtrlBytes = kSmemCtrlBytes;
  static constexpr int kRedBytes = RED ? 4 * BN * 4 : 0;
  // wide: per epilogue warp a 2 KB output staging buffer (its drain is partly
  // exposed, so its stores go out as 64-byte row segments) and a 1 KB buffer
  // of the tile's prefetched side inputs (column bias or mask words of its
  // 2 x 128 columns)
  // (+ the side-input ring of SRING 4 KB chunk slots per warp)
  static constexpr int kStgBytes =
      WIDE ? kEpiWarps * (2048 + (STG2 ? 2048 : 1024))
           : (STG ? kEpiWarps * (2048 + SRING * static_cast<int>(kSideSlotBytes)) : 0);
  static constexpr int kStages = ring_stages(kABytes + kStageBBytes, kRedBytes + kStgBytes);
  static constexpr int kSmemBytes = kSmemAlignSlack + kStages * (kABytes + kStageBBytes) +
                                    kCtrlBytes + kRedBytes + kStgBytes;
  static_assert(kStages >= 3 && kSmemBytes <= kSmemPerCta, "shared memory budget");
  static_assert(16 * kStages + 132 <= kCtrlBytes, "control region");
};

constexpr int kTileRing = 4;  // tile indices in flight between the roles (dynamic schedule)

// Pair tile t -> (256-row block, 256-column block), grouped like tile_coords.
__device__ __forceinline__ void pair_tile_coords(const GemmParams& p, int t, int& mb2, int& nb) {
  const int num_m2 = (p.num_m_blocks + 1) / 2;
  if (p.raster_n) {  // groups of group_m column blocks, columns fastest within a group
    const int group_size = p.group_m * num_m2;
    const int group = t / group_size;
    const int first_n = group * p.group_m;
    const int gn = min(p.num_n_blocks - first_n, p.group_m);
    const int r = t - group * group_size;
    nb = first_n + r % gn;
    mb2 = r / gn;
    return;
  }
  const int group_size = p.group_m * p.num_n_blocks;
  const int group = t / group_size;
  const int first_m = group * p.group_m;
  const int gm = min(num_m2 - first_m, p.group_m);
  const int r = t - group * group_size;
  mb2 = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// relu_aux words of one TMA-store drain (4 chunks of 32 columns from n0h)
// for the 32 rows of the warp starting at row0w; words past M or N are not
// stored. Called by all 32 lanes.
__device__ __forceinline__ void store_aux_words(const GemmParams& p, int row0w, int n0h,
                                                uint32_t lane, const AuxWords& aw) {
  if (row0w >= p.M) return;
  uint32_t* dst = p.aux_out + (size_t)(row0w >> 5) * p.N;
  const uint32_t w[4] = {aw.w0, aw.w1, aw.w2, aw.w3};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int col = n0h + 32 * c + (int)lane;
    if (col < p.N) dst[col] = w[c];
  }
}

// SPLITK (256 x 256 or wide tiles, one B operand): the tiles from
// p.split_from on run as p.k_splits work units of consecutive k-blocks each;
// a unit's CTAs leave their fp32 partial sums in the workspace, and the last
// CTA of each rank of a tile to finish adds them in split order and runs the
// epilogue.
template <int EPI, typename T, bool B_MN, bool WIDE = false, bool SPLITK = false>
__global__ void __launch_bounds__(PairCfg<epi_dual(EPI) ? 2 : 1, epi_has_bgrad(EPI), WIDE,
                                          pair_epi8(EPI, WIDE), pair_stg(EPI, WIDE),
                                          pair_side_ring(EPI, WIDE),
                                          pair_stg2(EPI, WIDE)>::kThreads,
                                  1)
    gemm_epilog_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                            const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmB2,
                            const __grid_constant__ CUtensorMap tmOut,
                            const __grid_constant__ CUtensorMap tmAux, const GemmParams p) {
  constexpr int NB = epi_dual(EPI) ? 2 : 1;
  using C = PairCfg<NB, epi_has_bgrad(EPI), WIDE, pair_epi8(EPI, WIDE), pair_stg(EPI, WIDE),
                    pair_side_ring(EPI, WIDE), pair_stg2(EPI, WIDE)>;
  static_assert(!SPLITK || (NB == 1 && (WIDE || C::kEpiWarps == 4)),
                "split k: one B operand, 256 x 256 or wide tiles");
  constexpr int kRing = pair_side_ring(EPI, WIDE);
  constexpr int S = C::kStages;
  constexpr int BN = C::BN;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + S * C::kABytes;
  const uint32_t ctrl = sB + S * C::kStageBBytes;
  uint8_t* gctrl = gbase + (ctrl - base);
  const uint32_t full0 = ctrl;              // leader: S barriers, stage filled (both CTAs' bytes)
  const uint32_t empty0 = ctrl + 8u * S;    // both: S barriers, stage consumed
  // both: 2 barriers, accumulator buffer ready (wide: only the first is used)
  const uint32_t tfull0 = ctrl + 16u * S;
  // leader: 2 barriers, accumulator buffer drained by the 8 epilogue warps
  // (wide: half 0 drained, half 1 drained)
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t done_bar = tempty0 + 16u;  // leader: MMA teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gctrl + 16 * S + 40);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gctrl + 16 * S + 44);
  const uint32_t tile_full0 = ctrl + 16u * S + 48u;   // both: kTileRing barriers, index ready
  const uint32_t tile_empty0 = ctrl + 16u * S + 80u;  // leader: kTileRing barriers, index read
  const uint32_t ring_s = ctrl + 16u * S + 112u;      // both: kTileRing tile indices
  volatile int* ring = reinterpret_cast<volatile int*>(gctrl + 16 * S + 112);
  // split k: whether this CTA's epilogue counted last for its tile and rank
  volatile int* last_flag = reinterpret_cast<volatile int*>(gctrl + 16 * S + 128);
  float* red = reinterpret_cast<float*>(gctrl + C::kCtrlBytes);
  const uint32_t stg0 = ctrl + C::kCtrlBytes + C::kRedBytes;  // 2 KB output staging per warp
  const uint32_t side0 = stg0 + C::kEpiWarps * 2048u;           // wide: 1 KB side inputs per warp

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  // dSwiGLU: an epilogue warp's side-input ring (kRing slots) after the staging buffers
  const int ew = warp - C::kCtlWarps;  // epilogue warp index (negative: other roles)
  const uint32_t sring = side0 + kRing * kSideSlotBytes * (uint32_t)(ew >= 0 ? ew : 0);
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x >> 1;
  const int num_clusters = gridDim.x >> 1;
  // work units: the pair tiles (the host counts pair tiles for this kernel),
  // with split k the split tiles' units in their place
  const int num_pair_tiles =
      SPLITK ? p.split_from + (p.num_tiles - p.split_from) * p.k_splits : p.num_tiles;
  const bool dynamic = p.tile_counter != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(tfull0, 1);
    mbar_init(tfull0 + 8u, 1);
    mbar_init(tempty0, 2 * C::kEpiWarps);
    mbar_init(tempty0 + 8u, 2 * C::kEpiWarps);
    mbar_init(done_bar, 1);
    for (int r = 0; r < kTileRing; ++r) {
      mbar_init(tile_full0 + 8u * r, 1);
      mbar_init(tile_empty0 + 8u * r, C::kTileConsumers);
    }
    *abort_flag = 0;
    fence_mbar_init();
    if (p.num_k_blocks > 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (NB == 2) prefetch_tmap(&tmB2);
    }
    if constexpr (WIDE) {
      prefetch_tmap(&tmOut);
      if constexpr (EPI == EPI_GELU_AUX_BIAS || EPI == EPI_DSWIGLU) prefetch_tmap(&tmAux);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the set-up above overlaps the previous kernel on the stream; its outputs
  // (this kernel's inputs) are complete from here on
  grid_dep_wait();
  grid_dep_launch();
  bool aborted = false;
  const uint32_t tile_empty_leader = mapa_shared(tile_empty0, 0);

  // Tile index number `it` of this pair for a consumer role (every role but
  // the leader's producer): static, or read from the ring and released on
  // the leader's barrier by lane 0 of the calling warp. -1 ends the loop;
  // -2 is a wait that gave up.
  auto consume_tile = [&](int it, bool release) -> int {
    if (!dynamic) {
      const int t = cluster_id + it * num_clusters;
      return t < num_pair_tiles ? t : -1;
    }
    const int slot = it % kTileRing;
    const uint32_t ph = (uint32_t)(it / kTileRing) & 1u;
    if (!mbar_wait_bounded_cluster(tile_full0 + 8u * slot, ph, abort_flag, p.wait_limit_ns))
      return -2;
    const int t = ring[slot];
    if (release) mbar_arrive_remote(tile_empty_leader + 8u * slot);
    return t;
  };

  // work unit u -> tile, split (-1: the whole tile) and k-blocks [kb0, kb1)
  auto unit_tile = [&](int u, int& split, int& kb0, int& kb1) -> int {
    split = -1;
    kb0 = 0;
    kb1 = p.num_k_blocks;
    if (!SPLITK || u < p.split_from) return u;
    const int v = u - p.split_from;
    split = v % p.k_splits;
    kb0 = split * p.kb_per_split;
    kb1 = min(p.num_k_blocks, kb0 + p.kb_per_split);
    return p.split_from + v / p.k_splits;
  };

  if (warp < C::kCtlWarps) {
    // control warps: warpgroup 0 of the wide tiles gives registers to the
    // two epilogue warpgroups (the host checks the launch's register count)
    if constexpr (WIDE) setmaxnreg_dec<C::kCtlRegs>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && (p.num_k_blocks > 0 || dynamic)) {
      int issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      int loads = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(p.l2_hint_a);
      const uint64_t pol_b = l2_policy(p.l2_hint_b);
      const int ha = p.l2_hint_a, hb = p.l2_hint_b;
      for (int it = 0; ok; ++it) {
        int t;
        if (dynamic && leader) {
          // take the next tile and hand its index to both CTAs
          const int slot = it % kTileRing;
          const uint32_t ph = (uint32_t)(it / kTileRing) & 1u;
          if (!mbar_wait_bounded_cluster(tile_empty0 + 8u * slot, ph ^ 1u, abort_flag,
                                         p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_PRODUCER);
            aborted = true;
            break;
          }
          t = atomicAdd(p.tile_counter, 1);
          if (t >= num_pair_tiles) {
            t = -1;
            // this pair takes no more tiles: count it; the last pair of the
            // launch sets both counters back to zero for the next launch (every
            // pair's last take of a tile comes before its count)
            __threadfence();
            if (atomicAdd(p.tile_counter + 1, 1) == num_clusters - 1) {
              __threadfence();
              atomicExch(p.tile_counter, 0);
              atomicExch(p.tile_counter + 1, 0);
            }
          }
          ring[slot] = t;
          st_shared_cluster_u32(mapa_shared(ring_s + 4u * slot, 1), (uint32_t)t);
          mbar_arrive_remote(mapa_shared(tile_full0 + 8u * slot, 0));
          mbar_arrive_remote(mapa_shared(tile_full0 + 8u * slot, 1));
        } else {
          t = consume_tile(it, true);
          if (t == -2) {
            raise_error(p, abort_flag, ST_TIMEOUT_PRODUCER);
            aborted = true;
            break;
          }
        }
        if (t < 0) break;
        // this unit's k-blocks [kb0, kb1) (the whole k of a whole tile)
        int split = -1, kb0 = 0, kb1 = p.num_k_blocks;
        if constexpr (SPLITK) t = unit_tile(t, split, kb0, kb1);
        int mb2, nb;
        pair_tile_coords(p, t, mb2, nb);
        const int m_row = mb2 * 256 + 128 * (int)rank;  // this CTA's A rows
        // this CTA's B columns (two operands: the tile's columns of its own
        // operand; wide: part h at n_col + 256 h)
        const int n_col = NB == 2 ? nb * BN : nb * BN + 128 * (int)rank;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_PRODUCER);
            ok = false;
            aborted = true;
            break;
          }
          ++loads;
          if (loads != p.drop_load) {
            const uint32_t fb_local = full0 + 8u * stage;
            const uint32_t fb = mapa_shared(fb_local, 0);  // the leader's barrier
            if (leader) mbar_arrive_expect_tx(fb_local, 2u * (C::kABytes + C::kStageBBytes));
            tma_load_pair(sA + stage * C::kABytes, &tmA, fb, kb * kBK, m_row, ha, pol_a);
#pragma unroll
            for (int h = 0; h < (WIDE ? 2 : 1); ++h) {
              const uint32_t dst = sB + stage * C::kStageBBytes + h * C::kBPartBytes;
              // (two operands: part h is output columns 128 h of the tile)
              const int col = n_col + (NB == 2 ? 128 : 256) * h;
              if (B_MN && p.b_mn_3d) {
                tma_load3_pair(dst, &tmB, fb, 0, kb * kBK, col / 64, hb, pol_b);
              } else if (B_MN) {
                tma_load_pair(dst, &tmB, fb, col, kb * kBK, hb, pol_b);
                tma_load_pair(dst + 64 * kBK * 2, &tmB, fb, col + 64, kb * kBK, hb, pol_b);
              } else {
                tma_load_pair(dst, NB == 2 && rank == 1 ? &tmB2 : &tmB, fb, kb * kBK, col, hb,
                              pol_b);
              }
            }
            issued[stage] = (int)phase;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the leader's full barriers count both CTAs' bytes: when they have
      // completed, every load of the pair has landed
      if (leader) {
#pragma unroll
        for (int s = 0; s < S; ++s)
          if (issued[s] >= 0 &&
              !mbar_wait_bounded(full0 + 8u * s, (uint32_t)issued[s], nullptr, p.wait_limit_ns))
            raise_error(p, abort_flag, ST_TIMEOUT_DRAIN);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------- MMA (leader)
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = idesc_f16(kBf16, B_MN, 256, 256);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int t = consume_tile(it, true);
        if (t == -2) {
          raise_error(p, abort_flag, ST_TIMEOUT_MMA_TMEM);
          aborted = true;
          break;
        }
        if (t < 0) break;
        int split = -1, kb0 = 0, kb1 = p.num_k_blocks;
        if constexpr (SPLITK) unit_tile(t, split, kb0, kb1);
        // double buffer: tile it uses buffer it & 1, whose previous use (tile
        // it - 2) must be drained; wide: one buffer in two halves, released
        // by the epilogue of tile it - 1 one after the other
        const int buf = WIDE ? 0 : (it & 1);
        const uint32_t use = WIDE ? (uint32_t)it & 1u : (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded_cluster(tempty0 + 8u * buf, use ^ 1u, abort_flag,
                                       p.wait_limit_ns)) {
          raise_error(p, abort_flag, ST_TIMEOUT_MMA_TMEM);
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * C::kAccCols);
        if (p.num_k_blocks == 0) {
          if (WIDE &&
              !mbar_wait_bounded_cluster(tempty0 + 8u, use ^ 1u, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_MMA_TMEM);
            aborted = true;
            break;
          }
          umma_commit_pair(tfull0 + 8u * buf, 0x3);  // nothing to multiply: acc is zero
          if (WIDE) umma_commit_pair(tfull0 + 8u, 0x3);
          continue;
        }
        // the MMAs of one k-slice into accumulator half h (wide) or the whole
        // accumulator
        auto mma_kslice = [&](int st, int kb, int h) {
          const uint32_t a_base = sA + st * C::kABytes;
          const uint32_t b_base = sB + st * C::kStageBBytes + h * C::kBPartBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t adesc = sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bdesc = B_MN ? sdesc_sw128(b_base + kk * 2048, 64 * kBK * 2, 1024)
                                        : sdesc_sw128(b_base + kk * 32, 16, 1024);
            umma_f16_pair(d_tmem + 256u * (uint32_t)h, adesc, bdesc, idesc,
                          ((kb - kb0) | kk) != 0 ? 1u : 0u);
          }
        };
        // this unit's k-blocks
        const int kbeg = kb0;
        const int kend = kb1;
        int kb = kbeg;
        if constexpr (WIDE) {
          // half 0 over the first stages that the producer has loaded while
          // the previous tile drained, then half 1 of the same stages
          const int pre = kend - kbeg < S ? kend - kbeg : S;
          int st = stage;
          uint32_t ph = phase;
          for (int j = 0; j < pre && ok; ++j) {
            if (!mbar_wait_bounded(full0 + 8u * st, ph, abort_flag, p.wait_limit_ns)) {
              raise_error(p, abort_flag, ST_TIMEOUT_MMA_SMEM);
              ok = false;
              aborted = true;
              break;
            }
            tc_fence_after();
            mma_kslice(st, kbeg + j, 0);
            if (++st == S) {
              st = 0;
              ph ^= 1u;
            }
          }
          if (!ok) break;
          if (!mbar_wait_bounded_cluster(tempty0 + 8u, use ^ 1u, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_MMA_TMEM);
            aborted = true;
            break;
          }
          tc_fence_after();
          for (int j = 0; j < pre; ++j) {
            mma_kslice(stage, kbeg + j, 1);
            umma_commit_pair(empty0 + 8u * stage, 0x3);  // frees the stage in both CTAs
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          kb = kbeg + pre;
        }
        // wide: the last S k-slices go half 0 first, then half 1, so that
        // half 0 is complete (and its drain starts) S k-slices early
        const int tail = WIDE && kend - kb >= 2 * S ? S : 0;
        for (; kb < kend - tail; ++kb) {
          if (!mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_MMA_SMEM);
            ok = false;
            aborted = true;
            break;
          }
          tc_fence_after();
          mma_kslice(stage, kb, 0);
          if constexpr (WIDE) mma_kslice(stage, kb, 1);
          umma_commit_pair(empty0 + 8u * stage, 0x3);  // frees the stage in both CTAs
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (WIDE) {
          if (tail > 0) {
            int st = stage;
            uint32_t ph = phase;
            for (int j = 0; j < tail; ++j) {
              if (!mbar_wait_bounded(full0 + 8u * st, ph, abort_flag, p.wait_limit_ns)) {
                raise_error(p, abort_flag, ST_TIMEOUT_MMA_SMEM);
                ok = false;
                aborted = true;
                break;
              }
              tc_fence_after();
              mma_kslice(st, kb + j, 0);
              if (++st == S) {
                st = 0;
                ph ^= 1u;
              }
            }
            if (!ok) break;
            umma_commit_pair(tfull0, 0x3);  // half 0 complete
            for (int j = 0; j < tail; ++j) {
              mma_kslice(stage, kb + j, 1);
              umma_commit_pair(empty0 + 8u * stage, 0x3);
              if (++stage == S) {
                stage = 0;
                phase ^= 1u;
              }
            }
          } else {
            umma_commit_pair(tfull0, 0x3);
          }
          umma_commit_pair(tfull0 + 8u, 0x3);  // half 1 complete
        } else {
          umma_commit_pair(tfull0 + 8u * buf, 0x3);
        }
      }
      umma_commit_pair(done_bar, 0x1);
      if (!mbar_wait_bounded(done_bar, 0, nullptr, p.wait_limit_ns))
        raise_error(p, abort_flag, ST_TIMEOUT_DRAIN);
    }
    __syncwarp();
  }  // warps 2 and 3 of the wide tiles' control warpgroup have no role
  } else {
    if constexpr (WIDE) setmaxnreg_inc<C::kEpiRegs>();
    // ------------------------------------------------------------ epilogue
    // warp w drains TMEM lanes 32 (w % 4)..; with 8 epilogue warps (wide) the
    // two warps of a lane quarter take column halves `sub` 0 and 1
    constexpr int NT = 32 * C::kEpiWarps;  // epilogue threads
    const int q = warp & 3;
    const int sub = ew >> 2;
    const int ep_tid = threadIdx.x - 32 * C::kCtlWarps;
    const uint32_t tempty_leader = mapa_shared(tempty0, 0);
    for (int it = 0;; ++it) {
      // every lane reads the index; lane 0 releases the slot for the warp
      int t = consume_tile(it, false);
      if (dynamic && t != -2) {
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tile_empty_leader + 8u * (it % kTileRing));
      }
      bool ok = t != -2;
      // (the epilogs with a barrier of all epilogue warps agree on the outcome)
      if constexpr (epi_has_bgrad(EPI) || SPLITK) ok = !named_bar_red_or(1, NT, !ok);
      if (!ok) {
        raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
        aborted = true;
        break;
      }
      if (t < 0) break;
      int split = -1, kb0 = 0, kb1 = p.num_k_blocks;
      if constexpr (SPLITK) t = unit_tile(t, split, kb0, kb1);
      int mb2, nb;
      pair_tile_coords(p, t, mb2, nb);
      const int row0 = mb2 * 256 + 128 * (int)rank;
      const int n0 = nb * BN;
      // wide: this warp's 128 columns of each accumulator half, their side
      // inputs (bias or mask words) prefetched while the mainloop runs
      constexpr bool kSide = WIDE && (EPI == EPI_DRELU_BGRAD || epi_has_bias(EPI));
      constexpr uint32_t kSideHalf = EPI == EPI_DRELU_BGRAD ? 512u : 256u;  // 128 columns
      const int c_sub = 128 * sub;
      const uint32_t side = side0 + 1024u * (uint32_t)ew;
      if constexpr (kSide) {
        prefetch_side<EPI, T, 128>(p, row0 + 32 * q, n0 + c_sub, lane, side);
        prefetch_side<EPI, T, 128>(p, row0 + 32 * q, n0 + 256 + c_sub, lane, side + kSideHalf);
      }
      if constexpr (kRing > 0)  // the first chunks' saved g and u, under the mainloop
        side_ring_prefetch<T, kRing>(p, row0 + 32 * q, n0, min(BN / 32, (p.N - n0 + 31) / 32),
                                     lane, sring);
      const int buf = WIDE ? 0 : (it & 1);
      const uint32_t use = WIDE ? (uint32_t)it & 1u : (uint32_t)(it >> 1) & 1u;
      // the accumulator (wide: accumulator half h) is complete; all epilogue
      // warps take part (the bias-gradient and split-k epilogs agree on the
      // outcome)
      auto wait_acc = [&](uint32_t h) -> bool {
        bool okh = mbar_wait_bounded(tfull0 + 8u * (buf + h), use, abort_flag, p.wait_limit_ns);
        if constexpr (epi_has_bgrad(EPI) || SPLITK) okh = !named_bar_red_or(1, NT, !okh);
        if (okh) tc_fence_after();
        return okh;
      };
      // (wide: each half's drain waits for its half itself, after issuing
      // the loads of its first side inputs)
      if (!WIDE && !wait_acc(0u)) {
        raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
        aborted = true;
        break;
      }
      const uint32_t t_row =
          tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * C::kAccCols);
      if constexpr (WIDE) {
        // half 0, then half 1: each warp loads its 128 columns of the half
        // out of tensor memory and releases the half at once (the next
        // tile's first MMAs go to half 0), then applies the epilog from
        // registers. The 16-bit outputs leave by TMA stores and the relu_aux
        // words are stored after the release, so that the release (a
        // cluster-scope release) has no global stores to wait for.
        const uint32_t stg = stg0 + 2048u * (uint32_t)ew;
        // dSwiGLU: d_gate's staging buffer (in place of the side buffer)
        const uint32_t stg2 = pair_stg2(EPI, WIDE) ? side0 + 2048u * (uint32_t)ew : 0u;
        AuxWords aw;
        // (a relaxed arrive: the accumulator's reads have completed before
        // it, and it must not wait for this warp's TMA stores in flight)
        auto release_half = [&](uint32_t h) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_remote_relaxed(tempty_leader + 8u * h);
        };
        if constexpr (NB == 2) {
          // two operands: half h holds g (columns 0..127) and u (128..255) of
          // output columns n0 + 128 h ..; this warp takes 64 of them
          const uint32_t c64 = 64u * (uint32_t)sub;
          if (!epilogue_drain_dual_wide<EPI, T>(
                  p, t_row + c64, t_row + 128u + c64, row0, n0 + (int)c64, q, lane, stg, &tmOut,
                  [&]() { release_half(0u); }, [&]() { return wait_acc(0u); })) {
            raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
            aborted = true;
            break;
          }
          if (!epilogue_drain_dual_wide<EPI, T>(
                  p, t_row + 256u + c64, t_row + 384u + c64, row0, n0 + 128 + (int)c64, q, lane,
                  stg, &tmOut, [&]() { release_half(1u); }, [&]() { return wait_acc(1u); })) {
            raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
            aborted = true;
            break;
          }
        } else {
          if constexpr (SPLITK) {
            if (split >= 0) {
              // split k: both halves complete, this unit's partial sums go to
              // the workspace; the last CTA of this rank of the tile to count
              // adds all of them, in split order, into its accumulator and
              // drains it, the others release both halves
              if (!wait_acc(0u) || !wait_acc(1u)) {
                raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
                aborted = true;
                break;
              }
              if (!splitk_reduce<BN, NT, 128, 256>(p, t_row, 2 * (t - p.split_from) + (int)rank,
                                                   split, p.k_splits, q, lane, ep_tid, last_flag,
                                                   0u, 0u, c_sub)) {
                release_half(0u);
                release_half(1u);
                continue;
              }
            }
          }
          if (!epilogue_drain<EPI, T, 128, BN, true, kSide, 0, true, true>(
                  p, t_row + (uint32_t)c_sub, row0, n0 + c_sub, q, lane, red + c_sub, stg, side,
                  &tmOut, &tmAux, &aw, [&]() { release_half(0u); }, stg2,
                  [&]() { return wait_acc(0u); })) {
            raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
            aborted = true;
            break;
          }
          if constexpr (EPI == EPI_RELU_AUX_BIAS) store_aux_words(p, row0 + 32 * q, n0 + c_sub, lane, aw);
          // half 1 is complete a few k-slices after half 0
          if (!epilogue_drain<EPI, T, 128, BN, true, kSide, 0, true, true>(
                  p, t_row + 256u + (uint32_t)c_sub, row0, n0 + 256 + c_sub, q, lane,
                  red + 256 + c_sub, stg, side + kSideHalf, &tmOut, &tmAux, &aw,
                  [&]() { release_half(1u); }, stg2, [&]() { return wait_acc(1u); })) {
            raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
            aborted = true;
            break;
          }
          if constexpr (EPI == EPI_RELU_AUX_BIAS)
            store_aux_words(p, row0 + 32 * q, n0 + 256 + c_sub, lane, aw);
        }
      } else if constexpr (C::kEpiWarps == 8) {
        // this warp's half of the tile's columns
        constexpr int H = BN / 2;
        epilogue_drain<EPI, T, H, BN>(p, t_row + (uint32_t)(H * sub), row0, n0 + H * sub, q, lane,
                                      red + H * sub);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_leader + 8u * buf);
      } else {
        constexpr bool kStg = pair_stg(EPI, false);
        // split k: this unit's partial sums go to the workspace; the last
        // CTA of this rank of the tile to count adds all of them, in split
        // order, into its accumulator and drains it
        bool drain = true;
        if constexpr (SPLITK) {
          if (split >= 0)
            drain = splitk_reduce<BN>(p, t_row, 2 * (t - p.split_from) + (int)rank, split,
                                      p.k_splits, q, lane, ep_tid, last_flag, 0u, 0u);
        }
        if (drain)
          epilogue_drain<EPI, T, BN, BN, kStg, false, kRing>(
              p, t_row, row0, n0, q, lane, red, stg0 + 2048u * (uint32_t)ew, sring);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(tempty_leader + 8u * buf);
      }
      if constexpr (epi_has_bgrad(EPI)) epilogue_bgrad<BN, NT>(p, red, ep_tid, n0, row0 / kBM);
    }
    if constexpr (kRing > 0) cp_async_wait_all();  // no copy lands after the CTA is gone
    if constexpr (WIDE) {
      if (lane == 0) bulk_wait_all();  // this warp's TMA stores have completed
      __syncwarp();
    }
  }

  // a CTA that gave up may still have loads in flight towards its shared
  // memory that no barrier of its own tracks: give them time to land
  if (__syncthreads_or(aborted ? 1 : 0) || *abort_flag) sleep_ns(200000);
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

}  // namespace gf
