// Persistent, warp-specialised fused GEMM + epilogue kernel for sm_103a.
//
//   warp 0      : TMA producer -- loads A and B k-slices into a ring of
//                 shared-memory stages (128-byte swizzle, no multicast).
//   warp 1      : allocates tensor memory and issues tcgen05.mma (one thread)
//                 into a double-buffered fp32 accumulator in TMEM.
//   warps 2..5  : epilogue -- drain TMEM with tcgen05.ld (warp w reads TMEM
//                 lanes 32*(w%4)..+31, i.e. 32 rows of the tile), apply the
//                 epilog and store. The second accumulator buffer lets the
//                 epilogue of tile t run under the mainloop of tile t+1.
//
// Epilogs (web pages on fused matmul epilogs: "Fusing Matmul Epilogs with
// nvmath-python", sections "The problem addressed by fused epilogs",
// "Forward-pass capabilities in the source", "Backward-pass path shown in the
// example"; nvmath-python / cuBLASLt page, step 2 and "other epilogs"):
//   NONE          out = acc
//   BIAS          out = acc + bias
//   RELU_BIAS     out = max(acc + bias, 0)
//   RELU_AUX_BIAS RELU_BIAS, plus the ReLU mask (z > 0) packed with
//                 __ballot_sync into column words: a warp's 32 lanes are 32
//                 consecutive rows, so one ballot is one word.
//   DRELU_BGRAD   dz = acc where the mask bit is set, else 0; out = dz; the
//                 column sums of dz are reduced in the CTA (warp shuffles,
//                 then the four warps in a fixed order) and written as one
//                 partial per tile, or added with one atomicAdd per column.
//
// Every mbarrier wait is bounded; on time-out the kernel records an error in
// the plan's status word, tells the other roles to stop, waits for its own
// copies and MMAs in flight and frees its tensor memory before returning.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include <type_traits>

#include "params.h"
#include "ptx.cuh"

namespace gf {

constexpr int kBM = 128;
constexpr int kBK = 64;  // 64 x 16-bit = 128 bytes = one swizzle row
constexpr int kThreads = 192;

// NB = number of B operands (2 for the gate+up SwiGLU: two accumulators);
// RED = the epilog reduces a bias gradient and needs the [4][BN] scratch.
template <int BN, int NB = 1, bool RED = false>
struct TileCfg {
  static_assert(BN == 128 || BN == 256, "tile N");
  static_assert(NB == 1 || (NB == 2 && BN == 128), "two B operands need 128-wide tiles");
  static constexpr int kABytes = kBM * kBK * 2;
  static constexpr int kBBytes = BN * kBK * 2;            // one B operand
  static constexpr int kStageBBytes = NB * kBBytes;       // all B operands of a stage
  static constexpr int kAccCols = NB * BN;                // TMEM columns of one accumulator set
  static constexpr int kTmemCols = 2 * kAccCols;          // two accumulator buffers
  static constexpr int kCtrlBytes = kSmemCtrlBytes;
  static constexpr int kRedBytes = RED ? 4 * BN * 4 : 0;
  static constexpr int kStages = ring_stages(kABytes + kStageBBytes, kRedBytes);
  static constexpr int kSmemBytes =
      kSmemAlignSlack + kStages * (kABytes + kStageBBytes) + kCtrlBytes + kRedBytes;
  static_assert(kStages >= 3 && kSmemBytes <= kSmemPerCta, "shared memory budget");
};

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) {
  return __half2float(x);
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// 8 consecutive 16-bit values -> fp32
template <typename T>
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  const T* h = reinterpret_cast<const T*>(&u);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = to_f32<T>(h[i]);
}

// Hardware tanh (tanh.approx.f32, relative error about 2^-11: below the
// rounding of the 16-bit outputs these epilogues store).
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// tanh form of GELU (Hendrycks & Gimpel, "Gaussian Error Linear Units",
// 2016): 0.5 z (1 + tanh(c (z + k z^3))) with c = sqrt(2/pi), k = 0.044715,
// and its derivative 0.5 (1 + t) + 0.5 z (1 - t^2) c (1 + 3 k z^2), t the
// tanh. Written as u = z (c + c k z^2) and 0.5 z + 0.5 z t, in fused
// multiply-adds with c k and 3 c k folded: five operations and one tanh per
// element for the forward, nine and one for the derivative.
constexpr float kGeluC = 0.7978845608028654f;     // sqrt(2 / pi)
constexpr float kGeluCK = 0.035677408136300125f;  // sqrt(2 / pi) * 0.044715
constexpr float kGelu3CK = 0.10703222440890038f;  // 3 sqrt(2 / pi) * 0.044715

__device__ __forceinline__ float gelu_tanh(float z) {
  const float z2 = z * z;
  const float u = z * fmaf(kGeluCK, z2, kGeluC);
  const float h = 0.5f * z;
  return fmaf(h, tanh_fast(u), h);
}

__device__ __forceinline__ float dgelu_tanh(float z) {
  const float z2 = z * z;
  const float t = tanh_fast(z * fmaf(kGeluCK, z2, kGeluC));
  const float b = fmaf(kGelu3CK, z2, kGeluC);  // c (1 + 3 k z^2)
  const float s = fmaf(-t, t, 1.f);            // 1 - t^2
  return fmaf(0.5f * z * s, b, fmaf(0.5f, t, 0.5f));
}

// SiLU and the logistic function of the SwiGLU epilogues (gate+up
// forward, dSwiGLU backward): sigmoid(g) = 1 / (1 + e^-g) = (1 + tanh(g/2)) / 2,
// silu(g) = g sigmoid(g).
__device__ __forceinline__ float sigmoid_f(float g) { return fmaf(0.5f, tanh_fast(0.5f * g), 0.5f); }

__device__ __forceinline__ float silu_f(float g) { return g * sigmoid_f(g); }

// 32 consecutive values of one row -> 4 x 16-byte stores of T (columns at or
// past N are skipped; N is a multiple of 8)
template <typename T>
__device__ __forceinline__ void store_row32(T* dst, const float* v, int col0, int N) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (col0 + 8 * g < N) {
      uint4 u;
      u.x = pack2<T>(v[8 * g + 0], v[8 * g + 1]);
      u.y = pack2<T>(v[8 * g + 2], v[8 * g + 3]);
      u.z = pack2<T>(v[8 * g + 4], v[8 * g + 5]);
      u.w = pack2<T>(v[8 * g + 6], v[8 * g + 7]);
      *reinterpret_cast<uint4*>(dst + 8 * g) = u;
    }
  }
}

// 32 x 32 bit-matrix transpose across a warp (lane i holds row i): five
// butterfly stages, each swapping the off-diagonal s x s blocks between lanes
// i and i ^ s with one shuffle. Returns column `lane`: bit i = bit `lane` of
// lane i's input. Called by all 32 lanes.
__device__ __forceinline__ uint32_t bit_transpose32(uint32_t x, uint32_t lane) {
  const uint32_t lo[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int sh = 16 >> k;
    const uint32_t y = __shfl_xor_sync(0xFFFFFFFFu, x, sh);
    x = (lane & (uint32_t)sh) ? ((x & ~lo[k]) | ((y >> sh) & lo[k]))
                              : ((x & lo[k]) | ((y << sh) & ~lo[k]));
  }
  return x;
}

// The same 32 columns for all 32 rows of a warp (lane l holds row row0w + l),
// through a 2 KB shared-memory transpose at `stg`: each global store
// instruction then writes 8 rows x 64 contiguous bytes instead of 32 rows x
// 16 bytes. The 16-byte pieces of a staged row are XOR-permuted by
// (row / 2) % 4 so that both the row-wise writes and the piece-wise reads hit
// 8 distinct 16-byte bank groups. Rows at or past M and columns at or past N
// (a multiple of 8) are not written. Called by all 32 lanes.
template <typename T>
__device__ __forceinline__ void store_rows32_staged(T* base, int M, int N, int row0w, int col0,
                                                    const float* v, uint32_t lane, uint32_t stg) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack2<T>(v[2 * i], v[2 * i + 1]);
  const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
  for (uint32_t pc = 0; pc < 4; ++pc)
    st_shared_v4(stg + lane * 64u + ((pc ^ sw) << 4), w[4 * pc], w[4 * pc + 1], w[4 * pc + 2],
                 w[4 * pc + 3]);
  __syncwarp();
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t r = 8u * g + (lane >> 2);
    const uint32_t pc = lane & 3u;
    const uint4 val = ld_shared_v4(stg + r * 64u + ((pc ^ ((r >> 1) & 3u)) << 4));
    const int row = row0w + (int)r;
    const int col = col0 + 8 * (int)pc;
    if (row < M && col < N) *reinterpret_cast<uint4*>(base + (size_t)row * N + col) = val;
  }
  __syncwarp();
}

// The same 32 x 32 block written by one 2-D TMA store from the staging buffer
// (its XOR permutation of 16-byte pieces by (row / 2) % 4 is the tensor map's
// 64-byte swizzle, so the box's rows land where the map expects them; rows
// and columns outside the tensor are not written). The store is issued by
// lane 0 and tracked by its bulk groups; the buffer is written again only
// after that store has read it. Nothing of it is left in flight for a later
// release fence of the warp to wait for. Called by all 32 lanes.
// PEND: bulk groups that may still be reading (0; 1 when the warp alternates
// two staging buffers, each store waiting only for the one before the last).
template <typename T, int PEND = 0>
__device__ __forceinline__ void store_rows32_tma(const CUtensorMap* map, int row0w, int col0,
                                                 const float* v, uint32_t lane, uint32_t stg) {
  uint32_t w[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = pack2<T>(v[2 * i], v[2 * i + 1]);
  if (lane == 0) bulk_wait_read<PEND>();  // the previous store from this buffer has read it
  __syncwarp();
  const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
  for (uint32_t pc = 0; pc < 4; ++pc)
    st_shared_v4(stg + lane * 64u + ((pc ^ sw) << 4), w[4 * pc], w[4 * pc + 1], w[4 * pc + 2],
                 w[4 * pc + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stg, col0, row0w);
    bulk_commit();
  }
}

// relu_aux words of a drain over 4 chunks kept in registers, so that they are
// stored after the accumulator release (TMA-store drains)
struct AuxWords {
  uint32_t w0, w1, w2, w3;
};

// this lane's 32 values of row `row` (direct) or the warp's 32 rows (staged)
template <typename T, bool STG>
__device__ __forceinline__ void emit_row32(T* base, int M, int N, int row0w, int col0,
                                           const float* v, uint32_t lane, uint32_t stg) {
  if constexpr (STG) {
    store_rows32_staged<T>(base, M, N, row0w, col0, v, lane, stg);
  } else {
    const int row = row0w + (int)lane;
    if (row < M) store_row32<T>(base + (size_t)row * N + col0, v, col0, N);
  }
}

// Tile t -> (m block, n block): groups of group_m row blocks are swept
// column by column so that CTAs running together share A and B in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mb, int& nb) {
  if (p.raster_n) {  // groups of group_m column blocks, columns fastest within a group
    const int group_size = p.group_m * p.num_m_blocks;
    const int group = t / group_size;
    const int first_n = group * p.group_m;
    const int gn = min(p.num_n_blocks - first_n, p.group_m);
    const int r = t - group * group_size;
    nb = first_n + r % gn;
    mb = r / gn;
    return;
  }
  const int group_size = p.group_m * p.num_n_blocks;
  const int group = t / group_size;
  const int first_m = group * p.group_m;
  const int gm = min(p.num_m_blocks - first_m, p.group_m);
  const int r = t - group * group_size;
  mb = first_m + r % gm;
  nb = r / gm;
}

__device__ __forceinline__ void raise_error(const GemmParams& p, volatile int* abort_flag,
                                            int code) {
  *abort_flag = 1;
  atomicOr(p.status, code);
}

// Per-tile side inputs of a drain, fetched into this warp's shared buffer at
// `side` before the accumulator is ready (the loads overlap the mainloop):
// the column bias of columns n0 .. n0 + NC - 1 (T, zero past N; bias epilogs
// with a per-column bias), or the mask words of this warp's 32 rows for the
// same columns (uint32, zero past N or M; DRELU_BGRAD). Called by all 32 lanes.
template <int EPI, typename T, int NC>
__device__ __forceinline__ void prefetch_side(const GemmParams& p, int row0w, int n0,
                                              uint32_t lane, uint32_t side) {
  if constexpr (EPI == EPI_DRELU_BGRAD) {
    const int wrow = row0w >> 5;
    const bool wrow_ok = row0w < p.M;
#pragma unroll
    for (int i = 0; i < NC / 32; ++i) {
      const int col = n0 + 32 * i + (int)lane;
      const uint32_t w = wrow_ok && col < p.N ? __ldg(p.aux_in + (size_t)wrow * p.N + col) : 0u;
      st_shared_u32(side + 4u * (uint32_t)(32 * i + (int)lane), w);
    }
  } else if constexpr (epi_has_bias(EPI)) {
    if (p.bias_axis == 0) {
      const T* bias = reinterpret_cast<const T*>(p.bias);
      // NC columns of 2 bytes: 16-byte pieces, lane-strided
#pragma unroll
      for (int pc = (int)lane; pc < NC / 8; pc += 32) {
        const int col = n0 + 8 * pc;
        const uint4 b = col < p.N ? __ldg(reinterpret_cast<const uint4*>(bias + col))
                                  : make_uint4(0u, 0u, 0u, 0u);
        st_shared_v4(side + 16u * (uint32_t)pc, b.x, b.y, b.z, b.w);
      }
    }
  }
  __syncwarp();
}

// Drain one 128-row x BN accumulator from tensor memory and apply the
// epilog. Warp quarter q owns TMEM lanes 32q..32q+31 = output rows
// row0 + 32q + lane; t_row addresses (lane 32q, first column of the buffer).
// The drain is software-pipelined over 32-column chunks: the tensor-memory
// load and the global side inputs (bias, mask word, saved activations) of
// chunk c + 1 are issued before chunk c is processed, so their latencies
// overlap its arithmetic and stores.
// A bias-gradient epilog leaves the warp's 32-row column sums in
// red[q * RS + column] (RS = BN unless the caller drains a wider tile in parts).
// STG: 16-bit outputs go through this warp's 2 KB staging buffer at `stg`
// (store_rows32_staged), else straight from registers. SIDE: the column bias
// (T) or this warp's mask words (uint32) of columns n0.. were prefetched into
// shared memory at `side` (prefetch_side), and are read from there.
// dSwiGLU side-input ring: per epilogue warp, slots of one 32-column chunk's
// saved g (2 KB: 32 rows x 64 bytes) and u (2 KB), filled by asynchronous
// copies several chunks ahead of the drain (and before the accumulator is
// ready), in the staging buffer's layout (16-byte piece pc of row r at
// r * 64 + ((pc ^ (r / 2 % 4)) * 16)).
constexpr uint32_t kSideSlotBytes = 4096;

// Issue (without committing) the copies of one chunk into `slot`: lane l
// copies 16 bytes of rows 8 g + l / 4 (g = 0..3) at column col0 + 8 (l % 4),
// of g and of u; rows at or past M and columns at or past N read nothing and
// leave zeros.
template <typename T>
__device__ __forceinline__ void side_ring_issue(const GemmParams& p, int row0w, int col0,
                                                uint32_t lane, uint32_t slot) {
  const uint32_t pc = lane & 3u;
  const int col = col0 + 8 * (int)pc;
#pragma unroll
  for (int in = 0; in < 2; ++in) {
    const T* base = reinterpret_cast<const T*>(in == 0 ? p.aux_in : p.aux_in2);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t r = 8u * g + (lane >> 2);
      const int row = row0w + (int)r;
      const bool ok = row < p.M && col < p.N;
      cp_async_16(slot + 2048u * in + r * 64u + ((pc ^ ((r >> 1) & 3u)) << 4),
                  ok ? static_cast<const void*>(base + (size_t)row * p.N + col)
                     : static_cast<const void*>(base),
                  ok ? 16u : 0u);
    }
  }
}

// The first `SRING` chunks of a drain over columns n0.. (one commit group per
// slot, empty past N), issued before the accumulator is ready.
template <typename T, int SRING>
__device__ __forceinline__ void side_ring_prefetch(const GemmParams& p, int row0w, int n0,
                                                   int nch, uint32_t lane, uint32_t ring) {
#pragma unroll
  for (int s = 0; s < SRING; ++s) {
    if (s < nch) side_ring_issue<T>(p, row0w, n0 + 32 * s, lane, ring + kSideSlotBytes * s);
    cp_async_commit();
  }
}

// SRING > 0 (dSwiGLU with the staging buffer): the side inputs come from
// this warp's ring of SRING chunk slots at `side`, whose first SRING chunks
// side_ring_prefetch has issued; the drain keeps SRING chunks in flight.
// TMA: the 16-bit outputs leave through the staging buffer by TMA stores
// (tm_out for out, tm_aux for the 16-bit aux_out), and relu_aux words are
// left in `words` for the caller to store after releasing the accumulator
// (BN <= 128: at most 4 chunks).
// PRELOAD (with TMA, one B operand, no side ring, 4 chunks): every chunk of
// the accumulator is loaded from tensor memory first (128 fp32 registers per
// thread: the caller runs with a raised register allowance), then `release`
// is called -- the accumulator may be overwritten from then on -- and the
// chunks are processed from registers. The MMAs that wait for this
// accumulator then wait only for its tensor-memory reads, not for the
// epilogue's arithmetic and stores. With PRELOAD the drain also waits for
// the accumulator itself (`wait_acc`, false: the wait gave up, nothing is
// drained and the drain returns false), after issuing the first chunk's
// side-input loads, so that their latency runs under the end of the
// mainloop instead of at the start of the drain.
struct NoRelease {
  __device__ __forceinline__ void operator()() const {}
};
struct NoWait {
  __device__ __forceinline__ bool operator()() const { return true; }
};

template <int EPI, typename T, int BN, int RS = BN, bool STG = false, bool SIDE = false,
          int SRING = 0, bool TMA = false, bool PRELOAD = false, typename Release = NoRelease,
          typename WaitAcc = NoWait>
__device__ __forceinline__ bool epilogue_drain(const GemmParams& p, uint32_t t_row, int row0,
                                               int n0, int q, uint32_t lane, float* red,
                                               uint32_t stg = 0, uint32_t side = 0,
                                               const CUtensorMap* tm_out = nullptr,
                                               const CUtensorMap* tm_aux = nullptr,
                                               AuxWords* words = nullptr,
                                               Release release = Release(),
                                               uint32_t stg2 = 0, WaitAcc wait_acc = WaitAcc()) {
  static_assert(!TMA || (STG && BN <= 128), "TMA-store drains: staged, at most 4 chunks");
  static_assert(!PRELOAD || (TMA && !epi_dual(EPI) && SRING == 0 && BN == 128),
                "preloaded drains: TMA stores, one operand, 4 chunks");
  constexpr bool kDual = epi_dual(EPI);
  // 16-byte side inputs per chunk: g and u (DSWIGLU), the pre-activation
  // (DGELU_BGRAD), the column bias (bias epilogs), the mask word (DRELU_BGRAD)
  constexpr int kSide = EPI == EPI_DSWIGLU ? 8
                        : (EPI == EPI_DGELU_BGRAD || epi_has_bias(EPI)) ? 4
                        : EPI == EPI_DRELU_BGRAD ? 1
                                                 : 0;
  constexpr int kSideN = kSide > 0 ? kSide : 1;
  const int row0w = row0 + 32 * q;  // this warp's first row
  const int row = row0w + (int)lane;
  const bool row_ok = row < p.M;
  const int wrow = (row0 >> 5) + q;  // relu_aux word row of this warp's 32 rows
  const bool wrow_ok = row0w < p.M;
  const T* bias = reinterpret_cast<const T*>(p.bias);
  float row_bias = 0.f;
  if constexpr (epi_has_bias(EPI)) {
    if (p.bias_axis == 1 && row_ok) row_bias = to_f32<T>(bias[row]);
  }
  const bool has_acc = p.num_k_blocks > 0;
  const int nch = min(BN / 32, (p.N - n0 + 31) / 32);  // chunks with columns below N
  constexpr bool kRing = SRING > 0;
  static_assert(!kRing || (STG && EPI == EPI_DSWIGLU), "side ring: dSwiGLU with staging");
  if (nch <= 0) {
    if constexpr (kRing) cp_async_wait_all();
    if constexpr (PRELOAD) {
      if (!wait_acc()) return false;
      release();
    }
    return true;
  }

  // one 32 x 32 block of a 16-bit output: `aux` selects aux_out over out
  // stg2 != 0 (TMA): out leaves through the second staging buffer, aux_out
  // and the saved activations' transposes through the first, and a buffer
  // waits only for the store before the last one
  const bool two_stg = TMA && stg2 != 0;
  auto emit = [&](bool aux, int col0, const float* vals) {
    if constexpr (TMA) {
      if (two_stg)
        store_rows32_tma<T, 1>(aux ? tm_aux : tm_out, row0w, col0, vals, lane, aux ? stg : stg2);
      else
        store_rows32_tma<T>(aux ? tm_aux : tm_out, row0w, col0, vals, lane, stg);
    } else {
      emit_row32<T, STG>(reinterpret_cast<T*>(aux ? p.aux_out : p.out), p.M, p.N, row0w, col0,
                         vals, lane, stg);
    }
  };

  // the saved 16-bit activations are read coalesced when the staging buffer
  // is there: lane l loads 16 bytes of row 8g + l/4 (4 lanes per 64-byte row
  // segment), and transpose_side() hands each lane its own row afterwards
  constexpr bool kCoalesced = STG && (EPI == EPI_DSWIGLU || EPI == EPI_DGELU_BGRAD);
  auto load_side = [&](int col0, uint4 (&sd)[kSideN]) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    if constexpr (kCoalesced) {
      const uint32_t pc = lane & 3u;
      const int col = col0 + 8 * (int)pc;
#pragma unroll
      for (int in = 0; in < (EPI == EPI_DSWIGLU ? 2 : 1); ++in) {
        const T* base = reinterpret_cast<const T*>(in == 0 ? p.aux_in : p.aux_in2);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int r = row0w + 8 * g + (int)(lane >> 2);
          sd[4 * in + g] = r < p.M && col < p.N
                               ? __ldg(reinterpret_cast<const uint4*>(base + (size_t)r * p.N + col))
                               : zero;
        }
      }
    } else if constexpr (EPI == EPI_DSWIGLU || EPI == EPI_DGELU_BGRAD) {
      const T* ap = reinterpret_cast<const T*>(p.aux_in) + (size_t)row * p.N + col0;
#pragma unroll
      for (int g = 0; g < 4; ++g)
        sd[g] = row_ok && col0 + 8 * g < p.N ? __ldg(reinterpret_cast<const uint4*>(ap + 8 * g))
                                             : zero;
      if constexpr (EPI == EPI_DSWIGLU) {
        const T* up = reinterpret_cast<const T*>(p.aux_in2) + (size_t)row * p.N + col0;
#pragma unroll
        for (int g = 0; g < 4; ++g)
          sd[4 + g] = row_ok && col0 + 8 * g < p.N
                          ? __ldg(reinterpret_cast<const uint4*>(up + 8 * g))
                          : zero;
      }
    } else if constexpr (EPI == EPI_DRELU_BGRAD) {
      sd[0] = zero;
      if constexpr (SIDE) {
        sd[0].x = ld_shared_u32(side + 4u * (uint32_t)(col0 - n0 + (int)lane));
      } else if (wrow_ok && col0 + (int)lane < p.N) {
        sd[0].x = __ldg(p.aux_in + (size_t)wrow * p.N + col0 + lane);
      }
    } else if constexpr (epi_has_bias(EPI)) {
      if constexpr (SIDE) {
#pragma unroll
        for (int g = 0; g < 4; ++g) sd[g] = ld_shared_v4(side + 2u * (uint32_t)(col0 - n0) + 16u * g);
      } else {
#pragma unroll
        for (int g = 0; g < 4; ++g)
          sd[g] = p.bias_axis == 0 && col0 + 8 * g < p.N
                      ? __ldg(reinterpret_cast<const uint4*>(bias + col0 + 8 * g))
                      : zero;
      }
    } else {
      sd[0] = zero;
    }
  };

  // saved activations of the staging path: rows as loaded -> this lane's row
  auto side_to_rows = [&](const uint4 (&sd)[kSideN], uint4 (&cur)[kSideN]) {
    if constexpr (kCoalesced) {
      if constexpr (TMA) {
        if (lane == 0) {  // a TMA store may still be reading it
          if (two_stg)
            bulk_wait_read<1>();
          else
            bulk_wait_read<0>();
        }
        __syncwarp();
      }
#pragma unroll
      for (int in = 0; in < (EPI == EPI_DSWIGLU ? 2 : 1); ++in) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const uint32_t r = 8u * g + (lane >> 2);
          const uint32_t pc = lane & 3u;
          const uint4 v4 = sd[4 * in + g];
          st_shared_v4(stg + r * 64u + ((pc ^ ((r >> 1) & 3u)) << 4), v4.x, v4.y, v4.z, v4.w);
        }
        __syncwarp();
        const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
        for (uint32_t pc = 0; pc < 4; ++pc)
          cur[4 * in + pc] = ld_shared_v4(stg + lane * 64u + ((pc ^ sw) << 4));
        __syncwarp();
      }
    } else {
#pragma unroll
      for (int i = 0; i < kSideN; ++i) cur[i] = sd[i];
    }
  };

  // the epilog of chunk c (columns col0 = n0 + 32 c ..): v = the accumulator
  // (u2 = the second one of the dual epilogs), cur = its side inputs
  auto finish_chunk = [&](int c, float (&v)[32], float (&u2)[kDual ? 32 : 1],
                          const uint4 (&cur)[kSideN]) {
    const int col0 = n0 + 32 * c;
    if constexpr (kDual) {
      // gate+up SwiGLU: v = g = x Wg^T, u2 = u = x Wu^T; h = silu(g) * u
      if constexpr (EPI == EPI_SWIGLU_SAVE) {
        emit_row32<T, STG>(reinterpret_cast<T*>(p.aux_out), p.M, p.N, row0w, col0, v, lane, stg);
        emit_row32<T, STG>(reinterpret_cast<T*>(p.aux_out2), p.M, p.N, row0w, col0, u2, lane,
                           stg);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = silu_f(v[j]) * u2[j];
    } else if constexpr (EPI == EPI_DSWIGLU) {
      // v = dh = dout Wd; saved g and u of this row's 32 columns; out = d_gate,
      // aux_out = d_up
      float dup[32];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float g8[8], u8[8];
        unpack8<T>(cur[g], g8);
        unpack8<T>(cur[4 + g], u8);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float s = sigmoid_f(g8[i]);
          const float dh = v[8 * g + i];
          dup[8 * g + i] = dh * (g8[i] * s);
          v[8 * g + i] = dh * u8[i] * s * (1.f + g8[i] * (1.f - s));
        }
      }
      emit(true, col0, dup);
    } else if constexpr (EPI == EPI_DGELU_BGRAD) {
      // saved pre-activation z of this row's 32 columns
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        float z8[8];
        unpack8<T>(cur[g], z8);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[8 * g + i] = v[8 * g + i] * dgelu_tanh(z8[i]);
      }
    } else if constexpr (EPI == EPI_DRELU_BGRAD) {
      // lane j holds the mask word of column col0 + j; transposed, lane i
      // holds its row's bits of the 32 columns
      const uint32_t bits = bit_transpose32(cur[0].x, lane);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = ((bits >> j) & 1u) ? v[j] : 0.f;
    } else if constexpr (EPI != EPI_NONE) {
      if (p.bias_axis == 0) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          float b8[8];
          unpack8<T>(cur[g], b8);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[8 * g + i] = v[8 * g + i] + b8[i];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = v[j] + row_bias;
      }
      if constexpr (EPI == EPI_RELU_AUX_BIAS) {
        // this lane's row bits (bit j: column col0 + j), transposed across the
        // warp into column words (bit i of lane j's word: row row0w + i)
        // four independent OR chains (a short dependency path), then merged
        uint32_t b4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int j = 0; j < 32; ++j) b4[j & 3] |= (v[j] > 0.f ? 1u : 0u) << j;
        const uint32_t bits = row_ok ? (b4[0] | b4[1]) | (b4[2] | b4[3]) : 0u;
        const uint32_t my_word = bit_transpose32(bits, lane);
        if constexpr (TMA) {
          if (c == 0) words->w0 = my_word;
          else if (c == 1) words->w1 = my_word;
          else if (c == 2) words->w2 = my_word;
          else words->w3 = my_word;
        } else if (wrow_ok && col0 + (int)lane < p.N) {
          p.aux_out[(size_t)wrow * p.N + col0 + lane] = my_word;
        }
      }
      if constexpr (EPI == EPI_RELU_BIAS || EPI == EPI_RELU_AUX_BIAS) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = v[j] > 0.f ? v[j] : 0.f;
      }
      if constexpr (EPI == EPI_GELU_AUX_BIAS) {
        // the pre-activation, rounded to T, for the backward
        emit(true, col0, v);
      }
      if constexpr (EPI == EPI_GELU_BIAS || EPI == EPI_GELU_AUX_BIAS) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = gelu_tanh(v[j]);
      }
    }

    emit(false, col0, v);

    if constexpr (epi_has_bgrad(EPI)) {
      // transpose-reduce: after 5 halving steps (31 shuffles) lane l
      // holds the sum of column col0 + l over this warp's 32 rows
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & (uint32_t)o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
          const float send = upper ? v[i] : v[i + o];
          const float keep = upper ? v[i + o] : v[i];
          v[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
      }
      red[q * RS + 32 * c + (int)lane] = v[0];
    }
  };

  uint4 sd[kSideN];
  if constexpr (PRELOAD) {
    // the first chunk's side inputs in flight, then the accumulator; every
    // chunk of it out of tensor memory (BN registers per thread), and the
    // accumulator is free again
    load_side(n0, sd);
    if (!wait_acc()) return false;
    uint32_t pre[BN / 32][32];
    float u2[1];
    if (has_acc) {
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_ld_32x32b_x32(t_row + 32u * c, pre[c]);
      tmem_ld_wait();
#pragma unroll
      for (int c = 0; c < BN / 32; ++c) tmem_tie(pre[c]);
    } else {
#pragma unroll
      for (int c = 0; c < BN / 32; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) pre[c][j] = 0u;  // nothing multiplied: zero
    }
    release();
#pragma unroll
    for (int c = 0; c < BN / 32; ++c) {
      if (c < nch) {
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(pre[c][j]);
        uint4 cur[kSideN];
        side_to_rows(sd, cur);
        if (c + 1 < nch) load_side(n0 + 32 * (c + 1), sd);
        finish_chunk(c, v, u2, cur);
      }
    }
    return true;
  }

  uint32_t ra[32];
  uint32_t rb[kDual ? 32 : 1];
  if (has_acc) {
    tmem_ld_32x32b_x32(t_row, ra);
    if constexpr (kDual) tmem_ld_32x32b_x32(t_row + (uint32_t)BN, rb);
  }
  if constexpr (!kRing) load_side(n0, sd);

#pragma unroll 1
  for (int c = 0; c < nch; ++c) {
    const int col0 = n0 + 32 * c;
    float v[32];
    float u2[kDual ? 32 : 1];  // the second accumulator (the SwiGLU "up" product)
    if (has_acc) {
      tmem_ld_wait_tied(ra);
      if constexpr (kDual) tmem_tie(rb);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(ra[j]);
      if constexpr (kDual) {
#pragma unroll
        for (int j = 0; j < 32; ++j) u2[j] = __uint_as_float(rb[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
      if constexpr (kDual) {
#pragma unroll
        for (int j = 0; j < 32; ++j) u2[j] = 0.f;
      }
    }
    uint4 cur[kSideN];
    if constexpr (kRing) {
      // this chunk's slot is complete once at most SRING - 1 groups are pending
      cp_async_wait_group<SRING - 1>();
      __syncwarp();
      const uint32_t slot = side + kSideSlotBytes * (uint32_t)(c % SRING);
      const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
      for (int in = 0; in < 2; ++in) {
#pragma unroll
        for (uint32_t pc = 0; pc < 4; ++pc)
          cur[4 * in + pc] = ld_shared_v4(slot + 2048u * in + lane * 64u + ((pc ^ sw) << 4));
      }
      __syncwarp();  // every lane has read the slot: refill it
      if (c + SRING < nch) side_ring_issue<T>(p, row0w, col0 + 32 * SRING, lane, slot);
      cp_async_commit();
    } else {
      side_to_rows(sd, cur);
    }
    if (c + 1 < nch) {  // next chunk's loads, in flight while this one is processed
      if (has_acc) {
        tmem_ld_32x32b_x32(t_row + 32u * (c + 1), ra);
        if constexpr (kDual) tmem_ld_32x32b_x32(t_row + (uint32_t)BN + 32u * (c + 1), rb);
      }
      if constexpr (!kRing) load_side(col0 + 32, sd);
    }
    finish_chunk(c, v, u2, cur);
  }
  return true;
}

// One warp's share of an accumulator half of the two-operand wide tile
// (gate+up SwiGLU): g of 64 output columns from n0 at t_g, u of the same
// columns at t_u, rows row0 + 32 q + lane. Waits for the half (`wait_acc`,
// false: the wait gave up, nothing is drained), loads both 64-column pieces
// into registers, releases the half, then per 32-column chunk stores g and u
// (SWIGLU_SAVE, through the staging buffer) and h = silu(g) * u (a TMA store
// from the staging buffer) -- the same arithmetic as the drain of the 256 x
// 128 two-operand tile.
template <int EPI, typename T, typename Release, typename WaitAcc>
__device__ __forceinline__ bool epilogue_drain_dual_wide(const GemmParams& p, uint32_t t_g,
                                                         uint32_t t_u, int row0, int n0, int q,
                                                         uint32_t lane, uint32_t stg,
                                                         const CUtensorMap* tm_out,
                                                         Release release, WaitAcc wait_acc) {
  const int row0w = row0 + 32 * q;
  const int nch = min(2, (p.N - n0 + 31) / 32);  // chunks with columns below N
  if (!wait_acc()) return false;
  uint32_t pre[4][32];  // g chunk 0, g chunk 1, u chunk 0, u chunk 1
  if (p.num_k_blocks > 0 && nch > 0) {
    tmem_ld_32x32b_x32(t_g, pre[0]);
    tmem_ld_32x32b_x32(t_g + 32u, pre[1]);
    tmem_ld_32x32b_x32(t_u, pre[2]);
    tmem_ld_32x32b_x32(t_u + 32u, pre[3]);
    tmem_ld_wait();
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_tie(pre[c]);
  } else {
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int j = 0; j < 32; ++j) pre[c][j] = 0u;  // nothing multiplied: zero
  }
  release();
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    if (c < nch) {
      const int col0 = n0 + 32 * c;
      float g[32], u[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        g[j] = __uint_as_float(pre[c][j]);
        u[j] = __uint_as_float(pre[2 + c][j]);
      }
      if constexpr (EPI == EPI_SWIGLU_SAVE) {
        if (lane == 0) bulk_wait_read<0>();  // the last h store has read the buffer
        __syncwarp();
        store_rows32_staged<T>(reinterpret_cast<T*>(p.aux_out), p.M, p.N, row0w, col0, g, lane,
                               stg);
        store_rows32_staged<T>(reinterpret_cast<T*>(p.aux_out2), p.M, p.N, row0w, col0, u, lane,
                               stg);
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) g[j] = silu_f(g[j]) * u[j];
      store_rows32_tma<T>(tm_out, row0w, col0, g, lane, stg);
    }
  }
  return true;
}

// Column sums of the tile's 128 rows: the four warps' 32-row sums (in red,
// [4][BN]) added in a fixed order, then one partial per 128-row block or one
// atomicAdd per column. Called by the NT epilogue threads (ep_tid 0..NT-1).
template <int BN, int NT = 128>
__device__ __forceinline__ void epilogue_bgrad(const GemmParams& p, const float* red, int ep_tid,
                                               int n0, int mb) {
  if (mb >= p.num_m_blocks) return;  // rows past M (same for all NT threads): nothing to add
  named_bar_sync(1, NT);
  for (int col = ep_tid; col < BN; col += NT) {
    if (n0 + col < p.N) {
      // the four warps' 32-row sums, always in the same order
      const float s = ((red[col] + red[BN + col]) + red[2 * BN + col]) + red[3 * BN + col];
      if (p.bgrad_atomic)
        atomicAdd(p.bgrad + n0 + col, s);
      else
        p.bgrad[(size_t)mb * p.N + n0 + col] = s;
    }
  }
  named_bar_sync(1, NT);
}

// Split k: the k-blocks of tile t are shared by `ks` CTAs. Each leaves its
// fp32 partial sum (its accumulator, one row per epilogue thread) in the
// workspace and counts itself in the tile's counter; the CTA that counts last
// adds the partials in split order -- the sum does not depend on which split
// finishes last -- writes it back into its accumulator and runs the epilogue.
// No CTA waits for another. Returns true in that last CTA. Called by the NT
// epilogue threads (ep_tid 0..NT-1, thread = accumulator row 32 q + lane).
// With NT = 128 a thread takes the whole row; with 256 (two warps per lane
// quarter) the row's BN / 2 columns of this warp, in segments of SEG columns
// SEG_STRIDE apart from column c_off.
// A partial is stored as [BN / 4][128 rows] float4 pieces, so that the 32
// lanes of a warp (32 consecutive rows) move 512 contiguous bytes per access.
template <int BN, int NT = 128, int SEG = BN, int SEG_STRIDE = BN>
__device__ __forceinline__ bool splitk_reduce(const GemmParams& p, uint32_t t_row, int t, int s,
                                              int ks, int q, uint32_t lane, int ep_tid,
                                              volatile int* last_flag, uint32_t ring,
                                              uint32_t ring_bytes, int c_off = 0) {
  constexpr int kPart = kBM * BN / 4;  // float4 pieces of one partial
  constexpr int kCols = BN * kBM / NT;  // columns of one thread
  static_assert(kCols % SEG == 0 && SEG % 32 == 0, "whole 32-column chunks");
  // accumulator column of this thread's column i (i a multiple of 32)
  auto col_of = [&](int i) { return c_off + (i / SEG) * SEG_STRIDE + i % SEG; };
  const int row = 32 * q + static_cast<int>(lane);
  float4* tile_ws = reinterpret_cast<float4*>(p.splitk_ws) + static_cast<size_t>(t) * ks * kPart;
  float4* mine = tile_ws + static_cast<size_t>(s) * kPart + row;
#pragma unroll 1
  for (int i = 0; i < kCols; i += 32) {
    const int c = col_of(i);
    uint32_t v[32];
    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c), v);
    tmem_ld_wait_tied(v);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      __stcg(mine + (c / 4 + j) * kBM,
             make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                         __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
  }
  __threadfence();
  named_bar_sync(1, NT);
  if (ep_tid == 0) {
    const int done = atomicAdd(p.splitk_cnt + t, 1);
    const int last = done == ks - 1 ? 1 : 0;
    if (last) p.splitk_cnt[t] = 0;  // every split has counted: ready for the next launch
    *last_flag = last;
  }
  named_bar_sync(1, NT);
  if (*last_flag == 0) return false;
  __threadfence();
  // When the operand ring is idle (`ring_bytes` > 0: this CTA's last unit,
  // every stage consumed) and holds the other splits' partials, they come in
  // by asynchronous copies all issued at once -- piece pc of this row from
  // the j-th other split at ((j * BN / 4 + pc) * 128 + row) * 16 -- instead
  // of a few loads in flight per thread (whole rows: NT = 128 only).
  const bool staged = NT == 128 && ring_bytes >= static_cast<uint32_t>((ks - 1) * kPart * 16);
  if (staged) {
    int j = 0;
#pragma unroll 1
    for (int sp = 0; sp < ks; ++sp) {
      if (sp == s) continue;
      const float4* src = tile_ws + static_cast<size_t>(sp) * kPart + row;
#pragma unroll 8
      for (int pc = 0; pc < BN / 4; ++pc)
        cp_async_16(ring + static_cast<uint32_t>(((j * (BN / 4) + pc) * kBM + row) * 16),
                    src + pc * kBM, 16u);
      ++j;
    }
    cp_async_commit();
    cp_async_wait_all();  // each thread reads back only what it copied itself
  }
#pragma unroll 1
  for (int i = 0; i < kCols; i += 32) {
    const int c = col_of(i);
    // this CTA's own partial is still in its accumulator
    uint32_t own[32];
    tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c), own);
    tmem_ld_wait_tied(own);
    const float4* src = tile_ws + (c / 4) * kBM + row;
    float acc[32];
    if (staged) {
#pragma unroll 1
      for (int sp = 0; sp < ks; ++sp) {
        float x[32];
        if (sp == s) {
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(own[i]);
        } else {
          const int j = sp < s ? sp : sp - 1;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const uint4 w = ld_shared_v4(
                ring + static_cast<uint32_t>(((j * (BN / 4) + c / 4 + k) * kBM + row) * 16));
            x[4 * k] = __uint_as_float(w.x);
            x[4 * k + 1] = __uint_as_float(w.y);
            x[4 * k + 2] = __uint_as_float(w.z);
            x[4 * k + 3] = __uint_as_float(w.w);
          }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = sp == 0 ? x[i] : acc[i] + x[i];
      }
    } else {
      // (two splits' pieces in flight at once with whole rows; one with the
      // 256-thread form, whose threads hold more live state)
      constexpr int kStep = NT == 128 ? 2 : 1;
#pragma unroll 1
      for (int sp = 0; sp < ks; sp += kStep) {
        // a split's own piece from TMEM
        float4 x[8], y[8];
        const float4* a = src + static_cast<size_t>(sp) * kPart;
        const float4* b = a + kPart;
        const bool has_b = kStep == 2 && sp + 1 < ks;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          x[j] = sp == s ? make_float4(__uint_as_float(own[4 * j]), __uint_as_float(own[4 * j + 1]),
                                       __uint_as_float(own[4 * j + 2]),
                                       __uint_as_float(own[4 * j + 3]))
                         : __ldcg(a + j * kBM);
          y[j] = !has_b ? make_float4(0.f, 0.f, 0.f, 0.f)
                 : sp + 1 == s
                     ? make_float4(__uint_as_float(own[4 * j]), __uint_as_float(own[4 * j + 1]),
                                   __uint_as_float(own[4 * j + 2]), __uint_as_float(own[4 * j + 3]))
                     : __ldcg(b + j * kBM);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (sp == 0) {
            acc[4 * j] = x[j].x;
            acc[4 * j + 1] = x[j].y;
            acc[4 * j + 2] = x[j].z;
            acc[4 * j + 3] = x[j].w;
          } else {
            acc[4 * j] += x[j].x;
            acc[4 * j + 1] += x[j].y;
            acc[4 * j + 2] += x[j].z;
            acc[4 * j + 3] += x[j].w;
          }
          if (has_b) {
            acc[4 * j] += y[j].x;
            acc[4 * j + 1] += y[j].y;
            acc[4 * j + 2] += y[j].z;
            acc[4 * j + 3] += y[j].w;
          }
        }
      }
    }
    uint32_t u[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(acc[j]);
    tmem_st_32x32b_x32(t_row + static_cast<uint32_t>(c), u);
  }
  tmem_st_wait();
  return true;
}

template <int EPI, typename T, bool B_MN, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_epilog_kernel(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmB2, const GemmParams p) {
  constexpr int NB = epi_dual(EPI) ? 2 : 1;
  using C = TileCfg<BN, NB, epi_has_bgrad(EPI)>;
  constexpr int S = C::kStages;
  constexpr bool kBf16 = std::is_same<T, __nv_bfloat16>::value;
  extern __shared__ uint8_t smem_raw[];

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sA = base;
  const uint32_t sB = base + S * C::kABytes;
  const uint32_t ctrl = sB + S * C::kStageBBytes;
  uint8_t* gctrl = gbase + (ctrl - base);
  const uint32_t full0 = ctrl;               // S barriers: stage filled
  const uint32_t empty0 = ctrl + 8u * S;     // S barriers: stage consumed
  const uint32_t tfull0 = ctrl + 16u * S;    // 2 barriers: accumulator ready
  const uint32_t tempty0 = tfull0 + 16u;     // 2 barriers: accumulator drained
  const uint32_t done_bar = tempty0 + 16u;   // MMA teardown
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gctrl + 16 * S + 40);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gctrl + 16 * S + 44);
  float* red = reinterpret_cast<float*>(gctrl + C::kCtrlBytes);  // [4][BN]

  volatile int* last_flag = reinterpret_cast<volatile int*>(gctrl + 16 * S + 48);

  const int warp = threadIdx.x >> 5;
  const uint32_t lane = lane_id();
  // work units: tile t, k-split s as unit t * ks + s (ks = 1: the tiles)
  const int ks = p.k_splits > 1 ? p.k_splits : 1;
  const int kps = ks > 1 ? p.kb_per_split : p.num_k_blocks;
  const int units = p.num_tiles * ks;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(tfull0, 1);
    mbar_init(tfull0 + 8u, 1);
    mbar_init(tempty0, 4);
    mbar_init(tempty0 + 8u, 4);
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    if (p.num_k_blocks > 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      if (NB == 2) prefetch_tmap(&tmB2);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *reinterpret_cast<volatile uint32_t*>(tmem_slot);
  // the set-up above overlaps the previous kernel on the stream; its outputs
  // (this kernel's inputs) are complete from here on
  grid_dep_wait();
  grid_dep_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && p.num_k_blocks > 0) {
      int issued[S];
#pragma unroll
      for (int s = 0; s < S; ++s) issued[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      int loads = 0;
      bool ok = true;
      const uint64_t pol_a = l2_policy(p.l2_hint_a);
      const uint64_t pol_b = l2_policy(p.l2_hint_b);
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
        const int t = u / ks;
        const int kb0 = (u - t * ks) * kps;
        const int kb1 = min(p.num_k_blocks, kb0 + kps);
        int mb, nb;
        tile_coords(p, t, mb, nb);
        const int m0 = mb * kBM, n0 = nb * BN;
        const int nbox = B_MN ? min(BN / 64, (p.N - n0 + 63) / 64) : 1;
        // a 3-D box always moves all BN / 64 chunks (zero fill past N)
        const uint32_t bytes =
            C::kABytes + (B_MN && !p.b_mn_3d ? nbox * 64 * kBK * 2 : C::kStageBBytes);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_PRODUCER);
            ok = false;
            break;
          }
          ++loads;
          if (loads != p.drop_load) {
            const uint32_t fb = full0 + 8u * stage;
            mbar_arrive_expect_tx(fb, bytes);
            tma_load(sA + stage * C::kABytes, &tmA, fb, kb * kBK, m0, p.l2_hint_a, pol_a);
            if (B_MN && p.b_mn_3d) {
              tma_load3(sB + stage * C::kStageBBytes, &tmB, fb, 0, kb * kBK, n0 / 64,
                        p.l2_hint_b, pol_b);
            } else if (B_MN) {
              for (int j = 0; j < nbox; ++j)
                tma_load(sB + stage * C::kStageBBytes + j * (64 * kBK * 2), &tmB, fb, n0 + 64 * j,
                         kb * kBK, p.l2_hint_b, pol_b);
            } else {
              tma_load(sB + stage * C::kStageBBytes, &tmB, fb, kb * kBK, n0, p.l2_hint_b, pol_b);
              if (NB == 2)  // the second B operand right after the first
                tma_load(sB + stage * C::kStageBBytes + C::kBBytes, &tmB2, fb, kb * kBK, n0,
                         p.l2_hint_b, pol_b);
            }
            issued[stage] = (int)phase;
          }
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every load issued must land before the CTA may exit
#pragma unroll
      for (int s = 0; s < S; ++s)
        if (issued[s] >= 0 &&
            !mbar_wait_bounded(full0 + 8u * s, (uint32_t)issued[s], nullptr, p.wait_limit_ns))
          raise_error(p, abort_flag, ST_TIMEOUT_DRAIN);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(kBf16, B_MN, kBM, BN);
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int it = 0;
      for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++it) {
        const int kb0 = (u % ks) * kps;
        const int kb1 = min(p.num_k_blocks, kb0 + kps);
        const int buf = it & 1;
        const uint32_t use = (uint32_t)(it >> 1) & 1u;
        if (!mbar_wait_bounded(tempty0 + 8u * buf, use ^ 1u, abort_flag, p.wait_limit_ns)) {
          raise_error(p, abort_flag, ST_TIMEOUT_MMA_TMEM);
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(buf * C::kAccCols);
        if (p.num_k_blocks == 0) {
          mbar_arrive(tfull0 + 8u * buf);  // acc is all zeros: nothing to multiply
          continue;
        }
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait_bounded(full0 + 8u * stage, phase, abort_flag, p.wait_limit_ns)) {
            raise_error(p, abort_flag, ST_TIMEOUT_MMA_SMEM);
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = sA + stage * C::kABytes;
          const uint32_t b_base = sB + stage * C::kStageBBytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            // K-major A: 16 k = 32 bytes along the swizzled 128-byte row;
            // 8-row groups 1024 bytes apart.
            const uint64_t adesc = sdesc_sw128(a_base + kk * 32, 16, 1024);
            // B K-major: as A. B MN-major: 16 k = 16 rows of 128 bytes;
            // 64-column chunks 64*128 bytes apart (LBO), 8-k groups 1024 (SBO).
            const uint64_t bdesc = B_MN ? sdesc_sw128(b_base + kk * 2048, 64 * kBK * 2, 1024)
                                        : sdesc_sw128(b_base + kk * 32, 16, 1024);
            const uint32_t accum = (kb != kb0 || kk != 0) ? 1u : 0u;
            umma_f16(d_tmem, adesc, bdesc, idesc, accum);
            if constexpr (NB == 2) {  // second accumulator: columns [BN, 2 BN) of the set
              const uint64_t bdesc2 = sdesc_sw128(b_base + C::kBBytes + kk * 32, 16, 1024);
              umma_f16(d_tmem + BN, adesc, bdesc2, idesc, accum);
            }
          }
          umma_commit(empty0 + 8u * stage);  // frees the stage once these MMAs finish
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) umma_commit(tfull0 + 8u * buf);
      }
      // all MMAs issued by this thread must finish before TMEM is freed
      umma_commit(done_bar);
      if (!mbar_wait_bounded(done_bar, 0, nullptr, p.wait_limit_ns))
        raise_error(p, abort_flag, ST_TIMEOUT_DRAIN);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // the TMEM lane quarter this warp may access
    const int ep_tid = threadIdx.x - 64;
    int it = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++it) {
      const int t = u / ks;
      const int buf = it & 1;
      const uint32_t use = (uint32_t)(it >> 1) & 1u;
      bool ok = mbar_wait_bounded(tfull0 + 8u * buf, use, abort_flag, p.wait_limit_ns);
      if (epi_has_bgrad(EPI) || ks > 1) {
        // the four warps meet at named barriers below: they must agree
        ok = !named_bar_red_or(1, 128, !ok);
      }
      if (!ok) {
        raise_error(p, abort_flag, ST_TIMEOUT_EPILOGUE);
        break;
      }
      tc_fence_after();
      int mb, nb;
      tile_coords(p, t, mb, nb);
      const int m0 = mb * kBM, n0 = nb * BN;
      const uint32_t t_row =
          tmem_base + ((uint32_t)(32 * q) << 16) + (uint32_t)(buf * C::kAccCols);

      // the operand ring is idle once this CTA's last unit has been multiplied
      const uint32_t ring_bytes =
          u + (int)gridDim.x >= units ? (uint32_t)(S * (C::kABytes + C::kStageBBytes)) : 0u;
      if (ks > 1 && !splitk_reduce<BN>(p, t_row, t, u - t * ks, ks, q, lane, ep_tid, last_flag,
                                       sA, ring_bytes)) {
        // a partial sum, handed over through the workspace: buffer free again
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8u * buf);
        continue;
      }
      epilogue_drain<EPI, T, BN>(p, t_row, m0, n0, q, lane, red);
      // accumulator buffer drained: the MMA warp may reuse it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8u * buf);

      if constexpr (epi_has_bgrad(EPI)) epilogue_bgrad<BN>(p, red, ep_tid, n0, mb);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

}  // namespace gf
