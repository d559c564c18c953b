// gf_drelu_bgrad_noalloc: the DRELU_BGRAD GEMM + epilogue for callers that
// cannot allocate device memory -- code running where cudaMalloc is not
// allowed or not wanted (inside a framework's memory pool that hands out
// only the tensors it manages, in a real-time loop that must not touch the
// allocator, or from a host API that forbids allocation while running).
//
// The DRELU_BGRAD kernel needs scratch memory beyond its inputs and outputs:
// one fp32 partial column sum per 128-row block (the deterministic two-pass
// bias gradient) and a status word. Here that scratch is one fixed,
// file-scope device array, set aside on every GPU that loads this library
// for as long as the process lives. Nothing is allocated per call.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "gf.h"
#include "launch.h"
#include "params.h"
#include "runtime_internal.h"

namespace {

constexpr int64_t kMaxPartials = GF_NOALLOC_MAX_PARTIALS;
constexpr size_t kStatusBytes = 256;

// [0, 256): status word; [256, ...): fp32 partials [ceil(m/128)][n].
// Device code reaches it through the pointer passed to the kernels; host
// code must not use its name as an address (it is a host-side stand-in).
static __device__ __align__(256) unsigned char g_noalloc_scratch[kStatusBytes + kMaxPartials * 4];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};
// the driver context each cached address belongs to: a device reset (or any
// teardown and re-creation of the context) reloads the module, and the
// address is then looked up again
CUcontext g_scratch_ctx[kMaxDevices] = {};

// the status is also the thread's last error (gf_last_error)
gf_status fail(gf_status s) { return gf::runtime_fail(s); }

// Once per device and context, with that device current: the device address
// of the scratch array.
gf_status scratch_for_device(int dev, unsigned char** out) {
  if (dev < 0 || dev >= kMaxDevices) return GF_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (cudaSetDevice(dev) != cudaSuccess) return GF_ERR_CUDA;
  const CUcontext ctx = gf::runtime_current_context();
  if (!g_scratch_addr[dev] || ctx == nullptr || ctx != g_scratch_ctx[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      g_scratch_addr[dev] = nullptr;
      return GF_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = gf::runtime_current_context();
  }
  *out = static_cast<unsigned char*>(g_scratch_addr[dev]);
  return GF_OK;
}

// The calling thread's device, checked to be one the kernels run on.
gf_status noalloc_device(int* dev, int* sms) {
  gf_status st = gf::runtime_current_device(dev);
  if (st != GF_OK) return st;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev) != cudaSuccess ||
      cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev) != cudaSuccess) {
    cudaGetLastError();
    return GF_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return GF_ERR_UNSUPPORTED;
  return GF_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

GF_API gf_status gf_drelu_bgrad_noalloc(int64_t m, int64_t n, int64_t k, gf_dtype dtype,
                                        gf_b_layout b_layout, const void* A, const void* B,
                                        void* out, const void* aux_in, float* bgrad,
                                        struct CUstream_st* stream) {
  const int64_t max_dim = (int64_t(1) << 31) - 1;
  if (m < 0 || n < 0 || k < 0 || m > max_dim || n > max_dim || k > max_dim)
    return fail(GF_ERR_INVALID_VALUE);
  if (dtype != GF_F16 && dtype != GF_BF16) return fail(GF_ERR_INVALID_VALUE);
  if (b_layout != GF_B_KN && b_layout != GF_B_NK) return fail(GF_ERR_INVALID_VALUE);
  if (n % 8 != 0 || k % 8 != 0) return fail(GF_ERR_UNSUPPORTED);
  const int64_t m_blocks = (m + 127) / 128;
  if (m_blocks * n > kMaxPartials) return fail(GF_ERR_UNSUPPORTED);  // beyond the fixed scratch
  const bool empty = m == 0 || n == 0;
  if (!empty) {
    if (!out || !aligned16(out) || !aux_in || !aligned16(aux_in)) return fail(GF_ERR_INVALID_VALUE);
    if (k > 0 && (!A || !B || !aligned16(A) || !aligned16(B))) return fail(GF_ERR_INVALID_VALUE);
  }
  if (n > 0 && (!bgrad || !aligned16(bgrad))) return fail(GF_ERR_INVALID_VALUE);

  int dev = 0, sms = 0;
  gf_status st = noalloc_device(&dev, &sms);
  if (st != GF_OK) return fail(st);
  unsigned char* scratch = nullptr;
  st = scratch_for_device(dev, &scratch);
  if (st != GF_OK) return fail(st);
  if (cudaSetDevice(dev) != cudaSuccess) return fail(GF_ERR_CUDA);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  if (empty) {
    if (n > 0 && cudaMemsetAsync(bgrad, 0, static_cast<size_t>(n) * 4, s) != cudaSuccess)
      return fail(GF_ERR_CUDA);
    return GF_OK;
  }

  // the single-CTA kernel, tile width as the plan would choose it
  const int64_t wide_tiles = m_blocks * ((n + 255) / 256);
  const int tile_n = wide_tiles >= sms ? 256 : 128;
  const int n_blocks = static_cast<int>((n + tile_n - 1) / tile_n);
  const int64_t tiles = m_blocks * n_blocks;

  CUtensorMap tmA, tmB;
  memset(&tmA, 0, sizeof tmA);
  memset(&tmB, 0, sizeof tmB);
  if (k > 0) {
    if (!gf::runtime_encode_2d(&tmA, A, dtype, k, m, 64, 128)) return fail(GF_ERR_INVALID_VALUE);
    const bool ok = b_layout == GF_B_KN ? gf::runtime_encode_2d(&tmB, B, dtype, n, k, 64, 64)
                                        : gf::runtime_encode_2d(&tmB, B, dtype, k, n, 64, tile_n);
    if (!ok) return fail(GF_ERR_INVALID_VALUE);
  }

  // the status word starts at zero for this call; the partials need no
  // clearing: every one that the finalize reads is written by the kernel
  int32_t* status = reinterpret_cast<int32_t*>(scratch);
  float* partials = reinterpret_cast<float*>(scratch + kStatusBytes);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return fail(GF_ERR_CUDA);

  gf::GemmParams prm;
  memset(&prm, 0, sizeof prm);
  prm.M = static_cast<int32_t>(m);
  prm.N = static_cast<int32_t>(n);
  prm.K = static_cast<int32_t>(k);
  prm.num_m_blocks = static_cast<int32_t>(m_blocks);
  prm.num_n_blocks = n_blocks;
  prm.num_k_blocks = static_cast<int32_t>((k + 63) / 64);
  prm.num_tiles = static_cast<int32_t>(tiles);
  prm.group_m = 8;
  prm.aux_in = static_cast<const uint32_t*>(aux_in);
  prm.out = out;
  prm.bgrad = partials;
  prm.bgrad_atomic = 0;
  prm.status = status;
  prm.wait_limit_ns = 2000000000ull;

  gf::LaunchArgs la;
  la.tmA = &tmA;
  la.tmB = &tmB;
  la.tmB2 = &tmB;
  la.tmOut = &tmA;  // the single-CTA kernel stores without tensor maps
  la.tmAux = &tmA;
  la.params = &prm;
  la.grid = static_cast<int>(tiles < sms ? tiles : sms);
  la.bf16 = dtype == GF_BF16 ? 1 : 0;
  la.b_mn = b_layout == GF_B_KN ? 1 : 0;
  la.tile_n = tile_n;
  la.pair = 0;
  la.wide = 0;
  la.pdl = 1;
  la.stream = s;
  if (gf::launch_drelu(la) != cudaSuccess) return fail(GF_ERR_CUDA);
  if (gf::launch_bgrad_finalize(partials, static_cast<int>(m_blocks), static_cast<int>(n), bgrad,
                                s, 1) != cudaSuccess)
    return fail(GF_ERR_CUDA);
  return GF_OK;
}

GF_API gf_status gf_noalloc_status(struct CUstream_st* stream) {
  int dev = 0, sms = 0;
  gf_status st = noalloc_device(&dev, &sms);
  if (st != GF_OK) return fail(st);
  unsigned char* scratch = nullptr;
  st = scratch_for_device(dev, &scratch);
  if (st != GF_OK) return fail(st);
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return fail(GF_ERR_CUDA);
  }
  int32_t word = 0;
  if (cudaMemcpy(&word, scratch, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return fail(GF_ERR_CUDA);
  }
  if (word != 0) {
    if (cudaMemset(scratch, 0, sizeof word) != cudaSuccess) {
      cudaGetLastError();
      return fail(GF_ERR_CUDA);
    }
    return fail(GF_ERR_DEVICE_TIMEOUT);
  }
  return GF_OK;
}

}  // extern "C"
