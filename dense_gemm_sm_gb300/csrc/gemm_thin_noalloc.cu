// gemm_thin_noalloc.cu -- the decode-shaped BF16 GEMM for callers that cannot allocate.
//
// gemm_bf16() gives the split-K decode kernel a workspace it obtains with cudaMalloc on first
// use.  Some callers cannot let a library do that: a host framework whose caching allocator
// has already reserved the device memory (a fresh cudaMalloc can fail or fragment its pool),
// or a latency-critical decode loop that cannot afford cudaMalloc's implicit device-wide
// synchronisation.  gemm_bf16_decode_noalloc() runs the same kernel with its scratch (FP32
// partial sums and per-tile arrival counters) in the fixed-size array below, which lives in
// the library's own device image: every GPU that loads the library holds it until exit.
//
// Limits: M <= 16 rows of X, N <= 1,048,576 columns, at most 160 CTAs; 2.5 MiB of partials
// plus 32 KiB of counters.  Every call shares the array: calls whose kernels overlap on the
// GPU (on different streams, or the same call issued from two threads) race on it and give
// wrong results; serialise them, e.g. on one stream.  Between calls the counters are zero
// (the kernel resets each one as it combines its tile), so a call enqueues only its kernel,
// which keeps back-to-back calls overlapping through programmatic dependent launch.
#include <cstdint>
#include <mutex>

#include "dg_internal.h"

namespace dg {

// Status word and SM count of a device (api.cu).
cudaError_t device_status_word(int dev, uint32_t** status, int* sms);

namespace {

constexpr int kNaMaxCtas = 160;
constexpr int kNaNtok = 16;
constexpr int64_t kNaMaxTiles = 8192;  // N <= 8192 * 128
constexpr size_t kNaPartialBytes = static_cast<size_t>(kNaMaxCtas) * 2 * kNaNtok * kThinBN * 4;
constexpr size_t kNaCounterBytes = static_cast<size_t>(kNaMaxTiles) * 4;
constexpr size_t kNaScratchBytes = kNaPartialBytes + kNaCounterBytes;
static_assert(kNaPartialBytes % 256 == 0, "counters must stay 256-byte aligned");
constexpr int kNaMaxDevices = 64;

// The scratch: partials [ctas][2][4][128] float4, then one uint32 counter per 128-column tile.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNaScratchBytes];

std::mutex g_na_mu;
unsigned char* g_na_addr[kNaMaxDevices] = {};
CUcontext g_na_ctx[kNaMaxDevices] = {};  // the context the cached address belongs to

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<CtxGetCurrentFn>(nullptr);
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of the scratch array on `dev` (the current device).  In host code the
// array's name is only a host-side stand-in, so the address is taken with
// cudaGetSymbolAddress and cached per device together with the current context: a new
// context (after cudaDeviceReset, say) loads the module again at a new address, so the
// address is looked up again when the context differs.  The array starts zeroed (module
// load), and the kernel leaves every arrival counter at zero when it finishes, so calls need
// no memset; the first call in a context still zeroes the counters on its stream once, and a
// call that gave up on a bounded wait is cleaned up by dg_device_status
// (noalloc_reset_counters below).
cudaError_t scratch_address(int dev, cudaStream_t s, unsigned char** out) {
  CUcontext ctx = nullptr;
  CtxGetCurrentFn get = ctx_get_current();
  if (!get || get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
  std::lock_guard<std::mutex> lock(g_na_mu);
  if (!g_na_addr[dev] || g_na_ctx[dev] != ctx) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(static_cast<unsigned char*>(p) + kNaPartialBytes, 0, kNaCounterBytes, s);
    if (e != cudaSuccess) return e;
    g_na_addr[dev] = static_cast<unsigned char*>(p);
    g_na_ctx[dev] = ctx;
  }
  *out = g_na_addr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

// Re-zeroes the arrival counters of `dev` (the current device) after a call gave up on a
// bounded wait and may have left some non-zero; synchronous (dg_device_status already
// synchronised the stream).  Nothing to do on a device that never ran this entry point.
cudaError_t noalloc_reset_counters(int dev) {
  std::lock_guard<std::mutex> lock(g_na_mu);
  if (dev < 0 || dev >= kNaMaxDevices || !g_na_addr[dev]) return cudaSuccess;
  return cudaMemset(g_na_addr[dev] + kNaPartialBytes, 0, kNaCounterBytes);
}

}  // namespace dg

using namespace dg;

extern "C" dg_status gemm_bf16_decode_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                              const uint16_t* A, int64_t lda, const uint16_t* B,
                                              int64_t ldb, float beta, void* C, int64_t ldc,
                                              dg_out c_type, void* stream) {
  if (M < 0 || N < 0 || K < 0) return DG_ERR_INVALID_ARG;
  if (c_type != DG_OUT_BF16 && c_type != DG_OUT_F32) return DG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return DG_OK;
  if (ldc < N || (K > 0 && (lda < K || ldb < N))) return DG_ERR_INVALID_ARG;
  if (M > kNaNtok || (N + kThinBN - 1) / kThinBN > kNaMaxTiles || K > INT32_MAX)
    return DG_ERR_UNSUPPORTED;  // beyond the fixed scratch
  if (!C) return DG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool c_f32 = c_type == DG_OUT_F32;
  if (K == 0 || alpha == 0.f)
    return launch_scale(C, c_f32, M, N, ldc, 0, 1, beta, s) == cudaSuccess ? DG_OK : DG_ERR_CUDA;
  if (!A || !B) return DG_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || lda % 8 != 0 || ldb % 8 != 0) return DG_ERR_MISALIGNED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_status_word(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  unsigned char* scratch = nullptr;
  if (scratch_address(dev, s, &scratch) != cudaSuccess) return DG_ERR_CUDA;

  ThinParams p;
  p.M = M; p.N = N; p.K = K;
  p.n_tiles = (N + kThinBN - 1) / kThinBN;
  p.kblocks = (K + kThinBK - 1) / kThinBK;
  p.units = p.n_tiles * p.kblocks;
  int64_t ctas = sms < kNaMaxCtas ? sms : kNaMaxCtas;
  if (p.units < ctas) ctas = p.units;
  p.ctas = ctas;
  p.alpha = alpha; p.beta = beta;
  p.C = C; p.ldc = ldc;
  p.c_f32 = c_f32 ? 1 : 0;
  p.ws = reinterpret_cast<float*>(scratch);
  p.counters = reinterpret_cast<uint32_t*>(scratch + kNaPartialBytes);
  p.status = status;
  // The arrival counters are zero between calls (the kernel resets each one when it combines
  // the tile); the partials are always written before they are read.
  return launch_gemm_thin(p, kNaNtok, A, lda, B, ldb, false, s) == cudaSuccess ? DG_OK
                                                                              : DG_ERR_CUDA;
}
