// quant.cu -- per-row FP8 E4M3 quantisation of BF16 activations for the FP8 GEMM
// ("Operator & Runtime", section 5.4.3, Example 5-7, and section 5.4.4, Example 5-8):
//   amax_i = max_k |x_ik|,  q_ik = E4M3(x_ik * (448 / amax_i)),  s_i = amax_i / 448,
// so that x_ik ~ q_ik * s_i.  The scale comes from the whole row, so the whole row is read
// before any element is quantised (from registers, or a second read hitting L1/L2).  The codes
// are written once; the GEMM then reads one byte per element instead of two (the separate
// quantisation the pages find cheaper than quantising inside every column block).
//
// Arithmetic, in the order the definition gives it: amax exact (a maximum of exact values),
// 448 / amax and amax / 448 as IEEE float32 divisions, the product x * (448 / amax) as one
// float32 multiplication, then round-to-nearest-even to E4M3 with saturation to +-448
// (cvt.rn.satfinite.e4m3x2.f32).  A row of zeros gets codes 0 and scale 0.
//
// HBM-bound: 2 bytes read and 1 byte written per element (plus 4 bytes per row).  One warp
// takes one row: rows of up to 4096 elements stay in the warp's registers between the two
// passes (one HBM read), the maximum is a warp shuffle reduction (no CTA barrier).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dg_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kQThreads = 256;

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %2, %1;\n\t"
      "mov.b16 %0, t;\n\t}"
      : "=h"(d)
      : "f"(lo), "f"(hi));
  return d;  // low byte: lo's code, high byte: hi's code
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// One warp per row.  R > 0: the row (cols <= 256 R, 16-byte aligned) is held in registers,
// R 16-byte chunks per lane, so it is read from HBM once and quantised from registers.
// R == 0: two passes over the row (the second from L1/L2), 16-byte chunks when VEC.
template <int R, bool VEC>
__global__ void __launch_bounds__(kQThreads)
    quantize_rows_kernel(int64_t rows, int64_t cols, const uint16_t* __restrict__ X, int64_t ldx,
                         uint8_t* __restrict__ Q, int64_t ldq, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQThreads / 32);
  pdl_trigger();
  pdl_wait();  // launched with programmatic serialisation: X may come from the previous kernel
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (kQThreads / 32) + (threadIdx.x >> 5); r < rows;
       r += warps) {
    const uint16_t* x = X + r * ldx;
    uint8_t* q = Q + r * ldq;
    const int64_t n8 = VEC ? cols / 8 : 0;  // whole 16-byte chunks
    uint4 v[R > 0 ? R : 1];
    float m = 0.f;
    // Pass 1: the row's absolute maximum.
    if (R > 0) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int64_t c = lane + 32 * i;
        v[i] = c < n8 ? __ldcs(reinterpret_cast<const uint4*>(x) + c) : make_uint4(0u, 0u, 0u, 0u);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v[i].x)), fabsf(bf16_hi(v[i].x))),
                           fmaxf(fabsf(bf16_lo(v[i].y)), fabsf(bf16_hi(v[i].y)))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v[i].z)), fabsf(bf16_hi(v[i].z))),
                           fmaxf(fabsf(bf16_lo(v[i].w)), fabsf(bf16_hi(v[i].w)))));
      }
    } else if (VEC) {
      for (int64_t c = lane; c < n8; c += 32) {
        const uint4 u = __ldg(reinterpret_cast<const uint4*>(x) + c);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(u.x)), fabsf(bf16_hi(u.x))),
                           fmaxf(fabsf(bf16_lo(u.y)), fabsf(bf16_hi(u.y)))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(u.z)), fabsf(bf16_hi(u.z))),
                           fmaxf(fabsf(bf16_lo(u.w)), fabsf(bf16_hi(u.w)))));
      }
    }
    for (int64_t i = n8 * 8 + lane; i < cols; i += 32)
      m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[i]) << 16)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float amax = m;
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    if (lane == 0) scales[r] = __fdiv_rn(amax, 448.f);
    // Pass 2: quantise, 8 codes (8 bytes) per 16-byte chunk.
    auto codes8 = [&](const uint4& u) {
      uint2 o;
      o.x = static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(u.x), inv), __fmul_rn(bf16_hi(u.x), inv))) |
            (static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(u.y), inv), __fmul_rn(bf16_hi(u.y), inv))) << 16);
      o.y = static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(u.z), inv), __fmul_rn(bf16_hi(u.z), inv))) |
            (static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(u.w), inv), __fmul_rn(bf16_hi(u.w), inv))) << 16);
      return o;
    };
    if (R > 0) {
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int64_t c = lane + 32 * i;
        if (c < n8) reinterpret_cast<uint2*>(q)[c] = codes8(v[i]);
      }
    } else if (VEC) {
      for (int64_t c = lane; c < n8; c += 32)
        reinterpret_cast<uint2*>(q)[c] = codes8(__ldg(reinterpret_cast<const uint4*>(x) + c));
    }
    for (int64_t i = n8 * 8 + lane; i < cols; i += 32) {
      const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[i]) << 16), inv);
      q[i] = static_cast<uint8_t>(e4m3x2(y, 0.f) & 0xFFu);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows(int64_t rows, int64_t cols, const void* X, int64_t ldx, void* Q,
                                 int64_t ldq, float* scales, bool vec, int sms, cudaStream_t s) {
  // One warp per row, up to 8 resident CTAs of 8 warps per SM.
  int64_t grid = (rows + kQThreads / 32 - 1) / (kQThreads / 32);
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
  if (grid > cap) grid = cap;
  const auto* x = static_cast<const uint16_t*>(X);
  auto* q = static_cast<uint8_t*>(Q);
  const dim3 g(static_cast<unsigned>(grid)), b(kQThreads);
  const int64_t chunks = vec ? (cols / 8 + 31) / 32 : 0;  // 16-byte chunks per lane
  if (vec && chunks <= 4) return launch_pdl(quantize_rows_kernel<4, true>, g, b, 0, s, rows, cols, x, ldx, q, ldq, scales);
  if (vec && chunks <= 16) return launch_pdl(quantize_rows_kernel<16, true>, g, b, 0, s, rows, cols, x, ldx, q, ldq, scales);
  if (vec) return launch_pdl(quantize_rows_kernel<0, true>, g, b, 0, s, rows, cols, x, ldx, q, ldq, scales);
  return launch_pdl(quantize_rows_kernel<0, false>, g, b, 0, s, rows, cols, x, ldx, q, ldq, scales);
}

}  // namespace dg
