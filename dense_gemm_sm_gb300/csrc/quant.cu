// quant.cu -- per-row FP8 E4M3 quantisation of BF16 activations for the FP8 GEMM
// ("Operator & Runtime", section 5.4.3, Example 5-7, and section 5.4.4, Example 5-8):
//   amax_i = max_k |x_ik|,  q_ik = E4M3(x_ik * (448 / amax_i)),  s_i = amax_i / 448,
// so that x_ik ~ q_ik * s_i.  The scale comes from the whole row, so the row is read twice:
// once for its maximum, once to quantise (the second read hits L1/L2).  The quantised codes
// are written once; the GEMM then reads one byte per element instead of two (the separate
// quantisation the pages find cheaper than quantising inside every column block).
//
// Arithmetic, in the order the definition gives it: amax exact (a maximum of exact values),
// 448 / amax and amax / 448 as IEEE float32 divisions, the product x * (448 / amax) as one
// float32 multiplication, then round-to-nearest-even to E4M3 with saturation to +-448
// (cvt.rn.satfinite.e4m3x2.f32).  A row of zeros gets codes 0 and scale 0.
//
// HBM-bound: 2 bytes read and 1 byte written per element (plus 4 bytes per row).  A CTA of
// 256 threads takes one row at a time, 8 elements (16 bytes) per thread per step.
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

template <bool VEC>
__global__ void __launch_bounds__(kQThreads, 1)
    quantize_rows_kernel(int64_t rows, int64_t cols, const uint16_t* __restrict__ X, int64_t ldx,
                         uint8_t* __restrict__ Q, int64_t ldq, float* __restrict__ scales) {
  __shared__ float red[kQThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();  // launched with programmatic serialisation: X may come from the previous kernel
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t* x = X + r * ldx;
    uint8_t* q = Q + r * ldq;
    // Pass 1: the row's absolute maximum.
    float m = 0.f;
    if (VEC) {
      const int64_t n8 = cols / 8;
      for (int64_t i = tid; i < n8; i += kQThreads) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x))),
                           fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y)))));
        m = fmaxf(m, fmaxf(fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))),
                           fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w)))));
      }
      for (int64_t i = n8 * 8 + tid; i < cols; i += kQThreads)
        m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[i]) << 16)));
    } else {
      for (int64_t i = tid; i < cols; i += kQThreads)
        m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(x[i]) << 16)));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    float amax = red[0];
#pragma unroll
    for (int w = 1; w < kQThreads / 32; ++w) amax = fmaxf(amax, red[w]);
    __syncthreads();  // red is rewritten for the next row
    const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
    if (tid == 0) scales[r] = __fdiv_rn(amax, 448.f);
    // Pass 2: quantise.
    if (VEC) {
      const int64_t n8 = cols / 8;
      for (int64_t i = tid; i < n8; i += kQThreads) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(x) + i);
        uint2 o;
        o.x = static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(v.x), inv), __fmul_rn(bf16_hi(v.x), inv))) |
              (static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(v.y), inv), __fmul_rn(bf16_hi(v.y), inv))) << 16);
        o.y = static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(v.z), inv), __fmul_rn(bf16_hi(v.z), inv))) |
              (static_cast<uint32_t>(e4m3x2(__fmul_rn(bf16_lo(v.w), inv), __fmul_rn(bf16_hi(v.w), inv))) << 16);
        reinterpret_cast<uint2*>(q)[i] = o;
      }
      for (int64_t i = n8 * 8 + tid; i < cols; i += kQThreads) {
        const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[i]) << 16), inv);
        q[i] = static_cast<uint8_t>(e4m3x2(y, 0.f) & 0xFFu);
      }
    } else {
      for (int64_t i = tid; i < cols; i += kQThreads) {
        const float y = __fmul_rn(__uint_as_float(static_cast<uint32_t>(x[i]) << 16), inv);
        q[i] = static_cast<uint8_t>(e4m3x2(y, 0.f) & 0xFFu);
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_rows(int64_t rows, int64_t cols, const void* X, int64_t ldx, void* Q,
                                 int64_t ldq, float* scales, bool vec, int sms, cudaStream_t s) {
  int64_t grid = static_cast<int64_t>(sms > 0 ? sms : 1) * 8;
  if (grid > rows) grid = rows;
  const auto* x = static_cast<const uint16_t*>(X);
  auto* q = static_cast<uint8_t*>(Q);
  if (vec)
    return launch_pdl(quantize_rows_kernel<true>, dim3(static_cast<unsigned>(grid)), dim3(kQThreads),
                      0, s, rows, cols, x, ldx, q, ldq, scales);
  return launch_pdl(quantize_rows_kernel<false>, dim3(static_cast<unsigned>(grid)), dim3(kQThreads), 0,
                    s, rows, cols, x, ldx, q, ldq, scales);
}

}  // namespace dg
