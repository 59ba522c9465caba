// dg_internal.h -- declarations shared by the C-ABI layer and the kernel translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/dgemm.h"

namespace dg {

// ------------------------------------------------------------------ FP32 SIMT path
struct SimtParams {
  int64_t M, N, K;
  float alpha, beta;
  const float* A; int64_t lda, strideA;
  const float* B; int64_t ldb, strideB;
  float* C; int64_t ldc, strideC;
  int64_t batch;
  int64_t tiles_m, tiles_n;
  int32_t group;
  // Schedule: the first dp_tiles CTAs of the grid compute one whole tile each; the next
  // sk_tiles * sk_splits CTAs each compute one of sk_splits equal K chunks of the remaining
  // (tail) tiles.  Grid = dp_tiles + sk_tiles * sk_splits.
  int64_t dp_tiles, sk_tiles;
  int32_t sk_splits;
  // Stream-K schedule instead (TMA kernel, sk_ctas > 0): CTA c computes the units
  // [c*U/G, (c+1)*U/G) of the U = sk_units (tile, K tile) pairs, G = sk_ctas = grid; a tile
  // shared by several CTAs is finished by the last of them, adding their parts in CTA order.
  int64_t sk_units, sk_ctas;
  float* ws;           // partials: [sk_tiles][sk_splits] or, stream-K, [sk_ctas][2], x [16][256] float4
  uint32_t* counters;  // [sk_tiles] or, stream-K, [tiles]; zero between calls
  uint32_t* status;    // device status word (bounded-wait expiry)
};
// Stream-K SIMT ranges span at most this many segments (whole tiles or pieces of tiles).
constexpr int kSimtMaxSegments = 10;
// vec: all rows 16-byte aligned (bases aligned, ld % 4 == 0): TMA-staged kernel; otherwise
// the cp.async kernel with 4-byte copies.
cudaError_t launch_sgemm_simt(const SimtParams& p, bool trans_b, bool vec, cudaStream_t s);
// Small problems: 32 x 32 tiles (p.tiles_m, p.tiles_n count them), K cut into p.sk_splits
// chunks; partials [tiles][splits][1024] floats and counters [tiles] when splits > 1.
cudaError_t launch_sgemm_simt_small(const SimtParams& p, bool trans_b, bool vec, cudaStream_t s);
constexpr int kSimtSmallT = 32, kSimtSmallKP = 128;
// CTAs of the SIMT kernel that fit on one SM at once (occupancy query, cached).
int sgemm_simt_ctas_per_sm(bool trans_b, bool vec);
inline int64_t simt_ws_floats(int64_t partial_tiles) { return partial_tiles * 16 * 256 * 4; }
#ifndef DG_SIMT_BK
#define DG_SIMT_BK 32
#endif
#ifndef DG_SIMT_STAGES
#define DG_SIMT_STAGES 2
#endif
constexpr int kSimtBM = 128, kSimtBN = 128, kSimtBK = DG_SIMT_BK, kSimtThreads = 256,
              kSimtStages = DG_SIMT_STAGES;
static_assert(kSimtBK == 16 || kSimtBK == 32, "SIMT K tile");

// ------------------------------------------------------------------ BF16 tcgen05 tile path
struct TcParams {
  int64_t M, N, K;
  int64_t batch;
  int64_t tiles_m, tiles_n, total_tiles;
  int32_t kblocks;
  int32_t group;
  float alpha, beta;
  void* C; int64_t ldc, strideC;
  int32_t c_f32;     // 1: C is float32, 0: bfloat16
  int32_t c_vec;     // 1: 16-byte vector stores/loads of C rows are legal
  int32_t c_tma;     // 1: epilogue writes C with TMA tensor stores (beta == 0, aligned C)
  uint32_t* status;  // device status word
  // Stream-K phase: the last sk_tiles tiles of the raster order run first, their K blocks
  // spread evenly over CTAs 0 .. sk_ctas-1 (sk_tiles = 0: none); then tiles 0 .. dp_tiles-1
  // run one per CTA per wave.  Partial tiles go to ws, [sk_ctas][2][BN / 4][128] float4,
  // and the last contributor of a tile adds them; counters[sk_tiles] are zero between calls.
  int64_t dp_tiles, sk_tiles;
  int32_t sk_ctas;
  float* ws;
  uint32_t* counters;
  // FP8 (E4M3) operands: C = acc * scale_a[row] * scale_b[column] (null otherwise).
  const float* scale_a;
  const float* scale_b;
};
inline int64_t tc_ws_floats(int64_t sk_ctas, int bn) { return sk_ctas * 2 * 128 * bn; }
// A: [batch][M][lda] bf16 (K contiguous).  B: op N -> [batch][K][ldb] (N contiguous),
// op T -> [batch][N][ldb] (K contiguous).
// pair: launch clusters of two CTAs that each compute half of a 256 x bn tile (bn = 256, or
// 224 for FP8; batch 1, num_ctas even; p.tiles_m then counts 256-row tile rows).
// B2 non-null: the FFN gate/up form -- B = W_g, B2 = W_u (both K x N, N-major, batch 1),
// bn = 256 covers 128 output columns of each, and C = SiLU(bf16(X W_g)) * bf16(X W_u).
// fp8: A [M][lda] and B [N][ldb] are E4M3 codes (bytes, K contiguous; b_kmajor), batch 1, and
// p.scale_a / p.scale_b scale the rows and columns of the FP32 accumulator.
cudaError_t launch_gemm_tc(const TcParams& p, int bn, const void* A, int64_t lda, int64_t strideA,
                           const void* B, int64_t ldb, int64_t strideB, bool b_kmajor,
                           bool pair, int num_ctas, cudaStream_t s, const void* B2 = nullptr,
                           int64_t ldb2 = 0, bool fp8 = false);
constexpr int kTcBM = 128, kTcBK = 64;

// ------------------------------------------------------------------ BF16 thin (decode) path
struct ThinParams {
  int64_t M, N, K;
  int64_t n_tiles;     // ceil(N / 128)
  int64_t kblocks;     // ceil(K / 64)
  int64_t units;       // n_tiles * kblocks
  int64_t ctas;        // grid size G
  float alpha, beta;
  void* C; int64_t ldc;
  int32_t c_f32;
  float* ws;           // partials: [ctas][2][ntok / 4][128 columns] float4
  uint32_t* counters;  // [n_tiles], zero between calls
  uint32_t* status;
};
cudaError_t launch_gemm_thin(const ThinParams& p, int ntok, const void* X, int64_t ldx,
                             const void* W, int64_t ldw, bool w_kmajor, cudaStream_t s);
constexpr int kThinBN = 128, kThinBK = 64;
inline int64_t thin_ws_floats(int64_t ctas, int ntok) { return ctas * 2 * ntok * 128; }

// Zeroes the arrival counters of the no-allocation decode entry point's fixed scratch on
// `dev` (after a bounded wait gave up); a no-op where that entry point never ran.
cudaError_t noalloc_reset_counters(int dev);

// ------------------------------------------------------------------ persistent decode chain
// y_{l+1} = bf16(y_l W_l) for l < layers (y_0 = X, M <= 16 rows), one cooperative launch of
// `ctas` CTAs; every layer is split stream-K over the same CTAs as gemm_thin_kernel splits
// one call; a layer's X loads wait for the previous layer's last output tile.
constexpr int kChainMax = 8;
struct ChainLayer {
  int64_t N, K;
  uint32_t n_tiles, kblocks, units;  // ceil(N / 128), ceil(K / 64), n_tiles * kblocks
  uint32_t ctas;                     // CTAs sharing the layer: min(units, grid), as one call
  void* C; int64_t ldc;              // the layer's BF16 output [M][ldc]
  float* ws;                         // partials: [ctas][2][4][128] float4
  uint32_t* counters;                // [n_tiles] split-K tickets, zero between calls
  uint32_t* tiles_done;              // output tiles written so far, zero between calls
};
struct ChainParams {
  int32_t layers;
  int64_t M;
  uint32_t ctas;
  uint32_t prefetch;  // W blocks of a later layer's range asked of L2 at the layer boundary
  uint32_t poll_ns;   // sleep between polls of the previous layer's tile count
  ChainLayer L[kChainMax];
  uint32_t* done;   // CTAs finished in this call, zero between calls
  uint32_t* status;
};
// W_l [K_l][ldw_l] N-major BF16; X [M][ldx].
cudaError_t launch_gemm_chain(const ChainParams& p, const void* X, int64_t ldx,
                              const void* const* W, const int64_t* ldw, cudaStream_t s,
                              bool pdl, bool coop);

// ------------------------------------------------------------------ FP8 row quantiser
// Q[i][:] = E4M3(X[i][:] * (448 / amax_i)), scales[i] = amax_i / 448 (X BF16, Q bytes).
// vec: rows 16-byte aligned (X ld % 8 == 0, Q ld % 16 == 0, bases aligned).
cudaError_t launch_quantize_rows(int64_t rows, int64_t cols, const void* X, int64_t ldx, void* Q,
                                 int64_t ldq, float* scales, bool vec, int sms, cudaStream_t s);

// ------------------------------------------------------------------ fused attention
struct AttnParams {
  int64_t batch, Lq, Lkv;
  int64_t q_tiles;     // ceil(Lq / 128)
  int64_t kv_blocks;   // ceil(Lkv / 128)
  float c_log2;        // scale * log2(e)
  int32_t rank3;       // batch > 1: 3-D tensor maps
  // Split over keys (0: none): a query tile's key blocks are cut into chunks of `chunk`
  // blocks, one CTA each; the chunks' (m, l, u) go to ws, [item][32 column groups][128
  // rows] float4 then m[128], l[128], and the last chunk to finish (counters[b * q_tiles +
  // tile], zero between calls) merges them in chunk order.
  int64_t chunk;
  int64_t items;       // grid size: work items (query tiles, or their key chunks)
  int32_t sms;         // SMs of the device
  float* ws;
  uint32_t* counters;
  uint32_t* status;
};
// Floats of one split-key partial: u (128 x 128) and the row statistics m, l.
constexpr int64_t kAttnPartFloats = 128 * 128 + 2 * 128;
// Q, O: [batch][Lq][ld] bf16; K, V: [batch][Lkv][ld] bf16 (d = 128 contiguous columns).
cudaError_t launch_attention(const AttnParams& p, bool causal, const void* Q, int64_t ldq,
                             int64_t sQ, const void* K, int64_t ldk, int64_t sK, const void* V,
                             int64_t ldv, int64_t sV, void* O, int64_t ldo, int64_t sO,
                             cudaStream_t s);

// Tensor map over a (batch x) outer x inner row-major view (cached by address, shape, box).
bool make_tile_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t esz, const void* base,
                   uint64_t inner, uint64_t outer, uint64_t ld, uint64_t batch, uint64_t stride,
                   uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                   uint32_t box_batch);

// ------------------------------------------------------------------ misc
// C = beta * C over a (batch, M, N) strided view (K == 0 or alpha == 0).
cudaError_t launch_scale(void* C, bool c_f32, int64_t M, int64_t N, int64_t ldc, int64_t strideC,
                         int64_t batch, float beta, cudaStream_t s);

// Sets the dynamic shared-memory limit of a kernel once per device (the attribute is
// per function and context; setting it on every call costs host time on the launch path).
template <typename Kernel>
inline cudaError_t ensure_smem_attr(Kernel kern, int bytes, std::atomic<uint64_t>& done_mask) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done_mask.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done_mask.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launches `kern` with programmatic stream serialisation: the launch may overlap the tail of
// the previous kernel in the stream; the kernel itself waits (griddepcontrol.wait) before it
// touches global memory, so stream order is kept for every memory effect.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Fault injection for the bounded-wait tests (host-set, read by the kernels at launch).
extern int g_fault_injection;

}  // namespace dg
