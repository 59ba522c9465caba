// sgemm_simt.cu -- FP32 SGEMM on CUDA cores for sm_103a.
//
// The SGEMM tutorial ("4.1 Toi uu hieu nang toan tu GEMM tren CUDA") builds the kernel in
// steps: block tiling in shared memory along K (section 4), a register-blocked outer
// product per thread (section 5), a 4 x 8 lane arrangement per warp (section 6), 16-byte
// vector accesses (section 7), a bank-conflict-free shared layout (section 8) and
// asynchronous multistage copies (sections 9-10).  These kernels keep those ideas and set
// them for this GPU:
//   * 128 x 128 block tile, BK = 32, 256 threads, an 8 x 8 FP32 accumulator per thread
//     (4 x 8 lanes per warp, warp tile 32 x 64), 2 CTAs per SM;
//   * operands staged by the tensor memory accelerator when every row is 16-byte aligned
//     (sgemm_tma_kernel): a 3-stage ring whose stages one thread fills with two bulk tensor
//     copies, completion counted in bytes on a per-stage mbarrier; the last warp to finish
//     reading a stage refills it, so no thread waits at a CTA barrier and no thread spends
//     issue slots on per-element copies;
//   * otherwise (unaligned rows) a 2-stage cp.async ring with zero-filled edges
//     (sgemm_simt_kernel);
//   * A stays K-contiguous in shared memory with a 36-float row stride: a thread reads 4
//     K-steps of one A row with one 16-byte load, and the 4 rows a warp reads at once fall
//     in 4 different bank quads (conflict-free without the tutorial's register transpose);
//   * B rows are read as two 16-byte vectors per K-step, 8 lanes covering 128 contiguous
//     bytes (conflict-free);
//   * thread rows are interleaved (row = base + 4*i) so C rows are written by 8 lanes
//     with 16-byte stores, 128 contiguous bytes per row segment;
//   * strictly FP32 fused multiply-add (packed two per instruction with fma.rn.f32x2, which
//     halves the issue slots the FMAs take); no TF32.
// Epilogue: C = fma(alpha, acc, beta*C_old) in FP32 (C_old not read when beta == 0), masked
// at the edges.
#include "dg_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dg {
namespace {

constexpr int BM = kSimtBM, BN = kSimtBN, BK = kSimtBK, NT = kSimtThreads, STAGES = kSimtStages;
constexpr int LDS_K = BK + 4;            // K-contiguous tile row stride (floats)
constexpr int A_STAGE = BM * LDS_K;      // floats per A stage
constexpr int B_STAGE = BM * LDS_K;      // floats per B stage (>= BK*BN for the N layout)
static_assert(BK * BN <= B_STAGE, "B stage too small");
constexpr int SMEM_BYTES = STAGES * (A_STAGE + B_STAGE) * 4;

__device__ __forceinline__ int clamp_bytes(int64_t remaining_elems) {
  return remaining_elems <= 0 ? 0 : (remaining_elems >= 4 ? 16 : static_cast<int>(remaining_elems) * 4);
}

// Copies one BM x BK tile of a K-contiguous matrix (rows r0.., columns k0..) into a
// [BM][LDS_K] shared tile, zero-filling outside [0,rows) x [0,K).
template <bool VEC>
__device__ __forceinline__ void load_kmajor(float* dst, const float* src, int64_t ld, int64_t r0,
                                            int64_t rows, int64_t k0, int64_t K, int tid) {
  if (VEC) {
#pragma unroll
    for (int h = 0; h < (BM * BK / 4) / NT; ++h) {
      const int q = tid + h * NT;
      const int r = q / (BK / 4), c4 = q % (BK / 4);
      const int64_t gr = r0 + r, gk = k0 + c4 * 4;
      const int bytes = gr < rows ? clamp_bytes(K - gk) : 0;
      const float* g = bytes ? src + gr * ld + gk : src;
      cp_async_16(smem_u32(dst + r * LDS_K + c4 * 4), g, bytes);
    }
  } else {
#pragma unroll
    for (int h = 0; h < (BM * BK) / NT; ++h) {
      const int e = tid + h * NT;
      const int r = e / BK, k = e % BK;
      const int64_t gr = r0 + r, gk = k0 + k;
      const bool ok = gr < rows && gk < K;
      cp_async_4(smem_u32(dst + r * LDS_K + k), ok ? src + gr * ld + gk : src, ok ? 4 : 0);
    }
  }
}

// Copies one BK x BN tile of an N-contiguous matrix (rows k0.., columns n0..) into a
// [BK][BN] shared tile, zero-filling outside [0,K) x [0,N).
template <bool VEC>
__device__ __forceinline__ void load_nmajor(float* dst, const float* src, int64_t ld, int64_t k0,
                                            int64_t K, int64_t n0, int64_t N, int tid) {
  if (VEC) {
#pragma unroll
    for (int h = 0; h < (BK * BN / 4) / NT; ++h) {
      const int q = tid + h * NT;
      const int r = q >> 5, c = q & 31;
      const int64_t gk = k0 + r, gn = n0 + c * 4;
      const int bytes = gk < K ? clamp_bytes(N - gn) : 0;
      const float* g = bytes ? src + gk * ld + gn : src;
      cp_async_16(smem_u32(dst + r * BN + c * 4), g, bytes);
    }
  } else {
#pragma unroll
    for (int h = 0; h < (BK * BN) / NT; ++h) {
      const int e = tid + h * NT;
      const int r = e >> 7, n = e & 127;
      const int64_t gk = k0 + r, gn = n0 + n;
      const bool ok = gk < K && gn < N;
      cp_async_4(smem_u32(dst + r * BN + n), ok ? src + gk * ld + gn : src, ok ? 4 : 0);
    }
  }
}

__device__ __forceinline__ float f4get(const float4& v, int i) {
  return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

#ifndef DG_SIMT_FFMA2
#define DG_SIMT_FFMA2 1
#endif
#ifndef DG_SIMT_MIN_BLOCKS
#define DG_SIMT_MIN_BLOCKS 2
#endif

// (d0, d1) += (a, a) * (b0, b1) with one packed FP32 instruction (fma.rn.f32x2): two IEEE
// single-precision fused multiply-adds, the same arithmetic as two fmaf calls, half the
// issue slots.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a, float b0, float b1) {
#if DG_SIMT_FFMA2
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %2};\n\t"
      "mov.b64 rb, {%3, %4};\n\t"
      "mov.b64 rd, {%0, %1};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rd;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "+f"(d0), "+f"(d1)
      : "f"(a), "f"(b0), "f"(b1));
#else
  d0 = fmaf(a, b0, d0);
  d1 = fmaf(a, b1, d1);
#endif
}

// The end of one work item: a tail chunk publishes its partial accumulator and the last
// chunk of the tile to arrive sums all chunks in chunk (= K) order; then C = alpha*acc +
// beta*C_old with one FP32 rounding per operation, masked at the edges.  Called by every
// thread of the CTA.
template <bool TRANS_B, bool VEC>
__device__ __forceinline__ void simt_finish(const SimtParams& p, float (&acc)[8][8], int64_t b,
                                            int64_t m0, int64_t n0, int64_t tile, int chunk,
                                            uint32_t* s_is_last) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;
  const int lm = lane >> 3, ln = lane & 7;
  const int row_base = wm * 32 + lm;          // thread rows: row_base + 4*i
  const int col_base_n = wn * 64 + ln * 4;    // N layout: cols col_base_n + {0..3}, +32
  const int col_base_t = wn * 64 + ln;        // T layout: cols col_base_t + 8*j
  float* C = p.C + b * p.strideC;

  if (chunk >= 0) {
    // One of the sk_splits K chunks of a tail tile: publish the partial accumulator; the last
    // chunk to arrive sums all chunks in chunk (= K) order -- a fixed order -- and writes C.
    const int64_t sk_tile = tile - p.dp_tiles;
    const int S = p.sk_splits;
    float4* mine = reinterpret_cast<float4*>(p.ws) + ((sk_tile * S + chunk) * 16) * NT + tid;
#pragma unroll
    for (int q = 0; q < 16; ++q)
      mine[q * NT] = make_float4(acc[q >> 1][4 * (q & 1)], acc[q >> 1][4 * (q & 1) + 1],
                                 acc[q >> 1][4 * (q & 1) + 2], acc[q >> 1][4 * (q & 1) + 3]);
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const uint32_t prev = atomicAdd(&p.counters[sk_tile], 1u);
      const bool last = prev + 1u == static_cast<uint32_t>(S);
      if (last) __threadfence();
      *s_is_last = last ? 1u : 0u;
    }
    __syncthreads();
    if (!*s_is_last) return;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
    for (int cc = 0; cc < S; ++cc) {
      const float4* src = reinterpret_cast<const float4*>(p.ws) + ((sk_tile * S + cc) * 16) * NT + tid;
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // 8 independent 16-byte loads in flight
        float4 part[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) part[q] = __ldcg(src + (8 * half + q) * NT);
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          const int q = 8 * half + q8;
          acc[q >> 1][4 * (q & 1)] += part[q8].x;
          acc[q >> 1][4 * (q & 1) + 1] += part[q8].y;
          acc[q >> 1][4 * (q & 1) + 2] += part[q8].z;
          acc[q >> 1][4 * (q & 1) + 3] += part[q8].w;
        }
      }
    }
    // The partials are scratch that nothing reads again before the next call rewrites them:
    // drop their L2 lines so they are never written back.  A warp drops the lines holding
    // its own 32 float4 of each of the 16 groups (4 x 128 bytes) once its lanes have read them.
    __syncwarp();
    for (int cc = 0; cc < S; ++cc) {
      const uint8_t* pb = reinterpret_cast<const uint8_t*>(reinterpret_cast<const float4*>(p.ws) +
                                                           ((sk_tile * S + cc) * 16) * NT + warp * 32);
#pragma unroll
      for (int i = lane; i < 16 * 4; i += 32) discard_l2(pb + static_cast<size_t>(i >> 2) * NT * 16 + (i & 3) * 128);
    }
    if (tid == 0) p.counters[sk_tile] = 0u;  // ready for the next call
  }

  // Epilogue: C = alpha*acc + beta*C_old, one FP32 rounding per operation.
  const float alpha = p.alpha, beta = p.beta;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int64_t gm = m0 + row_base + 4 * i;
    if (gm >= p.M) continue;
    float* crow = C + gm * p.ldc;
    if (TRANS_B) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t gn = n0 + col_base_t + 8 * j;
        if (gn < p.N)
          crow[gn] = beta != 0.f ? fmaf(alpha, acc[i][j], beta * crow[gn]) : alpha * acc[i][j];
      }
    } else {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t gn = n0 + col_base_n + 32 * h;
        const float* a4 = &acc[i][4 * h];
        if (VEC && gn + 3 < p.N) {
          float4* dst = reinterpret_cast<float4*>(crow + gn);
          float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
          if (beta != 0.f) o = *dst;
          *dst = make_float4(fmaf(alpha, a4[0], beta * o.x), fmaf(alpha, a4[1], beta * o.y),
                             fmaf(alpha, a4[2], beta * o.z), fmaf(alpha, a4[3], beta * o.w));
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (gn + j < p.N)
              crow[gn + j] = beta != 0.f ? fmaf(alpha, a4[j], beta * crow[gn + j]) : alpha * a4[j];
          }
        }
      }
    }
  }
}

// One work item: the K tiles [kbeg, kend) of output tile `tile`.  sk_cta < 0 marks a
// data-parallel tile (always the whole K range); otherwise the item is stream-K CTA
// sk_cta's piece of the tile and, when it covers only part of K, goes through the partial
// protocol (publish, count arrivals, the last arriver sums in CTA order).
template <bool TRANS_B, bool VEC>
__device__ __forceinline__ void simt_item(const SimtParams& p, float* As, float* Bs,
                                          const int64_t tile, const int kbeg, const int kend,
                                          const int chunk, uint32_t* s_is_last) {
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int wm = warp >> 1, wn = warp & 1;
  const int lm = lane >> 3, ln = lane & 7;
  const int K = static_cast<int>(p.K);

  int64_t b, tm, tn;
  raster_tile(tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
  const int64_t m0 = tm * BM, n0 = tn * BN;
  const float* A = p.A + b * p.strideA;
  const float* B = p.B + b * p.strideB;

  float acc[8][8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;

  // Copy plan of this thread for the 16-byte path.  A (and B in the T layout): CPR = BK/4
  // chunks per row, rows ar + h*RS (RS = NT/CPR) at K offset ac.  B in the N layout: rows
  // br + 8h of the K tile, column bc.  Only two running global pointers are kept; the other
  // chunks are reached through the leading dimension (a kernel parameter), so few registers
  // stay live across the main loop.
  constexpr int CPR = BK / 4, RS = NT / CPR, HA = BM / RS, HB = BK / 8;
  const int ar = tid / CPR, ac = (tid % CPR) * 4;
  const int br = tid >> 5, bc = (tid & 31) * 4;
  const int64_t a_rows_left = p.M - (m0 + ar), bt_rows_left = p.N - (n0 + ar);
  const int b_nbytes = TRANS_B ? 0 : clamp_bytes(p.N - (n0 + bc));
  const int64_t kofs = static_cast<int64_t>(kbeg) * BK;
  const float* ga = A + (m0 + ar) * p.lda + ac + kofs;
  const float* gb = TRANS_B ? B + (n0 + ar) * p.ldb + ac + kofs
                            : B + (br + kofs) * p.ldb + n0 + bc;

  int next_tile = kbeg;  // K tile the next issued stage copies
  auto load_stage = [&](int stage) {
    const int k0 = next_tile * BK;
    if (VEC) {
      const uint32_t as_ = smem_u32(As + stage * A_STAGE);
      const uint32_t bs_ = smem_u32(Bs + stage * B_STAGE);
      const int ka = clamp_bytes(K - (k0 + ac));
#pragma unroll
      for (int h = 0; h < HA; ++h) {
        const int a = a_rows_left > h * RS ? ka : 0;
        cp_async_16(as_ + ((ar + h * RS) * LDS_K + ac) * 4, a ? ga + h * RS * p.lda : p.A, a);
      }
      ga += BK;
      if (TRANS_B) {
#pragma unroll
        for (int h = 0; h < HA; ++h) {
          const int bb = bt_rows_left > h * RS ? ka : 0;
          cp_async_16(bs_ + ((ar + h * RS) * LDS_K + ac) * 4, bb ? gb + h * RS * p.ldb : p.B, bb);
        }
        gb += BK;
      } else {
#pragma unroll
        for (int h = 0; h < HB; ++h) {
          const int bb = k0 + br + 8 * h < K ? b_nbytes : 0;
          cp_async_16(bs_ + ((br + 8 * h) * BN + bc) * 4, bb ? gb + 8 * h * p.ldb : p.B, bb);
        }
        gb += BK * p.ldb;
      }
    } else {
      load_kmajor<false>(As + stage * A_STAGE, A, p.lda, m0, p.M, k0, p.K, tid);
      if (TRANS_B)
        load_kmajor<false>(Bs + stage * B_STAGE, B, p.ldb, n0, p.N, k0, p.K, tid);
      else
        load_nmajor<false>(Bs + stage * B_STAGE, B, p.ldb, k0, p.K, n0, p.N, tid);
    }
    ++next_tile;
  };

#pragma unroll
  for (int s = 0; s < STAGES - 1; ++s) {
    if (kbeg + s < kend) load_stage(s);
    cp_async_commit();
  }

  const int row_base = wm * 32 + lm;          // thread rows: row_base + 4*i
  const int col_base_n = wn * 64 + ln * 4;    // N layout: cols col_base_n + {0..3}, +32
  const int col_base_t = wn * 64 + ln;        // T layout: cols col_base_t + 8*j

  int stage = 0;                  // stage computed this iteration
  int load_slot = STAGES - 1;     // stage the next copy goes to
  for (int kt = kbeg; kt < kend; ++kt) {
    cp_async_wait<STAGES - 2>();
    __syncthreads();
    if (kt + STAGES - 1 < kend) load_stage(load_slot);
    cp_async_commit();
    load_slot = load_slot + 1 == STAGES ? 0 : load_slot + 1;
    const float* as = As + stage * A_STAGE;
    const float* bs = Bs + stage * B_STAGE;
#pragma unroll
    for (int kk = 0; kk < BK / 4; ++kk) {
      float4 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        a[i] = *reinterpret_cast<const float4*>(as + (row_base + 4 * i) * LDS_K + kk * 4);
      if (TRANS_B) {
        float4 bt[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          bt[j] = *reinterpret_cast<const float4*>(bs + (col_base_t + 8 * j) * LDS_K + kk * 4);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
          for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 8; j += 2)
              ffma2(acc[i][j], acc[i][j + 1], f4get(a[i], k4), f4get(bt[j], k4), f4get(bt[j + 1], k4));
      } else {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int k = kk * 4 + k4;
          const float4 b0 = *reinterpret_cast<const float4*>(bs + k * BN + col_base_n);
          const float4 b1 = *reinterpret_cast<const float4*>(bs + k * BN + col_base_n + 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float av = f4get(a[i], k4);
            ffma2(acc[i][0], acc[i][1], av, b0.x, b0.y);
            ffma2(acc[i][2], acc[i][3], av, b0.z, b0.w);
            ffma2(acc[i][4], acc[i][5], av, b1.x, b1.y);
            ffma2(acc[i][6], acc[i][7], av, b1.z, b1.w);
          }
        }
      }
    }
    stage = stage + 1 == STAGES ? 0 : stage + 1;
  }
  cp_async_wait<0>();
  simt_finish<TRANS_B, VEC>(p, acc, b, m0, n0, tile, chunk, s_is_last);
}

template <bool TRANS_B, bool VEC>
__global__ void __launch_bounds__(NT, DG_SIMT_MIN_BLOCKS) sgemm_simt_kernel(const SimtParams p) {
  extern __shared__ __align__(16) float smem[];
  float* As = smem;
  float* Bs = smem + STAGES * A_STAGE;
  __shared__ uint32_t s_is_last;

  // Launched with programmatic serialisation: wait for the previous kernel before the first
  // global access, and let the next one launch early.
  pdl_trigger();
  pdl_wait();

  const int KT = static_cast<int>((p.K + BK - 1) / BK);
  if (blockIdx.x < p.dp_tiles) {
    // Data-parallel part of the grid: one whole tile per CTA.
    simt_item<TRANS_B, VEC>(p, As, Bs, blockIdx.x, 0, KT, -1, &s_is_last);
    return;
  }
  // Tail of the grid: tile dp_tiles + j / S, K chunk j % S (S = sk_splits equal chunks).
  const int64_t j = blockIdx.x - p.dp_tiles;
  const int S = p.sk_splits;
  const int chunk = static_cast<int>(j % S);
  const int kbeg = static_cast<int>(static_cast<int64_t>(chunk) * KT / S);
  const int kend = static_cast<int>(static_cast<int64_t>(chunk + 1) * KT / S);
  simt_item<TRANS_B, VEC>(p, As, Bs, p.dp_tiles + j / S, kbeg, kend, chunk, &s_is_last);
}

// ------------------------------------------------------------------ TMA-staged kernel
// Work item of CTA `cta`: the first dp_tiles CTAs take one whole tile each; CTA
// dp_tiles + j takes K chunk j % S (of S equal chunks) of tail tile dp_tiles + j / S.
struct SimtItem {
  int64_t tile, b, m0, n0;
  int kbeg, kend, chunk;  // chunk -1: a whole tile
};
__device__ __forceinline__ SimtItem simt_item_of(const SimtParams& p, int64_t cta) {
  SimtItem it;
  const int KT = static_cast<int>((p.K + BK - 1) / BK);
  if (cta < p.dp_tiles) {
    it.tile = cta; it.kbeg = 0; it.kend = KT; it.chunk = -1;
  } else {
    const int64_t j = cta - p.dp_tiles;
    const int S = p.sk_splits;
    it.chunk = static_cast<int>(j % S);
    it.kbeg = static_cast<int>(static_cast<int64_t>(it.chunk) * KT / S);
    it.kend = static_cast<int>(static_cast<int64_t>(it.chunk + 1) * KT / S);
    it.tile = p.dp_tiles + j / S;
  }
  int64_t tm, tn;
  raster_tile(it.tile, p.tiles_m, p.tiles_n, p.group, &it.b, &tm, &tn);
  it.m0 = tm * BM;
  it.n0 = tn * BN;
  return it;
}

// A (and B^T) arrive as boxes of 128 rows x LDS_K = 36 floats: the copy carries 4 columns
// of the next K tile (or zeros past K) that are never read, and in exchange the rows land
// with the padded 144-byte pitch, so the 4 rows a warp reads at once fall in 4 different bank
// quads and every shared address is a register plus an immediate offset.  B [K][N] arrives
// as dense [32][128] rows.
constexpr int T_STAGES = 3;
constexpr uint32_t T_A_BYTES = BM * LDS_K * 4;                     // 18 KiB
template <bool TRANS_B>
struct TmaCfg {
  static constexpr uint32_t B_BYTES = TRANS_B ? BN * LDS_K * 4 : BK * BN * 4;  // 18 / 16 KiB
  static constexpr uint32_t STAGE_BYTES = T_A_BYTES + B_BYTES;
  static constexpr int SMEM_BYTES = 1024 + T_STAGES * STAGE_BYTES + 128;
};
constexpr int T_WARPS = NT / 32;


// Bounded wait for a stage (mbar_wait with the abort flag addressed in the shared window,
// so that few registers stay live in the main loop).
__device__ __forceinline__ bool stage_wait(uint32_t bar, uint32_t parity, uint32_t abort_s,
                                           const SimtParams& p) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0) {
      uint32_t ab;
      asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(ab) : "r"(abort_s) : "memory");
      if (ab) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        asm volatile("st.volatile.shared.u32 [%0], 1;" ::"r"(abort_s) : "memory");
        atomicCAS(p.status, 0u, static_cast<uint32_t>(kDevTimeoutMma));
        return false;
      }
    }
  }
}

// A CTA's work in (tile, K tile) units is one contiguous range, cut into segments at tile
// boundaries: one segment (a whole tile or one K chunk of a tail tile) in the data-parallel
// schedule, a few in the stream-K schedule.  The segment table is built once per CTA.
constexpr int T_MAX_SEG = kSimtMaxSegments;
struct SegInfo {
  int64_t tile;
  int32_t start, len;       // relative unit index of the first K tile, number of K tiles
  int32_t kbeg, kend;       // K tiles of the tile
  int32_t kx0, x_m, x_n, x_b;  // copy coordinates of the first K tile
};

struct TmaCtl {
  SegInfo seg[T_MAX_SEG];
  int32_t nseg, total;      // segments, K tiles over all of them
  int32_t chunk;            // data-parallel schedule: the K chunk (-1: whole tile)
  uint64_t full[T_STAGES];  // stage s holds K tile i (bytes counted by the copies)
  uint32_t done[T_STAGES];  // warps that have finished reading stage s, over all its uses
  uint32_t abort;
  uint32_t is_last;
};

// Shared-memory add with acquire and release at CTA scope: the warps' reads of a stage are
// ordered before the count that tells the last of them to refill it.
__device__ __forceinline__ uint32_t atom_add_acq_rel_cta(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// Global add with acquire and release at GPU scope (the stream-K ticket).
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// Stream-K end of a segment that covers only part of its tile's K range: the CTA publishes
// its partial accumulator (slot 0 for its range's first segment, 1 for its last) and takes a
// ticket; the last contributor to take one adds every contributor's part in CTA (= K) order
// -- a fixed order, so results repeat bit for bit whoever is last -- and writes C.
template <bool TRANS_B>
__device__ __forceinline__ void sk_segment_finish(const SimtParams& p, float (&acc)[8][8],
                                                  const SegInfo& sg, int slot, uint32_t* s_is_last) {
  const int tid = threadIdx.x;
  const int64_t KT = (p.K + BK - 1) / BK, U = p.sk_units, G = p.sk_ctas;
  const int64_t c = blockIdx.x;
  const int64_t first = sk_cta_of<int64_t>(sg.tile * KT, U, G);
  const int64_t last = sk_cta_of<int64_t>((sg.tile + 1) * KT - 1, U, G);
  float4* mine = reinterpret_cast<float4*>(p.ws) + ((c * 2 + slot) * 16) * NT + tid;
#pragma unroll
  for (int q = 0; q < 16; ++q)
    __stcg(mine + q * NT, make_float4(acc[q >> 1][4 * (q & 1)], acc[q >> 1][4 * (q & 1) + 1],
                                      acc[q >> 1][4 * (q & 1) + 2], acc[q >> 1][4 * (q & 1) + 3]));
  __syncthreads();
  if (tid == 0) {
    const uint32_t prev = atom_add_acq_rel_gpu(&p.counters[sg.tile], 1u);
    const bool is_last = prev + 1u == static_cast<uint32_t>(last - first + 1);
    if (is_last) p.counters[sg.tile] = 0u;  // ready for the next call
    *s_is_last = is_last ? 1u : 0u;
  }
  __syncthreads();
  if (!*s_is_last) return;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[i][j] = 0.f;
  for (int64_t cc = first; cc <= last; ++cc) {
    const int sl = sk_start<int64_t>(cc, U, G) >= sg.tile * KT ? 0 : 1;
    const float4* src = reinterpret_cast<const float4*>(p.ws) + ((cc * 2 + sl) * 16) * NT + tid;
#pragma unroll
    for (int half = 0; half < 2; ++half) {  // 8 independent 16-byte loads in flight
      float4 part[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) part[q] = __ldcg(src + (8 * half + q) * NT);
#pragma unroll
      for (int q8 = 0; q8 < 8; ++q8) {
        const int q = 8 * half + q8;
        acc[q >> 1][4 * (q & 1)] += part[q8].x;
        acc[q >> 1][4 * (q & 1) + 1] += part[q8].y;
        acc[q >> 1][4 * (q & 1) + 2] += part[q8].z;
        acc[q >> 1][4 * (q & 1) + 3] += part[q8].w;
      }
    }
  }
  // The partials are dead scratch now: drop their L2 lines (see simt_finish).
  {
    const int warp = tid >> 5, lane = tid & 31;
    __syncwarp();
    for (int64_t cc = first; cc <= last; ++cc) {
      const int sl = sk_start<int64_t>(cc, U, G) >= sg.tile * KT ? 0 : 1;
      const uint8_t* pb = reinterpret_cast<const uint8_t*>(reinterpret_cast<const float4*>(p.ws) +
                                                           ((cc * 2 + sl) * 16) * NT + warp * 32);
#pragma unroll
      for (int i = lane; i < 16 * 4; i += 32) discard_l2(pb + static_cast<size_t>(i >> 2) * NT * 16 + (i & 3) * 128);
    }
  }
  simt_finish<TRANS_B, true>(p, acc, sg.x_b, sg.x_m, sg.x_n, sg.tile, -1, s_is_last);
}

// One CTA's range of (tile, K tile) units, operands staged by TMA.  Every thread waits on the
// stage's barrier (bounded); after reading a stage, each warp counts itself done, and the warp
// completing the count issues the copies of the K tile that goes to that stage next -- across
// segment boundaries too, so the next tile's operands stream in during an epilogue.
template <bool TRANS_B, bool RANK3, bool STREAMK>
__global__ void __launch_bounds__(NT, DG_SIMT_MIN_BLOCKS)
    sgemm_tma_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const SimtParams p) {
  using Cfg = TmaCfg<TRANS_B>;
  constexpr uint32_t T_STAGE_BYTES = Cfg::STAGE_BYTES;
  extern __shared__ __align__(16) float smem_f[];
  const uint32_t raw = smem_u32(smem_f);
  const uint32_t base = (raw + 1023u) & ~1023u;
  float* const stages = smem_f + (base - raw) / 4;
  TmaCtl* ctl = reinterpret_cast<TmaCtl*>(stages + T_STAGES * T_STAGE_BYTES / 4);

  // Launched with programmatic serialisation: wait for the previous kernel before the first
  // global access, and let the next one launch early.
  pdl_trigger();

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // The segment table (64-bit index arithmetic here, once; the main loop reads the table).
    const int64_t KT = (p.K + BK - 1) / BK;
    int64_t u, u1;
    ctl->chunk = -1;
    if (STREAMK) {
      u = sk_start<int64_t>(blockIdx.x, p.sk_units, p.sk_ctas);
      u1 = sk_start<int64_t>(blockIdx.x + 1, p.sk_units, p.sk_ctas);
    } else {
      const SimtItem it = simt_item_of(p, blockIdx.x);
      u = it.tile * KT + it.kbeg;
      u1 = it.tile * KT + it.kend;
      ctl->chunk = it.chunk;
    }
    int n = 0, start = 0;
    while (u < u1 && n < T_MAX_SEG) {
      SegInfo& sg = ctl->seg[n];
      sg.tile = u / KT;
      sg.kbeg = static_cast<int32_t>(u - sg.tile * KT);
      sg.kend = static_cast<int32_t>(u1 - sg.tile * KT < KT ? u1 - sg.tile * KT : KT);
      sg.start = start;
      sg.len = sg.kend - sg.kbeg;
      int64_t b, tm, tn;
      raster_tile(sg.tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
      sg.kx0 = sg.kbeg * BK;
      sg.x_m = static_cast<int32_t>(tm * BM);
      sg.x_n = static_cast<int32_t>(tn * BN);
      sg.x_b = static_cast<int32_t>(b);
      start += sg.len;
      u += sg.len;
      ++n;
    }
    ctl->nseg = n;
    ctl->total = start;
    for (int s = 0; s < T_STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      ctl->done[s] = 0;
    }
    ctl->abort = 0;
    ctl->is_last = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
  }
  __syncthreads();
  pdl_wait();
  const int total = ctl->total;

  // Copies of relative K tile i into its stage, by one thread.
  auto issue = [&](int i) {
    int g = 0;
    if (STREAMK)
      while (g + 1 < ctl->nseg && ctl->seg[g + 1].start <= i) ++g;
    const SegInfo& sg = ctl->seg[g];
    const int32_t x_m = sg.x_m, x_n = sg.x_n, x_b = sg.x_b;
    const int32_t kx = sg.kx0 + (i - sg.start) * BK;
    const int s = i % T_STAGES;
    const uint32_t fb = smem_u32(&ctl->full[s]);
    const uint32_t dst = base + s * T_STAGE_BYTES;
    static_assert(T_STAGE_BYTES % 128 == 0 && T_A_BYTES % 128 == 0, "TMA destinations");
    fence_proxy_async_smem();  // earlier reads of the stage come before the async writes
    mbar_arrive_expect_tx(fb, T_STAGE_BYTES);
    if (RANK3) {
      tma_load_3d(dst, &tmA, fb, kx, x_m, x_b);
      if (TRANS_B)
        tma_load_3d(dst + T_A_BYTES, &tmB, fb, kx, x_n, x_b);
      else
        tma_load_3d(dst + T_A_BYTES, &tmB, fb, x_n, kx, x_b);
    } else {
      tma_load_2d(dst, &tmA, fb, kx, x_m);
      if (TRANS_B)
        tma_load_2d(dst + T_A_BYTES, &tmB, fb, kx, x_n);
      else
        tma_load_2d(dst + T_A_BYTES, &tmB, fb, x_n, kx);
    }
  };
  if (tid == 0)
    for (int i = 0; i < T_STAGES && i < total; ++i) issue(i);

  const int wm = warp >> 1, wn = warp & 1;
  const int lm = lane >> 3, ln = lane & 7;
  const int row_base = wm * 32 + lm;          // thread rows: row_base + 4*i
  const int col_base_n = wn * 64 + ln * 4;    // N layout: cols col_base_n + {0..3}, +32
  const int col_base_t = wn * 64 + ln;        // T layout: cols col_base_t + 8*j

  int i = 0;  // relative K tile across the range
  bool failed = false;
  const int nseg = STREAMK ? ctl->nseg : 1;
  for (int g = 0; g < nseg && !failed; ++g) {
    const int seg_end = STREAMK ? ctl->seg[g].start + ctl->seg[g].len : total;
    float acc[8][8];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[r][j] = 0.f;
    for (; i < seg_end; ++i) {
      const int s = i % T_STAGES;
      if (!stage_wait(smem_u32(&ctl->full[s]), static_cast<uint32_t>(i / T_STAGES) & 1u,
                      smem_u32(&ctl->abort), p)) {
        failed = true;
        break;
      }
      const float* as = stages + s * (T_STAGE_BYTES / 4);
      const float* bs = as + T_A_BYTES / 4;
#pragma unroll
      for (int kk = 0; kk < BK / 4; ++kk) {
        float4 a[8];
#pragma unroll
        for (int r = 0; r < 8; ++r)
          a[r] = *reinterpret_cast<const float4*>(as + (row_base + 4 * r) * LDS_K + kk * 4);
        if (TRANS_B) {
          float4 bt[8];
#pragma unroll
          for (int j = 0; j < 8; ++j)
            bt[j] = *reinterpret_cast<const float4*>(bs + (col_base_t + 8 * j) * LDS_K + kk * 4);
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
            for (int r = 0; r < 8; ++r)
#pragma unroll
              for (int j = 0; j < 8; j += 2)
                ffma2(acc[r][j], acc[r][j + 1], f4get(a[r], k4), f4get(bt[j], k4), f4get(bt[j + 1], k4));
        } else {
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int k = kk * 4 + k4;
            const float4 b0 = *reinterpret_cast<const float4*>(bs + k * BN + col_base_n);
            const float4 b1 = *reinterpret_cast<const float4*>(bs + k * BN + col_base_n + 32);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
              const float av = f4get(a[r], k4);
              ffma2(acc[r][0], acc[r][1], av, b0.x, b0.y);
              ffma2(acc[r][2], acc[r][3], av, b0.z, b0.w);
              ffma2(acc[r][4], acc[r][5], av, b1.x, b1.y);
              ffma2(acc[r][6], acc[r][7], av, b1.z, b1.w);
            }
          }
        }
      }
      // This warp is done with the stage; the warp that completes its count refills it.
      __syncwarp();
      if (lane == 0) {
        const uint32_t prev = atom_add_acq_rel_cta(smem_u32(&ctl->done[s]), 1u);
        if (prev + 1u == static_cast<uint32_t>(T_WARPS * (i / T_STAGES + 1)) && i + T_STAGES < total)
          issue(i + T_STAGES);
      }
    }
    // Every thread leaves the K loop at the same K tile (a stage whose copies never land
    // times all of them out), so the barriers of the segment's end are reached by all.
    __syncthreads();
    if (failed || *reinterpret_cast<volatile uint32_t*>(&ctl->abort)) {
      failed = true;
      break;
    }
    const SegInfo& sg = ctl->seg[g];
    if (STREAMK && sg.len < static_cast<int32_t>((p.K + BK - 1) / BK))
      sk_segment_finish<TRANS_B>(p, acc, sg, g == 0 ? 0 : 1, &ctl->is_last);
    else
      simt_finish<TRANS_B, true>(p, acc, sg.x_b, sg.x_m, sg.x_n, sg.tile,
                                 STREAMK ? -1 : ctl->chunk, &ctl->is_last);
    if (STREAMK) __syncthreads();  // is_last is rewritten by the next segment's end
  }
  if (failed && tid == 0) {
    // A wait gave up: no copy may still be landing in shared memory when the CTA exits.
    uint32_t never = 0;
    const int issued_end = i + T_STAGES < total ? i + T_STAGES : total;
    for (int j = i; j < issued_end; ++j)
      mbar_wait(smem_u32(&ctl->full[j % T_STAGES]), static_cast<uint32_t>(j / T_STAGES) & 1u,
                &never, p.status, kDevTimeoutDrain);
  }
}

template <bool TRANS_B, bool RANK3, bool STREAMK>
cudaError_t launch_tma_variant(const CUtensorMap& ma, const CUtensorMap& mb, const SimtParams& p,
                               cudaStream_t s) {
  auto kern = sgemm_tma_kernel<TRANS_B, RANK3, STREAMK>;
  constexpr int smem = TmaCfg<TRANS_B>::SMEM_BYTES;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.sk_ctas > 0 ? p.sk_ctas : p.dp_tiles + p.sk_tiles * p.sk_splits;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NT), smem, s, ma, mb, p);
}

template <bool TRANS_B, bool VEC>
cudaError_t launch_variant(const SimtParams& p, cudaStream_t s) {
  auto kern = sgemm_simt_kernel<TRANS_B, VEC>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.dp_tiles + p.sk_tiles * p.sk_splits;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NT), SMEM_BYTES, s, p);
}

}  // namespace

namespace {
template <bool TRANS_B, bool VEC>
int ctas_per_sm_variant() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n > 0) return n;
  auto kern = sgemm_simt_kernel<TRANS_B, VEC>;
  static std::atomic<uint64_t> attr_done{0};
  n = 0;
  if (ensure_smem_attr(kern, SMEM_BYTES, attr_done) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, SMEM_BYTES) != cudaSuccess ||
      n < 1)
    n = 1;
  cached.store(n, std::memory_order_relaxed);
  return n;
}
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// ------------------------------------------------------------------ small problems
// When the 128 x 128 tiles would fill under a quarter of the resident CTA slots (256^3: 4
// tiles), one tile's whole K on one SM is the call's time, and splitting K over CTAs in
// 128 x 128 pieces leaves the last CTA adding eight 64 KiB partial tiles.  Here a CTA
// computes a 32 x 32 tile instead: its 8 warps split each staged K piece 8 ways (16 K-steps
// each, a 4 x 8 register tile per lane), then add their 8 partial tiles through shared
// memory in warp order.  K may also be cut into S chunks over CTAs (partials of 4 KiB,
// added in chunk order by the last chunk to arrive).
constexpr int SM_T = 32, SM_KP = 128, SM_STAGES = 2;
constexpr int SM_LDA = SM_KP + 4;   // K-contiguous rows (A, and B^T): 132 floats
constexpr int SM_LDB = SM_T + 4;    // B rows [k][36]
constexpr int SM_A_FLOATS = SM_T * SM_LDA;                    // 4224
constexpr int SM_B_FLOATS = SM_KP * SM_LDB > SM_T * SM_LDA ? SM_KP * SM_LDB : SM_T * SM_LDA;
constexpr int SM_STAGE_FLOATS = SM_A_FLOATS + SM_B_FLOATS;
constexpr int SM_SMEM_BYTES = SM_STAGES * SM_STAGE_FLOATS * 4;
static_assert(SM_SMEM_BYTES >= 8 * SM_T * SM_T * 4, "reduction buffer fits in the ring");

// Copies rows [r0, r0 + 32) x K columns [k0, k0 + 128) of a K-contiguous matrix into a
// [32][SM_LDA] tile (zero outside [0, rows) x [0, K)).
template <bool VEC>
__device__ __forceinline__ void small_load_kmajor(float* dst, const float* src, int64_t ld,
                                                  int64_t r0, int64_t rows, int64_t k0, int64_t K,
                                                  int tid) {
  if (VEC) {
#pragma unroll
    for (int h = 0; h < (SM_T * SM_KP / 4) / NT; ++h) {
      const int q = tid + h * NT;
      const int r = q / (SM_KP / 4), c4 = q % (SM_KP / 4);
      const int64_t gr = r0 + r, gk = k0 + c4 * 4;
      const int bytes = gr < rows ? clamp_bytes(K - gk) : 0;
      cp_async_16(smem_u32(dst + r * SM_LDA + c4 * 4), bytes ? src + gr * ld + gk : src, bytes);
    }
  } else {
#pragma unroll 4
    for (int h = 0; h < (SM_T * SM_KP) / NT; ++h) {
      const int e = tid + h * NT;
      const int r = e / SM_KP, k = e % SM_KP;
      const int64_t gr = r0 + r, gk = k0 + k;
      const bool ok = gr < rows && gk < K;
      cp_async_4(smem_u32(dst + r * SM_LDA + k), ok ? src + gr * ld + gk : src, ok ? 4 : 0);
    }
  }
}

// Copies K rows [k0, k0 + 128) x columns [n0, n0 + 32) of an N-contiguous matrix into a
// [128][SM_LDB] tile (zero outside [0, K) x [0, N)).
template <bool VEC>
__device__ __forceinline__ void small_load_nmajor(float* dst, const float* src, int64_t ld,
                                                  int64_t k0, int64_t K, int64_t n0, int64_t N,
                                                  int tid) {
  if (VEC) {
#pragma unroll
    for (int h = 0; h < (SM_KP * SM_T / 4) / NT; ++h) {
      const int q = tid + h * NT;
      const int r = q / (SM_T / 4), c4 = q % (SM_T / 4);
      const int64_t gk = k0 + r, gn = n0 + c4 * 4;
      const int bytes = gk < K ? clamp_bytes(N - gn) : 0;
      cp_async_16(smem_u32(dst + r * SM_LDB + c4 * 4), bytes ? src + gk * ld + gn : src, bytes);
    }
  } else {
#pragma unroll 4
    for (int h = 0; h < (SM_KP * SM_T) / NT; ++h) {
      const int e = tid + h * NT;
      const int r = e / SM_T, n = e % SM_T;
      const int64_t gk = k0 + r, gn = n0 + n;
      const bool ok = gk < K && gn < N;
      cp_async_4(smem_u32(dst + r * SM_LDB + n), ok ? src + gk * ld + gn : src, ok ? 4 : 0);
    }
  }
}

// Grid: tiles32 * S CTAs; CTA j computes K chunk j % S (of S equal chunks, in 128-wide
// pieces) of 32 x 32 tile j / S.  Lane l of warp w holds rows (l >> 2) + 8 r (r < 4) and
// columns 8 (l & 3) + c (c < 8) for the K-steps [16 w, 16 w + 16) of every piece.
template <bool TRANS_B, bool VEC>
__global__ void __launch_bounds__(NT) sgemm_small_kernel(const SimtParams p) {
  extern __shared__ __align__(16) float sm[];
  __shared__ uint32_t s_is_last;
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.sk_splits;
  const int64_t tile = blockIdx.x / S;
  const int chunk = static_cast<int>(blockIdx.x % S);
  const int64_t tiles_mn = p.tiles_m * p.tiles_n;
  const int64_t b = tile / tiles_mn;
  const int64_t t_in = tile - b * tiles_mn;
  const int64_t m0 = (t_in / p.tiles_n) * SM_T, n0 = (t_in % p.tiles_n) * SM_T;
  const float* A = p.A + b * p.strideA;
  const float* B = p.B + b * p.strideB;
  const int64_t KP_total = (p.K + SM_KP - 1) / SM_KP;
  const int64_t pbeg = static_cast<int64_t>(chunk) * KP_total / S;
  const int64_t pend = static_cast<int64_t>(chunk + 1) * KP_total / S;
  const int npieces = static_cast<int>(pend - pbeg);

  // The first piece's operands go to L2 while the previous grid of the stream drains: a
  // prefetch returns nothing to the program, and L2 is the device's point of coherence, so
  // loads issued after the wait still see every write of the previous grid.  One 128-byte
  // line per thread for each of A and B (32 rows x 512 bytes, and 128 K rows x 128 bytes or
  // 32 rows x 512 bytes for B^T).
  if (npieces > 0) {
    const int64_t k0 = pbeg * SM_KP;
    const int r = tid >> 3, seg = (tid & 7) * 32;  // 32 rows x 8 lines of 32 floats
    if (m0 + r < p.M && k0 + seg < p.K) prefetch_l2(A + (m0 + r) * p.lda + k0 + seg);
    if (TRANS_B) {
      if (n0 + r < p.N && k0 + seg < p.K) prefetch_l2(B + (n0 + r) * p.ldb + k0 + seg);
    } else {
      const int kr = tid >> 1, cs = (tid & 1) * 16;  // 128 K rows x 2 half-lines
      if (k0 + kr < p.K && n0 + cs < p.N) prefetch_l2(B + (k0 + kr) * p.ldb + n0 + cs);
    }
  }
  pdl_wait();

  auto load_piece = [&](int piece, int stage) {
    float* as = sm + stage * SM_STAGE_FLOATS;
    float* bs = as + SM_A_FLOATS;
    const int64_t k0 = (pbeg + piece) * SM_KP;
    small_load_kmajor<VEC>(as, A, p.lda, m0, p.M, k0, p.K, tid);
    if (TRANS_B)
      small_load_kmajor<VEC>(bs, B, p.ldb, n0, p.N, k0, p.K, tid);
    else
      small_load_nmajor<VEC>(bs, B, p.ldb, k0, p.K, n0, p.N, tid);
  };

  const int lr = lane >> 2, lc = lane & 3;
  float acc[4][8];
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 8; ++c) acc[r][c] = 0.f;

  if (npieces > 0) load_piece(0, 0);
  cp_async_commit();
  for (int pc = 0; pc < npieces; ++pc) {
    if (pc + 1 < npieces) load_piece(pc + 1, (pc + 1) & 1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const float* as = sm + (pc & 1) * SM_STAGE_FLOATS;
    const float* bs = as + SM_A_FLOATS;
#pragma unroll
    for (int kg = 0; kg < 4; ++kg) {
      const int kk = warp * 16 + kg * 4;
      float4 a[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) a[r] = *reinterpret_cast<const float4*>(as + (lr + 8 * r) * SM_LDA + kk);
      if (TRANS_B) {
        float4 bt[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)
          bt[c] = *reinterpret_cast<const float4*>(bs + (lc * 8 + c) * SM_LDA + kk);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
#pragma unroll
          for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int c = 0; c < 8; c += 2)
              ffma2(acc[r][c], acc[r][c + 1], f4get(a[r], k4), f4get(bt[c], k4), f4get(bt[c + 1], k4));
      } else {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const float4 b0 = *reinterpret_cast<const float4*>(bs + (kk + k4) * SM_LDB + lc * 8);
          const float4 b1 = *reinterpret_cast<const float4*>(bs + (kk + k4) * SM_LDB + lc * 8 + 4);
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            const float av = f4get(a[r], k4);
            ffma2(acc[r][0], acc[r][1], av, b0.x, b0.y);
            ffma2(acc[r][2], acc[r][3], av, b0.z, b0.w);
            ffma2(acc[r][4], acc[r][5], av, b1.x, b1.y);
            ffma2(acc[r][6], acc[r][7], av, b1.z, b1.w);
          }
        }
      }
    }
    __syncthreads();  // the stage is refilled by the next iteration's copies
  }
  cp_async_wait<0>();
  __syncthreads();

  // The 8 warps' partial tiles, added in warp order; thread t then owns outputs 4t..4t+3
  // (row 4t / 32, columns 4t % 32 ..).
  float* red = sm;
#pragma unroll
  for (int r = 0; r < 4; ++r)
#pragma unroll
    for (int c = 0; c < 8; c += 4)
      *reinterpret_cast<float4*>(red + warp * SM_T * SM_T + (lr + 8 * r) * SM_T + lc * 8 + c) =
          make_float4(acc[r][c], acc[r][c + 1], acc[r][c + 2], acc[r][c + 3]);
  __syncthreads();
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int w = 0; w < 8; ++w) {
    const float4 x = *reinterpret_cast<const float4*>(red + w * SM_T * SM_T + tid * 4);
    v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
  }
  if (S > 1) {
    float4* mine = reinterpret_cast<float4*>(p.ws) + (tile * S + chunk) * (SM_T * SM_T / 4) + tid;
    __stcg(mine, v);
    __syncthreads();
    if (tid == 0) {
      uint32_t prev;
      asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&p.counters[tile]) : "memory");
      const bool last = prev + 1u == static_cast<uint32_t>(S);
      if (last) p.counters[tile] = 0u;  // ready for the next call
      s_is_last = last ? 1u : 0u;
    }
    __syncthreads();
    if (!s_is_last) return;
    v = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int cc = 0; cc < S; ++cc) {
      const float4 x = __ldcg(reinterpret_cast<const float4*>(p.ws) + (tile * S + cc) * (SM_T * SM_T / 4) + tid);
      v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
    }
  }
  const int64_t gm = m0 + (tid * 4) / SM_T, gn = n0 + (tid * 4) % SM_T;
  if (gm >= p.M) return;
  float* crow = p.C + b * p.strideC + gm * p.ldc;
  const float alpha = p.alpha, beta = p.beta;
  const float vv[4] = {v.x, v.y, v.z, v.w};
  if (VEC && gn + 3 < p.N) {
    float4* dst = reinterpret_cast<float4*>(crow + gn);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (beta != 0.f) o = *dst;
    *dst = make_float4(fmaf(alpha, vv[0], beta * o.x), fmaf(alpha, vv[1], beta * o.y),
                       fmaf(alpha, vv[2], beta * o.z), fmaf(alpha, vv[3], beta * o.w));
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (gn + j < p.N)
        crow[gn + j] = beta != 0.f ? fmaf(alpha, vv[j], beta * crow[gn + j]) : alpha * vv[j];
  }
}

template <bool TRANS_B, bool VEC>
cudaError_t launch_small_variant(const SimtParams& p, cudaStream_t s) {
  auto kern = sgemm_small_kernel<TRANS_B, VEC>;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, SM_SMEM_BYTES, attr_done);
  if (e != cudaSuccess) return e;
  const int64_t grid = p.batch * p.tiles_m * p.tiles_n * p.sk_splits;
  return launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(NT), SM_SMEM_BYTES, s, p);
}

template <bool TRANS_B>
int ctas_per_sm_tma() {
  static std::atomic<int> cached{0};
  int n = cached.load(std::memory_order_relaxed);
  if (n > 0) return n;
  auto kern = sgemm_tma_kernel<TRANS_B, false, false>;
  constexpr int smem = TmaCfg<TRANS_B>::SMEM_BYTES;
  static std::atomic<uint64_t> attr_done{0};
  n = 0;
  if (ensure_smem_attr(kern, smem, attr_done) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, NT, smem) != cudaSuccess ||
      n < 1)
    n = 1;
  cached.store(n, std::memory_order_relaxed);
  return n;
}
}  // namespace

int sgemm_simt_ctas_per_sm(bool trans_b, bool vec) {
  if (vec) return trans_b ? ctas_per_sm_tma<true>() : ctas_per_sm_tma<false>();
  return trans_b ? ctas_per_sm_variant<true, false>() : ctas_per_sm_variant<false, false>();
}

cudaError_t launch_sgemm_simt_small(const SimtParams& p, bool trans_b, bool vec, cudaStream_t s) {
  if (trans_b) return vec ? launch_small_variant<true, true>(p, s) : launch_small_variant<true, false>(p, s);
  return vec ? launch_small_variant<false, true>(p, s) : launch_small_variant<false, false>(p, s);
}

cudaError_t launch_sgemm_simt(const SimtParams& p, bool trans_b, bool vec, cudaStream_t s) {
  if (vec) {
    // Tensor maps over A [batch][M][lda] (box 36 K x 128 rows) and B: [K][ldb] (box 128 N x
    // 32 K rows) or, transposed, [N][ldb] (box 36 K x 128 rows); no swizzle.
    const uint64_t batch = p.batch > 1 ? static_cast<uint64_t>(p.batch) : 1;
    CUtensorMap ma, mb;
    if (!make_tile_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.A, p.K, p.M, p.lda, batch,
                       p.strideA, LDS_K, BM, CU_TENSOR_MAP_SWIZZLE_NONE, 1))
      return cudaErrorInvalidValue;
    const bool okb = trans_b ? make_tile_map(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.B, p.K, p.N,
                                             p.ldb, batch, p.strideB, LDS_K, BN,
                                             CU_TENSOR_MAP_SWIZZLE_NONE, 1)
                             : make_tile_map(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.B, p.N, p.K,
                                             p.ldb, batch, p.strideB, BN, BK,
                                             CU_TENSOR_MAP_SWIZZLE_NONE, 1);
    if (!okb) return cudaErrorInvalidValue;
    const bool sk = p.sk_ctas > 0;
#define DG_TMA_CASE(TB, R3, SK) \
    if (trans_b == TB && (batch > 1) == R3 && sk == SK) return launch_tma_variant<TB, R3, SK>(ma, mb, p, s);
    DG_TMA_CASE(false, false, false)
    DG_TMA_CASE(true, false, false)
    DG_TMA_CASE(false, true, false)
    DG_TMA_CASE(true, true, false)
    DG_TMA_CASE(false, false, true)
    DG_TMA_CASE(true, false, true)
    DG_TMA_CASE(false, true, true)
    DG_TMA_CASE(true, true, true)
#undef DG_TMA_CASE
    return cudaErrorInvalidValue;
  }
  return trans_b ? launch_variant<true, false>(p, s) : launch_variant<false, false>(p, s);
}

}  // namespace dg
