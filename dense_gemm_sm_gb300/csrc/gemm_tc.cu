// gemm_tc.cu -- BF16-in / FP32-accumulate GEMM on the 5th-generation tensor cores (sm_103a).
//
// Structure (the pages' ideas, set for tcgen05):
//   * The output is cut into 128 x BN tiles (BN = 256 or 128) and walked by a persistent
//     grid (one CTA per SM) in the grouped raster order of tile_sched.h; the linear tile index
//     is the "fuse the tile grid into one linear index" transform of "Operator & Runtime"
//     section 5.4.2.
//   * Operands move global -> shared with TMA (cp.async.bulk.tensor, 128-byte swizzle)
//     into a STAGES-deep ring guarded by "full" and "empty" mbarriers with byte-counted
//     completion: the producer / consumer warp specialisation of "Operator & Runtime"
//     section 5.1.5 and the async-transaction barrier of the MUSA lesson m11-l5.  The
//     swizzle replaces padding, which a tensor-descriptor copy cannot do (section 5.1.5).
//   * One thread issues tcgen05.mma (M = 128, N = BN, K = 16) into an FP32 accumulator in
//     tensor memory; tcgen05.commit releases each smem stage when its MMAs finish.
//   * Two accumulators in TMEM (2 x BN columns) let the epilogue of tile i overlap the
//     main loop of tile i+1.
//   * Epilogue warps read the accumulator with tcgen05.ld, apply C = alpha*acc + beta*C_old
//     in FP32 and round once to the output type (BF16 nearest-even or FP32), after the
//     whole K reduction ("Operator & Runtime" sections 5.4.2-5.4.3).
//   * When the tiles do not fill the last wave, the tail tiles are computed first, stream-K
//     style: their (tile, K block) units are spread evenly over the CTAs, each CTA stores
//     its partial tile, and the last contributor of a tile (atomic ticket, release/acquire
//     fences) adds the partials in CTA (= K) order -- a fixed order, so results repeat run
//     to run ("Operator & Runtime" section 5.2.4).  Done first, these combines overlap the
//     whole-wave tiles that follow instead of extending the kernel.
//   * Every mbarrier wait is bounded; a CTA that gives up records an error in the status
//     word, waits (bounded) for its in-flight copies and MMAs, frees TMEM and exits.
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2-5 = epilogue (warp w reads TMEM lanes 32*(w%4) .. 32*(w%4)+31).
#include <cuda_bf16.h>

#include <cstring>
#include <mutex>
#include <unordered_map>

#include "dg_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dg {
namespace {

constexpr int BM = kTcBM, BK = kTcBK;
constexpr uint32_t A_BYTES = BM * BK * 2;  // 16 KiB per stage
constexpr int NUM_THREADS = 192;

template <int BN, bool B_KMAJOR>
struct TcCfg {
  // N-major B arrives as 64-column boxes (8 KiB each), K-major B as one BN-row box.
  static constexpr int NBOX = (BN + 63) / 64;
  static constexpr uint32_t B_BYTES = NBOX * 8192;  // stage footprint
  static constexpr uint32_t B_LOAD_BYTES = B_KMAJOR ? BN * BK * 2 : NBOX * 8192;  // expect_tx
  static constexpr int STAGES = BN >= 192 ? 4 : 6;
  // Two accumulators of BN columns; the allocation is a power of two.
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr uint32_t RING_BYTES = STAGES * (A_BYTES + B_BYTES);
  // Epilogue staging for TMA stores: 4 warps x 2 buffers x (32 rows x 128 bytes).
  static constexpr uint32_t STAGE_OUT_BYTES = 4 * 2 * 4096;
  static constexpr uint32_t BAR_BYTES = 256;
  static constexpr uint32_t SMEM_BYTES =
      1024 /*alignment slack*/ + RING_BYTES + STAGE_OUT_BYTES + BAR_BYTES;
  static_assert(BN % 32 == 0 && BN <= 256 && 2 * BN <= 512, "tile width");
};

struct SmemCtl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t is_last;
};

// One item of a CTA's work: K blocks [kbeg, kend) of output tile `tile` (raster order).
struct TcItem {
  int64_t tile;
  int32_t kbeg, kend;
  bool sk;  // a stream-K piece of a tail tile
};

// The work of CTA c, in order: its stream-K pieces of the tail tiles, then its whole-wave
// tiles c, c + G, c + 2G, ... below dp_tiles.
struct TcWalk {
  int64_t u, u1, t, step;
  __device__ TcWalk(const TcParams& p, int64_t c, int64_t G) : t(c), step(G) {
    const int64_t units = p.sk_tiles * p.kblocks;
    if (c < p.sk_ctas) {
      u = sk_start<int64_t>(c, units, p.sk_ctas);
      u1 = sk_start<int64_t>(c + 1, units, p.sk_ctas);
    } else {
      u = u1 = 0;
    }
  }
  __device__ bool next(const TcParams& p, TcItem* it) {
    if (u < u1) {
      const int64_t kb = p.kblocks;
      const int64_t st = u / kb;
      const int64_t lim = u1 - st * kb;
      it->tile = p.dp_tiles + st;
      it->kbeg = static_cast<int32_t>(u - st * kb);
      it->kend = static_cast<int32_t>(lim < kb ? lim : kb);
      it->sk = true;
      u = st * kb + it->kend;
      return true;
    }
    if (t < p.dp_tiles) {
      it->tile = t;
      it->kbeg = 0;
      it->kend = p.kblocks;
      it->sk = false;
      t += step;
      return true;
    }
    return false;
  }
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, uint32_t* status) {
  uint32_t never = 0;
  return mbar_wait(bar, parity, &never, status, kDevTimeoutDrain);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Writes 32 consecutive outputs of one row: out[j] = alpha*acc[j] + beta*old[j], j < 32,
// columns gn0 .. gn0+31 (masked against N).
__device__ __forceinline__ void store_row_chunk(const TcParams& p, void* crow_v, int64_t gn0,
                                                const uint32_t (&r)[32]) {
  const float alpha = p.alpha, beta = p.beta;
  const bool full = p.c_vec && gn0 + 32 <= p.N;
  if (p.c_f32) {
    float* crow = static_cast<float*>(crow_v) + gn0;
    if (full) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (beta != 0.f) o = reinterpret_cast<const float4*>(crow)[q];
        float4 v;
        v.x = fmaf(alpha, __uint_as_float(r[4 * q + 0]), beta * o.x);
        v.y = fmaf(alpha, __uint_as_float(r[4 * q + 1]), beta * o.y);
        v.z = fmaf(alpha, __uint_as_float(r[4 * q + 2]), beta * o.z);
        v.w = fmaf(alpha, __uint_as_float(r[4 * q + 3]), beta * o.w);
        reinterpret_cast<float4*>(crow)[q] = v;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (gn0 + j < p.N) {
          const float a = __uint_as_float(r[j]);
          crow[j] = beta != 0.f ? fmaf(alpha, a, beta * crow[j]) : alpha * a;
        }
      }
    }
  } else {
    __nv_bfloat16* crow = static_cast<__nv_bfloat16*>(crow_v) + gn0;
    if (full) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (beta != 0.f) o = reinterpret_cast<const uint4*>(crow)[q];
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float a0 = __uint_as_float(r[8 * q + 2 * h]);
          const float a1 = __uint_as_float(r[8 * q + 2 * h + 1]);
          w[h] = pack_bf16x2(fmaf(alpha, a0, beta * bf16_lo(ow[h])),
                             fmaf(alpha, a1, beta * bf16_hi(ow[h])));
        }
        reinterpret_cast<uint4*>(crow)[q] = make_uint4(w[0], w[1], w[2], w[3]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (gn0 + j < p.N) {
          const float a = __uint_as_float(r[j]);
          const float v = beta != 0.f ? fmaf(alpha, a, beta * __bfloat162float(crow[j])) : alpha * a;
          crow[j] = __float2bfloat16_rn(v);
        }
      }
    }
  }
}

// B3D: N-major B is read through a 3-D view (64 columns, K rows, 64-column chunks), so one
// TMA copy brings a stage's whole B tile instead of one per 64-column box (the copies per
// stage, not the bytes, were the producer's limit).  Only when N is a multiple of 64.
template <int BN, bool B_KMAJOR, bool RANK3, bool B3D>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p, const int fault) {
  using Cfg = TcCfg<BN, B_KMAJOR>;
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;            // 1024-byte aligned swizzle atoms
  const uint32_t a_ring = ring;
  const uint32_t b_ring = ring + STAGES * A_BYTES;
  const uint32_t out_stage = ring + Cfg::RING_BYTES;  // 1024-byte aligned
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem_raw + (ring - raw) + Cfg::RING_BYTES +
                                            Cfg::STAGE_OUT_BYTES);
  volatile uint32_t* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), 4);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ctl->is_last = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (p.c_tma) tma_prefetch_map(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // Only shared memory, TMEM and parameters above: this may overlap the previous kernel.
  pdl_trigger();
  pdl_wait();

  const int kblocks = p.kblocks;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      TcWalk walk(p, blockIdx.x, gridDim.x);
      TcItem item;
      while (ok && walk.next(p, &item)) {
        int64_t b, tm, tn;
        raster_tile(item.tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
        const int32_t ym = static_cast<int32_t>(tm * BM);
        const int32_t xn = static_cast<int32_t>(tn * BN);
        const int32_t zb = static_cast<int32_t>(b);
        for (int kb = item.kbeg; kb < item.kend; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, A_BYTES + Cfg::B_LOAD_BYTES);
          const int32_t kx = kb * BK;
          const uint32_t adst = a_ring + s * A_BYTES, bdst = b_ring + s * Cfg::B_BYTES;
          if (RANK3) tma_load_3d(adst, &tmA, fb, kx, ym, zb);
          else tma_load_2d(adst, &tmA, fb, kx, ym);
          if (B_KMAJOR) {
            if (RANK3) tma_load_3d(bdst, &tmB, fb, kx, xn, zb);
            else tma_load_2d(bdst, &tmB, fb, kx, xn);
          } else if (B3D) {
            tma_load_3d(bdst, &tmB, fb, 0, kx, xn / 64);
          } else {
#pragma unroll
            for (int j = 0; j < Cfg::NBOX; ++j) {
              if (RANK3) tma_load_3d(bdst + j * 8192u, &tmB, fb, xn + 64 * j, kx, zb);
              else tma_load_2d(bdst + j * 8192u, &tmB, fb, xn + 64 * j, kx);
            }
          }
          ++it;
        }
      }
      if (!ok) {
        // Do not leave copies landing in shared memory after exit.
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_drain(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1u, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, false, !B_KMAJOR);
      uint32_t it = 0, lt = 0;
      bool ok = true;
      TcWalk walk(p, blockIdx.x, gridDim.x);
      TcItem item;
      for (; ok && walk.next(p, &item); ++lt) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        if (!mbar_wait(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort, p.status, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = item.kbeg; kb < item.kend; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = a_ring + s * A_BYTES, b0 = b_ring + s * Cfg::B_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            // A (K-major, 128B swizzle): K step of 16 elements = 32 bytes inside the atom.
            const uint64_t adesc = sdesc_sw128(a0 + k * 32, 16, 1024);
            // B: K-major like A, or N-major: 64-column atoms 8 KiB apart (LBO), 8-row
            // groups 1 KiB apart (SBO), K step of 16 rows = 2 KiB.
            const uint64_t bdesc = B_KMAJOR ? sdesc_sw128(b0 + k * 32, 16, 1024)
                                            : sdesc_sw128(b0 + k * 2048, 8192, 1024);
            umma_bf16(d, adesc, bdesc, idesc, (kb > item.kbeg || k > 0) ? 1u : 0u);
          }
          if (fault != 1) umma_commit(smem_u32(&ctl->empty[s]));
          ++it;
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctl->tfull[acc]));
      }
      // All MMAs of this CTA finished before TMEM is released.
      umma_commit(smem_u32(&ctl->drain));
      wait_drain(smem_u32(&ctl->drain), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int row = q * 32 + lane;
    // Two 4 KiB staging buffers per warp for the TMA-store path (32 rows x 128 bytes each,
    // 128-byte swizzled like the tensor map's box).
    const uint32_t stg = out_stage + static_cast<uint32_t>(warp - 2) * 8192u;
    uint32_t sbuf = 0;
    uint32_t lt = 0;
    const int etid = threadIdx.x - 64;
    TcWalk walk(p, blockIdx.x, gridDim.x);
    TcItem item;
    for (; walk.next(p, &item); ++lt) {
      int64_t b, tm, tn;
      raster_tile(item.tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
      const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
      if (!mbar_wait(smem_u32(&ctl->tfull[acc]), aph, abort, p.status, kDevTimeoutEpilogue)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (item.sk && !(item.kbeg == 0 && item.kend == kblocks)) {
        // Stream-K piece of a tail tile: publish the partial tile, then take a ticket; the
        // last contributor adds the partials in CTA order and writes C.
        const int64_t kb = kblocks;
        const int64_t units = p.sk_tiles * kb, ctas = p.sk_ctas;
        const int64_t st = item.tile - p.dp_tiles;
        const int64_t c = blockIdx.x;
        float4* const ws4 = reinterpret_cast<float4*>(p.ws);
        // Partial of CTA cc: [BN / 4 column groups][128 rows] float4, so a warp's stores and
        // loads of one group cover 512 contiguous bytes.
        auto part_of = [&](int64_t cc) {
          const int sl = sk_slot<int64_t>(cc, st, kb, units, ctas);
          return ws4 + (cc * 2 + sl) * (BN / 4) * BM + row;
        };
        {
          float4* dst = part_of(c);
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + ch * 32, r);
            tmem_ld_wait();
#pragma unroll
            for (int g = 0; g < 8; ++g)
              __stcg(dst + (ch * 8 + g) * BM,
                     make_float4(__uint_as_float(r[4 * g]), __uint_as_float(r[4 * g + 1]),
                                 __uint_as_float(r[4 * g + 2]), __uint_as_float(r[4 * g + 3])));
          }
        }
        // The accumulator is in the workspace now: hand TMEM back to the MMA issuer.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
        // The barrier orders the 128 threads' stores before thread 0's release fence, and the
        // fence (cumulative) orders them before the ticket; the last contributor's acquire
        // fence orders the others' partials before its loads.
        epi_bar();
        if (etid == 0) {
          const uint32_t need = static_cast<uint32_t>(sk_contributors<int64_t>(st, kb, units, ctas));
          fence_acq_rel_gpu();
          const uint32_t prev = atomicAdd(&p.counters[st], 1u);
          const bool is_last = prev + 1u == need;
          if (is_last) {
            fence_acq_rel_gpu();
            p.counters[st] = 0u;  // every contributor holds its ticket: ready for the next call
          }
          ctl->is_last = is_last ? 1u : 0u;
        }
        epi_bar();
        if (ctl->is_last) {
          const int64_t first = sk_cta_of<int64_t>(st * kb, units, ctas);
          const int64_t lastc = sk_cta_of<int64_t>((st + 1) * kb - 1, units, ctas);
          const int64_t gm = tm * BM + row;
          uint8_t* cbase = static_cast<uint8_t*>(p.C) +
                           (b * p.strideC + gm * p.ldc) * (p.c_f32 ? 4 : 2);
#pragma unroll 1
          for (int ch = 0; ch < BN / 32; ++ch) {
            float sum[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[j] = 0.f;
            // Contributors in CTA order, two per round trip.
            for (int64_t cc = first; cc <= lastc; cc += 2) {
              const bool two = cc + 1 <= lastc;
              const float4* pa = part_of(cc) + ch * 8 * BM;
              const float4* pb = two ? part_of(cc + 1) + ch * 8 * BM : pa;
              float4 va[8], vb[8];
#pragma unroll
              for (int g = 0; g < 8; ++g) va[g] = __ldcg(pa + g * BM);
              if (two) {
#pragma unroll
                for (int g = 0; g < 8; ++g) vb[g] = __ldcg(pb + g * BM);
              }
#pragma unroll
              for (int g = 0; g < 8; ++g) {
                sum[4 * g] += va[g].x; sum[4 * g + 1] += va[g].y;
                sum[4 * g + 2] += va[g].z; sum[4 * g + 3] += va[g].w;
              }
              if (two) {
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  sum[4 * g] += vb[g].x; sum[4 * g + 1] += vb[g].y;
                  sum[4 * g + 2] += vb[g].z; sum[4 * g + 3] += vb[g].w;
                }
              }
            }
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(sum[j]);
            if (gm < p.M) store_row_chunk(p, cbase, tn * BN + ch * 32, r);
          }
        }
        epi_bar();  // is_last is rewritten only after everyone read it
        continue;
      }
      if (p.c_tma) {
        // C = alpha * acc, in pieces of 32 rows x 32 columns: registers -> swizzled shared
        // staging -> one TMA tensor store (rows / columns beyond M / N are clipped).  An FP32
        // piece is 32 x 128 bytes (128-byte swizzle), a BF16 piece 32 x 64 bytes (64-byte).
        const int32_t y = static_cast<int32_t>(tm * BM + q * 32);
        const int32_t zb = static_cast<int32_t>(b);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t w[32];
          tmem_ld_32x32b_x32(taddr + c * 32, w);
          tmem_ld_wait();
          if (c == BN / 32 - 1) {
            // The accumulator is in registers now: hand TMEM back to the MMA issuer.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
          }
          // The store issued from this buffer two pieces ago must have finished reading it.
          if (lane == 0) bulk_wait_read<1>();
          __syncwarp();
          const uint32_t buf = stg + sbuf * 4096u;
          if (p.c_f32) {
            const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              const float a0 = p.alpha * __uint_as_float(w[4 * j]);
              const float a1 = p.alpha * __uint_as_float(w[4 * j + 1]);
              const float a2 = p.alpha * __uint_as_float(w[4 * j + 2]);
              const float a3 = p.alpha * __uint_as_float(w[4 * j + 3]);
              st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ (lane & 7u)) << 4),
                           __float_as_uint(a0), __float_as_uint(a1), __float_as_uint(a2),
                           __float_as_uint(a3));
            }
          } else {
            const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 64u;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                h[e] = pack_bf16x2(p.alpha * __uint_as_float(w[8 * j + 2 * e]),
                                   p.alpha * __uint_as_float(w[8 * j + 2 * e + 1]));
              st_shared_v4(rowaddr + ((static_cast<uint32_t>(j) ^ ((lane >> 1) & 3u)) << 4), h[0],
                           h[1], h[2], h[3]);
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int32_t x = static_cast<int32_t>(tn * BN + c * 32);
            if (y < p.M && x < p.N) {  // skip pieces wholly outside C
              if (RANK3) tma_store_3d(&tmC, buf, x, y, zb);
              else tma_store_2d(&tmC, buf, x, y);
            }
            bulk_commit();
          }
          sbuf ^= 1u;
        }
      } else {
        const int64_t gm = tm * BM + row;
        uint8_t* cbase = static_cast<uint8_t*>(p.C) +
                         (b * p.strideC + gm * p.ldc) * (p.c_f32 ? 4 : 2);
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          tmem_ld_wait();
          if (gm < p.M) store_row_chunk(p, cbase, tn * BN + c * 32, r);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
      }
    }
    // Stores must have finished reading shared memory (and landed) before the CTA exits.
    if (p.c_tma && lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

EncodeTiledFn get_encode_tiled();

namespace {
struct MapKey {
  const void* base;
  uint64_t inner, outer, ld, batch, stride;
  uint32_t box_inner, box_outer;
  bool operator==(const MapKey& o) const { return std::memcmp(this, &o, sizeof(MapKey)) == 0; }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    uint64_t h = reinterpret_cast<uintptr_t>(k.base);
    const uint64_t v[7] = {k.inner, k.outer, k.ld, k.batch, k.stride, k.box_inner, k.box_outer};
    for (uint64_t x : v) h = (h ^ x) * 0x100000001B3ull;
    return static_cast<size_t>(h);
  }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;
}  // namespace

// Builds a tensor map over a (batch x) outer x inner row-major view of elements of `esz`
// bytes with a box_inner x box_outer box and 128-byte swizzle.  Out-of-range elements read
// as zero (and are not written by stores).  Encoded maps are cached by (address, shape,
// type, box): repeated calls on the same buffers (the usual inference loop) skip the
// encoding on the launch path.
bool make_tile_map(CUtensorMap* map, CUtensorMapDataType dtype, uint32_t esz, const void* base,
                   uint64_t inner, uint64_t outer, uint64_t ld, uint64_t batch, uint64_t stride,
                   uint32_t box_inner, uint32_t box_outer,
                   CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B, uint32_t box_batch = 1) {
  MapKey key;
  std::memset(&key, 0, sizeof key);
  key.base = base; key.inner = inner; key.outer = outer; key.ld = ld;
  key.batch = batch > 1 ? batch : 1; key.stride = batch > 1 ? stride : 0;
  key.box_inner = box_inner | (static_cast<uint32_t>(dtype) << 16);
  key.box_outer = box_outer | (static_cast<uint32_t>(swizzle) << 16) | (box_batch << 20);
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    auto it = g_map_cache.find(key);
    if (it != g_map_cache.end()) {
      *map = it->second;
      return true;
    }
  }
  static EncodeTiledFn fn = get_encode_tiled();
  if (!fn) return false;
  const bool rank3 = batch > 1;
  cuuint64_t dims[3] = {inner, outer, batch};
  cuuint64_t strides[2] = {ld * esz, stride * esz};
  cuuint32_t box[3] = {box_inner, box_outer, box_batch};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, dtype, rank3 ? 3 : 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  if (g_map_cache.size() >= 4096) g_map_cache.clear();
  g_map_cache.emplace(key, *map);
  return true;
}

bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint64_t batch, uint64_t stride, uint32_t box_inner, uint32_t box_outer) {
  return make_tile_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, inner, outer, ld, batch,
                       stride, box_inner, box_outer);
}

EncodeTiledFn get_encode_tiled() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<EncodeTiledFn>(p);
}

namespace {
template <int BN, bool B_KMAJOR, bool RANK3, bool B3D = false>
cudaError_t launch_tc_variant(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mc,
                              const TcParams& p, int num_ctas, cudaStream_t s) {
  auto kern = gemm_tc_kernel<BN, B_KMAJOR, RANK3, B3D>;
  constexpr uint32_t smem = TcCfg<BN, B_KMAJOR>::SMEM_BYTES;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(num_ctas), dim3(NUM_THREADS), smem, s, ma, mb, mc, p,
                    g_fault_injection);
}
}  // namespace

cudaError_t launch_gemm_tc(const TcParams& p, int bn, const void* A, int64_t lda, int64_t strideA,
                           const void* B, int64_t ldb, int64_t strideB, bool b_kmajor,
                           int num_ctas, cudaStream_t s) {
  CUtensorMap ma, mb;
  const uint64_t batch = static_cast<uint64_t>(p.batch);
  if (!make_bf16_map(&ma, A, p.K, p.M, lda, batch, strideA, BK, BM)) return cudaErrorInvalidValue;
  // N-major B as one 3-D box per stage when the 64-column chunks tile N exactly (so no box
  // reaches past a row) and the tile width is whole chunks.
  const bool b3d = !b_kmajor && batch <= 1 && p.N % 64 == 0 && bn % 64 == 0 && p.N >= bn;
  bool ok_b;
  if (b_kmajor)
    ok_b = make_bf16_map(&mb, B, p.K, p.N, ldb, batch, strideB, BK, bn);
  else if (b3d)
    ok_b = make_tile_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, 64, p.K, ldb,
                         static_cast<uint64_t>(p.N / 64), 64, 64, BK, CU_TENSOR_MAP_SWIZZLE_128B,
                         static_cast<uint32_t>(bn / 64));
  else
    ok_b = make_bf16_map(&mb, B, p.N, p.K, ldb, batch, strideB, 64, BK);
  if (!ok_b) return cudaErrorInvalidValue;
  CUtensorMap mc;
  std::memset(&mc, 0, sizeof mc);
  TcParams q = p;
  if (q.c_tma) {
    // Stores of 32 rows x 32 columns: 128-byte FP32 rows, 64-byte BF16 rows.
    const bool ok_c = q.c_f32 ? make_tile_map(&mc, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, q.C, q.N, q.M,
                                              q.ldc, batch, q.strideC, 32, 32,
                                              CU_TENSOR_MAP_SWIZZLE_128B)
                              : make_tile_map(&mc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q.C, q.N,
                                              q.M, q.ldc, batch, q.strideC, 32, 32,
                                              CU_TENSOR_MAP_SWIZZLE_64B);
    if (!ok_c) q.c_tma = 0;  // fall back to direct stores from registers
  }
  const bool rank3 = batch > 1;
  if (b3d) {
    if (bn == 256) return launch_tc_variant<256, false, false, true>(ma, mb, mc, q, num_ctas, s);
    if (bn == 192) return launch_tc_variant<192, false, false, true>(ma, mb, mc, q, num_ctas, s);
    if (bn == 128) return launch_tc_variant<128, false, false, true>(ma, mb, mc, q, num_ctas, s);
  }
#define DG_TC_CASE(BNV, KM, R3)                                                     \
  if (bn == BNV && b_kmajor == KM && rank3 == R3)                                   \
    return launch_tc_variant<BNV, KM, R3>(ma, mb, mc, q, num_ctas, s);
  DG_TC_CASE(256, false, false)
  DG_TC_CASE(256, false, true)
  DG_TC_CASE(256, true, false)
  DG_TC_CASE(256, true, true)
  DG_TC_CASE(224, false, false)
  DG_TC_CASE(224, false, true)
  DG_TC_CASE(224, true, false)
  DG_TC_CASE(224, true, true)
  DG_TC_CASE(192, false, false)
  DG_TC_CASE(192, false, true)
  DG_TC_CASE(192, true, false)
  DG_TC_CASE(192, true, true)
  DG_TC_CASE(128, false, false)
  DG_TC_CASE(128, false, true)
  DG_TC_CASE(128, true, false)
  DG_TC_CASE(128, true, true)
#undef DG_TC_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dg
