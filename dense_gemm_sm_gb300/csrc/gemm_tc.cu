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

// PAIR: a CTA pair (cluster of 2) computes a 256 x BN tile with tcgen05.mma.cta_group::2;
// each CTA holds its 128 rows of A and BN / 2 columns of B, so a stage is half as large.
// A stage holds KA K atoms of 128 bytes per row (64 BF16 or 128 FP8 elements each): BF16 pairs
// take two (8 MMAs per stage), the rest one.  Every stage costs the MMA issuer a barrier wait,
// a fence and a commit that the tensor pipe does not hide: measured without operand loads, the
// FFN's stage took ~240 cycles beyond its 4 MMAs in BF16, added in full when the stage's MMAs
// were doubled; two atoms per stage pay it half as often (4096^3 1707 -> 1741 TFLOPS, gate/up
// 1633 -> 1662, FFN equal).  FP8 pairs keep one atom and six stages: with three stages of two
// atoms the FFN shape lost 2% (2537 -> 2480 TFLOPS).
template <int BN, bool B_KMAJOR, bool PAIR = false, bool FP8 = false>
struct TcCfg {
  static constexpr int BNC = PAIR ? BN / 2 : BN;  // B columns held by this CTA
  static constexpr int KA = PAIR && !FP8 ? 2 : 1;  // K atoms per stage
  static constexpr uint32_t A_STAGE = KA * A_BYTES;
  // N-major B arrives as 64-column boxes (8 KiB per atom each), K-major B as one BNC-row box
  // per atom.
  static constexpr int NBOX = (BNC + 63) / 64;
  static constexpr uint32_t B_ATOM = NBOX * 8192;   // one atom's footprint
  static constexpr uint32_t B_BYTES = KA * B_ATOM;  // stage footprint
  static constexpr uint32_t B_LOAD_BYTES = KA * (B_KMAJOR ? BNC * BK * 2 : NBOX * 8192);  // expect_tx
  static constexpr int STAGES = PAIR ? (KA == 2 ? 3 : 6) : (BN >= 192 ? 4 : 6);
  // Two accumulators of BN columns; the allocation is a power of two.
  static constexpr uint32_t TMEM_COLS = 2 * BN <= 256 ? 256 : 512;
  static constexpr uint32_t RING_BYTES = STAGES * (A_STAGE + B_BYTES);
  // Epilogue staging for TMA stores: 4 warps x 2 buffers x (32 rows x 128 bytes).
  static constexpr uint32_t STAGE_OUT_BYTES = 4 * 2 * 4096;
  static constexpr uint32_t BAR_BYTES = 256;
  static constexpr uint32_t SMEM_BYTES =
      1024 /*alignment slack*/ + RING_BYTES + STAGE_OUT_BYTES + BAR_BYTES;
  static_assert(BN % 32 == 0 && BN <= 256 && 2 * BN <= 512, "tile width");
};

struct SmemCtl;
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
static_assert(sizeof(SmemCtl) <= 256, "barrier block");

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

// ---------------------------------------------------------------- CTA-pair (cluster of 2)
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                   "memory");
}

// Arrives (release, cluster scope) on the barrier at the same shared-memory offset in CTA
// `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(bar), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// mbar_wait for a barrier that the peer CTA arrives on: acquire at cluster scope.  Bounded
// like mbar_wait.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  volatile uint32_t* abort, uint32_t* status,
                                                  uint32_t code) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicCAS(status, 0u, code);
        return false;
      }
    }
  }
}

// TMA loads into this CTA's shared memory whose completion counts on `bar`, a shared::cluster
// barrier address that may be the pair peer's (rank 1 signals rank 0's stage barrier).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                 int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t local, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local), "r"(rank));
  return a;
}

// tcgen05 forms for the pair (every tcgen05 instruction of a kernel uses one CTA group).
__device__ __forceinline__ void tmem_alloc2(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish2() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc2(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void umma2_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives on the barrier at this offset in both CTAs of the pair once the issuing thread's
// earlier MMAs have completed.
__device__ __forceinline__ void umma2_commit_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(bar), "h"(static_cast<uint16_t>(3))
      : "memory");
}
__device__ __forceinline__ void umma2_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// FP8 (E4M3 x E4M3 -> FP32) forms: kind::f8f6f4, K = 32 per instruction (32 bytes of K, as
// for BF16), so the shared-memory descriptors and their K steps are the BF16 ones.
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma2_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Instruction descriptor for kind::f8f6f4 with E4M3 A and B (format code 0) and FP32 D;
// the other fields as idesc_bf16_f32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t m, uint32_t n, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((n >> 3) << 17) | ((m >> 4) << 24);
}

// FP8 epilogue: acc[i][j] * scale_a[i] * scale_b[j] for the 32 columns gn0 .. gn0+31 of row
// gm (columns past N get scale 0; they are not stored).
__device__ __forceinline__ void fp8_scale(uint32_t (&r)[32], const TcParams& p, int64_t gm,
                                          int64_t gn0) {
  const float sa = gm < p.M ? __ldg(p.scale_a + gm) : 0.f;
  float sb[32];
  if (gn0 + 32 <= p.N) {
    const float4* s4 = reinterpret_cast<const float4*>(p.scale_b + gn0);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 v = __ldg(s4 + q);
      sb[4 * q] = v.x; sb[4 * q + 1] = v.y; sb[4 * q + 2] = v.z; sb[4 * q + 3] = v.w;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) sb[j] = gn0 + j < p.N ? __ldg(p.scale_b + gn0 + j) : 0.f;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) r[j] = __float_as_uint((__uint_as_float(r[j]) * sa) * sb[j]);
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

// FFN activation chain ("Operator & Runtime" sections 5.3.1 and 5.4.3): z = SiLU(G) * U
// with G and U rounded to BF16 first (the unfused program stores them as BF16), SiLU(x) =
// x / (1 + e^-x) and the product in FP32; the store rounds z to BF16 once more.
__device__ __forceinline__ void silu_mul_bf16(uint32_t (&g)[32], const uint32_t (&u)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const float gb = __bfloat162float(__float2bfloat16_rn(__uint_as_float(g[j])));
    const float ub = __bfloat162float(__float2bfloat16_rn(__uint_as_float(u[j])));
    g[j] = __float_as_uint(gb / (1.f + expf(-gb)) * ub);
  }
}
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
//
// PAIR (launched as clusters of 2): tile i of the walk is a 256 x BN tile; CTA rank r of the
// pair computes its rows 128r .. 128r + 127 into its own TMEM, from its own A rows and with
// B split by columns between the two CTAs' shared memories.  Rank 0 issues the MMAs for both
// (tcgen05.mma.cta_group::2) once both CTAs' stage has landed (rank 1's copies count on rank
// 0's stage barrier), and its commits reach the stage and accumulator barriers of both CTAs.  Each CTA's epilogue writes its own rows;
// both hand the accumulator back to rank 0.  Halving each CTA's B halves the bytes that
// move through each SM's shared memory per FLOP (TMA writes plus MMA reads), which bounds
// the single-CTA tile.
//
// DUAL (FFN gate and up projections): B is [W_g tile | W_u tile], BN / 2 columns each, so the
// accumulator holds G and U side by side; the epilogue writes z = SiLU(bf16(G)) * bf16(U),
// BN / 2 output columns per tile.  Pair: rank 0 holds the W_g tile and rank 1 the W_u tile.
//
// FP8: A and B are E4M3 codes (K-major, 128 codes = 128 bytes per stage row, so a stage holds
// 128 K elements), the MMA is kind::f8f6f4, and the epilogue scales the accumulator by the
// per-row scale of A and the per-column scale of op(B) (alpha = 1, beta = 0).
template <int BN, bool B_KMAJOR, bool RANK3, bool B3D, bool PAIR, bool DUAL, bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                   const TcParams p, const int fault) {
  using Cfg = TcCfg<BN, B_KMAJOR, PAIR, FP8>;
  static_assert(!PAIR || ((BN == 256 || (BN == 224 && FP8)) && !RANK3),
                "pair tiles are 256 x 256 (FP8 also 256 x 224), one problem");
  static_assert(!DUAL || (BN == 256 && !B_KMAJOR && !RANK3), "gate/up: 2 x 128 columns, N-major");
  static_assert(!FP8 || (B_KMAJOR && !RANK3 && !DUAL), "FP8: one problem, K-major B");
  constexpr int ATOM_K = FP8 ? 128 : BK;           // K elements per 128-byte atom row
  constexpr int KA = Cfg::KA;
  constexpr int BK_ELEMS = KA * ATOM_K;            // K elements per stage
  constexpr int OUT_N = DUAL ? BN / 2 : BN;  // output columns per tile
  constexpr int STAGES = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;            // 1024-byte aligned swizzle atoms
  const uint32_t a_ring = ring;
  const uint32_t b_ring = ring + STAGES * Cfg::A_STAGE;
  const uint32_t out_stage = ring + Cfg::RING_BYTES;  // 1024-byte aligned
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem_raw + (ring - raw) + Cfg::RING_BYTES +
                                            Cfg::STAGE_OUT_BYTES);
  volatile uint32_t* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Pair: rank in the cluster, the pair's index and count; otherwise the CTA's.
  const uint32_t rank = PAIR ? cluster_rank() : 0u;
  const int64_t cid = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t ncl = PAIR ? (gridDim.x >> 1) : gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&ctl->tfull[a]), 1);
      mbar_init(smem_u32(&ctl->tempty[a]), PAIR ? 8 : 4);  // pair: both CTAs' epilogue warps
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    ctl->is_last = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if (PAIR) {
      tmem_alloc2(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);  // one warp of each CTA, together
      tmem_relinquish2();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);
      tmem_relinquish();
    }
  }
  if (threadIdx.x == 0) {
    tma_prefetch_map(&tmA);
    tma_prefetch_map(&tmB);
    if (DUAL) tma_prefetch_map(&tmB2);
    if (p.c_tma) tma_prefetch_map(&tmC);
  }
  tc_fence_before();
  __syncthreads();
  // Pair: both CTAs' barriers are initialised and TMEM allocated before either signals the
  // other or issues an MMA into it.
  if (PAIR) cluster_sync();
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
      TcWalk walk(p, cid, ncl);
      TcItem item;
      while (ok && walk.next(p, &item)) {
        int64_t b, tm, tn;
        raster_tile(item.tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
        if (PAIR) tm = 2 * tm + rank;  // pair row -> this CTA's 128-row tile
        const int32_t ym = static_cast<int32_t>(tm * BM);
        // This CTA's B columns (gate/up: the output tile's columns in W_g and W_u).
        const int32_t xn = static_cast<int32_t>(DUAL ? tn * OUT_N : tn * BN + rank * Cfg::BNC);
        const CUtensorMap* mb1 = (DUAL && PAIR && rank == 1) ? &tmB2 : &tmB;
        const int32_t zb = static_cast<int32_t>(b);
        for (int kb = item.kbeg; kb < item.kend; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) {
            ok = false;
            break;
          }
          const int32_t kx = kb * BK_ELEMS;
          const uint32_t adst = a_ring + s * Cfg::A_STAGE, bdst = b_ring + s * Cfg::B_BYTES;
          if (PAIR) {
            // Both CTAs' loads of stage s count on rank 0's full[s]; rank 0 posts the bytes
            // of both (a load may land before the post: the count is signed within a phase).
            // A and K-major B: one box per atom, the atoms B_ATOM / 16 KiB apart; N-major B:
            // 64-column boxes KA atoms deep (KA * 64 rows of K), chunks KA * 8 KiB apart.
            const uint32_t fb = cluster_addr(smem_u32(&ctl->full[s]), 0u);
            if (rank == 0) mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), 2 * (Cfg::A_STAGE + Cfg::B_LOAD_BYTES));
#pragma unroll
            for (int a = 0; a < KA; ++a) tma_load_2d_pair(adst + a * A_BYTES, &tmA, fb, kx + a * ATOM_K, ym);
            if (B_KMAJOR) {
#pragma unroll
              for (int a = 0; a < KA; ++a) tma_load_2d_pair(bdst + a * Cfg::B_ATOM, &tmB, fb, kx + a * ATOM_K, xn);
            } else if (B3D) {
              tma_load_3d_pair(bdst, mb1, fb, 0, kx, xn / 64);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::NBOX; ++j) tma_load_2d_pair(bdst + j * (KA * 8192u), mb1, fb, xn + 64 * j, kx);
            }
            ++it;
            continue;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, Cfg::A_STAGE + Cfg::B_LOAD_BYTES);
          if (RANK3) tma_load_3d(adst, &tmA, fb, kx, ym, zb);
          else tma_load_2d(adst, &tmA, fb, kx, ym);
          if (B_KMAJOR) {
            if (RANK3) tma_load_3d(bdst, &tmB, fb, kx, xn, zb);
            else tma_load_2d(bdst, &tmB, fb, kx, xn);
          } else if (DUAL) {
            // W_g's columns into the first half of the stage's B, W_u's into the second.
            if (B3D) {
              tma_load_3d(bdst, &tmB, fb, 0, kx, xn / 64);
              tma_load_3d(bdst + Cfg::B_BYTES / 2, &tmB2, fb, 0, kx, xn / 64);
            } else {
#pragma unroll
              for (int j = 0; j < Cfg::NBOX / 2; ++j) {
                tma_load_2d(bdst + j * 8192u, &tmB, fb, xn + 64 * j, kx);
                tma_load_2d(bdst + Cfg::B_BYTES / 2 + j * 8192u, &tmB2, fb, xn + 64 * j, kx);
              }
            }
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
      if (!ok && (!PAIR || rank == 0)) {
        // Do not leave copies landing in shared memory after exit (pair: rank 0's stage
        // barriers count both CTAs' copies; the final cluster barrier holds rank 1 until
        // rank 0 has seen them land).
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          wait_drain(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1u, p.status);
      } else if (ok && PAIR) {
        // Rank 0's last commits arrive on this CTA's stage barriers: see them land before
        // the CTA can exit.
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait(smem_u32(&ctl->empty[j % STAGES]), (j / STAGES) & 1u, abort, p.status,
                    kDevTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && (!PAIR || rank == 0)) {
      constexpr uint32_t idesc = FP8 ? idesc_e4m3_f32(PAIR ? 2 * BM : BM, BN, false, !B_KMAJOR)
                                     : idesc_bf16_f32(PAIR ? 2 * BM : BM, BN, false, !B_KMAJOR);
      uint32_t it = 0, lt = 0;
      uint32_t s = 0, ph = 0;  // ring stage of block `it` and its phase parity
      // Operand descriptors of the ring bases, advanced by the start-address field alone
      // (16-byte units; every offset stays inside the 256 KiB the field spans), so an MMA costs
      // the issuing thread a few integer additions.
      const uint64_t dA = sdesc_sw128(a_ring, 16, 1024);
      const uint64_t dB = B_KMAJOR ? sdesc_sw128(b_ring, 16, 1024) : sdesc_sw128(b_ring, KA * 8192, 1024);
      bool ok = true;
      TcWalk walk(p, cid, ncl);
      TcItem item;
      for (; ok && walk.next(p, &item); ++lt) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        const uint32_t te = smem_u32(&ctl->tempty[acc]);
        if (!(PAIR ? mbar_wait_cluster(te, aph ^ 1u, abort, p.status, kDevTimeoutMma)
                   : mbar_wait(te, aph ^ 1u, abort, p.status, kDevTimeoutMma))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        for (int kb = item.kbeg; kb < item.kend; ++kb) {
          // Pair: full[s] counts the bytes of both CTAs' stage s (acquire at cluster scope).
          if (!(PAIR ? mbar_wait_cluster(smem_u32(&ctl->full[s]), ph, abort, p.status, kDevTimeoutMma)
                     : mbar_wait(smem_u32(&ctl->full[s]), ph, abort, p.status, kDevTimeoutMma))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t dAs = dA + ((s * Cfg::A_STAGE) >> 4), dBs = dB + ((s * Cfg::B_BYTES) >> 4);
#pragma unroll
          for (int k = 0; k < KA * (BK / 16); ++k) {
            const int a = k / (BK / 16), kk = k % (BK / 16);  // atom, MMA inside the atom
            // A (K-major, 128B swizzle): atoms 16 KiB apart; K step of one MMA = 32 bytes
            // inside the atom (16 BF16 or 32 FP8 elements).
            const uint64_t adesc = dAs + ((a * A_BYTES + kk * 32) >> 4);
            // B: K-major like A (atoms B_ATOM apart), or N-major: 64-column chunks KA * 8 KiB
            // apart (LBO), 8-row groups 1 KiB apart (SBO), K step of 16 rows = 2 KiB through
            // the KA atoms' rows.  For the pair the same offsets describe each CTA's share.
            const uint64_t bdesc = dBs + ((B_KMAJOR ? a * Cfg::B_ATOM + kk * 32 : k * 2048) >> 4);
            const uint32_t accum = (kb > item.kbeg || k > 0) ? 1u : 0u;
            if (FP8) {
              if (PAIR) umma2_f8(d, adesc, bdesc, idesc, accum);
              else umma_f8(d, adesc, bdesc, idesc, accum);
            } else {
              if (PAIR) umma2_bf16(d, adesc, bdesc, idesc, accum);
              else umma_bf16(d, adesc, bdesc, idesc, accum);
            }
          }
          if (fault != 1) {
            if (PAIR) umma2_commit_both(smem_u32(&ctl->empty[s]));
            else umma_commit(smem_u32(&ctl->empty[s]));
          }
          ++it;
          if (++s == static_cast<uint32_t>(STAGES)) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        if (PAIR) umma2_commit_both(smem_u32(&ctl->tfull[acc]));
        else umma_commit(smem_u32(&ctl->tfull[acc]));
      }
      // All MMAs of this CTA (pair: of both CTAs) finished before TMEM is released.
      if (PAIR) umma2_commit(smem_u32(&ctl->drain));
      else umma_commit(smem_u32(&ctl->drain));
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
    // Hands the accumulator back to the MMA issuer (pair: to rank 0, from both CTAs).
    auto release_acc = [&](uint32_t acc) {
      if (PAIR) mbar_arrive_remote(smem_u32(&ctl->tempty[acc]), 0u);
      else mbar_arrive(smem_u32(&ctl->tempty[acc]));
    };
    TcWalk walk(p, cid, ncl);
    TcItem item;
    for (; walk.next(p, &item); ++lt) {
      int64_t b, tm, tn;
      raster_tile(item.tile, p.tiles_m, p.tiles_n, p.group, &b, &tm, &tn);
      if (PAIR) tm = 2 * tm + rank;
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
        const int64_t c = cid;
        float4* const ws4 = reinterpret_cast<float4*>(p.ws);
        // Partial of contributor cc (pair: cc's CTA of this rank): [BN / 4 column groups][128
        // rows] float4, so a warp's stores and loads of one group cover 512 contiguous bytes.
        auto part_of = [&](int64_t cc) {
          const int sl = sk_slot<int64_t>(cc, st, kb, units, ctas);
          const int64_t who = PAIR ? 2 * cc + rank : cc;
          return ws4 + (who * 2 + sl) * (BN / 4) * BM + row;
        };
        uint32_t* const counter = &p.counters[PAIR ? 2 * st + rank : st];
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
        if (lane == 0) release_acc(acc);
        // The barrier orders the 128 threads' stores before thread 0's release fence, and the
        // fence (cumulative) orders them before the ticket; the last contributor's acquire
        // fence orders the others' partials before its loads.
        epi_bar();
        if (etid == 0) {
          const uint32_t need = static_cast<uint32_t>(sk_contributors<int64_t>(st, kb, units, ctas));
          fence_acq_rel_gpu();
          const uint32_t prev = atomicAdd(counter, 1u);
          const bool is_last = prev + 1u == need;
          if (is_last) {
            fence_acq_rel_gpu();
            *counter = 0u;  // every contributor holds its ticket: ready for the next call
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
          // The contributors' partials of accumulator columns ch*32 .. ch*32+31, in CTA
          // order, two per round trip.
          auto sum_chunk = [&](int ch, float (&sum)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[j] = 0.f;
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
          };
#pragma unroll 1
          for (int ch = 0; ch < OUT_N / 32; ++ch) {
            float sum[32];
            sum_chunk(ch, sum);
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(sum[j]);
            if (DUAL) {
              float usum[32];
              sum_chunk(ch + OUT_N / 32, usum);
              uint32_t u[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(usum[j]);
              silu_mul_bf16(r, u);
            }
            if (FP8) fp8_scale(r, p, gm, tn * OUT_N + ch * 32);
            if (gm < p.M) store_row_chunk(p, cbase, tn * OUT_N + ch * 32, r);
          }
          // The partials are scratch that nothing reads again before the next call rewrites
          // them: drop their L2 lines so they are never written back to DRAM.  A warp drops
          // the lines of its own 32 rows (4 x 128 bytes per column group) once all its lanes
          // have read them.
          __syncwarp();
          for (int64_t cc = first; cc <= lastc; ++cc) {
            const uint8_t* pbase = reinterpret_cast<const uint8_t*>(part_of(cc) - row + q * 32);
#pragma unroll 4
            for (int i = lane; i < (BN / 4) * 4; i += 32)
              discard_l2(pbase + (static_cast<size_t>(i >> 2) * BM * 16) + (i & 3) * 128);
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
        for (int c = 0; c < OUT_N / 32; ++c) {
          uint32_t w[32];
          tmem_ld_32x32b_x32(taddr + c * 32, w);
          if (DUAL) {
            uint32_t u[32];
            tmem_ld_32x32b_x32(taddr + OUT_N + c * 32, u);
            tmem_ld_wait();
            silu_mul_bf16(w, u);
          } else {
            tmem_ld_wait();
          }
          if (FP8) fp8_scale(w, p, tm * BM + row, tn * OUT_N + c * 32);
          if (c == OUT_N / 32 - 1) {
            // The accumulator is in registers now: hand TMEM back to the MMA issuer.
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release_acc(acc);
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
            const int32_t x = static_cast<int32_t>(tn * OUT_N + c * 32);
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
        for (int c = 0; c < OUT_N / 32; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + c * 32, r);
          if (DUAL) {
            uint32_t u[32];
            tmem_ld_32x32b_x32(taddr + OUT_N + c * 32, u);
            tmem_ld_wait();
            silu_mul_bf16(r, u);
          } else {
            tmem_ld_wait();
          }
          if (FP8) fp8_scale(r, p, gm, tn * OUT_N + c * 32);
          if (gm < p.M) store_row_chunk(p, cbase, tn * OUT_N + c * 32, r);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release_acc(acc);
      }
    }
    // Stores must have finished reading shared memory (and landed) before the CTA exits.
    if (p.c_tma && lane == 0) bulk_wait<0>();
  }

  tc_fence_before();
  __syncthreads();
  // Pair: neither CTA frees TMEM or exits while the other may still touch its shared memory
  // or barriers; the TMEM release is collective.
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if (PAIR) tmem_dealloc2(tmem_base, Cfg::TMEM_COLS);
    else tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
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
template <int BN, bool B_KMAJOR, bool RANK3, bool B3D = false, bool PAIR = false, bool DUAL = false,
          bool FP8 = false>
cudaError_t launch_tc_variant(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mb2,
                              const CUtensorMap& mc, const TcParams& p, int num_ctas,
                              cudaStream_t s) {
  auto kern = gemm_tc_kernel<BN, B_KMAJOR, RANK3, B3D, PAIR, DUAL, FP8>;
  constexpr uint32_t smem = TcCfg<BN, B_KMAJOR, PAIR, FP8>::SMEM_BYTES;
  static_assert(smem <= 232448, "shared memory per CTA");
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  if (!PAIR)
    return launch_pdl(kern, dim3(num_ctas), dim3(NUM_THREADS), smem, s, ma, mb, mb2, mc, p,
                      g_fault_injection);
  // Clusters of two CTAs, with programmatic stream serialisation as for the other kernels.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(num_ctas);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, mb2, mc, p, g_fault_injection);
}
}  // namespace

cudaError_t launch_gemm_tc(const TcParams& p, int bn, const void* A, int64_t lda, int64_t strideA,
                           const void* B, int64_t ldb, int64_t strideB, bool b_kmajor,
                           bool pair, int num_ctas, cudaStream_t s, const void* B2,
                           int64_t ldb2, bool fp8) {
  CUtensorMap ma, mb, mb2;
  const uint64_t batch = static_cast<uint64_t>(p.batch);
  const bool dual = B2 != nullptr;
  if (pair && ((bn != 256 && !(fp8 && bn == 224)) || batch > 1 || num_ctas % 2 != 0))
    return cudaErrorInvalidValue;
  if (dual && (bn != 256 || batch > 1 || b_kmajor)) return cudaErrorInvalidValue;
  // B columns one tensor map box set covers: the CTA's share of the tile (the pair splits the
  // tile's columns between its two CTAs; gate/up reads BN / 2 from each of W_g and W_u).
  const int bnc = dual ? bn / 2 : (pair ? bn / 2 : bn);
  if (fp8 && (!b_kmajor || dual || batch > 1)) return cudaErrorInvalidValue;
  // FP8: E4M3 codes as bytes, boxes of 128 codes (128-byte rows) along K.
  if (fp8 ? !make_tile_map(&ma, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, p.K, p.M, lda, 1, 0, 128, BM,
                           CU_TENSOR_MAP_SWIZZLE_128B, 1)
          : !make_bf16_map(&ma, A, p.K, p.M, lda, batch, strideA, BK, BM))
    return cudaErrorInvalidValue;
  // N-major B as one 3-D box per stage when the 64-column chunks tile N exactly (so no box
  // reaches past a row) and the tile width is whole chunks.
  const bool b3d = !fp8 && !b_kmajor && batch <= 1 && p.N % 64 == 0 && bn % 64 == 0 &&
                   p.N >= (dual ? bn / 2 : bn);
  // BF16 pairs stage two K atoms: N-major B boxes are 2 * BK rows of K deep (A and K-major B
  // take one box per atom).
  const uint32_t bk_rows = pair && !fp8 ? 2 * BK : BK;
  bool ok_b;
  if (fp8)
    ok_b = make_tile_map(&mb, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, p.K, p.N, ldb, 1, 0, 128,
                         static_cast<uint32_t>(bnc), CU_TENSOR_MAP_SWIZZLE_128B, 1);
  else if (b_kmajor)
    ok_b = make_bf16_map(&mb, B, p.K, p.N, ldb, batch, strideB, BK, bnc);
  else if (b3d)
    ok_b = make_tile_map(&mb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, 64, p.K, ldb,
                         static_cast<uint64_t>(p.N / 64), 64, 64, bk_rows, CU_TENSOR_MAP_SWIZZLE_128B,
                         static_cast<uint32_t>(bnc / 64));
  else
    ok_b = make_bf16_map(&mb, B, p.N, p.K, ldb, batch, strideB, 64, bk_rows);
  if (!ok_b) return cudaErrorInvalidValue;
  mb2 = mb;
  if (dual) {
    const bool ok_b2 =
        b3d ? make_tile_map(&mb2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B2, 64, p.K, ldb2,
                            static_cast<uint64_t>(p.N / 64), 64, 64, bk_rows,
                            CU_TENSOR_MAP_SWIZZLE_128B, static_cast<uint32_t>(bnc / 64))
            : make_bf16_map(&mb2, B2, p.N, p.K, ldb2, 1, 0, 64, bk_rows);
    if (!ok_b2) return cudaErrorInvalidValue;
  }
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
  if (fp8) {
    if (pair && bn == 224) return launch_tc_variant<224, true, false, false, true, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (pair) return launch_tc_variant<256, true, false, false, true, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (bn == 256) return launch_tc_variant<256, true, false, false, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (bn == 128) return launch_tc_variant<128, true, false, false, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    return cudaErrorInvalidValue;
  }
  if (dual) {
    if (pair && b3d) return launch_tc_variant<256, false, false, true, true, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (pair) return launch_tc_variant<256, false, false, false, true, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (b3d) return launch_tc_variant<256, false, false, true, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    return launch_tc_variant<256, false, false, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
  }
  if (pair) {
    if (b_kmajor) return launch_tc_variant<256, true, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (b3d) return launch_tc_variant<256, false, false, true, true>(ma, mb, mb2, mc, q, num_ctas, s);
    return launch_tc_variant<256, false, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
  }
  if (b3d) {
    if (bn == 256) return launch_tc_variant<256, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (bn == 192) return launch_tc_variant<192, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
    if (bn == 128) return launch_tc_variant<128, false, false, true>(ma, mb, mb2, mc, q, num_ctas, s);
  }
#define DG_TC_CASE(BNV, KM, R3)                                                     \
  if (bn == BNV && b_kmajor == KM && rank3 == R3)                                   \
    return launch_tc_variant<BNV, KM, R3>(ma, mb, mb2, mc, q, num_ctas, s);
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
