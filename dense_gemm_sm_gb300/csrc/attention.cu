// attention.cu -- fused attention forward on the tcgen05 tensor cores:
//   O = softmax(scale * Q K^T) V  per head, BF16 in, FP32 accumulate, BF16 out, d = 128
// ("Operator & Runtime", section 5.3.3: tiling with the online softmax, so the score and
// probability matrices never leave the SM).
//
// One CTA computes one 128-row query tile of one head and streams the head's keys and values
// through shared memory in blocks of 128 rows:
//   warp 0     TMA producer of Q (once) and K_j into a 3-slot ring;
//   warp 1     allocates TMEM and issues the MMAs: S_j = Q K_j^T into one of two TMEM score
//              buffers, O += P_j V_j into the TMEM output accumulator;
//   warps 2-5  softmax and epilogue, one query row per thread (the TMEM lane of that row):
//              the running maximum m and sum l in registers, p = 2^(s * scale * log2 e - m)
//              rounded to BF16 into TMEM as the A operand of the P V product;
//   warp 6     TMA producer of V_j into a 3-slot ring.
// K and V have producers of their own so that a K load waits only for the S product that
// frees its slot: with one producer issuing K_j, V_j, K_j+1, ... in order, the next K load
// queued behind a V load whose slot frees only after the softmax and P V of an earlier block,
// and the S products (and with them the softmax) waited for K.
// The recurrence is the pages' (m' = max(m, max s), r = e^(m - m'), l' = r l + sum p,
// u' = r u + sum p v), with one change that leaves the result unchanged: the reference
// point m is moved only when the block maximum exceeds it by more than 2^8 in the weights,
// so the rescale of the TMEM accumulator (a TMEM load/multiply/store of the row) runs only
// on the few blocks that raise the maximum that much; between moves the weights stay below
// 2^8, far inside FP32 and BF16 range.  Any common reference point gives the same u / l.
// Causal attention (key j visible to query i iff j <= i) skips the blocks past the
// diagonal and masks inside the diagonal block.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>

#include "dg_internal.h"
#include "ptx.cuh"

namespace dg {
namespace {

constexpr int kBQ = 128, kBKV = 128, kHD = 128;
// Softmax warps per 128 rows: 4 (one row per thread, all 128 keys of a block) or 8 (two
// warps per row quadrant, 64 keys each).  Measured: 4 is faster (1007 vs 900 TFLOPS on 64
// heads x 2048): with 8 every row's maximum is taken twice and the exponential / conversion
// pipe, not latency, bounds the softmax.
constexpr int kSoftWarps = 4;
constexpr int kHalves = kSoftWarps / 4;       // key / column parts per row
constexpr int kKeysPer = kBKV / kHalves;      // keys of a block per thread
constexpr int kVWarp = 2 + kSoftWarps;          // the V producer
constexpr int kThreads = 64 + 32 * kSoftWarps + 32;
constexpr int kKStages = 3, kVStages = 3;        // K and V ring slots (32 KiB each)
constexpr uint32_t kTile = 128 * kHD * 2;  // 128 rows x 128 BF16: two 64-column boxes, 32 KiB
constexpr uint32_t kHalf = kTile / 2;      // one 128-row x 64-column box (128-byte rows)
constexpr uint32_t kTmemCols = 512;        // S[0] at 0, S[1] at 128, O at 256, P[0..1] at 384
constexpr uint32_t kOCol = 256;
constexpr uint32_t kPCol = 384;            // P in TMEM: 64 columns (128 BF16 pairs) per buffer
constexpr float kMoveLog2 = 8.f;           // move m when the block raises it by > 8 (log2)

// Shared memory: Q | K[3] | V[3] (32 KiB each, 1024-byte aligned) | control | l exchange.
struct AttnCtl {
  uint64_t qfull;
  uint64_t kfull[kKStages], kempty[kKStages], vfull[kVStages], vempty[kVStages];
  uint64_t sfull[2], sfree[2], pfull[2], odone[2];
  uint64_t drain;
  uint64_t mfull;  // split over keys: the other chunks' partials in shared memory
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t is_last;  // split over keys: this CTA merges the tile's chunks
  uint32_t epi_ok;   // the softmax warps' common verdict before the epilogue
};
static_assert(sizeof(AttnCtl) <= 256, "control block");
// Q | K[3] | V[3] (32 KiB each) | control (256 B) | the halves' l exchange (1 KiB).
constexpr uint32_t kRingTiles = 1 + kKStages + kVStages;
constexpr uint32_t kSmemBytes = 1024 + kRingTiles * kTile + 256 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Three-input maximum (one instruction on sm_100 and later).
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two FP32 lanes in one 64-bit register (low lane first) and the packed FP32 operations on
// them: each lane is rounded exactly as the scalar instruction would round it.
__device__ __forceinline__ uint64_t f2_pack(uint32_t lo, uint32_t hi) {
  return static_cast<uint64_t>(hi) << 32 | lo;
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// The maximum of a row's 128 scores of one block (TMEM words, FP32): 64 three-input maxima
// over 8 independent chains.
__device__ __forceinline__ float block_row_max(const uint32_t (&sv)[4][32]) {
  float mx8[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) mx8[t] = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < 32; k += 2)
      mx8[(k >> 1) & 7] = max3f(mx8[(k >> 1) & 7], __uint_as_float(sv[c][k]), __uint_as_float(sv[c][k + 1]));
  return max3f(max3f(mx8[0], mx8[1], mx8[2]), max3f(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
}

// The weights p = 2^(s * cl + nb) of keys 32 c0 .. 32 (c0 + NC) - 1 of a row, two keys per
// packed FMA, rounded to BF16 pairs into pw (32-key chunk c in pw[c / 2], words 16 (c % 2) ..);
// returns their sum, kept in eight FP32 lanes (four packed partial sums) and added in a fixed
// order, so every kernel that calls this gets the same bits for the same scores.
template <int NC>
__device__ __forceinline__ float block_weights(const uint32_t (&sv)[4][32], int c0, float cl, float nb,
                                               uint32_t (&pw)[NC / 2][32]) {
  const uint64_t cl2 = f2_pack(__float_as_uint(cl), __float_as_uint(cl));
  const uint64_t nb2 = f2_pack(__float_as_uint(nb), __float_as_uint(nb));
  uint64_t ls4[4];
#pragma unroll
  for (int t = 0; t < 4; ++t) ls4[t] = 0;
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint64_t x = f2_fma(f2_pack(sv[c0 + c][2 * k], sv[c0 + c][2 * k + 1]), cl2, nb2);
      const float p0 = ex2(f2_lo(x));
      const float p1 = ex2(f2_hi(x));
      ls4[k & 3] = f2_add(ls4[k & 3], f2_pack(__float_as_uint(p0), __float_as_uint(p1)));
      pw[c >> 1][(c & 1) * 16 + k] = pack2(p0, p1);
    }
  return ((f2_lo(ls4[0]) + f2_hi(ls4[0])) + (f2_lo(ls4[1]) + f2_hi(ls4[1]))) +
         ((f2_lo(ls4[2]) + f2_hi(ls4[2])) + (f2_lo(ls4[3]) + f2_hi(ls4[3])));
}

// 32 lanes x 32 consecutive 32-bit TMEM columns from registers (thread i -> lane base+i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc] (the A operand read from tensor memory: row m in lane
// m, K elements packed two BF16 per 32-bit column, low half first).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void softmax_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kSoftWarps) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

__device__ __forceinline__ void load_box(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                         int32_t x, int32_t y, int32_t z, bool rank3) {
  if (rank3) tma_load_3d(dst, m, bar, x, y, z);
  else tma_load_2d(dst, m, bar, x, y);
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16), completing
// on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

__device__ __forceinline__ bool drain_wait(uint32_t bar, uint32_t parity, uint32_t* status) {
  uint32_t never = 0;
  return mbar_wait(bar, parity, &never, status, kDevTimeoutDrain);
}

// Softmax-warp wait: every lane waits (and acquires), then the warp agrees on the outcome,
// so the warp-collective TMEM instructions and votes after it never run diverged.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                          uint32_t* status) {
  const bool ok = mbar_wait(bar, parity, abort, status, kDevTimeoutEpilogue);
  return __all_sync(0xffffffffu, ok);
}

// The softmax writes P into TMEM (tcgen05.st) and the P V MMA reads its A operand from there,
// so only V passes through shared memory for that product.
template <bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                    const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // swizzle atoms need 1024-byte alignment
  const uint32_t sQ = base, sK = base + kTile, sV = base + (1 + kKStages) * kTile;
  AttnCtl* ctl = reinterpret_cast<AttnCtl*>(smem_raw + (base - raw) + kRingTiles * kTile);
  float* xl = reinterpret_cast<float*>(smem_raw + (base - raw) + kRingTiles * kTile + 256);  // [2][128]
  volatile uint32_t* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: causal, query tiles in decreasing order (the longest rows start first); not
  // causal, head by head; with a split over keys, the tile's chunk `kc` of nch covers its
  // key blocks j0 .. j0 + nkv - 1.
  int64_t qt, b, j0 = 0, kc = 0, nch = 1, nkv;
  {
    int64_t id = blockIdx.x;
    if (p.chunk > 0) {
      // Tile t has ch(t) = ceil(nk(t) / chunk) chunks, numbered tile by tile from the top
      // tile down, batch index fastest.  Non-causal: ch is the same for every tile.  Causal
      // (nk = t + 1): ch(t) = k on the band of tiles (k - 1) * chunk .. k * chunk - 1, so the
      // walk goes band by band (a few steps) instead of tile by tile.
      const int64_t C = p.chunk, B = p.batch;
      int64_t k = CAUSAL ? (p.q_tiles + C - 1) / C : (p.kv_blocks + C - 1) / C;
      int64_t hi = p.q_tiles - 1;  // the band's highest tile
      for (;;) {
        const int64_t lo = CAUSAL ? (k - 1) * C : 0;
        const int64_t n = (hi - lo + 1) * k * B;  // items of the band
        if (id < n || k <= 1 || !CAUSAL) {
          const int64_t u = id / (k * B), r = id - u * (k * B);
          qt = hi - u;
          b = r % B;
          kc = r / B;
          nch = k;
          j0 = kc * C;
          const int64_t nk = CAUSAL ? qt + 1 : p.kv_blocks;
          nkv = nk - j0 < C ? nk - j0 : C;
          break;
        }
        id -= n;
        hi = lo - 1;
        --k;
      }
    } else if (CAUSAL) {
      qt = p.q_tiles - 1 - id / p.batch;
      b = id % p.batch;
      nkv = qt + 1;
    } else {
      // Head by head, so that the CTAs running together share few heads' K and V, which then
      // stay in L2 while all of the head's query tiles stream them.
      b = id / p.q_tiles;
      qt = id - b * p.q_tiles;
      nkv = p.kv_blocks;
    }
  }
  const int64_t q0 = qt * kBQ;
  const bool rank3 = p.rank3 != 0;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->qfull), 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(smem_u32(&ctl->kfull[s]), 1);
      mbar_init(smem_u32(&ctl->kempty[s]), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(smem_u32(&ctl->vfull[s]), 1);
      mbar_init(smem_u32(&ctl->vempty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->sfull[s]), 1);
      mbar_init(smem_u32(&ctl->sfree[s]), kSoftWarps);  // one arrival per softmax warp
      mbar_init(smem_u32(&ctl->pfull[s]), kSoftWarps);
      mbar_init(smem_u32(&ctl->odone[s]), 1);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    mbar_init(smem_u32(&ctl->mfull), 1);
    ctl->abort = 0;
    ctl->is_last = 1;
    fence_barrier_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  pdl_wait();

  const int32_t zb = static_cast<int32_t>(b);
  if (warp == 0 || warp == kVWarp) {
    // ------------------------------------------------------------ TMA producers (Q, K | V)
    if (lane == 0) {
      const bool isk = warp == 0;
      const int stages = isk ? kKStages : kVStages;
      const uint32_t ring = isk ? sK : sV;
      const CUtensorMap* map = isk ? &tmK : &tmV;
      uint64_t* full = isk ? ctl->kfull : ctl->vfull;
      uint64_t* empty = isk ? ctl->kempty : ctl->vempty;
      const uint32_t qf = smem_u32(&ctl->qfull);
      if (isk) {
        mbar_arrive_expect_tx(qf, kTile);
        load_box(sQ, &tmQ, qf, 0, static_cast<int32_t>(q0), zb, rank3);
        load_box(sQ + kHalf, &tmQ, qf, 64, static_cast<int32_t>(q0), zb, rank3);
      }
      int64_t issued = 0;
      uint32_t s = 0, ph = 0;  // ring slot and its phase parity for block j
      for (int64_t j = 0; j < nkv; ++j) {
        if (!mbar_wait(smem_u32(&empty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) break;
        const uint32_t f = smem_u32(&full[s]);
        const int32_t y = static_cast<int32_t>((j0 + j) * kBKV);
        mbar_arrive_expect_tx(f, kTile);
        load_box(ring + s * kTile, map, f, 0, y, zb, rank3);
        load_box(ring + s * kTile + kHalf, map, f, 64, y, zb, rank3);
        ++issued;
        if (++s == static_cast<uint32_t>(stages)) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (*abort) {
        // No copy may still be landing in shared memory when the CTA exits: wait for the
        // last loads issued into each slot (earlier ones were consumed before the reuse).
        if (isk) drain_wait(qf, 0, p.status);
        for (int64_t j = issued > stages ? issued - stages : 0; j < issued; ++j)
          drain_wait(smem_u32(&full[j % stages]), static_cast<uint32_t>((j / stages) & 1), p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // S = Q K^T: A = Q and B = K both K-major (d contiguous).  O += P V: A = P K-major
      // (keys contiguous), B = V N-major (d contiguous, keys along K).
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, 128, false, true);
      bool ok = mbar_wait(smem_u32(&ctl->qfull), 0, abort, p.status, kDevTimeoutMma);
      // Operand descriptors of the ring bases, advanced per MMA by the start-address field
      // alone (16-byte units; every offset stays inside the 256 KiB the field spans), so each
      // MMA costs the issuing thread a few integer additions: the issuing thread shares its
      // SM sub-partition with a softmax warp, and its instruction count per MMA showed in the
      // tensor pipe's rate (1001 -> 1048 TFLOPS on 64 heads x 2048).
      const uint64_t dQ = sdesc_sw128(sQ, 16, 1024), dK = sdesc_sw128(sK, 16, 1024);
      const uint64_t dV = sdesc_sw128(sV, kHalf, 1024);
      // S products are issued in block order: ks / kph track the K ring slot of the next one.
      uint32_t ks = 0, kph = 0;
      auto issue_s = [&](int64_t j) -> bool {
        const uint32_t sb = j & 1;  // score buffer
        if (!mbar_wait(smem_u32(&ctl->kfull[ks]), kph, abort, p.status, kDevTimeoutMma)) return false;
        tc_fence_after();
        const uint64_t dKs = dK + ks * (kTile >> 4);
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k) {
          // 16 columns of d per MMA: 32 bytes inside a 128-byte swizzle row, the second
          // 64 columns in the second box.
          const uint32_t off = ((k >> 2) * kHalf + (k & 3) * 32) >> 4;
          umma_bf16(tmem + sb * 128, dQ + off, dKs + off, idS, k > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&ctl->kempty[ks]));
        umma_commit(smem_u32(&ctl->sfull[sb]));
        if (++ks == kKStages) {
          ks = 0;
          kph ^= 1u;
        }
        return true;
      };
      // Per block j: S_j+2 goes into score buffer j % 2 as soon as the softmax has read S_j
      // into registers, so it runs while the softmax of block j exponentiates; P_j V_j follows
      // once the weights are in TMEM.  (Issuing S_j+2 only after P_j V_j queued every score
      // product behind the softmax of the block two earlier.)
      if (ok) ok = issue_s(0);
      if (ok && nkv > 1) ok = issue_s(1);
      uint32_t vs = 0, vph = 0;  // V ring slot of block j
      for (int64_t j = 0; ok && j < nkv; ++j) {
        const uint32_t s = j & 1, ph = (j >> 1) & 1;
        if (j + 2 < nkv) {
          if (!mbar_wait(smem_u32(&ctl->sfree[s]), ph, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!issue_s(j + 2)) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait(smem_u32(&ctl->pfull[s]), ph, abort, p.status, kDevTimeoutMma) ||
            !mbar_wait(smem_u32(&ctl->vfull[vs]), vph, abort, p.status, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t dVs = dV + vs * (kTile >> 4);
#pragma unroll
        for (int k = 0; k < kBKV / 16; ++k) {
          // V: 16 key rows = 2 KiB per MMA; its two 64-column halves of d are one box apart
          // (LBO).  A = P: 16 keys = 8 packed columns of the TMEM P buffer.
          umma_bf16_ts(tmem + kOCol, tmem + kPCol + s * 64 + k * 8, dVs + k * (2048 >> 4), idO,
                       (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(smem_u32(&ctl->vempty[vs]));
        umma_commit(smem_u32(&ctl->odone[s]));
        if (++vs == kVStages) {
          vs = 0;
          vph ^= 1u;
        }
      }
      // Every MMA finished before TMEM is released.
      umma_commit(smem_u32(&ctl->drain));
      drain_wait(smem_u32(&ctl->drain), 0, p.status);
    }
  } else if (warp < kVWarp) {
    // ------------------------------------------------------------ softmax + epilogue
    // One query row per thread (the TMEM lane of warp w % 4's quadrant).  With 8 warps, warps
    // w and w + 4 split each block's keys and the row's columns of O in halves; both read the
    // whole row of scores for its maximum, so both take the same reference point without
    // exchanging anything, and their parts of l are added at the end.
    const int qd = warp & 3;                 // TMEM lane quadrant this warp may access
    const int half = kHalves == 1 ? 0 : (warp - 2) >> 2;  // which keys of a block / columns of O
    const int row = qd * 32 + lane;          // query row in the tile = TMEM lane
    const int64_t qrow = q0 + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qd * 32) << 16);
    const uint32_t swz = static_cast<uint32_t>(row & 7);
    const uint32_t prow = static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128);
    const float cl = p.c_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int64_t j = 0; j < nkv; ++j) {
      const uint32_t s = j & 1, ph = (j >> 1) & 1;
      if (!warp_wait(smem_u32(&ctl->sfull[s]), ph, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tl + s * 128 + c * 32, sv[c]);
      tmem_ld_wait();
      // S_j is in registers: its buffer may take S_j+2.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->sfree[s]));
      const int64_t kv0 = (j0 + j) * kBKV;
      const bool masked = kv0 + kBKV > p.Lkv || (CAUSAL && j0 + j == qt);
      if (masked) {
        // Keys at or past `lim` are not visible to this row: weight 0.
        const int64_t lim = CAUSAL ? (qrow + 1 < p.Lkv ? qrow + 1 : p.Lkv) : p.Lkv;
        const int64_t nv = lim - kv0;
        const int nvis = nv < 0 ? 0 : (nv > kBKV ? kBKV : static_cast<int>(nv));
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (c * 32 + k >= nvis) sv[c][k] = 0xFF800000u;  // -inf
      }
      const float m_blk = block_row_max(sv) * cl;  // the block's maximum in log2 units (scale > 0)
      float r = 1.f;
      if (m_blk > m_run + kMoveLog2) {
        r = ex2(m_run - m_blk);  // 0 on the first block (m_run = -inf)
        m_run = m_blk;
      }
      const bool rescale = j > 0 && __any_sync(0xffffffffu, r != 1.f);
      const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
      // P buffer s is free once P V of block j - 2 has completed.
      if (j >= 2 && !warp_wait(smem_u32(&ctl->odone[s]), ((j - 2) >> 1) & 1, abort, p.status)) {
        ok = false;
        break;
      }
      uint32_t pw[kKeysPer / 64][32];  // this thread's weights as packed BF16 pairs
      const float lsum = block_weights<kKeysPer / 32>(sv, half * (kKeysPer / 32), cl, nb, pw);
      l_run = l_run * r + lsum;
#pragma unroll
      for (int c = 0; c < kKeysPer / 64; ++c)
        tmem_st_32x32b_x32(tl + kPCol + s * 64 + half * (kKeysPer / 2) + c * 32, pw[c]);
      tmem_st_wait();
      if (rescale) {
        // The reference point moved: scale this half's 64 columns of the row of O by r once
        // P V of block j - 1 has landed in TMEM (lanes whose point did not move multiply by 1).
        if (!warp_wait(smem_u32(&ctl->odone[(j - 1) & 1]), ((j - 1) >> 1) & 1, abort, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4 / kHalves; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tl + kOCol + half * (128 / kHalves) + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * r);
          tmem_st_32x32b_x32(tl + kOCol + half * (128 / kHalves) + c * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->pfull[s]));
    }
    if (ok) {
      const int64_t jl = nkv - 1;
      ok = warp_wait(smem_u32(&ctl->odone[jl & 1]), (jl >> 1) & 1, abort, p.status);
    }
    // Writes 32 values of this row's O (columns 32c .. 32c+31, already divided by l) as BF16
    // into the (no longer read) Q tile, in the layout of the output map's 128B-swizzled boxes.
    const uint32_t ob = sQ + prow;
    auto stage = [&](int c, const float (&f)[32]) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const uint32_t chunk = static_cast<uint32_t>((c & 1) * 4 + q4);
        st_shared_v4(ob + (c >> 1) * kHalf + ((chunk ^ swz) << 4), pack2(f[8 * q4], f[8 * q4 + 1]),
                     pack2(f[8 * q4 + 2], f[8 * q4 + 3]), pack2(f[8 * q4 + 4], f[8 * q4 + 5]),
                     pack2(f[8 * q4 + 6], f[8 * q4 + 7]));
      }
    };
    // The eight softmax warps take one decision (the split path below has group barriers):
    // any failed wait has set the abort flag before this barrier.  The row's l is the sum
    // of the two halves' parts, half 0's first.
    xl[half * 128 + row] = l_run;
    softmax_bar();
    if (threadIdx.x == 64) ctl->epi_ok = (ok && !*abort) ? 1u : 0u;
    softmax_bar();
    ok = ctl->epi_ok != 0;
    const float l_tot = kHalves == 1 ? l_run : xl[row] + xl[128 + row];
    constexpr int kCols = 4 / kHalves;  // 32-column chunks of O per thread
    if (ok && nch == 1) {
      // O = u / l, rounded once to BF16.
      tc_fence_after();
      const float inv = 1.f / l_tot;
#pragma unroll
      for (int c = kCols * half; c < kCols * half + kCols; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + kOCol + c * 32, o);
        tmem_ld_wait();
        float f[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) f[k] = __uint_as_float(o[k]) * inv;
        stage(c, f);
      }
      fence_proxy_async_smem();
    } else if (ok) {
      // Split over keys: publish this chunk's state (u unnormalised in FP32, m and l per row),
      // take a ticket; the chunk that takes the last merges all chunks in chunk order with
      // the pages' recurrence: m* = max m_k, l* = sum 2^(m_k - m*) l_k,
      // u* = sum 2^(m_k - m*) u_k, O = u* / l*.
      tc_fence_after();
      float* mine = p.ws + static_cast<int64_t>(blockIdx.x) * kAttnPartFloats;
      {
        float4* u4 = reinterpret_cast<float4*>(mine);
#pragma unroll
        for (int c = kCols * half; c < kCols * half + kCols; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tl + kOCol + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 8; ++g)
            __stcg(u4 + (c * 8 + g) * 128 + row,
                   make_float4(__uint_as_float(o[4 * g]), __uint_as_float(o[4 * g + 1]),
                               __uint_as_float(o[4 * g + 2]), __uint_as_float(o[4 * g + 3])));
        }
        if (half == 0) {
          __stcg(mine + 128 * 128 + row, m_run);
          __stcg(mine + 128 * 128 + 128 + row, l_tot);
        }
      }
      softmax_bar();
      uint32_t* counter = &p.counters[b * p.q_tiles + qt];
      if (threadIdx.x == 64) {
        fence_acq_rel_gpu();  // cumulative: the 128 threads' stores, ordered by the barrier
        const uint32_t prev = atomicAdd(counter, 1u);
        const bool last = prev + 1u == static_cast<uint32_t>(nch);
        if (last) {
          fence_acq_rel_gpu();
          *counter = 0u;  // every chunk holds its ticket: ready for the next call
        }
        ctl->is_last = last ? 1u : 0u;
      }
      softmax_bar();
      if (ctl->is_last) {
        // The tile's chunks are the items blockIdx.x + (k - kc) * batch, k < nch; the sums run
        // in chunk order.  With at most four chunks, the other chunks' u come into the idle K / V
        // rings (3 x 64 KiB) by bulk copies and this chunk's own u is read from TMEM (the same
        // FP32 values it published); more chunks read their partials from L2.
        const float* first = mine - kc * p.batch * kAttnPartFloats;
        auto part = [&](int64_t k) { return first + k * p.batch * kAttnPartFloats; };
        constexpr uint32_t kPartBytes = 128 * 128 * 4;
        const bool via_smem = nch <= 4;
        const uint32_t mb = smem_u32(&ctl->mfull);
        if (via_smem && threadIdx.x == 64) {
          asm volatile("fence.proxy.async.global;" ::: "memory");  // the acquired partials, for the copy engine
          mbar_arrive_expect_tx(mb, static_cast<uint32_t>(nch - 1) * kPartBytes);
          for (int64_t k = 0, slot = 0; k < nch; ++k)
            if (k != kc) bulk_g2s(sK + static_cast<uint32_t>(slot++) * kPartBytes, part(k), kPartBytes, mb);
        }
        float ms = -INFINITY;
#pragma unroll 4
        for (int64_t k = 0; k < nch; ++k) ms = fmaxf(ms, __ldcg(part(k) + 128 * 128 + row));
        float ls = 0.f;
#pragma unroll 4
        for (int64_t k = 0; k < nch; ++k)
          ls += ex2(__ldcg(part(k) + 128 * 128 + row) - ms) * __ldcg(part(k) + 128 * 128 + 128 + row);
        const float inv = 1.f / ls;
        bool mok = true;
        if (via_smem) {
          // The chunks' weights 2^(m_k - m*), k < 4, in registers (selected, not indexed).
          const float w0 = ex2(__ldcg(part(0) + 128 * 128 + row) - ms);
          const float w1 = ex2(__ldcg(part(1) + 128 * 128 + row) - ms);
          const float w2 = nch > 2 ? ex2(__ldcg(part(2) + 128 * 128 + row) - ms) : 0.f;
          const float w3 = nch > 3 ? ex2(__ldcg(part(3) + 128 * 128 + row) - ms) : 0.f;
          mok = warp_wait(mb, 0, abort, p.status);
          if (!mok && threadIdx.x == 64) drain_wait(mb, 0, p.status);
          const float4* ring4 = reinterpret_cast<const float4*>(smem_raw + (sK - raw));
#pragma unroll 1
          for (int c = kCols * half; mok && c < kCols * half + kCols; ++c) {
            float f[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) f[k] = 0.f;
            for (int k = 0; k < nch; ++k) {
              const float w = k == 0 ? w0 : k == 1 ? w1 : k == 2 ? w2 : w3;
              if (k == kc) {
                uint32_t o[32];
                tmem_ld_32x32b_x32(tl + kOCol + c * 32, o);
                tmem_ld_wait();
#pragma unroll
                for (int q = 0; q < 32; ++q) f[q] = fmaf(w, __uint_as_float(o[q]), f[q]);
              } else {
                const float4* u4 = ring4 + (k < kc ? k : k - 1) * (kPartBytes / 16) + c * 8 * 128 + row;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                  const float4 v = u4[g * 128];
                  f[4 * g] = fmaf(w, v.x, f[4 * g]);
                  f[4 * g + 1] = fmaf(w, v.y, f[4 * g + 1]);
                  f[4 * g + 2] = fmaf(w, v.z, f[4 * g + 2]);
                  f[4 * g + 3] = fmaf(w, v.w, f[4 * g + 3]);
                }
              }
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) f[k] *= inv;
            stage(c, f);
          }
        } else {
#pragma unroll 1
          for (int c2 = kCols * half; c2 < kCols * half + kCols; c2 += 2) {
            float f[2][32];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int k = 0; k < 32; ++k) f[h][k] = 0.f;
            for (int64_t k = 0; k < nch; ++k) {
              const float* pk = part(k);
              const float w = ex2(__ldcg(pk + 128 * 128 + row) - ms);
              const float4* u4 = reinterpret_cast<const float4*>(pk) + c2 * 8 * 128 + row;
              float4 v[16];
#pragma unroll
              for (int g = 0; g < 16; ++g) v[g] = __ldcg(u4 + g * 128);
#pragma unroll
              for (int g = 0; g < 16; ++g) {
                float* fh = f[g >> 3];
                const int b4 = 4 * (g & 7);
                fh[b4] = fmaf(w, v[g].x, fh[b4]);
                fh[b4 + 1] = fmaf(w, v[g].y, fh[b4 + 1]);
                fh[b4 + 2] = fmaf(w, v[g].z, fh[b4 + 2]);
                fh[b4 + 3] = fmaf(w, v[g].w, fh[b4 + 3]);
              }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
              for (int k = 0; k < 32; ++k) f[h][k] *= inv;
              stage(c2 + h, f[h]);
            }
          }
        }
        if (!mok) *abort = 1;
        fence_proxy_async_smem();
      }
    }
    softmax_bar();
    if (warp == 2 && lane == 0 && !*abort && ctl->is_last) {
      // Rows past Lq are clipped by the tensor map.
      if (rank3) {
        tma_store_3d(&tmO, sQ, 0, static_cast<int32_t>(q0), zb);
        tma_store_3d(&tmO, sQ + kHalf, 64, static_cast<int32_t>(q0), zb);
      } else {
        tma_store_2d(&tmO, sQ, 0, static_cast<int32_t>(q0));
        tma_store_2d(&tmO, sQ + kHalf, 64, static_cast<int32_t>(q0));
      }
      bulk_commit();
      bulk_wait_read<0>();  // the CTA may retire once the store has read shared memory
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------------
// Two query tiles per CTA (non-causal attention with enough tiles to fill the GPU; opt-in,
// see launch_attention).  The
// tiles A and B share every K and V block; each has its own softmax group of four warps
// (warps 2-5: A, 6-9: B) and its own S and O in TMEM (S_A 0, O_A 128, S_B 256, O_B 384; the
// weights P are written over the first 64 columns of their S after S has been read).  While
// one group exponentiates, the tensor core runs the other group's P V and S products, so
// the two groups' softmax latencies and the MMAs overlap.  The MMA issuer waits for P V of
// block j to complete before it overwrites that tile's S (and P) with block j + 1.
constexpr uint32_t kPairSmemBytes = 1024 + 6 * kTile + 256;  // Q_A, Q_B, K[2], V[2], control
constexpr int kPairThreads = 320;

struct PairCtl {
  uint64_t qfull;
  uint64_t kfull[2], kempty[2], vfull[2], vempty[2];
  uint64_t sfull[2], pfull[2], odone[2];  // per tile (A, B)
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
};
static_assert(sizeof(PairCtl) <= 256, "control block");

__device__ __forceinline__ void group_bar(int g) {
  // Named barriers 2 and 3: the four warps of softmax group g.
  asm volatile("bar.sync %0, 128;" ::"r"(2 + g) : "memory");
}

__global__ void __launch_bounds__(kPairThreads, 1)
    attn_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                     const AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t sQ = base, sK = base + 2 * kTile, sV = base + 4 * kTile;  // Q_A, Q_B, K[2], V[2]
  PairCtl* ctl = reinterpret_cast<PairCtl*>(smem_raw + (base - raw) + 6 * kTile);
  volatile uint32_t* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int64_t pairs = (p.q_tiles + 1) / 2;
  const int64_t pi = static_cast<int64_t>(blockIdx.x) / p.batch;
  const int64_t b = static_cast<int64_t>(blockIdx.x) % p.batch;
  const int64_t qtA = 2 * pi;
  const bool hasB = qtA + 1 < p.q_tiles;
  const int64_t nkv = p.kv_blocks;
  const bool rank3 = p.rank3 != 0;
  (void)pairs;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&ctl->qfull), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&ctl->kfull[s]), 1);
      mbar_init(smem_u32(&ctl->kempty[s]), 1);
      mbar_init(smem_u32(&ctl->vfull[s]), 1);
      mbar_init(smem_u32(&ctl->vempty[s]), 1);
      mbar_init(smem_u32(&ctl->sfull[s]), 1);
      mbar_init(smem_u32(&ctl->pfull[s]), 4);
      mbar_init(smem_u32(&ctl->odone[s]), 1);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort = 0;
    fence_barrier_init();
    tma_prefetch_map(&tmQ);
    tma_prefetch_map(&tmK);
    tma_prefetch_map(&tmV);
    tma_prefetch_map(&tmO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_trigger();
  pdl_wait();

  const int32_t zb = static_cast<int32_t>(b);
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t qf = smem_u32(&ctl->qfull);
      mbar_arrive_expect_tx(qf, hasB ? 2 * kTile : kTile);
      for (int t = 0; t < (hasB ? 2 : 1); ++t) {
        const int32_t y = static_cast<int32_t>((qtA + t) * kBQ);
        load_box(sQ + t * kTile, &tmQ, qf, 0, y, zb, rank3);
        load_box(sQ + t * kTile + kHalf, &tmQ, qf, 64, y, zb, rank3);
      }
      int64_t issued = 0;
      bool k_only = false;
      for (int64_t j = 0; j < nkv; ++j) {
        const uint32_t s = j & 1, ph = (j >> 1) & 1;
        const int32_t y = static_cast<int32_t>(j * kBKV);
        if (!mbar_wait(smem_u32(&ctl->kempty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) break;
        const uint32_t kf = smem_u32(&ctl->kfull[s]);
        mbar_arrive_expect_tx(kf, kTile);
        load_box(sK + s * kTile, &tmK, kf, 0, y, zb, rank3);
        load_box(sK + s * kTile + kHalf, &tmK, kf, 64, y, zb, rank3);
        k_only = true;
        if (!mbar_wait(smem_u32(&ctl->vempty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) break;
        const uint32_t vf = smem_u32(&ctl->vfull[s]);
        mbar_arrive_expect_tx(vf, kTile);
        load_box(sV + s * kTile, &tmV, vf, 0, y, zb, rank3);
        load_box(sV + s * kTile + kHalf, &tmV, vf, 64, y, zb, rank3);
        k_only = false;
        ++issued;
      }
      if (*abort) {
        drain_wait(qf, 0, p.status);
        const int64_t kl = issued + (k_only ? 1 : 0);
        for (int64_t j = kl > 2 ? kl - 2 : 0; j < kl; ++j)
          drain_wait(smem_u32(&ctl->kfull[j & 1]), (j >> 1) & 1, p.status);
        for (int64_t j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
          drain_wait(smem_u32(&ctl->vfull[j & 1]), (j >> 1) & 1, p.status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, 128, false, true);
      const int nt = hasB ? 2 : 1;
      bool ok = mbar_wait(smem_u32(&ctl->qfull), 0, abort, p.status, kDevTimeoutMma);
      // S_t = Q_t K_j^T into tile t's S columns.
      auto issue_s = [&](int t, uint32_t kb) {
        const uint32_t qb = sQ + t * kTile;
#pragma unroll
        for (int k = 0; k < kHD / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
          umma_bf16(tmem + t * 256, sdesc_sw128(qb + off, 16, 1024), sdesc_sw128(kb + off, 16, 1024),
                    idS, k > 0 ? 1u : 0u);
        }
        umma_commit(smem_u32(&ctl->sfull[t]));
      };
      if (ok) ok = mbar_wait(smem_u32(&ctl->kfull[0]), 0, abort, p.status, kDevTimeoutMma);
      if (ok) {
        tc_fence_after();
        for (int t = 0; t < nt; ++t) issue_s(t, sK);
        umma_commit(smem_u32(&ctl->kempty[0]));
      }
      for (int64_t j = 0; ok && j < nkv; ++j) {
        const uint32_t s = j & 1, ph = (j >> 1) & 1, jp = j & 1;
        if (!mbar_wait(smem_u32(&ctl->vfull[s]), ph, abort, p.status, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        const uint32_t vb = sV + s * kTile;
        for (int t = 0; t < nt; ++t) {
          if (!mbar_wait(smem_u32(&ctl->pfull[t]), jp, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kBKV / 16; ++k)
            umma_bf16_ts(tmem + t * 256 + 128, tmem + t * 256 + k * 8, sdesc_sw128(vb + k * 2048, kHalf, 1024),
                         idO, (j > 0 || k > 0) ? 1u : 0u);
          umma_commit(smem_u32(&ctl->odone[t]));
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctl->vempty[s]));
        if (j + 1 < nkv) {
          const uint32_t s1 = (j + 1) & 1, ph1 = ((j + 1) >> 1) & 1;
          if (!mbar_wait(smem_u32(&ctl->kfull[s1]), ph1, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          for (int t = 0; t < nt; ++t) {
            // Tile t's S columns hold P of block j until its P V has run.
            if (!mbar_wait(smem_u32(&ctl->odone[t]), jp, abort, p.status, kDevTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(t, sK + s1 * kTile);
          }
          if (!ok) break;
          umma_commit(smem_u32(&ctl->kempty[s1]));
        }
      }
      umma_commit(smem_u32(&ctl->drain));
      drain_wait(smem_u32(&ctl->drain), 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue, per tile
    const int g = (warp - 2) >> 2;  // tile: 0 = A, 1 = B
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const bool active = g == 0 || hasB;
    const uint32_t tl = tmem + (static_cast<uint32_t>(qd * 32) << 16) + g * 256;
    const uint32_t swz = static_cast<uint32_t>(row & 7);
    const uint32_t prow = static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128);
    const float cl = p.c_log2;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = active;
    for (int64_t j = 0; ok && j < nkv; ++j) {
      const uint32_t jp = j & 1;
      if (!warp_wait(smem_u32(&ctl->sfull[g]), jp, abort, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld_32x32b_x32(tl + c * 32, sv[c]);
      tmem_ld_wait();
      const int64_t kv0 = j * kBKV;
      const bool masked = kv0 + kBKV > p.Lkv;
      if (masked) {
        const int64_t nv = p.Lkv - kv0;
        const int nvis = nv > kBKV ? kBKV : static_cast<int>(nv);
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k)
            if (c * 32 + k >= nvis) sv[c][k] = 0xFF800000u;
      }
      const float m_blk = block_row_max(sv) * cl;
      float r = 1.f;
      if (m_blk > m_run + kMoveLog2) {
        r = ex2(m_run - m_blk);
        m_run = m_blk;
      }
      const bool rescale = j > 0 && __any_sync(0xffffffffu, r != 1.f);
      const float nb = (m_run == -INFINITY) ? 0.f : -m_run;
      uint32_t pw[2][32];
      const float lsum = block_weights<4>(sv, 0, cl, nb, pw);
      l_run = l_run * r + lsum;
      // P over the first 64 columns of this tile's S (already read into registers).
      tmem_st_32x32b_x32(tl, pw[0]);
      tmem_st_32x32b_x32(tl + 32, pw[1]);
      tmem_st_wait();
      if (rescale) {
        // P V of block j - 1 has completed: the MMA issuer waited for it before computing S
        // of block j into these columns.
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tl + 128 + c * 32, o);
          tmem_ld_wait();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * r);
          tmem_st_32x32b_x32(tl + 128 + c * 32, o);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->pfull[g]));
    }
    if (ok) {
      const int64_t jl = nkv - 1;
      ok = warp_wait(smem_u32(&ctl->odone[g]), jl & 1, abort, p.status);
    }
    // The group's four warps agree, then write O = u / l through the tile's Q buffer.
    group_bar(g);
    const bool store = active && !*abort;
    group_bar(g);
    if (store && ok) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      const uint32_t ob = sQ + g * kTile + prow;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld_32x32b_x32(tl + 128 + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          const uint32_t chunk = static_cast<uint32_t>((c & 1) * 4 + q4);
          const float* f = reinterpret_cast<const float*>(o) + 8 * q4;
          st_shared_v4(ob + (c >> 1) * kHalf + ((chunk ^ swz) << 4), pack2(f[0] * inv, f[1] * inv),
                       pack2(f[2] * inv, f[3] * inv), pack2(f[4] * inv, f[5] * inv),
                       pack2(f[6] * inv, f[7] * inv));
        }
      }
      fence_proxy_async_smem();
    }
    group_bar(g);
    if (store && (warp & 3) == 2 && lane == 0 && !*abort) {
      const int32_t y = static_cast<int32_t>((qtA + g) * kBQ);
      const uint32_t src = sQ + g * kTile;
      if (rank3) {
        tma_store_3d(&tmO, src, 0, y, zb);
        tma_store_3d(&tmO, src + kHalf, 64, y, zb);
      } else {
        tma_store_2d(&tmO, src, 0, y);
        tma_store_2d(&tmO, src + kHalf, 64, y);
      }
      bulk_commit();
      bulk_wait<0>();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

std::atomic<uint64_t> g_pair_attr{0};

std::atomic<uint64_t> g_attr_done[2];

template <bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
                           const CUtensorMap& mo, const AttnParams& p, cudaStream_t s) {
  auto kern = attn_fwd_kernel<CAUSAL>;
  constexpr uint32_t smem = kSmemBytes;
  cudaError_t e = ensure_smem_attr(kern, static_cast<int>(smem), g_attr_done[CAUSAL ? 1 : 0]);
  if (e != cudaSuccess) return e;
  const dim3 grid(static_cast<unsigned>(p.items));
  return launch_pdl(kern, grid, dim3(kThreads), smem, s, mq, mk, mv, mo, p);
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, bool causal, const void* Q, int64_t ldq,
                             int64_t sQ, const void* K, int64_t ldk, int64_t sK, const void* V,
                             int64_t ldv, int64_t sV, void* O, int64_t ldo, int64_t sO,
                             cudaStream_t s) {
  const uint64_t batch = static_cast<uint64_t>(p.batch);
  CUtensorMap mq, mk, mv, mo;
  // Every operand is a (batch x) rows x 128 row-major BF16 view read or written in boxes of
  // 128 rows x 64 columns (128-byte rows, 128-byte swizzle).
  auto map = [&](CUtensorMap* m, const void* ptr, int64_t rows, int64_t ld, int64_t stride) {
    return make_tile_map(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, ptr, kHD,
                         static_cast<uint64_t>(rows), static_cast<uint64_t>(ld), batch,
                         static_cast<uint64_t>(stride), 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, 1);
  };
  if (!map(&mq, Q, p.Lq, ldq, sQ) || !map(&mk, K, p.Lkv, ldk, sK) || !map(&mv, V, p.Lkv, ldv, sV) ||
      !map(&mo, O, p.Lq, ldo, sO))
    return cudaErrorInvalidValue;
  // DG_ATTN_PAIR=1: non-causal attention with at least one pair of query tiles per SM takes
  // the two-tile kernel.  Measured slower (890 vs 1004 TFLOPS on 64 heads x 2048): each
  // tile's chain softmax -> P V -> (wait) -> next S serialises, and two softmax groups per
  // SM sub-partition slow each other down more than their overlap gains; so one tile per CTA
  // is the default.
  const char* pe = std::getenv("DG_ATTN_PAIR");
  if (!causal && p.chunk == 0 && pe && pe[0] == '1' &&
      p.batch * ((p.q_tiles + 1) / 2) >= static_cast<int64_t>(p.sms)) {
    cudaError_t e = ensure_smem_attr(attn_pair_kernel, static_cast<int>(kPairSmemBytes), g_pair_attr);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(p.batch * ((p.q_tiles + 1) / 2)));
    return launch_pdl(attn_pair_kernel, grid, dim3(kPairThreads), kPairSmemBytes, s, mq, mk, mv, mo, p);
  }
  return causal ? launch_variant<true>(mq, mk, mv, mo, p, s)
                : launch_variant<false>(mq, mk, mv, mo, p, s);
}

}  // namespace dg
