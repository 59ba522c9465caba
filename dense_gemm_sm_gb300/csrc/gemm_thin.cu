// gemm_thin.cu -- decode-shaped BF16 GEMM (M <= 32 rows of X) on tcgen05, stream-K split.
//
// C[M,N] = alpha * X[M,K] * W[K,N] + beta * C with M tiny: every weight element is used
// by at most 32 rows, so the cost is streaming W (K*N*2 bytes) from HBM once; the MUSA
// lesson m11-l5 ("Batch GEMV" for [m,k] x [k,4]) and the Little's-law argument of
// "Operator & Runtime" section 5.1.5 (enough bytes in flight per SM) drive the design:
//   * swap A/B: the MMA's M dimension (128) runs over 128 columns of W, its N dimension
//     (16 or 32) over the rows of X, so D^T = W^T X^T sits in TMEM as 128 lanes x ntok;
//   * the (W column tile, K block) pairs are flattened into U units and split evenly over
//     one CTA per SM (stream-K); each CTA streams its contiguous range of W through a deep
//     TMA ring (8 stages x 16 KiB of W);
//   * a tile split across CTAs ("split K", "Operator & Runtime" section 5.2.4) is combined
//     by one of its contributors.  Each contributor stores its part, fences and takes a
//     ticket from the tile's atomic counter; the last to take one adds the parts in a fixed
//     order -- the contributors after the tile's first CTA in CTA order, then the first
//     CTA's part -- so results are identical run to run whoever combines (same section:
//     atomics give arrival-dependent rounding, a fixed combination order does not).  The
//     tile's first CTA reaches its part at the very end of its range, when the others have
//     usually finished theirs: while its own part still streams it watches the counter, and
//     once every other contributor holds a ticket it adds their parts ahead of time,
//     leaving only its own for the end;
//   * alpha/beta and the single rounding to BF16 (or FP32 output) happen after the full
//     K reduction (sections 5.4.2-5.4.3).
// Warp roles (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA issuer,
// warps 2-5 epilogue / combine (thread = one W column of the tile).
#include <cuda_bf16.h>

#include "dg_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dg {

bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint64_t batch, uint64_t stride, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int BNW = kThinBN, BK = kThinBK;
constexpr uint32_t W_BYTES = BNW * BK * 2;  // 16 KiB per stage
#ifndef DG_THIN_STAGES
#define DG_THIN_STAGES 8
#endif
constexpr int STAGES = DG_THIN_STAGES;
// W blocks of its range a CTA asks L2 for before the previous grid of the stream has
// finished (0: none).
#ifndef DG_THIN_PREFETCH
#define DG_THIN_PREFETCH 32
#endif
constexpr int PREFETCH = DG_THIN_PREFETCH;

constexpr int NUM_THREADS = 192;

template <int NTOK>
struct ThinCfg {
  static constexpr uint32_t X_BYTES = NTOK * BK * 2;  // 2 or 4 KiB (multiple of 1 KiB)
  static constexpr uint32_t RING_BYTES = STAGES * (W_BYTES + X_BYTES);
  static constexpr uint32_t TMEM_COLS = NTOK == 16 ? 32 : 64;  // two accumulators
  static constexpr uint32_t SMEM_BYTES = 1024 + RING_BYTES + 256;
};

struct SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t is_last;
  uint32_t seg_ok;
  uint32_t pre;  // the tile's other parts were added ahead of this CTA's own
};

// Brings one box of the tensor into L2 (no shared memory, no completion signal).  The
// prefetch returns nothing to the program, so it may run before the previous grid of the
// stream has finished: L2 is the device's point of coherence, and writes that the previous
// grid makes later land there too, so loads issued after the wait still see them.
__device__ __forceinline__ void tma_prefetch_l2_2d(const CUtensorMap* map, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t* a, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}

// Ticket with release and acquire semantics in one instruction: the parts stored before it
// (by all 128 epilogue threads, ordered by their group barrier) are visible to whoever sees
// the new count, and the parts of earlier ticket-takers are visible after it.  Measured
// 0.3-0.4 us a call faster than a fence followed by a relaxed atomic.
__device__ __forceinline__ uint32_t atom_add_acq_rel(uint32_t* a, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(a), "r"(v) : "memory");
  return old;
}

// A split-K part is [ntok / 4 float4 groups][128 columns]: a warp's stores and loads of one
// group cover 512 contiguous bytes.  Adds one column's values of one or two parts into s[],
// A's before B's (srcB may be null; the first nq groups carry rows of X), with all loads in
// flight together: under a full HBM stream an L2 round trip costs about a microsecond.
template <int NTOK, bool TWO>
__device__ __forceinline__ void add_parts(float (&s)[NTOK], const float4* srcA, const float4* srcB,
                                          int nq) {
  float4 a[NTOK / 4], b[TWO ? NTOK / 4 : 1];
  const bool two = TWO && srcB != nullptr;
#pragma unroll
  for (int q = 0; q < NTOK / 4; ++q)
    if (q < nq) a[q] = __ldcg(srcA + q * BNW);
  if (TWO && two) {
#pragma unroll
    for (int q = 0; q < NTOK / 4; ++q)
      if (q < nq) b[q] = __ldcg(srcB + q * BNW);
  }
#pragma unroll
  for (int q = 0; q < NTOK / 4; ++q) {
    if (q < nq) {
      s[4 * q] += a[q].x; s[4 * q + 1] += a[q].y; s[4 * q + 2] += a[q].z; s[4 * q + 3] += a[q].w;
    }
  }
  if (TWO && two) {
#pragma unroll
    for (int q = 0; q < NTOK / 4; ++q) {
      if (q < nq) {
        s[4 * q] += b[q].x; s[4 * q + 1] += b[q].y; s[4 * q + 2] += b[q].z; s[4 * q + 3] += b[q].w;
      }
    }
  }
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// One contiguous piece of a CTA's stream-K range that lies in a single W column tile.
template <typename IDX>
struct Segment {
  IDX tile;
  IDX kbeg, kend;  // K blocks [kbeg, kend) of that tile
};

// Walks CTA c's range [u0, u1) tile by tile.  IDX is uint32_t when units * ctas < 2^32, so
// the divisions on this path are 32-bit.
template <typename IDX>
struct SegmentWalk {
  IDX u, u1, kb;
  __device__ SegmentWalk(const ThinParams& p, IDX c)
      : u(sk_start<IDX>(c, static_cast<IDX>(p.units), static_cast<IDX>(p.ctas))),
        u1(sk_start<IDX>(c + 1, static_cast<IDX>(p.units), static_cast<IDX>(p.ctas))),
        kb(static_cast<IDX>(p.kblocks)) {}
  __device__ bool next(Segment<IDX>* s) {
    if (u >= u1) return false;
    s->tile = u / kb;
    s->kbeg = u - s->tile * kb;
    const IDX lim = u1 - s->tile * kb;
    s->kend = lim < kb ? lim : kb;
    u = s->tile * kb + s->kend;
    return true;
  }
};

// Writes column n of C for rows 0..M-1 from vals[] (one value per row of X).
template <int NTOK>
__device__ __forceinline__ void store_row(const ThinParams& p, int64_t n, const float (&vals)[NTOK]) {
  const int m = p.M < NTOK ? static_cast<int>(p.M) : NTOK;
  const float alpha = p.alpha, beta = p.beta;
  if (p.c_f32) {
    float* c = static_cast<float*>(p.C) + n;
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      if (t < m) *c = beta != 0.f ? fmaf(alpha, vals[t], beta * *c) : alpha * vals[t];
      c += p.ldc;
    }
  } else {
    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(p.C) + n;
#pragma unroll
    for (int t = 0; t < NTOK; ++t) {
      if (t < m) {
        const float x = beta != 0.f ? fmaf(alpha, vals[t], beta * __bfloat162float(*c)) : alpha * vals[t];
        *c = __float2bfloat16_rn(x);
      }
      c += p.ldc;
    }
  }
}

template <int NTOK, bool W_KMAJOR, typename IDX>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_thin_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                     const ThinParams p) {
  using Cfg = ThinCfg<NTOK>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t w_ring = ring;
  const uint32_t x_ring = ring + STAGES * W_BYTES;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem_raw + (ring - raw) + Cfg::RING_BYTES);
  volatile uint32_t* abort = &ctl->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const IDX c = blockIdx.x;
  const IDX units = static_cast<IDX>(p.units), ctas = static_cast<IDX>(p.ctas);
  const IDX kblocks = static_cast<IDX>(p.kblocks);

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
    ctl->seg_ok = 0;
    ctl->pre = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0) {
    tma_prefetch_map(&tmW);
    tma_prefetch_map(&tmX);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // Everything above touches only shared memory, TMEM and kernel parameters; it may overlap
  // the previous kernel of the stream.  The producer and the epilogue wait for the previous
  // grid (pdl_wait) before their first global access; the MMA issuer waits too, so that its
  // bounded waits start only once this grid's data can arrive.  The next grid is released
  // (pdl_trigger) by the producer once it has issued its last load: one CTA per SM fits, so
  // the next grid's CTAs take an SM only as this grid's leave it, and an earlier release
  // measured 1-1.5% slower.

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegmentWalk<IDX> walk(p, c);
      Segment<IDX> sg;
      uint32_t it = 0;
      bool ok = true;
      bool have = walk.next(&sg);  // index arithmetic before the wait
      if (PREFETCH > 0) {
        // The head of this CTA's range goes to L2 while the previous grid drains; the
        // loads below then find it there.
        const IDX u0 = sk_start<IDX>(c, units, ctas), u1 = sk_start<IDX>(c + 1, units, ctas);
        const IDX ue = u1 - u0 > static_cast<IDX>(PREFETCH) ? u0 + static_cast<IDX>(PREFETCH) : u1;
        for (IDX u = u0; u < ue; ++u) {
          const IDX tile = u / kblocks;
          const int32_t xn = static_cast<int32_t>(tile * BNW);
          const int32_t kx = static_cast<int32_t>((u - tile * kblocks) * BK);
          if (W_KMAJOR) {
            tma_prefetch_l2_2d(&tmW, kx, xn);
          } else {
            tma_prefetch_l2_2d(&tmW, xn, kx);
            if (xn + 64 < p.N) tma_prefetch_l2_2d(&tmW, xn + 64, kx);
          }
        }
      }
      pdl_wait();
      for (; ok && have; have = walk.next(&sg)) {
        const int32_t xn = static_cast<int32_t>(sg.tile * BNW);
        for (IDX kbi = sg.kbeg; kbi < sg.kend; ++kbi) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, W_BYTES + Cfg::X_BYTES);
          const int32_t kx = static_cast<int32_t>(kbi * BK);
          const uint32_t wdst = w_ring + s * W_BYTES;
          if (W_KMAJOR) {
            tma_load_2d(wdst, &tmW, fb, kx, xn);
          } else {
            tma_load_2d(wdst, &tmW, fb, xn, kx);
            tma_load_2d(wdst + 8192u, &tmW, fb, xn + 64, kx);
          }
          tma_load_2d(x_ring + s * Cfg::X_BYTES, &tmX, fb, kx, 0);
          ++it;
        }
      }
      pdl_trigger();
      if (!ok) {
        const uint32_t first = it > static_cast<uint32_t>(STAGES) ? it - STAGES : 0u;
        uint32_t never = 0;
        for (uint32_t j = first; j < it; ++j)
          mbar_wait(smem_u32(&ctl->full[j % STAGES]), (j / STAGES) & 1u, &never, p.status,
                    kDevTimeoutDrain);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      // A = W^T tile (128 W columns x 64 K): N-contiguous W is "MN-major" for the MMA.
      constexpr uint32_t idesc = idesc_bf16_f32(128, NTOK, !W_KMAJOR, false);
      SegmentWalk<IDX> walk(p, c);
      Segment<IDX> sg;
      uint32_t it = 0, lt = 0;
      bool ok = true;
      pdl_wait();
      while (ok && walk.next(&sg)) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        if (!mbar_wait(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort, p.status, kDevTimeoutMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + acc * NTOK;
        for (IDX kbi = sg.kbeg; kbi < sg.kend; ++kbi) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w0 = w_ring + s * W_BYTES, x0 = x_ring + s * Cfg::X_BYTES;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = W_KMAJOR ? sdesc_sw128(w0 + k * 32, 16, 1024)
                                            : sdesc_sw128(w0 + k * 2048, 8192, 1024);
            const uint64_t bdesc = sdesc_sw128(x0 + k * 32, 16, 1024);
            umma_bf16(d, adesc, bdesc, idesc, (kbi > sg.kbeg || k > 0) ? 1u : 0u);
          }
          umma_commit(smem_u32(&ctl->empty[s]));
          ++it;
        }
        if (!ok) break;
        umma_commit(smem_u32(&ctl->tfull[acc]));
        ++lt;
      }
      umma_commit(smem_u32(&ctl->drain));
      uint32_t never = 0;
      mbar_wait(smem_u32(&ctl->drain), 0, &never, p.status, kDevTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue / combine
    const int q = warp & 3;
    const int row = q * 32 + lane;  // W column within the tile
    const int etid = threadIdx.x - 64;
    // float4 groups per column that carry rows of X; the rest are never stored or read.
    const int nq = static_cast<int>(((p.M < NTOK ? p.M : NTOK) + 3) / 4);
    SegmentWalk<IDX> walk(p, c);
    Segment<IDX> sg;
    uint32_t lt = 0;
    pdl_wait();
    while (walk.next(&sg)) {
      const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
      const bool whole = sg.kbeg == 0 && sg.kend == kblocks;
      // kbeg == 0 on a shared tile: this CTA is the tile's first contributor, and this is
      // the last segment of its range.
      const bool head = sg.kbeg == 0 && !whole;
      const IDX first = sk_cta_of<IDX>(sg.tile * kblocks, units, ctas);
      const IDX last = sk_cta_of<IDX>((sg.tile + 1) * kblocks - 1, units, ctas);
      auto part_of = [&](IDX cc) {
        const int sl = sk_slot<IDX>(cc, sg.tile, kblocks, units, ctas);
        return reinterpret_cast<float4*>(p.ws) + (static_cast<int64_t>(cc) * 2 + sl) * BNW * (NTOK / 4) + row;
      };
      // Adds the first nk parts of the fixed order -- the contributors after the first in
      // CTA order, then the first CTA's part -- into acc_s[], this CTA's own from vals[] and
      // the others from the workspace, two per round trip.
      auto add_in_order = [&](float (&acc_s)[NTOK], const float (&vals)[NTOK], IDX nk) {
        auto order = [&](IDX k) { return k < last - first ? first + 1 + k : first; };
        for (IDX k = 0; k < nk;) {
          const IDX cc = order(k);
          if (cc == c) {
#pragma unroll
            for (int t = 0; t < NTOK; ++t) acc_s[t] += vals[t];
            ++k;
            continue;
          }
          const bool pair = k + 1 < nk && order(k + 1) != c;
          add_parts<NTOK, true>(acc_s, part_of(cc), pair ? part_of(order(k + 1)) : nullptr, nq);
          k += pair ? 2 : 1;
        }
      };
      float s[NTOK], v[NTOK];  // the combined sum; this CTA's own part
#pragma unroll
      for (int t = 0; t < NTOK; ++t) s[t] = 0.f;
      if (head) {
        // Watch the counter while this CTA's own part streams.  Once all other contributors
        // hold tickets none of them can be last, so this CTA combines: it resets the counter
        // and adds their parts now, leaving only its own for the end.  If its own part is
        // ready first, it takes a ticket like the others.
        if (etid == 0) {
          const uint32_t need = static_cast<uint32_t>(sk_contributors<IDX>(sg.tile, kblocks, units, ctas));
          uint32_t pre = 0;
          const uint64_t t0 = globaltimer_ns();
          for (;;) {
            if (ld_relaxed(&p.counters[sg.tile]) + 1u == need) {
              pre = 1;
              break;
            }
            if (mbar_test(smem_u32(&ctl->tfull[acc]), aph)) break;
            if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) break;  // the wait below reports
            __nanosleep(128);
          }
          if (pre) {
            fence_acq_rel_gpu();  // acquire: the parts are read after their tickets
            st_relaxed(&p.counters[sg.tile], 0u);  // ready for the next call
          }
          ctl->pre = pre;
        }
        epi_bar();
        if (ctl->pre) add_in_order(s, v, last - first);
      }
      const bool pre = head && ctl->pre;

      // One thread waits (bounded) and the 128 epilogue threads take the same decision
      // after the group barrier, so no thread is ever left alone in a barrier.
      if (etid == 0)
        ctl->seg_ok = mbar_wait(smem_u32(&ctl->tfull[acc]), aph, abort, p.status,
                                kDevTimeoutEpilogue) ? 1u : 0u;
      epi_bar();
      if (!ctl->seg_ok) break;
      tc_fence_after();
      {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * NTOK;
        if (NTOK == 16) {
          uint32_t r[16];
          tmem_ld_32x32b_x16(taddr, r);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < NTOK && t < 16; ++t) v[t] = __uint_as_float(r[t]);
        } else {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr, r);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < NTOK; ++t) v[t] = __uint_as_float(r[t]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
      ++lt;

      const int64_t n = static_cast<int64_t>(sg.tile) * BNW + row;
      if (whole) {
        // This CTA computed the whole K range of the tile: write C directly.
        if (n < p.N) store_row(p, n, v);
        epi_bar();  // seg_ok is rewritten for the next segment only after everyone read it
        continue;
      }
      if (pre) {
        // The other parts are in s[]; the first CTA's own part comes last.
#pragma unroll
        for (int t = 0; t < NTOK; ++t) s[t] += v[t];
        if (n < p.N) store_row(p, n, s);
        epi_bar();
        continue;
      }
      // Publish this CTA's part, then take a ticket.  The barrier orders the 128 threads'
      // stores before thread 0's ticket, whose release (cumulative) orders them before the
      // new count.  The last contributor to take a ticket combines (its own stored part goes
      // unused); the ticket's acquire orders the others' parts before its loads, and it
      // resets the counter at once, as every contributor already holds its ticket.
      {
        float4* dst = part_of(c);
#pragma unroll
        for (int g = 0; g < NTOK / 4; ++g)
          if (g < nq) __stcg(dst + g * BNW, make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
      }
      epi_bar();
      if (etid == 0) {
        const uint32_t need = static_cast<uint32_t>(sk_contributors<IDX>(sg.tile, kblocks, units, ctas));
        const uint32_t prev = atom_add_acq_rel(&p.counters[sg.tile], 1u);
        const bool is_last = prev + 1u == need;
        if (is_last) st_relaxed(&p.counters[sg.tile], 0u);
        ctl->is_last = is_last ? 1u : 0u;
      }
      epi_bar();
      if (ctl->is_last) {
        add_in_order(s, v, last - first + 1);
        if (n < p.N) store_row(p, n, s);
      }
      epi_bar();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

template <int NTOK, bool W_KMAJOR, typename IDX>
cudaError_t launch_thin_variant(const CUtensorMap& mw, const CUtensorMap& mx, const ThinParams& p,
                                cudaStream_t s) {
  auto kern = gemm_thin_kernel<NTOK, W_KMAJOR, IDX>;
  constexpr uint32_t smem = ThinCfg<NTOK>::SMEM_BYTES;
  static std::atomic<uint64_t> attr_done{0};
  cudaError_t e = ensure_smem_attr(kern, smem, attr_done);
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(static_cast<unsigned>(p.ctas)), dim3(NUM_THREADS), smem, s, mw, mx, p);
}

}  // namespace

cudaError_t launch_gemm_thin(const ThinParams& p, int ntok, const void* X, int64_t ldx,
                             const void* W, int64_t ldw, bool w_kmajor, cudaStream_t s) {
  CUtensorMap mw, mx;
  const bool ok_w = w_kmajor ? make_bf16_map(&mw, W, p.K, p.N, ldw, 1, 0, BK, BNW)
                             : make_bf16_map(&mw, W, p.N, p.K, ldw, 1, 0, 64, BK);
  if (!ok_w) return cudaErrorInvalidValue;
  if (!make_bf16_map(&mx, X, p.K, p.M, ldx, 1, 0, BK, ntok)) return cudaErrorInvalidValue;
  const bool small = sk_fits_u32(p.units, p.ctas);
#define DG_THIN_CASE(NT, KM)                                                          \
  if (ntok == NT && w_kmajor == KM)                                                   \
    return small ? launch_thin_variant<NT, KM, uint32_t>(mw, mx, p, s)                \
                 : launch_thin_variant<NT, KM, int64_t>(mw, mx, p, s);
  DG_THIN_CASE(16, false)
  DG_THIN_CASE(16, true)
  DG_THIN_CASE(32, false)
  DG_THIN_CASE(32, true)
#undef DG_THIN_CASE
  return cudaErrorInvalidValue;
}

}  // namespace dg
