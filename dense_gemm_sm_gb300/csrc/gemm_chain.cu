// gemm_chain.cu -- persistent multi-layer decode GEMM: y_{l+1} = bf16(y_l W_l), l < layers,
// for M <= 16 rows, in one launch ("Operator & Runtime", section 5.5.4: a kernel that stays
// resident, takes its tasks in order and checks with events that the data a task needs is
// ready; section 5.5.2: one submission instead of one per layer).
//
// Every layer is the decode GEMM of gemm_thin.cu -- 128 W columns x 64 K rows per unit, the
// layer's units split evenly (stream-K) over one CTA per SM, an 8-stage TMA ring, split
// tiles combined in a fixed order by one contributor -- and a CTA moves on to its range of
// the next layer as soon as it has finished its range of this one.  The event: the writer of
// each output tile (128 columns of y_{l+1}, all rows) counts it in the layer's tiles_done
// (release); the next layer's X loads wait for tiles_done == n_tiles (acquire).  Per-tile
// events would not let a layer start earlier: with a stream-K split almost every tile is
// shared by two or three CTAs and is finished only when its first CTA reaches the end of its
// range, i.e. at the end of the layer.  What the next layer must not wait for is its weight
// stream: the producer fills its whole ring with the next layer's W blocks (and has asked
// L2 for the head of its W range) before it waits, then adds the X blocks; so HBM keeps
// streaming while the previous layer's last tiles are combined.
//
// All CTAs must be resident at once (a CTA waits for tiles that other CTAs write): the grid
// is one CTA per SM, launched cooperatively, which the runtime guarantees or refuses.  The
// last CTA to finish resets the counters for the next call, so repeated calls (also from a
// replayed CUDA graph) need no host-side state; every wait is bounded.  Partition and
// combine order per layer are those of a single decode call, so each layer's result equals
// that call's bit for bit.
//
// Measured on GB300 (4 FFN-shaped layers of 96 MiB, M = 1): 86 us, against 78 us for the
// same four gemm_bf16 calls launched with programmatic dependent launch, which already
// overlaps each call's prologue and L2 prefetch with the previous call's tail -- the launch
// cost the pages' persistent kernel removes is mostly hidden there.  Without the
// cooperative attribute (DG_CHAIN_COOP=0: programmatic serialisation only, dependents launch
// only after every CTA of this grid has started, waits still bounded) the chain takes 81 us.
// Asking L2 for the head of a later layer's range at the boundary (DG_CHAIN_PREFETCH) made
// it slower at every depth tried (16 to 64 blocks): the previous layer still streams
// through L2 then.
#include <cuda_bf16.h>

#include <atomic>
#include <cstring>

#include "dg_internal.h"
#include "ptx.cuh"
#include "tile_sched.h"

namespace dg {

bool make_bf16_map(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t ld,
                   uint64_t batch, uint64_t stride, uint32_t box_inner, uint32_t box_outer);

namespace {

constexpr int NTOK = 16;
constexpr int BNW = kThinBN, BK = kThinBK;
constexpr uint32_t W_BYTES = BNW * BK * 2;   // 16 KiB per stage
constexpr uint32_t X_BYTES = NTOK * BK * 2;  // 2 KiB per stage
constexpr int STAGES = 8;
constexpr int PREFETCH = 32;
constexpr int NUM_THREADS = 192;
constexpr uint32_t TMEM_COLS = 32;  // two 16-column accumulators
constexpr uint32_t RING_BYTES = STAGES * (W_BYTES + X_BYTES);
constexpr uint32_t SMEM_BYTES = 1024 + RING_BYTES + 256;

struct ChainMaps {
  CUtensorMap w[kChainMax];
  CUtensorMap x[kChainMax];  // x[0] = X, x[l] = the output of layer l - 1
};

struct ChainCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort;
  uint32_t is_last;
  uint32_t seg_ok;
  uint32_t pre;
};
static_assert(sizeof(ChainCtl) <= 256, "control block");

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
__device__ __forceinline__ uint32_t ld_acquire(const uint32_t* a) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(uint32_t* a, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_acq_rel_gpu() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
}
// Orders this thread's generic-proxy global accesses with its async-proxy (TMA) ones.
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Waits (bounded) until *count >= want, with acquire semantics.
__device__ __forceinline__ bool wait_count(const uint32_t* count, uint32_t want, uint32_t sleep_ns,
                                           volatile uint32_t* abort, uint32_t* status) {
  if (ld_acquire(count) >= want) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ld_acquire(count) >= want) return true;
    if ((i & 15u) == 0) {
      if (*abort) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        atomicCAS(status, 0u, static_cast<uint32_t>(kDevTimeoutProducer));
        return false;
      }
    }
    __nanosleep(sleep_ns);
  }
}

template <bool TWO>
__device__ __forceinline__ void add_parts(float (&s)[NTOK], const float4* srcA, const float4* srcB,
                                          int nq) {
  float4 a[NTOK / 4], b[NTOK / 4];
  const bool two = TWO && srcB != nullptr;
#pragma unroll
  for (int q = 0; q < NTOK / 4; ++q)
    if (q < nq) a[q] = __ldcg(srcA + q * BNW);
  if (two) {
#pragma unroll
    for (int q = 0; q < NTOK / 4; ++q)
      if (q < nq) b[q] = __ldcg(srcB + q * BNW);
  }
#pragma unroll
  for (int q = 0; q < NTOK / 4; ++q)
    if (q < nq) {
      s[4 * q] += a[q].x; s[4 * q + 1] += a[q].y; s[4 * q + 2] += a[q].z; s[4 * q + 3] += a[q].w;
    }
  if (two) {
#pragma unroll
    for (int q = 0; q < NTOK / 4; ++q)
      if (q < nq) {
        s[4 * q] += b[q].x; s[4 * q + 1] += b[q].y; s[4 * q + 2] += b[q].z; s[4 * q + 3] += b[q].w;
      }
  }
}

struct Seg {
  uint32_t tile, kbeg, kend;
};
// CTA c's range of one layer, tile by tile.
struct SegWalk {
  uint32_t u, u1, kb;
  // CTAs c >= L.ctas take no part in the layer (a layer with fewer units than the grid is
  // split over L.ctas CTAs, one unit or more each, as a single decode call splits it).
  __device__ SegWalk(const ChainLayer& L, uint32_t c)
      : u(c < L.ctas ? sk_start<uint32_t>(c, L.units, L.ctas) : 0u),
        u1(c < L.ctas ? sk_start<uint32_t>(c + 1, L.units, L.ctas) : 0u), kb(L.kblocks) {}
  __device__ bool next(Seg* s) {
    if (u >= u1) return false;
    s->tile = u / kb;
    s->kbeg = u - s->tile * kb;
    const uint32_t lim = u1 - s->tile * kb;
    s->kend = lim < kb ? lim : kb;
    u = s->tile * kb + s->kend;
    return true;
  }
};

// Column n of the layer's output for rows 0 .. M-1, rounded once to BF16.
__device__ __forceinline__ void store_col(const ChainLayer& L, int64_t M, int64_t n,
                                          const float (&v)[NTOK]) {
  const int m = M < NTOK ? static_cast<int>(M) : NTOK;
  __nv_bfloat16* c = static_cast<__nv_bfloat16*>(L.C) + n;
#pragma unroll
  for (int t = 0; t < NTOK; ++t) {
    if (t < m) *c = __float2bfloat16_rn(v[t]);
    c += L.ldc;
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_chain_kernel(const __grid_constant__ ChainMaps maps, const ChainParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t ring = (raw + 1023u) & ~1023u;
  const uint32_t w_ring = ring;
  const uint32_t x_ring = ring + STAGES * W_BYTES;
  ChainCtl* ctl = reinterpret_cast<ChainCtl*>(smem_raw + (ring - raw) + RING_BYTES);
  volatile uint32_t* abort = &ctl->abort;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t c = blockIdx.x, G = p.ctas;

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
    for (int l = 0; l < p.layers; ++l) {
      tma_prefetch_map(&maps.w[l]);
      tma_prefetch_map(&maps.x[l]);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  // Shared memory, TMEM and parameters only above: this may overlap the previous kernel.
  pdl_trigger();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int l = 0; ok && l < p.layers; ++l) {
        const ChainLayer& L = p.L[l];
        const uint32_t kb = L.kblocks;
        const uint32_t Gl = L.ctas;
        const uint32_t u0 = c < Gl ? sk_start<uint32_t>(c, L.units, Gl) : 0u;
        const uint32_t u1 = c < Gl ? sk_start<uint32_t>(c + 1, L.units, Gl) : 0u;
        // The head of this layer's range goes to L2 now; it does not depend on the events.
        // (Layer 0 before the wait for the previous grid; later layers p.prefetch blocks,
        // 0 by default, since the previous layer still streams through L2.)
        const uint32_t pf = l == 0 ? static_cast<uint32_t>(PREFETCH) : p.prefetch;
        const uint32_t ue = u1 - u0 > pf ? u0 + pf : u1;
        for (uint32_t u = u0; u < ue; ++u) {
          const uint32_t tile = u / kb;
          const int32_t xn = static_cast<int32_t>(tile * BNW);
          const int32_t kx = static_cast<int32_t>((u - tile * kb) * BK);
          tma_prefetch_l2_2d(&maps.w[l], xn, kx);
          if (xn + 64 < L.N) tma_prefetch_l2_2d(&maps.w[l], xn + 64, kx);
        }
        if (l == 0) pdl_wait();  // first global loads: after the previous grid of the stream
        // Layer l > 0: the first min(STAGES, range) stages get their W blocks before the
        // wait for the previous layer, their X blocks after it.
        const uint32_t n_pre = l == 0 ? 0u : (u1 - u0 < static_cast<uint32_t>(STAGES) ? u1 - u0 : STAGES);
        for (uint32_t u = u0; ok && u < u1; ++u) {
          const uint32_t tile = u / kb, kbi = u - tile * kb;
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
          if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort, p.status, kDevTimeoutProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&ctl->full[s]);
          mbar_arrive_expect_tx(fb, W_BYTES + X_BYTES);
          const int32_t xn = static_cast<int32_t>(tile * BNW);
          const uint32_t wdst = w_ring + s * W_BYTES;
          tma_load_2d(wdst, &maps.w[l], fb, xn, static_cast<int32_t>(kbi * BK));
          tma_load_2d(wdst + 8192u, &maps.w[l], fb, xn + 64, static_cast<int32_t>(kbi * BK));
          if (u - u0 + 1 == n_pre) {
            // The ring is full of this layer's W: now wait for the previous layer's output
            // (on a timeout the X copies are still issued, so the stages complete and the
            // drain below ends; the status word reports the error), then load its X blocks.
            const ChainLayer& P = p.L[l - 1];
            if (!wait_count(P.tiles_done, P.n_tiles, p.poll_ns, abort, p.status)) ok = false;
            fence_proxy_async_global();
            for (uint32_t v = u0; v <= u; ++v) {
              const uint32_t jt = it - (u - v);
              const uint32_t vt = v / kb;
              tma_load_2d(x_ring + (jt % STAGES) * X_BYTES, &maps.x[l], smem_u32(&ctl->full[jt % STAGES]),
                          static_cast<int32_t>((v - vt * kb) * BK), 0);
            }
          } else if (u - u0 >= n_pre) {
            tma_load_2d(x_ring + s * X_BYTES, &maps.x[l], fb, static_cast<int32_t>(kbi * BK), 0);
          }
          ++it;
        }
      }
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
      // A = W^T tile (N-contiguous W is MN-major), B = X block (K-major), D^T in TMEM.
      constexpr uint32_t idesc = idesc_bf16_f32(128, NTOK, true, false);
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int l = 0; ok && l < p.layers; ++l) {
        SegWalk walk(p.L[l], c);
        Seg sg;
        while (ok && walk.next(&sg)) {
          const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
          if (!mbar_wait(smem_u32(&ctl->tempty[acc]), aph ^ 1u, abort, p.status, kDevTimeoutMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem_base + acc * NTOK;
          for (uint32_t kbi = sg.kbeg; kbi < sg.kend; ++kbi) {
            const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
            if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort, p.status, kDevTimeoutMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t w0 = w_ring + s * W_BYTES, x0 = x_ring + s * X_BYTES;
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
              umma_bf16(d, sdesc_sw128(w0 + k * 2048, 8192, 1024), sdesc_sw128(x0 + k * 32, 16, 1024),
                        idesc, (kbi > sg.kbeg || k > 0) ? 1u : 0u);
            umma_commit(smem_u32(&ctl->empty[s]));
            ++it;
          }
          if (!ok) break;
          umma_commit(smem_u32(&ctl->tfull[acc]));
          ++lt;
        }
      }
      umma_commit(smem_u32(&ctl->drain));
      uint32_t never = 0;
      mbar_wait(smem_u32(&ctl->drain), 0, &never, p.status, kDevTimeoutDrain);
    }
  } else {
    // ------------------------------------------------------------ epilogue / combine / events
    const int q = warp & 3;
    const int row = q * 32 + lane;  // W column within the tile
    const int etid = threadIdx.x - 64;
    const int nq = static_cast<int>(((p.M < NTOK ? p.M : NTOK) + 3) / 4);
    uint32_t lt = 0;
    bool ok = true;
    pdl_wait();
    for (int l = 0; ok && l < p.layers; ++l) {
      const ChainLayer& L = p.L[l];
      const uint32_t kblocks = L.kblocks, units = L.units, Gl = L.ctas;
      const bool publish = l + 1 < p.layers;
      SegWalk walk(L, c);
      Seg sg;
      while (walk.next(&sg)) {
        const uint32_t acc = lt & 1u, aph = (lt >> 1) & 1u;
        const bool whole = sg.kbeg == 0 && sg.kend == kblocks;
        const bool head = sg.kbeg == 0 && !whole;
        const uint32_t first = sk_cta_of<uint32_t>(sg.tile * kblocks, units, Gl);
        const uint32_t last = sk_cta_of<uint32_t>((sg.tile + 1) * kblocks - 1, units, Gl);
        auto part_of = [&](uint32_t cc) {
          const int sl = sk_slot<uint32_t>(cc, sg.tile, kblocks, units, Gl);
          return reinterpret_cast<float4*>(L.ws) + (static_cast<int64_t>(cc) * 2 + sl) * BNW * (NTOK / 4) + row;
        };
        auto add_in_order = [&](float (&acc_s)[NTOK], const float (&vals)[NTOK], uint32_t nk) {
          auto order = [&](uint32_t k) { return k < last - first ? first + 1 + k : first; };
          for (uint32_t k = 0; k < nk;) {
            const uint32_t cc = order(k);
            if (cc == c) {
#pragma unroll
              for (int t = 0; t < NTOK; ++t) acc_s[t] += vals[t];
              ++k;
              continue;
            }
            const bool two = k + 1 < nk && order(k + 1) != c;
            add_parts<true>(acc_s, part_of(cc), two ? part_of(order(k + 1)) : nullptr, nq);
            k += two ? 2 : 1;
          }
        };
        // The tile's output is complete: count it for the next layer's loads.
        auto signal = [&]() {
          fence_proxy_async_global();
          epi_bar();
          if (etid == 0) {
            fence_acq_rel_gpu();  // cumulative: the 128 threads' stores, ordered by the barrier
            atomicAdd(L.tiles_done, 1u);
          }
        };
        float s[NTOK], v[NTOK];
#pragma unroll
        for (int t = 0; t < NTOK; ++t) s[t] = 0.f;
        if (head) {
          if (etid == 0) {
            const uint32_t need = sk_contributors<uint32_t>(sg.tile, kblocks, units, Gl);
            uint32_t pre = 0;
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
              if (ld_relaxed(&L.counters[sg.tile]) + 1u == need) {
                pre = 1;
                break;
              }
              if (mbar_test(smem_u32(&ctl->tfull[acc]), aph)) break;
              if (*abort || globaltimer_ns() - t0 > kWaitLimitNs) break;
              __nanosleep(128);
            }
            if (pre) {
              fence_acq_rel_gpu();
              st_relaxed(&L.counters[sg.tile], 0u);
            }
            ctl->pre = pre;
          }
          epi_bar();
          if (ctl->pre) add_in_order(s, v, last - first);
        }
        const bool pre = head && ctl->pre;
        if (etid == 0)
          ctl->seg_ok = mbar_wait(smem_u32(&ctl->tfull[acc]), aph, abort, p.status,
                                  kDevTimeoutEpilogue) ? 1u : 0u;
        epi_bar();
        if (!ctl->seg_ok) {
          ok = false;
          break;
        }
        tc_fence_after();
        {
          uint32_t r[16];
          tmem_ld_32x32b_x16(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * NTOK, r);
          tmem_ld_wait();
#pragma unroll
          for (int t = 0; t < NTOK; ++t) v[t] = __uint_as_float(r[t]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&ctl->tempty[acc]));
        ++lt;

        const int64_t n = static_cast<int64_t>(sg.tile) * BNW + row;
        if (whole) {
          if (n < L.N) store_col(L, p.M, n, v);
          if (publish) signal();
          epi_bar();
          continue;
        }
        if (pre) {
#pragma unroll
          for (int t = 0; t < NTOK; ++t) s[t] += v[t];
          if (n < L.N) store_col(L, p.M, n, s);
          if (publish) signal();
          epi_bar();
          continue;
        }
        {
          float4* dst = part_of(c);
#pragma unroll
          for (int g = 0; g < NTOK / 4; ++g)
            if (g < nq) __stcg(dst + g * BNW, make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]));
        }
        epi_bar();
        if (etid == 0) {
          const uint32_t need = sk_contributors<uint32_t>(sg.tile, kblocks, units, Gl);
          fence_acq_rel_gpu();
          const uint32_t prev = atomicAdd(&L.counters[sg.tile], 1u);
          const bool is_last = prev + 1u == need;
          if (is_last) {
            fence_acq_rel_gpu();
            st_relaxed(&L.counters[sg.tile], 0u);
          }
          ctl->is_last = is_last ? 1u : 0u;
        }
        epi_bar();
        const bool combine = ctl->is_last != 0;
        if (combine) {
          add_in_order(s, v, last - first + 1);
          if (n < L.N) store_col(L, p.M, n, s);
        }
        if (combine && publish) signal();
        epi_bar();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0) {
    // The last CTA to finish resets the call's counters for the next call.
    fence_acq_rel_gpu();
    const uint32_t prev = atomicAdd(p.done, 1u);
    if (prev + 1u == G) {
      fence_acq_rel_gpu();
      for (int l = 0; l < p.layers; ++l) st_relaxed(p.L[l].tiles_done, 0u);
      st_relaxed(p.done, 0u);
    }
  }
}

std::atomic<uint64_t> g_chain_attr{0};

}  // namespace

cudaError_t launch_gemm_chain(const ChainParams& p, const void* X, int64_t ldx,
                              const void* const* W, const int64_t* ldw, cudaStream_t s, bool pdl,
                              bool coop) {
  ChainMaps maps;
  std::memset(&maps, 0, sizeof maps);
  for (int l = 0; l < p.layers; ++l) {
    const ChainLayer& L = p.L[l];
    if (!make_bf16_map(&maps.w[l], W[l], static_cast<uint64_t>(L.N), static_cast<uint64_t>(L.K),
                       static_cast<uint64_t>(ldw[l]), 1, 0, 64, BK))
      return cudaErrorInvalidValue;
    const void* xin = l == 0 ? X : p.L[l - 1].C;
    const int64_t ld = l == 0 ? ldx : p.L[l - 1].ldc;
    if (!make_bf16_map(&maps.x[l], xin, static_cast<uint64_t>(L.K), static_cast<uint64_t>(p.M),
                       static_cast<uint64_t>(ld), 1, 0, BK, NTOK))
      return cudaErrorInvalidValue;
  }
  cudaError_t e = ensure_smem_attr(gemm_chain_kernel, static_cast<int>(SMEM_BYTES), g_chain_attr);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.ctas);
  cfg.blockDim = dim3(NUM_THREADS);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (coop) {
    attr[n].id = cudaLaunchAttributeCooperative;  // all CTAs resident at once, or no launch
    attr[n].val.cooperative = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, gemm_chain_kernel, maps, p);
}

}  // namespace dg
