// api.cu -- the C ABI: argument checks, shape-based dispatch, workspace, status word.
//
// Dispatch (a static table keyed on dtype and shape class; chosen by measurement):
//   FP32                       -> SIMT kernel (vector-copy variant when rows are aligned)
//   BF16, batch == 1, M <= 32  -> thin stream-K kernel (HBM-bound decode shapes)
//   BF16 otherwise             -> persistent tcgen05 tile kernel, BN = 256 (128 when the
//                                 256-wide tiling leaves most SMs idle)
//   K == 0 or alpha == 0       -> C = beta*C (scale kernel)
// This is the "specialise per shape class with precompiled kernels" option of
// "Operator & Runtime" section 5.5.3: no run-time compilation, a fixed table.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "dg_internal.h"
#include "tile_sched.h"

namespace dg {

int g_fault_injection = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kRasterGroup = 8;
constexpr int64_t kThinMaxM = 32;
constexpr int kSimtCtasPerSmPlan = 2;  // occupancy of the SIMT kernel (launch bounds 256 x 2)

// Device status word: kernels record the first bounded-wait expiry here.
__device__ uint32_t g_status_word;

std::mutex g_mu;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

struct Workspace {
  float* ws = nullptr;
  size_t ws_floats = 0;
  uint32_t* counters = nullptr;
  size_t n_counters = 0;
};
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

// State of the persistent decode chain, per (device, stream), never shared with the other
// kernels: partials, and a word array [done, tiles_done[8], tickets[cap]] zeroed when
// allocated; the kernel leaves every word zero again at the end of a call.
struct ChainState {
  float* ws = nullptr;
  size_t ws_floats = 0;
  uint32_t* words = nullptr;
  size_t cap = 0;
};
std::map<std::pair<int, cudaStream_t>, ChainState> g_chain_states;

bool log_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("DG_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

cudaError_t current_device(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return e;
  if (*dev < 0 || *dev >= kMaxDevices) return cudaErrorInvalidDevice;
  return cudaSuccess;
}

// Status-word address and SM count of the current device (cached per device).
cudaError_t device_info(int dev, uint32_t** status, int* sms) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
    if (e != cudaSuccess) return e;
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    g_status_ptr[dev] = static_cast<uint32_t*>(p);
    g_num_sms[dev] = n;
  }
  *status = g_status_ptr[dev];
  *sms = g_num_sms[dev];
  return cudaSuccess;
}

// Workspace of (device, stream), grown to at least the requested sizes.  New counters are
// zeroed on the stream; the kernels leave them at zero when they finish.
dg_status get_workspace(int dev, cudaStream_t s, size_t ws_floats, size_t n_counters,
                        Workspace* out) {
  std::lock_guard<std::mutex> lock(g_mu);
  Workspace& w = g_workspaces[{dev, s}];
  if (w.ws_floats < ws_floats || w.n_counters < n_counters) {
    if (w.ws || w.counters) {
      // Earlier work on this stream may still use the old buffers.
      if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
      cudaFree(w.ws);
      cudaFree(w.counters);
      w = Workspace{};
    }
    const size_t nf = ws_floats > 0 ? ws_floats : 1;
    const size_t nc = n_counters > 0 ? n_counters : 1;
    if (cudaMalloc(&w.ws, nf * sizeof(float)) != cudaSuccess) {
      w = Workspace{};
      return DG_ERR_NO_MEMORY;
    }
    if (cudaMalloc(&w.counters, nc * sizeof(uint32_t)) != cudaSuccess) {
      cudaFree(w.ws);
      w = Workspace{};
      return DG_ERR_NO_MEMORY;
    }
    if (cudaMemsetAsync(w.counters, 0, nc * sizeof(uint32_t), s) != cudaSuccess)
      return DG_ERR_CUDA;
    w.ws_floats = nf;
    w.n_counters = nc;
  }
  *out = w;
  return DG_OK;
}

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ planning
// FP32: whole waves of tiles run data-parallel (one tile per CTA).  The tiles of the last,
// partial wave are split along K into S equal chunks, one CTA each, S chosen so that the
// tail takes the fewest tile-times: ceil(tail * S / resident) / S, with at least 256 of K
// per chunk and at most three waves of tail CTAs; the chunks of a tile are summed
// in K order by the last one to finish (a fixed order).
void plan_f32(int64_t M, int64_t N, int64_t K, int64_t batch, int64_t resident, dg_plan* pl,
              int64_t* dp_tiles, int64_t* sk_tiles, int* sk_splits, bool vec = true) {
  pl->kernel = DG_KERNEL_SIMT_F32;
  {
    // Small problems (128 x 128 tiles for under a quarter of the resident slots): 32 x 32
    // tiles, K in chunks of at least 4 pieces of 128 over at most as many CTAs as are
    // resident (at most 16 chunks).  tile_k reports the staged K piece.
    const int64_t T128 = batch * cdiv(M, kSimtBM) * cdiv(N, kSimtBN);
    const int64_t G = resident > 0 ? resident : 1;
    if (4 * T128 <= G) {
      const int64_t T = batch * cdiv(M, kSimtSmallT) * cdiv(N, kSimtSmallT);
      const int64_t pieces = cdiv(K, kSimtSmallKP);
      int64_t S = G / T;
      if (S > cdiv(pieces, 4)) S = cdiv(pieces, 4);
      if (S > 16) S = 16;
      if (S < 1) S = 1;
      if (const char* f = std::getenv("DG_SIMT_SPLITS")) {  // tuning override (sweeps)
        const int64_t v = std::atoi(f);
        if (v >= 1) S = v < pieces ? v : pieces;
      }
      pl->tile_m = kSimtSmallT;
      pl->tile_n = kSimtSmallT;
      pl->tile_k = kSimtSmallKP;
      pl->stages = 2;
      pl->group = 1;
      pl->tiles = T;
      pl->kblocks = pieces;
      pl->vec = 1;
      pl->splits = static_cast<int32_t>(S);
      pl->tail_tiles = S > 1 ? T : 0;
      pl->grid = T * S;
      pl->workspace_bytes = S > 1 ? T * S * kSimtSmallT * kSimtSmallT * 4 + T * 4 : 0;
      *sk_splits = static_cast<int>(S);
      *sk_tiles = S > 1 ? T : 0;
      *dp_tiles = -1;  // marks the small-tile kernel
      return;
    }
  }
  pl->tile_m = kSimtBM;
  pl->tile_n = kSimtBN;
  pl->tile_k = kSimtBK;
  pl->stages = kSimtStages;
  // Groups of 16 tile rows: on 4096^3 the DRAM traffic per call was 453 / 427 / 707 / 564 MB
  // with groups of 8 / 16 / 32 / 4 rows (two 128 x 128 tiles per SM: about ten tile rows
  // run together), the time the same.
  pl->group = 2 * kRasterGroup;
  pl->tiles = batch * cdiv(M, kSimtBM) * cdiv(N, kSimtBN);
  pl->kblocks = cdiv(K, kSimtBK);
  pl->vec = 1;
  const int64_t T = pl->tiles, KT = pl->kblocks, G = resident > 0 ? resident : 1;
  const int64_t tail = T % G;
  int best_s = 1;
  // Tuning override (sweeps): DG_SIMT_SPLITS=S forces S K chunks for the tail tiles.
  const char* force = std::getenv("DG_SIMT_SPLITS");
  const int forced = force ? std::atoi(force) : 0;
  if (tail > 0 && forced >= 1) {
    best_s = static_cast<int>(forced < KT ? forced : KT);
  } else if (tail > 0) {
    double best = 1.0;  // tail time (in tile times) without splitting
    // At least 256 of K per chunk, so a chunk outweighs its partial tile.
    const int64_t min_chunk = cdiv(256, kSimtBK);
    for (int64_t S = 2; S <= KT / min_chunk && tail * S <= 3 * G; ++S) {
      const double t = static_cast<double>(cdiv(tail * S, G)) / static_cast<double>(S);
      if (t < best - 1e-9) {
        best = t;
        best_s = static_cast<int>(S);
      }
    }
  }
  *sk_splits = best_s;
  *sk_tiles = best_s > 1 ? tail : 0;
  *dp_tiles = T - *sk_tiles;
  pl->splits = best_s;
  pl->tail_tiles = *sk_tiles;
  pl->grid = *dp_tiles + *sk_tiles * best_s;
  pl->workspace_bytes = *sk_tiles > 0 ? simt_ws_floats(*sk_tiles * best_s) * 4 + *sk_tiles * 4 : 0;
  // Stream-K (16-byte-aligned rows: the TMA kernel) when the tiles fill under one wave but
  // over a quarter of it and every resident CTA gets at least 4 K tiles: the units of all
  // tiles are split evenly over one wave of CTAs, so no CTA waits on a tail and every CTA
  // pays one pipeline fill (1000x3000x777: 113 -> 106 us).  With several waves the
  // data-parallel raster keeps the concurrent tiles in one group of tile rows, which reuses
  // the operands in L2 (4096^3: 2.19 ms against 2.26 ms stream-K).  Ranges must span at
  // most kSimtMaxSegments segments.  DG_SIMT_STREAMK=0/1 forces it off or on (sweeps).
  const int64_t U = T * KT;
  const char* fsk = std::getenv("DG_SIMT_STREAMK");
  bool sk = vec && T < G && U >= 4 * G;
  if (fsk) sk = vec && fsk[0] == '1' && U >= G;
  if (sk && cdiv(U, G) + 2 * KT > static_cast<int64_t>(kSimtMaxSegments - 1) * KT) sk = false;
  if (sk) {
    *sk_splits = 0;
    *sk_tiles = T;
    *dp_tiles = 0;
    pl->splits = 0;
    pl->tail_tiles = T;
    pl->grid = G;
    pl->workspace_bytes = simt_ws_floats(2 * G) * 4 + T * 4;
  }
}

// dual: the FFN gate/up form, planned as one GEMM over [W_g | W_u] (N = 2 x the output
// columns): always the tile kernel, 256-column tiles (128 output columns).
void plan_bf16(int64_t M, int64_t N, int64_t K, int64_t batch, int sms, dg_plan* pl,
               bool dual = false, bool fp8 = false) {
  if (!dual && !fp8 && batch == 1 && M <= kThinMaxM) {
    pl->kernel = DG_KERNEL_THIN_BF16;
    pl->ntok = M <= 16 ? 16 : 32;
    pl->tile_m = pl->ntok;
    pl->tile_n = kThinBN;
    pl->tile_k = kThinBK;
    pl->stages = 8;
    pl->group = 1;
    pl->tiles = cdiv(N, kThinBN);
    pl->kblocks = cdiv(K, kThinBK);
    const int64_t units = pl->tiles * pl->kblocks;
    pl->grid = units < sms ? units : sms;
    pl->workspace_bytes =
        thin_ws_floats(pl->grid, pl->ntok) * 4 + pl->tiles * static_cast<int64_t>(sizeof(uint32_t));
    return;
  }
  pl->kernel = DG_KERNEL_TC_BF16;
  // Tile width, from a measured sweep over 128..256 on FFN, square (2048..8192) and wide
  // shapes: 256 is fastest everywhere (narrower tiles load more B bytes per FLOP, which
  // costs more than the better wave fill they buy), so 128 is used only when N <= 128.
  int bn = N <= 128 && !dual ? 128 : 256;
  // Tuning override (bench and sweeps): DG_TC_BN=256|224|192|128 forces the tile width.
  if (const char* e = (dual || fp8) ? nullptr : std::getenv("DG_TC_BN")) {
    const int f = std::atoi(e);
    if (f == 256 || f == 224 || f == 192 || f == 128) bn = f;
  }
  pl->tile_m = kTcBM;
  pl->tile_n = bn;
  pl->tile_k = kTcBK;
  pl->stages = bn >= 192 ? 4 : 6;
  pl->group = kRasterGroup;
  pl->tiles = batch * cdiv(M, kTcBM) * cdiv(N, bn);
  pl->grid = pl->tiles < sms ? pl->tiles : sms;
  // A stage row is 128 bytes: 64 BF16 or 128 FP8 elements of K.
  pl->tile_k = fp8 ? 2 * kTcBK : kTcBK;
  pl->kblocks = cdiv(K, pl->tile_k);
  // CTA pairs (tcgen05 cta_group::2, 256 x 256 tiles) for one problem with at least two
  // 128-row tile rows: each SM then moves half the B bytes per FLOP through its shared
  // memory, which bounds the single-CTA tile.  DG_TC_PAIR=0 keeps single CTAs (sweeps).
  const char* pe = std::getenv("DG_TC_PAIR");
  const bool pair = batch == 1 && bn == 256 && cdiv(M, kTcBM) >= 2 && sms >= 2 &&
                    !(pe && pe[0] == '0');
  if (pair) {
    pl->kernel = DG_KERNEL_TC2_BF16;
    pl->tile_m = 2 * kTcBM;
    // FP8 pairs also come 224 columns wide (112 B rows per CTA).  The width with the smaller
    // tile-waves x width wins, 256 on a tie: on the FFN shape 4 x 55 tiles of 224 fill 3
    // waves of 76 pairs to 96% where 4 x 48 tiles of 256 fill them to 84%.
    if (fp8) {
      const int64_t G2 = sms / 2, tm2 = cdiv(cdiv(M, kTcBM), 2);
      const int64_t w256 = cdiv(tm2 * cdiv(N, 256), G2) * 256, w224 = cdiv(tm2 * cdiv(N, 224), G2) * 224;
      if (w224 < w256) {
        bn = 224;
        pl->tile_n = bn;
      }
    }
    // BF16 pairs stage two 128-byte K atoms (128 elements) in 3 stages, FP8 pairs one atom
    // (128 elements) in 6 (gemm_tc.cu, TcCfg).
    pl->stages = fp8 ? 6 : 3;
    if (!fp8) pl->tile_k *= 2;
    pl->kblocks = cdiv(K, pl->tile_k);
    pl->group = kRasterGroup / 2;  // in 256-row tile rows: the same 8 rows of 128
    pl->tiles = cdiv(cdiv(M, kTcBM), 2) * cdiv(N, bn);
    const int64_t clusters = pl->tiles < sms / 2 ? pl->tiles : sms / 2;
    pl->grid = 2 * clusters;
  }
  const int64_t G = pair ? pl->grid / 2 : pl->grid;  // CTAs, or CTA pairs, that share the work
  // A partial last wave runs first, stream-K style (its tiles' K blocks spread over the
  // CTAs), when the whole waves that follow are long enough to hide the combine -- at
  // least 96 K blocks per CTA (measured: 2 waves of K = 4096 hide it, 1 wave of K = 1024
  // does not, where the combine made the call 2.3x slower) -- and a tile has at least 16
  // K blocks, so a piece is worth its partial tile (with 2, as in attention scores with
  // d = 128, the partials cost a quarter of the call).  Each tail tile is shared by at
  // most 4 CTAs.  tail_tiles = the stream-K tiles, splits = the CTAs sharing them.
  pl->splits = 1;
  pl->tail_tiles = 0;
  // The thresholds count 128-byte K atoms (a pair's stage holds two).
  const int64_t katoms = pl->kblocks * (pair && !fp8 ? 2 : 1);
  if (pl->tiles > G && pl->tiles % G != 0 && katoms >= 16 && (pl->tiles / G) * katoms >= 96) {
    pl->tail_tiles = pl->tiles % G;
    const int64_t c4 = 4 * pl->tail_tiles;
    pl->splits = static_cast<int32_t>(c4 < G ? c4 : G);
    const int64_t per = pair ? 2 : 1;  // partials and counters per stream-K unit
    pl->workspace_bytes = tc_ws_floats(per * pl->splits, bn) * 4 +
                          per * pl->tail_tiles * static_cast<int64_t>(sizeof(uint32_t));
  }
}

dg_status plan(int32_t dtype, int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
               int sms, dg_plan* pl) {
  *pl = dg_plan{};
  if (M == 0 || N == 0 || batch == 0) {
    pl->kernel = DG_KERNEL_NONE;
    return DG_OK;
  }
  if (K == 0 || alpha == 0.f) {
    pl->kernel = DG_KERNEL_SCALE;
    return DG_OK;
  }
  if (dtype == 0) {
    int64_t dp = 0, sk = 0;
    int splits = 1;
    plan_f32(M, N, K, batch, static_cast<int64_t>(sms) * kSimtCtasPerSmPlan, pl, &dp, &sk,
             &splits);
  } else {
    plan_bf16(M, N, K, batch, sms, pl, false, dtype == 2);
  }
  return DG_OK;
}

void log_plan(const char* who, int64_t M, int64_t N, int64_t K, int64_t batch, const dg_plan& pl) {
  if (!log_enabled()) return;
  std::fprintf(stderr,
               "[dgemm] %s M=%lld N=%lld K=%lld batch=%lld -> kernel=%d tile=%dx%dx%d stages=%d "
               "grid=%lld tiles=%lld ntok=%d\n",
               who, (long long)M, (long long)N, (long long)K, (long long)batch, pl.kernel,
               pl.tile_m, pl.tile_n, pl.tile_k, pl.stages, (long long)pl.grid, (long long)pl.tiles,
               pl.ntok);
}

dg_status check_common(int64_t M, int64_t N, int64_t K, int64_t batch, int64_t lda, int64_t ldb,
                       int64_t ldc, dg_op op_b, int64_t sA, int64_t sB, int64_t sC) {
  if (M < 0 || N < 0 || K < 0 || batch < 0) return DG_ERR_INVALID_ARG;
  if (op_b != DG_OP_N && op_b != DG_OP_T) return DG_ERR_INVALID_ARG;
  if (M == 0 || N == 0 || batch == 0) return DG_OK;
  if (ldc < N) return DG_ERR_INVALID_ARG;
  if (K > 0) {
    if (lda < K) return DG_ERR_INVALID_ARG;
    if (op_b == DG_OP_N ? ldb < N : ldb < K) return DG_ERR_INVALID_ARG;
  }
  if (batch > 1 && (sA < 0 || sB < 0 || sC < 0)) return DG_ERR_INVALID_ARG;
  // Tile coordinates and TMA coordinates are 32-bit.
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX || batch > INT32_MAX)
    return DG_ERR_UNSUPPORTED;
  return DG_OK;
}

dg_status from_cuda(cudaError_t e) { return e == cudaSuccess ? DG_OK : DG_ERR_CUDA; }

dg_status run_scale(void* C, bool f32, int64_t M, int64_t N, int64_t ldc, int64_t sC, int64_t batch,
                    float beta, cudaStream_t s) {
  if (!C) return DG_ERR_INVALID_ARG;
  return from_cuda(launch_scale(C, f32, M, N, ldc, sC, batch, beta, s));
}

dg_status f32_impl(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
                   int64_t sA, const float* B, int64_t ldb, int64_t sB, dg_op op_b, float beta,
                   float* C, int64_t ldc, int64_t sC, int64_t batch, void* stream) {
  dg_status st = check_common(M, N, K, batch, lda, ldb, ldc, op_b, sA, sB, sC);
  if (st != DG_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (M == 0 || N == 0 || batch == 0) return DG_OK;
  if (K == 0 || alpha == 0.f) return run_scale(C, true, M, N, ldc, sC, batch, beta, s);
  if (!A || !B || !C) return DG_ERR_INVALID_ARG;
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  const bool vec = aligned16(A) && aligned16(B) && aligned16(C) && lda % 4 == 0 &&
                   ldb % 4 == 0 && ldc % 4 == 0 &&
                   (batch <= 1 || (sA % 4 == 0 && sB % 4 == 0 && sC % 4 == 0));
  const bool trans_b = op_b == DG_OP_T;
  const int64_t resident =
      static_cast<int64_t>(sms) * sgemm_simt_ctas_per_sm(trans_b, vec);
  dg_plan pl = dg_plan{};
  int64_t dp = 0, sk = 0;
  int splits = 1;
  plan_f32(M, N, K, batch, resident, &pl, &dp, &sk, &splits, vec);
  log_plan("gemm_f32", M, N, K, batch, pl);
  if (pl.tiles > INT32_MAX || pl.grid > INT32_MAX) return DG_ERR_UNSUPPORTED;
  SimtParams p;
  p.M = M; p.N = N; p.K = K;
  p.alpha = alpha; p.beta = beta;
  p.A = A; p.lda = lda; p.strideA = batch > 1 ? sA : 0;
  p.B = B; p.ldb = ldb; p.strideB = batch > 1 ? sB : 0;
  p.C = C; p.ldc = ldc; p.strideC = batch > 1 ? sC : 0;
  p.batch = batch;
  p.tiles_m = cdiv(M, kSimtBM);
  p.tiles_n = cdiv(N, kSimtBN);
  p.group = pl.group;
  if (const char* e = std::getenv("DG_SIMT_GROUP")) {  // tuning override (sweeps)
    const int g = std::atoi(e);
    if (g >= 1 && g <= 4096) p.group = g;
  }
  p.dp_tiles = dp;
  p.sk_tiles = sk;
  p.sk_splits = splits;
  p.ws = nullptr;
  p.counters = nullptr;
  p.status = status;
  p.sk_units = 0;
  p.sk_ctas = 0;
  if (dp < 0) {  // small problem: 32 x 32 tiles
    p.tiles_m = cdiv(M, kSimtSmallT);
    p.tiles_n = cdiv(N, kSimtSmallT);
    p.dp_tiles = 0;
    p.sk_tiles = sk;
    p.sk_splits = splits;
    if (splits > 1) {
      Workspace w;
      st = get_workspace(dev, s, static_cast<size_t>(pl.tiles * splits * kSimtSmallT * kSimtSmallT),
                         static_cast<size_t>(pl.tiles), &w);
      if (st != DG_OK) return st;
      p.ws = w.ws;
      p.counters = w.counters;
    }
    return from_cuda(launch_sgemm_simt_small(p, trans_b, vec, s));
  }
  if (splits == 0) {  // stream-K over all tiles
    p.sk_units = pl.tiles * pl.kblocks;
    p.sk_ctas = pl.grid;
    p.dp_tiles = 0;
    p.sk_tiles = 0;
    p.sk_splits = 1;
    Workspace w;
    st = get_workspace(dev, s, static_cast<size_t>(simt_ws_floats(2 * pl.grid)),
                       static_cast<size_t>(pl.tiles), &w);
    if (st != DG_OK) return st;
    p.ws = w.ws;
    p.counters = w.counters;
  } else if (sk > 0) {
    Workspace w;
    st = get_workspace(dev, s, static_cast<size_t>(simt_ws_floats(sk * splits)),
                       static_cast<size_t>(sk), &w);
    if (st != DG_OK) return st;
    p.ws = w.ws;
    p.counters = w.counters;
  }
  return from_cuda(launch_sgemm_simt(p, trans_b, vec, s));
}

// The tile kernels (single CTAs or pairs) for a planned BF16 problem.  B2 non-null selects
// the FFN gate/up form (C = SiLU(bf16(A B)) * bf16(A B2), N output columns).
dg_status run_tile(const dg_plan& pl, int64_t M, int64_t N, int64_t K, int64_t batch, float alpha,
                   float beta, const uint16_t* A, int64_t lda, int64_t sA, const uint16_t* B,
                   int64_t ldb, int64_t sB, dg_op op_b, void* C, int64_t ldc, int64_t sC,
                   bool c_f32, bool c_vec, uint32_t* status, int dev, cudaStream_t s,
                   const uint16_t* B2, int64_t ldb2, const float* scale_a = nullptr,
                   const float* scale_b = nullptr) {
  dg_status st = DG_OK;
  TcParams p;
  p.M = M; p.N = N; p.K = K;
  p.batch = batch;
  const bool pair = pl.kernel == DG_KERNEL_TC2_BF16;
  p.tiles_m = pair ? cdiv(cdiv(M, kTcBM), 2) : cdiv(M, kTcBM);
  p.tiles_n = cdiv(N, B2 ? pl.tile_n / 2 : pl.tile_n);  // gate/up: 128 output columns a tile
  p.total_tiles = pl.tiles;
  p.kblocks = static_cast<int32_t>(pl.kblocks);
  p.group = pl.group;
  p.alpha = alpha; p.beta = beta;
  p.C = C; p.ldc = ldc; p.strideC = batch > 1 ? sC : 0;
  p.c_f32 = c_f32 ? 1 : 0;
  p.c_vec = c_vec ? 1 : 0;
  p.c_tma = (c_vec && beta == 0.f) ? 1 : 0;
  p.status = status;
  p.sk_tiles = pl.tail_tiles;
  p.dp_tiles = pl.tiles - pl.tail_tiles;
  p.sk_ctas = pl.tail_tiles > 0 ? pl.splits : 0;
  p.ws = nullptr;
  p.counters = nullptr;
  p.scale_a = scale_a;
  p.scale_b = scale_b;
  if (p.sk_tiles > 0) {
    Workspace w;
    const int64_t per = pair ? 2 : 1;
    st = get_workspace(dev, s, static_cast<size_t>(tc_ws_floats(per * p.sk_ctas, pl.tile_n)),
                       static_cast<size_t>(per * p.sk_tiles), &w);
    if (st != DG_OK) return st;
    p.ws = w.ws;
    p.counters = w.counters;
  }
  return from_cuda(launch_gemm_tc(p, pl.tile_n, A, lda, batch > 1 ? sA : 0, B, ldb,
                                  batch > 1 ? sB : 0, op_b == DG_OP_T, pair,
                                  static_cast<int>(pl.grid), s, B2, ldb2, scale_a != nullptr));
}


dg_status bf16_impl(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t* A, int64_t lda,
                    int64_t sA, const uint16_t* B, int64_t ldb, int64_t sB, dg_op op_b,
                    float beta, void* C, int64_t ldc, int64_t sC, int64_t batch, dg_out c_type,
                    void* stream) {
  dg_status st = check_common(M, N, K, batch, lda, ldb, ldc, op_b, sA, sB, sC);
  if (st != DG_OK) return st;
  if (c_type != DG_OUT_BF16 && c_type != DG_OUT_F32) return DG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool c_f32 = c_type == DG_OUT_F32;
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  dg_plan pl;
  plan(1, M, N, K, batch, alpha, sms, &pl);
  log_plan("gemm_bf16", M, N, K, batch, pl);
  if (pl.kernel == DG_KERNEL_NONE) return DG_OK;
  if (pl.kernel == DG_KERNEL_SCALE) return run_scale(C, c_f32, M, N, ldc, sC, batch, beta, s);
  if (!A || !B || !C) return DG_ERR_INVALID_ARG;
  // TMA: 16-byte aligned bases and row / batch strides that are multiples of 16 bytes.
  if (!aligned16(A) || !aligned16(B) || lda % 8 != 0 || ldb % 8 != 0) return DG_ERR_MISALIGNED;
  if (batch > 1 && (sA % 8 != 0 || sB % 8 != 0)) return DG_ERR_MISALIGNED;
  const int esz = c_f32 ? 4 : 2;
  const bool c_vec = aligned16(C) && (ldc * esz) % 16 == 0 && (batch <= 1 || (sC * esz) % 16 == 0);

  if (pl.kernel == DG_KERNEL_THIN_BF16) {
    Workspace w;
    st = get_workspace(dev, s, static_cast<size_t>(thin_ws_floats(pl.grid, pl.ntok)),
                       static_cast<size_t>(pl.tiles), &w);
    if (st != DG_OK) return st;
    ThinParams p;
    p.M = M; p.N = N; p.K = K;
    p.n_tiles = pl.tiles;
    p.kblocks = pl.kblocks;
    p.units = pl.tiles * pl.kblocks;
    p.ctas = pl.grid;
    p.alpha = alpha; p.beta = beta;
    p.C = C; p.ldc = ldc;
    p.c_f32 = c_f32 ? 1 : 0;
    p.ws = w.ws;
    p.counters = w.counters;
    p.status = status;
    return from_cuda(launch_gemm_thin(p, pl.ntok, A, lda, B, ldb, op_b == DG_OP_T, s));
  }

  return run_tile(pl, M, N, K, batch, alpha, beta, A, lda, sA, B, ldb, sB, op_b, C, ldc, sC,
                  c_f32, c_vec, status, dev, s, nullptr, 0);
}

// ------------------------------------------------------------------ scale kernel
template <typename T>
__global__ void scale_kernel(T* C, int64_t M, int64_t N, int64_t ldc, int64_t sC, int64_t batch,
                             float beta) {
  const int64_t total = batch * M * N;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t b = i / (M * N);
    const int64_t r = i - b * M * N;
    const int64_t m = r / N, n = r - m * N;
    T* c = C + b * sC + m * ldc + n;
    if constexpr (sizeof(T) == 4) {
      *c = beta != 0.f ? beta * *c : 0.f;
    } else {
      const float v = beta != 0.f ? beta * __bfloat162float(*c) : 0.f;
      *c = __float2bfloat16_rn(v);
    }
  }
}

}  // namespace

cudaError_t device_status_word(int dev, uint32_t** status, int* sms) {
  return device_info(dev, status, sms);
}

cudaError_t launch_scale(void* C, bool c_f32, int64_t M, int64_t N, int64_t ldc, int64_t strideC,
                         int64_t batch, float beta, cudaStream_t s) {
  const int64_t total = batch * M * N;
  // A grid-stride loop over at most 32 blocks of 256 threads per SM of this device.
  int dev = 0;
  cudaError_t e = current_device(&dev);
  if (e != cudaSuccess) return e;
  uint32_t* status = nullptr;
  int sms = 0;
  e = device_info(dev, &status, &sms);
  if (e != cudaSuccess) return e;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 1) * 32;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (c_f32)
    scale_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<float*>(C), M, N, ldc, strideC, batch, beta);
  else
    scale_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(C), M, N, ldc, strideC, batch, beta);
  return cudaGetLastError();
}

}  // namespace dg

// ==================================================================== C ABI
using namespace dg;

extern "C" {

dg_status gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
                   const float* B, int64_t ldb, float beta, float* C, int64_t ldc, void* stream) {
  return f32_impl(M, N, K, alpha, A, lda, 0, B, ldb, 0, DG_OP_N, beta, C, ldc, 0, 1, stream);
}

dg_status gemm_f32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                                   int64_t lda, int64_t strideA, const float* B, int64_t ldb,
                                   int64_t strideB, dg_op op_b, float beta, float* C, int64_t ldc,
                                   int64_t strideC, int64_t batch, void* stream) {
  return f32_impl(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, op_b, beta, C, ldc, strideC,
                  batch, stream);
}

dg_status gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t* A, int64_t lda,
                    const uint16_t* B, int64_t ldb, float beta, void* C, int64_t ldc,
                    dg_out c_type, void* stream) {
  return bf16_impl(M, N, K, alpha, A, lda, 0, B, ldb, 0, DG_OP_N, beta, C, ldc, 0, 1, c_type,
                   stream);
}

dg_status gemm_bf16_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                    const uint16_t* A, int64_t lda, int64_t strideA,
                                    const uint16_t* B, int64_t ldb, int64_t strideB, dg_op op_b,
                                    float beta, void* C, int64_t ldc, int64_t strideC,
                                    int64_t batch, dg_out c_type, void* stream) {
  return bf16_impl(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, op_b, beta, C, ldc, strideC,
                   batch, c_type, stream);
}

dg_status gemm_bf16_gate_up_silu(int64_t M, int64_t N, int64_t K, const uint16_t* X, int64_t ldx,
                                 const uint16_t* Wg, int64_t ldwg, const uint16_t* Wu,
                                 int64_t ldwu, uint16_t* Z, int64_t ldz, void* stream) {
  if (M < 0 || N < 0 || K < 0) return DG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return DG_OK;
  if (ldz < N || (K > 0 && (ldx < K || ldwg < N || ldwu < N))) return DG_ERR_INVALID_ARG;
  if (!Z) return DG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  // K == 0: G = U = 0 and SiLU(0) * 0 = 0.
  if (K == 0) return run_scale(Z, false, M, N, ldz, 0, 1, 0.f, s);
  if (!X || !Wg || !Wu) return DG_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(Wg) || !aligned16(Wu) || ldx % 8 != 0 || ldwg % 8 != 0 ||
      ldwu % 8 != 0)
    return DG_ERR_MISALIGNED;
  dg_plan pl;
  plan_bf16(M, 2 * N, K, 1, sms, &pl, true);
  log_plan("gemm_bf16_gate_up_silu", M, N, K, 1, pl);
  const bool c_vec = aligned16(Z) && (ldz * 2) % 16 == 0;
  return run_tile(pl, M, N, K, 1, 1.f, 0.f, X, ldx, 0, Wg, ldwg, 0, DG_OP_N, Z, ldz, 0, false,
                  c_vec, status, dev, s, Wu, ldwu);
}

dg_status quantize_rows_e4m3(int64_t rows, int64_t cols, const uint16_t* X, int64_t ldx,
                             uint8_t* Q, int64_t ldq, float* scales, void* stream) {
  if (rows < 0 || cols < 0) return DG_ERR_INVALID_ARG;
  if (rows == 0) return DG_OK;
  if (ldx < cols || ldq < cols || !scales || (cols > 0 && (!X || !Q))) return DG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  const bool vec = aligned16(X) && aligned16(Q) && ldx % 8 == 0 && ldq % 16 == 0;
  return from_cuda(launch_quantize_rows(rows, cols, X, ldx, Q, ldq, scales, vec, sms, s));
}

dg_status gemm_fp8_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                        const float* scale_a, const uint8_t* B, int64_t ldb, const float* scale_b,
                        void* C, int64_t ldc, dg_out c_type, void* stream) {
  if (M < 0 || N < 0 || K < 0) return DG_ERR_INVALID_ARG;
  if (c_type != DG_OUT_BF16 && c_type != DG_OUT_F32) return DG_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return DG_OK;
  if (ldc < N || !C || (K > 0 && (lda < K || ldb < K || !A || !B || !scale_a || !scale_b)))
    return DG_ERR_INVALID_ARG;
  const bool c_f32 = c_type == DG_OUT_F32;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  if (K == 0) return run_scale(C, c_f32, M, N, ldc, 0, 1, 0.f, s);  // empty sums: C = 0
  if (!aligned16(A) || !aligned16(B) || lda % 16 != 0 || ldb % 16 != 0 || !aligned16(scale_b) ||
      (reinterpret_cast<uintptr_t>(scale_a) & 3u) != 0)
    return DG_ERR_MISALIGNED;
  dg_plan pl;
  plan_bf16(M, N, K, 1, sms, &pl, false, true);
  log_plan("gemm_fp8_e4m3", M, N, K, 1, pl);
  const bool c_vec = aligned16(C) && (ldc * (c_f32 ? 4 : 2)) % 16 == 0;
  return run_tile(pl, M, N, K, 1, 1.f, 0.f, reinterpret_cast<const uint16_t*>(A), lda, 0,
                  reinterpret_cast<const uint16_t*>(B), ldb, 0, DG_OP_T, C, ldc, 0, c_f32, c_vec,
                  status, dev, s, nullptr, 0, scale_a, scale_b);
}

dg_status gemm_bf16_decode_chain(int32_t layers, int64_t M, const int64_t* dims, const uint16_t* X,
                                 int64_t ldx, const uint16_t* const* W, const int64_t* ldw,
                                 uint16_t* const* Y, void* stream) {
  if (layers < 1 || layers > kChainMax || M < 0 || !dims || !W || !ldw || !Y) return DG_ERR_INVALID_ARG;
  if (M == 0) return DG_OK;
  if (M > 16) return DG_ERR_UNSUPPORTED;
  for (int l = 0; l <= layers; ++l)
    if (dims[l] <= 0) return DG_ERR_INVALID_ARG;
  if (!X || ldx < dims[0]) return DG_ERR_INVALID_ARG;
  for (int l = 0; l < layers; ++l)
    if (!W[l] || !Y[l] || ldw[l] < dims[l + 1]) return DG_ERR_INVALID_ARG;
  if (!aligned16(X) || ldx % 8 != 0) return DG_ERR_MISALIGNED;
  for (int l = 0; l < layers; ++l)
    if (!aligned16(W[l]) || ldw[l] % 8 != 0 || !aligned16(Y[l]) ||
        (l + 1 < layers && dims[l + 1] % 8 != 0))
      return DG_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  ChainParams p;
  std::memset(&p, 0, sizeof p);
  p.layers = layers;
  p.M = M;
  p.ctas = static_cast<uint32_t>(sms);
  p.status = status;
  size_t tiles = 0;
  for (int l = 0; l < layers; ++l) {
    const int64_t n_tiles = cdiv(dims[l + 1], kThinBN), kb = cdiv(dims[l], kThinBK);
    if (!sk_fits_u32(n_tiles * kb, sms)) return DG_ERR_UNSUPPORTED;
    tiles += static_cast<size_t>(n_tiles);
  }
  const size_t per_layer = static_cast<size_t>(thin_ws_floats(sms, 16));
  ChainState st;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ChainState& cs = g_chain_states[{dev, s}];
    if (cs.ws_floats < per_layer * layers || cs.cap < tiles) {
      if (cs.ws || cs.words) {
        if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
        cudaFree(cs.ws);
        cudaFree(cs.words);
        cs = ChainState{};
      }
      size_t cap = 4096;
      while (cap < tiles) cap *= 2;
      const size_t nf = per_layer * kChainMax;
      if (cudaMalloc(&cs.ws, nf * sizeof(float)) != cudaSuccess) {
        cs = ChainState{};
        return DG_ERR_NO_MEMORY;
      }
      if (cudaMalloc(&cs.words, (1 + kChainMax + cap) * sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(cs.ws);
        cs = ChainState{};
        return DG_ERR_NO_MEMORY;
      }
      if (cudaMemsetAsync(cs.words, 0, (1 + kChainMax + cap) * sizeof(uint32_t), s) != cudaSuccess)
        return DG_ERR_CUDA;
      cs.ws_floats = nf;
      cs.cap = cap;
    }
    st = cs;
  }
  p.done = st.words;
  size_t off = 0;
  for (int l = 0; l < layers; ++l) {
    ChainLayer& L = p.L[l];
    L.N = dims[l + 1];
    L.K = dims[l];
    L.n_tiles = static_cast<uint32_t>(cdiv(L.N, kThinBN));
    L.kblocks = static_cast<uint32_t>(cdiv(L.K, kThinBK));
    L.units = L.n_tiles * L.kblocks;
    L.ctas = L.units < static_cast<uint32_t>(sms) ? L.units : static_cast<uint32_t>(sms);
    L.C = Y[l];
    L.ldc = dims[l + 1];
    L.ws = st.ws + per_layer * l;
    L.counters = st.words + 1 + kChainMax + off;
    L.tiles_done = st.words + 1 + l;
    off += L.n_tiles;
  }
  if (log_enabled())
    std::fprintf(stderr, "[dg] gemm_bf16_decode_chain layers=%d M=%lld grid=%d\n", layers,
                 static_cast<long long>(M), sms);
  // Tuning knobs (sweeps): DG_CHAIN_PREFETCH (W blocks per CTA asked of L2 at a layer
  // boundary), DG_CHAIN_POLL_NS (sleep between polls of a layer's tile count),
  // DG_CHAIN_PDL=0 (no programmatic overlap with the previous kernel), DG_CHAIN_COOP=0 (no
  // cooperative attribute; co-residency then rests on the grid of one CTA per SM).
  p.prefetch = 0;
  if (const char* e = std::getenv("DG_CHAIN_PREFETCH")) p.prefetch = static_cast<uint32_t>(std::atoi(e));
  p.poll_ns = 64;
  if (const char* e = std::getenv("DG_CHAIN_POLL_NS")) p.poll_ns = static_cast<uint32_t>(std::atoi(e));
  const char* pe = std::getenv("DG_CHAIN_PDL");
  const bool pdl = !(pe && pe[0] == '0');
  const char* ce = std::getenv("DG_CHAIN_COOP");
  const bool coop = !(ce && ce[0] == '0');
  const void* wp[kChainMax];
  for (int l = 0; l < layers; ++l) wp[l] = W[l];
  return from_cuda(launch_gemm_chain(p, X, ldx, wp, ldw, s, pdl, coop));
}

dg_status attention_bf16(int64_t batch, int64_t Lq, int64_t Lkv, int64_t d, float scale,
                         int32_t causal, const uint16_t* Q, int64_t ldq, int64_t strideQ,
                         const uint16_t* K, int64_t ldk, int64_t strideK, const uint16_t* V,
                         int64_t ldv, int64_t strideV, uint16_t* O, int64_t ldo, int64_t strideO,
                         void* stream) {
  if (batch < 0 || Lq < 0 || Lkv < 0 || d < 0) return DG_ERR_INVALID_ARG;
  if (batch == 0 || Lq == 0) return DG_OK;
  if (Lkv == 0 || !(scale > 0.f) || !std::isfinite(scale)) return DG_ERR_INVALID_ARG;
  if (causal && Lq != Lkv) return DG_ERR_INVALID_ARG;
  if (ldq < d || ldk < d || ldv < d || ldo < d) return DG_ERR_INVALID_ARG;
  if (batch > 1 && (strideQ < Lq * ldq || strideK < Lkv * ldk || strideV < Lkv * ldv ||
                    strideO < Lq * ldo))
    return DG_ERR_INVALID_ARG;
  if (!Q || !K || !V || !O) return DG_ERR_INVALID_ARG;
  if (d != 128 || Lq >= (int64_t(1) << 31) || Lkv >= (int64_t(1) << 31)) return DG_ERR_UNSUPPORTED;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || ldq % 8 || ldk % 8 ||
      ldv % 8 || ldo % 8 || (batch > 1 && (strideQ % 8 || strideK % 8 || strideV % 8 || strideO % 8)))
    return DG_ERR_MISALIGNED;
  const int64_t q_tiles = (Lq + 127) / 128;
  if (batch * q_tiles > 0x7FFFFFFF) return DG_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  AttnParams p;
  p.batch = batch;
  p.Lq = Lq;
  p.Lkv = Lkv;
  p.q_tiles = q_tiles;
  p.kv_blocks = cdiv(Lkv, 128);
  // Split over keys when the query tiles alone do not fill the GPU: chunks of `chunk` key
  // blocks, the smallest chunk for which the chunks still fit in one wave.
  p.chunk = 0;
  p.ws = nullptr;
  p.counters = nullptr;
  int64_t items = batch * q_tiles;
  {
    auto nk = [&](int64_t t) { return causal ? t + 1 : p.kv_blocks; };
    const int64_t max_nk = causal ? q_tiles : p.kv_blocks;
    const char* se = std::getenv("DG_ATTN_SPLIT");
    const bool allow = !(se && se[0] == '0');
    if (allow && items < sms && max_nk > 1) {
      int64_t total = 0;
      for (int64_t t = 0; t < q_tiles; ++t) total += nk(t);
      total *= batch;
      int64_t C = cdiv(total, sms);
      if (C < 1) C = 1;
      for (;; ++C) {
        int64_t cnt = 0;
        for (int64_t t = 0; t < q_tiles; ++t) cnt += cdiv(nk(t), C);
        if (cnt * batch <= sms || C >= max_nk) {
          items = cnt * batch;
          break;
        }
      }
      if (C < max_nk) p.chunk = C;
      else items = batch * q_tiles;
    }
  }
  if (p.chunk > 0) {
    Workspace w;
    const dg_status ws_st =
        get_workspace(dev, static_cast<cudaStream_t>(stream), static_cast<size_t>(items * kAttnPartFloats),
                      static_cast<size_t>(batch * q_tiles), &w);
    if (ws_st != DG_OK) return ws_st;
    p.ws = w.ws;
    p.counters = w.counters;
  }
  p.items = items;
  p.sms = sms;
  p.c_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);  // log2(e)
  p.rank3 = batch > 1 ? 1 : 0;
  p.status = status;
  if (std::getenv("DG_LOG_PLAN"))
    std::fprintf(stderr, "[dg] attention_bf16 batch=%lld Lq=%lld Lkv=%lld causal=%d grid=%lld chunk=%lld\n",
                 static_cast<long long>(batch), static_cast<long long>(Lq),
                 static_cast<long long>(Lkv), causal ? 1 : 0, static_cast<long long>(items),
                 static_cast<long long>(p.chunk));
  return from_cuda(launch_attention(p, causal != 0, Q, ldq, strideQ, K, ldk, strideK, V, ldv,
                                    strideV, O, ldo, strideO, s));
}

const char* dg_status_string(dg_status s) {
  switch (s) {
    case DG_OK: return "DG_OK";
    case DG_ERR_INVALID_ARG: return "DG_ERR_INVALID_ARG: invalid argument";
    case DG_ERR_MISALIGNED: return "DG_ERR_MISALIGNED: pointer or leading dimension violates the 16-byte TMA rule";
    case DG_ERR_UNSUPPORTED: return "DG_ERR_UNSUPPORTED: shape not covered by the kernels";
    case DG_ERR_CUDA: return "DG_ERR_CUDA: a CUDA runtime call failed";
    case DG_ERR_TIMEOUT: return "DG_ERR_TIMEOUT: a kernel gave up a bounded wait";
    case DG_ERR_NO_MEMORY: return "DG_ERR_NO_MEMORY: workspace allocation failed";
  }
  return "unknown dg_status";
}

dg_status dg_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int dev = 0;
  if (current_device(&dev) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t* status = nullptr;
  int sms = 0;
  if (device_info(dev, &status, &sms) != cudaSuccess) return DG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DG_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return DG_ERR_CUDA;
  if (word == 0) return DG_OK;
  const uint32_t zero = 0;
  if (cudaMemcpy(status, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return DG_ERR_CUDA;
  // A CTA that gave up may have left split-K arrival counters non-zero.
  {
    std::lock_guard<std::mutex> lock(g_mu);
    for (auto& kv : g_workspaces)
      if (kv.first.first == dev && kv.second.counters)
        cudaMemset(kv.second.counters, 0, kv.second.n_counters * sizeof(uint32_t));
  }
  if (noalloc_reset_counters(dev) != cudaSuccess) return DG_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return DG_ERR_CUDA;
  return DG_ERR_TIMEOUT;
}

dg_status dg_release_workspace(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_workspaces.empty() && g_chain_states.empty()) return DG_OK;
  if (cudaDeviceSynchronize() != cudaSuccess) return DG_ERR_CUDA;
  int cur = 0;
  cudaGetDevice(&cur);
  for (auto& kv : g_workspaces) {
    cudaSetDevice(kv.first.first);
    cudaFree(kv.second.ws);
    cudaFree(kv.second.counters);
  }
  for (auto& kv : g_chain_states) {
    cudaSetDevice(kv.first.first);
    cudaFree(kv.second.ws);
    cudaFree(kv.second.words);
  }
  cudaSetDevice(cur);
  g_workspaces.clear();
  g_chain_states.clear();
  return DG_OK;
}

dg_status dg_plan_gemm(int32_t dtype, int64_t M, int64_t N, int64_t K, int64_t batch, dg_op op_b,
                       dg_out c_type, int32_t num_sms, dg_plan* out) {
  if (!out || dtype < 0 || dtype > 2 || (dtype == 2 && batch > 1)) return DG_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0 || batch < 0) return DG_ERR_INVALID_ARG;
  if (op_b != DG_OP_N && op_b != DG_OP_T) return DG_ERR_INVALID_ARG;
  if (c_type != DG_OUT_BF16 && c_type != DG_OUT_F32) return DG_ERR_INVALID_ARG;
  int sms = num_sms;
  if (sms <= 0) {
    int dev = 0;
    uint32_t* status = nullptr;
    if (current_device(&dev) != cudaSuccess || device_info(dev, &status, &sms) != cudaSuccess)
      return DG_ERR_CUDA;
  }
  return plan(dtype, M, N, K, batch, 1.0f, sms, out);
}

void dg_raster_tile(int64_t t, int64_t tiles_m, int64_t tiles_n, int32_t group, int64_t* b,
                    int64_t* tm, int64_t* tn) {
  raster_tile(t, tiles_m, tiles_n, group, b, tm, tn);
}

int64_t dg_streamk_start(int64_t c, int64_t units, int64_t ctas) {
  return sk_start<int64_t>(c, units, ctas);
}

double dg_model_traffic_bytes(int64_t M, int64_t N, int64_t K, int64_t tile_m, int64_t tile_n,
                              int32_t elem_bytes, int32_t out_bytes) {
  const double e = elem_bytes, Md = M, Nd = N, Kd = K;
  return e * Md * Kd * (Nd / tile_n) + e * Kd * Nd * (Md / tile_m) + out_bytes * Md * Nd;
}

double dg_model_quant_traffic_bytes(int64_t M, int64_t K, int64_t N, int64_t tile_m,
                                    int64_t tile_n, int32_t in_bytes, int32_t q_bytes,
                                    int32_t out_bytes, int32_t fused) {
  const double Md = M, Kd = K, Nd = N;
  const double col_blocks = Nd / tile_n, row_blocks = Md / tile_m;
  // Both schedules read the input once for the row maxima; then either write the codes and
  // let every column block read them, or let every column block re-read the input.
  const double input = fused ? in_bytes * Md * Kd + col_blocks * in_bytes * Md * Kd
                             : in_bytes * Md * Kd + q_bytes * Md * Kd + col_blocks * q_bytes * Md * Kd;
  return input + row_blocks * q_bytes * Kd * Nd + out_bytes * Md * Nd;
}

int64_t dg_model_local_bytes(int64_t tile_m, int64_t tile_n, int64_t tile_k, int32_t elem_bytes) {
  return elem_bytes * tile_m * tile_k + elem_bytes * tile_k * tile_n + 4 * tile_m * tile_n;
}

const char* dg_version(void) { return "dgemm-sm103a 0.1.0"; }

void dg_set_fault_injection(int32_t mode) { g_fault_injection = mode; }

}  // extern "C"
