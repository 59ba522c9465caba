/*
 * dgemm.h -- C ABI of the GB300 (sm_103a) dense GEMM library.
 *
 * Operation (every entry point):
 *
 *     C = alpha * A * op(B) + beta * C          (row-major matrices)
 *
 *   - GEMM definition: "4.1 Toi uu hieu nang toan tu GEMM tren CUDA"
 *     (infra-guide), section 1.1, and MUSA learning centre lesson m11-l5,
 *     Case 4 "GEMM" (C_ij = sum_k A_ik B_kj).  Row-major element addressing
 *     follows section 3.1 of the GEMM page: A[i*lda + k], B[k*ldb + j],
 *     C[i*ldc + j].
 *   - Work: 2*M*N*K floating-point operations ("Operator & Runtime", AI infra
 *     book ch. 5, section 5.2.1, F_gemm = 2MKN).
 *   - BF16 path: BF16 inputs, FP32 accumulation over the whole K reduction,
 *     then alpha/beta and one rounding to the output type ("Operator &
 *     Runtime" chapter introduction: X, W, C in BF16 with FP32 accumulation;
 *     sections 5.4.2-5.4.3: round to BF16 once, after the K loop).
 *   - Strided-batched variants: `batch` independent problems whose operands
 *     start `stride*` elements apart ("Batched GEMM" in multi-head attention,
 *     GEMM page section 1.2).
 *
 * Conventions shared by all entry points:
 *   - Pointers A, B, C are DEVICE pointers (cudaMalloc / torch CUDA memory) on
 *     the current device, owned by the caller.  The library never frees them.
 *   - Dimensions and leading dimensions are in elements.  op(B) = B (DG_OP_N):
 *     B is K x N with B[k*ldb + j]; op(B) = B^T (DG_OP_T): B is stored N x K
 *     with op(B)[k][j] = B[j*ldb + k].
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting.  Faults in the kernels
 *     surface at the caller's next synchronisation; a kernel that gives up a
 *     bounded wait records DG_ERR_TIMEOUT, read with dg_device_status().
 *   - BLAS edge semantics (the pages are silent): M == 0, N == 0 or
 *     batch == 0 is a no-op; K == 0 or alpha == 0 gives C = beta*C; when
 *     beta == 0, C is not read (NaN/Inf in it do not propagate).
 *   - Return value: DG_OK, or an error status with nothing enqueued.  No
 *     exceptions cross the ABI.
 *   - Thread safety: calls may come from several host threads.  Calls that
 *     use the split-K workspace (thin BF16 shapes) on the SAME stream are
 *     ordered by the stream; each stream gets its own workspace.
 */
#ifndef DGEMM_SM103_H
#define DGEMM_SM103_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DG_OK = 0,
  DG_ERR_INVALID_ARG = 1,  /* negative size, ld smaller than a row, null pointer, bad enum */
  DG_ERR_MISALIGNED = 2,   /* BF16 path: a base pointer not 16-byte aligned, or an ld or
                              batch stride not a multiple of 8 elements (TMA rule) */
  DG_ERR_UNSUPPORTED = 3,  /* shape the kernels do not cover (e.g. > 2^31-1 rows) */
  DG_ERR_CUDA = 4,         /* a CUDA runtime call failed (launch, allocation, query) */
  DG_ERR_TIMEOUT = 5,      /* a kernel gave up a bounded wait; results are invalid */
  DG_ERR_NO_MEMORY = 6     /* workspace allocation failed */
} dg_status;

typedef enum { DG_OP_N = 0, DG_OP_T = 1 } dg_op;
typedef enum { DG_OUT_BF16 = 0, DG_OUT_F32 = 1 } dg_out;

/*
 * FP32 SGEMM on CUDA cores: C = alpha*A*B + beta*C, all float32, row-major.
 * A: M x K (lda >= K), B: K x N (ldb >= N), C: M x N (ldc >= N).
 * FP32 multiply-add throughout; no TF32 or other reduced-precision
 * substitution.  Any alignment is accepted (rows that are 16-byte aligned
 * take the vector-copy variant of the kernel).
 * Defined by: GEMM page sections 1.1, 3-10 (the SGEMM this path implements).
 */
dg_status gemm_f32(int64_t M, int64_t N, int64_t K, float alpha, const float* A, int64_t lda,
                   const float* B, int64_t ldb, float beta, float* C, int64_t ldc, void* stream);

/*
 * Strided-batched FP32 SGEMM: for b < batch,
 *   C_b = alpha*A_b*op(B_b) + beta*C_b with X_b = X + b*strideX.
 * op_b = DG_OP_T reads B_b as N x K (ldb >= K).
 */
dg_status gemm_f32_strided_batched(int64_t M, int64_t N, int64_t K, float alpha, const float* A,
                                   int64_t lda, int64_t strideA, const float* B, int64_t ldb,
                                   int64_t strideB, dg_op op_b, float beta, float* C, int64_t ldc,
                                   int64_t strideC, int64_t batch, void* stream);

/*
 * BF16 GEMM with FP32 accumulation on the 5th-generation tensor cores:
 * C = alpha*A*B + beta*C.  A: M x K bfloat16 (lda >= K), B: K x N bfloat16
 * (ldb >= N), C: M x N of type c_type (bfloat16 rounded to nearest-even, or
 * float32), ldc >= N.  bfloat16 values are passed as their 16-bit patterns.
 * Requirements (TMA): A and B 16-byte aligned, lda and ldb multiples of 8.
 * Shapes with M <= 32 use the split-K decode kernel and a library-owned
 * workspace (see dg_release_workspace).
 * Defined by: "Operator & Runtime" chapter introduction and section 5.2.1
 * (the FFN projection C = XW, BF16 with FP32 accumulate), sections 5.4.2-5.4.3.
 */
dg_status gemm_bf16(int64_t M, int64_t N, int64_t K, float alpha, const uint16_t* A, int64_t lda,
                    const uint16_t* B, int64_t ldb, float beta, void* C, int64_t ldc,
                    dg_out c_type, void* stream);

/*
 * Strided-batched BF16 GEMM: for b < batch, C_b = alpha*A_b*op(B_b) + beta*C_b.
 * op_b = DG_OP_T reads B_b as N x K (ldb >= K), e.g. attention scores
 * S = Q K^T / sqrt(d) with Q_b, K_b stored [seq][d].  strideA/strideB must
 * be multiples of 8 elements when batch > 1.
 */
dg_status gemm_bf16_strided_batched(int64_t M, int64_t N, int64_t K, float alpha,
                                    const uint16_t* A, int64_t lda, int64_t strideA,
                                    const uint16_t* B, int64_t ldb, int64_t strideB, dg_op op_b,
                                    float beta, void* C, int64_t ldc, int64_t strideC,
                                    int64_t batch, dg_out c_type, void* stream);

/*
 * gemm_bf16 for decode shapes, without any allocation.  The pages have no counterpart: this
 * entry point exists for callers that cannot let a library call cudaMalloc -- a framework
 * whose caching allocator already holds the device memory (a new cudaMalloc may fail or
 * fragment its pool), or a latency-critical decode loop that cannot take cudaMalloc's
 * implicit device-wide synchronisation.  gemm_bf16 gives its split-K decode kernel a
 * workspace it allocates on first use; this variant runs the same kernel with its scratch
 * (FP32 partial sums, per-tile arrival counters) in a fixed array inside the library's
 * device image, 2.5 MiB + 32 KiB, which every GPU that loads the library holds until exit.
 *   - Arguments, layout and result are those of gemm_bf16 (op(B) = B), restricted to
 *     M <= 16 and N <= 1,048,576; larger sizes return DG_ERR_UNSUPPORTED and enqueue
 *     nothing.  Alignment rules as gemm_bf16 (DG_ERR_MISALIGNED).
 *   - Calls no cudaMalloc, cudaFree or other allocating routine.  The first call in a
 *     device's context does that context's set-up: it looks up the array's device address
 *     (cudaGetSymbolAddress) and zeroes the arrival counters once (cudaMemsetAsync on
 *     `stream`); make that first call before any stream capture.  The address is cached
 *     with the context it belongs to; a call in another context (after cudaDeviceReset,
 *     say) does the set-up again.
 *   - Every call shares the one array and leaves its contents behind.  The kernel leaves
 *     every arrival counter at zero when it finishes, so later calls enqueue only the
 *     kernel; after a bounded wait gave up (dg_device_status returns DG_ERR_TIMEOUT) that
 *     call re-zeroes the counters.  Calls whose work overlaps on the GPU (other streams,
 *     other host threads) race on the array and give wrong results: serialise them.
 */
dg_status gemm_bf16_decode_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                   const uint16_t* A, int64_t lda, const uint16_t* B,
                                   int64_t ldb, float beta, void* C, int64_t ldc, dg_out c_type,
                                   void* stream);

/*
 * FFN gate and up projections with the activation chain fused into the epilogue
 * ("Operator & Runtime" section 5.3.1: G = X W_g, U = X W_u, Z = SiLU(G) (.) U, all
 * [M, N]; section 5.4.3: the FP32 accumulation is rounded to BF16 before the activation,
 * as the unfused program stores G and U in BF16):
 *     Z[i][j] = bf16( SiLU(bf16(G[i][j])) * bf16(U[i][j]) ),   SiLU(x) = x / (1 + e^-x),
 * with the activation and the product in FP32 and every rounding nearest-even.  G and U
 * never reach memory; only Z (BF16) is written.
 *   - X is M x K (ldx >= K); W_g and W_u are K x N (ldwg, ldwu >= N), row-major BF16, so
 *     X W_g is the op(B) = B case of gemm_bf16.  Z is M x N BF16 (ldz >= N).
 *   - Device pointers owned by the caller; no aliasing between Z and the inputs.
 *   - Errors as gemm_bf16: negative sizes or short leading dimensions DG_ERR_INVALID_ARG;
 *     X, W_g, W_u not 16-byte aligned or ldx, ldwg, ldwu not multiples of 8
 *     DG_ERR_MISALIGNED.  M == 0 or N == 0: nothing; K == 0: Z = 0.
 *   - Any M uses the tile kernel (CTA pairs from M > 128); there is no decode-shaped form.
 */
dg_status gemm_bf16_gate_up_silu(int64_t M, int64_t N, int64_t K, const uint16_t* X, int64_t ldx,
                                 const uint16_t* Wg, int64_t ldwg, const uint16_t* Wu,
                                 int64_t ldwu, uint16_t* Z, int64_t ldz, void* stream);

/*
 * A chain of decode GEMMs in one persistent launch ("Operator & Runtime" sections 5.5.2 and
 * 5.5.4: one submission instead of one per layer, and a dependent layer starts on each block
 * of its input as soon as that block is written):
 *     Y[0] = bf16(X W[0]),  Y[l] = bf16(Y[l-1] W[l])  for 0 < l < layers,
 * each layer FP32-accumulated and rounded once to BF16 (nearest-even), exactly what
 * `layers` calls of gemm_bf16 (alpha = 1, beta = 0, op N) compute -- and with the same
 * stream-K partition and combine order as those calls when a layer has at least as many
 * (128-column, 64-row) W blocks as the GPU has SMs, so bit for bit the same result.
 *   - dims[0 .. layers]: dims[0] = columns of X, dims[l+1] = columns of Y[l] (= rows of
 *     W[l]).  X is M x dims[0] (ldx); W[l] is dims[l] x dims[l+1] row-major (ldw[l] >=
 *     dims[l+1]); Y[l] is M x dims[l+1] with row stride dims[l+1].  dims, W, ldw and Y are
 *     host arrays (of device pointers for W and Y).  1 <= layers <= 8, M <= 16.
 *   - Device buffers owned by the caller; every Y[l] is written, Y buffers must not alias
 *     each other or the inputs.  The library keeps per-stream scratch for the chain
 *     (partials and per-tile flags), allocated on first use (cudaMalloc) and freed by
 *     dg_release_workspace.
 *   - Launched cooperatively, one CTA per SM (all resident at once): the call fails with
 *     DG_ERR_CUDA when the GPU cannot hold that grid.  Waits are bounded (DG_ERR_TIMEOUT via
 *     dg_device_status).
 *   - Errors: layers outside 1..8, non-positive dims, short leading dimensions or null
 *     pointers DG_ERR_INVALID_ARG; M > 16 DG_ERR_UNSUPPORTED; M == 0: nothing; X, W[l] or
 *     Y[l] not 16-byte aligned, ldx or ldw[l] not multiples of 8, or an intermediate width
 *     dims[l] (0 < l < layers) not a multiple of 8 DG_ERR_MISALIGNED.
 */
dg_status gemm_bf16_decode_chain(int32_t layers, int64_t M, const int64_t* dims, const uint16_t* X,
                                 int64_t ldx, const uint16_t* const* W, const int64_t* ldw,
                                 uint16_t* const* Y, void* stream);

/*
 * FP8 E4M3 quantisation of a BF16 matrix, one scale per row ("Operator & Runtime" section
 * 5.4.3, Example 5-7: the scale comes from the absolute maximum of the whole row, so the
 * row is read in full before any element is quantised):
 *     amax_i = max_k |X[i][k]|,   Q[i][k] = E4M3(X[i][k] * (448 / amax_i)),
 *     scales[i] = amax_i / 448,   so X[i][k] ~ Q[i][k] * scales[i].
 * E4M3 is the E4M3FN format (1 sign, 4 exponent, 3 mantissa bits, largest finite 448).  The
 * two divisions and the product are IEEE float32 operations, the conversion rounds to
 * nearest-even and saturates to +-448.  A row of zeros gets codes 0 and scale 0.  X must be
 * finite (a row holding Inf or NaN gets unspecified codes).
 *   - X: rows x cols BF16, row stride ldx >= cols.  Q: rows x cols E4M3 codes (bytes), row
 *     stride ldq >= cols.  scales: rows float32.  Device pointers owned by the caller.
 *   - Activations are quantised this way for gemm_fp8_e4m3; so are weights stored [N][K],
 *     whose row scales are then the per-output-column scales of the product.
 *   - Errors: negative sizes, short leading dimensions or null pointers DG_ERR_INVALID_ARG;
 *     rows == 0: nothing.  Any alignment is accepted (16-byte rows take the vector path).
 */
dg_status quantize_rows_e4m3(int64_t rows, int64_t cols, const uint16_t* X, int64_t ldx,
                             uint8_t* Q, int64_t ldq, float* scales, void* stream);

/*
 * FP8 E4M3 GEMM with per-row scales (tcgen05 kind::f8f6f4, FP32 accumulate):
 *     C[i][j] = scale_a[i] * scale_b[j] * sum_k A[i][k] * B[j][k]
 * with A and B E4M3 codes as written by quantize_rows_e4m3: A is M x K (activations, one
 * scale per row), B is N x K (weights stored by output column, one scale per output
 * column), both K contiguous.  The accumulation is FP32 over the exact code products; the
 * scales are applied to the finished sum (two FP32 multiplications) and C is rounded once
 * to BF16 (nearest-even) or kept FP32 (c_type).
 *   - C is M x N row-major, ldc >= N.  Device pointers owned by the caller; C must not alias
 *     the inputs.
 *   - Errors: negative sizes, short leading dimensions, null pointers or another c_type
 *     DG_ERR_INVALID_ARG; A, B or scale_b not 16-byte aligned, lda or ldb not multiples of
 *     16, or scale_a not 4-byte aligned DG_ERR_MISALIGNED.  M == 0 or N == 0: nothing;
 *     K == 0: C = 0.
 *   - The tile kernel of gemm_bf16 (CTA pairs from M > 128), 128 K elements per stage; pair
 *     tiles are 256 x 256 or 256 x 224, whichever fills the waves of CTA pairs better.
 */
dg_status gemm_fp8_e4m3(int64_t M, int64_t N, int64_t K, const uint8_t* A, int64_t lda,
                        const float* scale_a, const uint8_t* B, int64_t ldb, const float* scale_b,
                        void* C, int64_t ldc, dg_out c_type, void* stream);

/*
 * Fused attention forward ("Operator & Runtime" section 5.3.3: S = Q K^T / sqrt(d),
 * P = softmax(S) row by row, O = P V, computed block by block with the online softmax so
 * that S and P never reach memory), over a strided batch of heads:
 *     O[b][i][:] = sum_j softmax_j(scale * Q[b][i][:] . K[b][j][:]) V[b][j][:]
 * for b < batch, i < Lq, over the keys j < Lkv visible to query i (all of them, or j <= i
 * when `causal` is non-zero).  BF16 inputs, FP32 scores, weights and accumulation, the
 * weights rounded to BF16 for the P V product, O rounded once to BF16 (nearest-even).
 *   - Layout: row-major, element (b, i, c) of Q at Q[b * strideQ + i * ldq + c], likewise
 *     K, V (Lkv rows) and O (Lq rows); c < d.  Only d = 128 is implemented.
 *   - scale: the factor applied to the scores (1/sqrt(d) for the standard form); must be
 *     finite and > 0.
 *   - causal requires Lq == Lkv (queries and keys of one sequence).
 *   - Device pointers owned by the caller; O must not alias the inputs, and the batch
 *     entries of O must not overlap (strideO >= Lq * ldo when batch > 1; likewise the
 *     strides of the inputs are at least L * ld).
 *   - Errors: negative sizes, Lkv == 0 (softmax over no keys), ld < d, overlapping batch
 *     strides, causal with Lq != Lkv, or a scale that is not finite and positive:
 *     DG_ERR_INVALID_ARG.  d != 128, or Lq, Lkv >= 2^31: DG_ERR_UNSUPPORTED.  Base
 *     pointers not 16-byte aligned, or ld / strides not multiples of 8 elements:
 *     DG_ERR_MISALIGNED.  batch == 0 or Lq == 0: nothing.  Nothing is enqueued on an error.
 *   - Enqueued on `stream`; allocates nothing.  A kernel that gives up a bounded wait
 *     reports DG_ERR_TIMEOUT through dg_device_status.
 */
dg_status attention_bf16(int64_t batch, int64_t Lq, int64_t Lkv, int64_t d, float scale,
                         int32_t causal, const uint16_t* Q, int64_t ldq, int64_t strideQ,
                         const uint16_t* K, int64_t ldk, int64_t strideK, const uint16_t* V,
                         int64_t ldv, int64_t strideV, uint16_t* O, int64_t ldo, int64_t strideO,
                         void* stream);

/* Human-readable name of a status code (static storage). */
const char* dg_status_string(dg_status s);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns DG_ERR_TIMEOUT if a kernel gave up a bounded wait since the
 * last call, DG_ERR_CUDA if the stream reported an error, DG_OK otherwise.
 * After a timeout the split-K workspace counters are re-zeroed.
 */
dg_status dg_device_status(void* stream);

/* Synchronises the device and frees every library-owned workspace. */
dg_status dg_release_workspace(void);

/* ----------------------------------------------------------------------
 * Introspection (host only; no GPU needed).  Used by the tests and the bench.
 * ---------------------------------------------------------------------- */

typedef enum {
  DG_KERNEL_NONE = 0,      /* no-op (empty problem) */
  DG_KERNEL_SCALE = 1,     /* C = beta*C only (K == 0 or alpha == 0) */
  DG_KERNEL_SIMT_F32 = 2,  /* FP32 CUDA-core SGEMM */
  DG_KERNEL_TC_BF16 = 3,   /* tcgen05 tile kernel (persistent, TMA ring, TMEM accumulators) */
  DG_KERNEL_THIN_BF16 = 4, /* tcgen05 stream-K decode kernel (M <= 32) */
  DG_KERNEL_TC2_BF16 = 5   /* tile kernel on CTA pairs (cta_group::2, 256 x 256 tiles;
                              FP8 also 256 x 224) */
} dg_kernel;

typedef struct {
  int32_t kernel;          /* dg_kernel */
  int32_t tile_m, tile_n, tile_k;
  int32_t stages;          /* shared-memory ring depth */
  int32_t group;           /* raster group height, in tile rows */
  int32_t ntok;            /* thin path: MMA N (tokens padded to 16 or 32) */
  int32_t vec;             /* SIMT path: 16-byte copy variant */
  int32_t splits;          /* SIMT: K chunks of each tail tile (1: no split);
                              tile kernel: CTAs sharing the stream-K tail's K blocks */
  int64_t tiles;           /* output tiles over all batches */
  int64_t tail_tiles;      /* tiles of the last partial wave split along K (SIMT) or
                              computed stream-K before the whole waves (tile kernel) */
  int64_t grid;            /* CTAs launched */
  int64_t kblocks;         /* K blocks per tile */
  int64_t workspace_bytes; /* library workspace needed (split-K partials and counters) */
} dg_plan;

/*
 * The kernel choice and launch shape for a problem, without running it.
 * dtype: 0 = FP32 path, 1 = BF16 path, 2 = FP8 E4M3 path (gemm_fp8_e4m3: batch
 * at most 1, B K-major whatever op_b says).  num_sms <= 0 queries the current
 * device (needs a GPU); pass the SM count explicitly to plan on a CPU.
 * Pointer alignment is not considered (vec assumes aligned rows).
 */
dg_status dg_plan_gemm(int32_t dtype, int64_t M, int64_t N, int64_t K, int64_t batch, dg_op op_b,
                       dg_out c_type, int32_t num_sms, dg_plan* out);

/* Tile raster: linear tile id -> (batch, tile row, tile column). */
void dg_raster_tile(int64_t t, int64_t tiles_m, int64_t tiles_n, int32_t group, int64_t* b,
                    int64_t* tm, int64_t* tn);

/* Stream-K partition of `units` work units over `ctas` CTAs: first unit of CTA c. */
int64_t dg_streamk_start(int64_t c, int64_t units, int64_t ctas);

/*
 * Interface-traffic model of a tiled GEMM ("Operator & Runtime" section 5.2.2,
 * Example 5-3): every m x n output tile reads its own A and B panels once,
 * V = e*M*K*(N/n) + e*K*N*(M/m) + e_out*M*N bytes, and needs
 * S = e*m*k + e*k*n + 4*m*n bytes of local memory (FP32 accumulator).
 */
double dg_model_traffic_bytes(int64_t M, int64_t N, int64_t K, int64_t tile_m, int64_t tile_n,
                              int32_t elem_bytes, int32_t out_bytes);
int64_t dg_model_local_bytes(int64_t tile_m, int64_t tile_n, int64_t tile_k, int32_t elem_bytes);
/*
 * Traffic model of an FP8 GEMM whose input A (M x K, in_bytes per element) is quantised
 * per row ("Operator & Runtime" section 5.4.4, Example 5-8), output tiles tile_m x tile_n,
 * every tile reading what it needs: fused == 0 quantises once (read A for the maxima and
 * codes, write the q_bytes codes, every column block reads the codes); fused != 0 lets
 * every column block re-read A and quantise locally.  Plus, for both, every row block reads
 * the q_bytes weights (K x N) and the output is written once (out_bytes).
 */
double dg_model_quant_traffic_bytes(int64_t M, int64_t K, int64_t N, int64_t tile_m,
                                    int64_t tile_n, int32_t in_bytes, int32_t q_bytes,
                                    int32_t out_bytes, int32_t fused);

/* Library version string. */
const char* dg_version(void);

/* Test hook: 0 = off.  1 = the tcgen05 tile kernel's MMA issuer skips its stage
 * releases, so the bounded waits expire and DG_ERR_TIMEOUT is reported (no hang,
 * no fault).  Affects launches made after the call. */
void dg_set_fault_injection(int32_t mode);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_SM103_H */
