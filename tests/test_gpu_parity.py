"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle.

Acceptance (the stated tolerance):
  * small-integer inputs: bit-exact (sums are exact in FP32 for any order);
  * FP32 output:  |C - C_ref| <= 1e-5 * D,  D = sum_k |alpha a b| + |beta c0|;
  * BF16 output:  |C - C_ref| <= 2e-4 * D + ulp_bf16(|C_ref|).
Every configuration is compared element by element: the full-size FP32 4096^3, BF16 FFN
and BF16 4096^3 outputs whole, the batched QK^T on eight whole heads (the rest on sampled
outputs computed one dot product at a time); C past 2^31 elements on sampled outputs.
"""
import numpy as np
import pytest

import oracle
import dense_gemm_sm_gb300 as dg
from dense_gemm_sm_gb300 import inputs

from .helpers import (assert_bf16_close, assert_f32_close, dev_bf16, dev_f32, host_bf16_bits,
                      host_f32, sample_indices, torch_mod)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    dg.load()
    return t


def sync(torch):
    torch.cuda.synchronize()
    st = dg.dg_device_status()
    assert st == dg.DG_OK, dg.status_string(st)


# ------------------------------------------------------------------------- FP32 path

def run_f32(torch, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc):
    dA, dB = dev_f32(A), dev_f32(B)
    dC = dev_f32(C0) if C0 is not None else torch.full((M * ldc,), float("nan"), device="cuda")
    dg.gemm_f32(M, N, K, float(alpha), dA, lda, dB, ldb, float(beta), dC, ldc)
    sync(torch)
    return host_f32(dC).reshape(-1)


def check_f32_full(torch, w):
    M, N, K, lda, ldb, ldc = w["M"], w["N"], w["K"], w["lda"], w["ldb"], w["ldc"]
    C = run_f32(torch, M, N, K, w["alpha"], w["A"], lda, w["B"], ldb, w["beta"], w["C0"], ldc)
    ref, den = oracle.gemm(M, N, K, w["alpha"], w["A"], lda, w["B"], ldb, w["beta"], w["C0"], ldc,
                           absden=True)
    Cv = C.reshape(-1, ldc)[:M, :N] if ldc != N else C.reshape(M, N)
    return Cv, ref[0], den[0]


def test_f32_256_integer_bit_exact(torch):
    w = inputs.sgemm_256(integer=True)
    C, ref, _ = check_f32_full(torch, w)
    assert np.array_equal(C.astype(np.float64), ref)


def test_f32_256_uniform(torch):
    w = inputs.sgemm_256()
    C, ref, den = check_f32_full(torch, w)
    assert_f32_close(C, ref, den, "sgemm 256^3")


def test_f32_ragged_padded_ld(torch):
    w = inputs.sgemm_ragged()
    C, ref, den = check_f32_full(torch, w)
    assert_f32_close(C, ref, den, "sgemm 1000x3000x777")
    # padding columns of C (beyond N) are not written
    M, ldc, N = w["M"], w["ldc"], w["N"]
    assert ldc == N or np.all(np.isnan(C.reshape(M, -1)[:, N:]))


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (7, 9, 5), (127, 129, 33), (129, 127, 17),
                                   (1, 300, 64), (300, 1, 64), (64, 64, 1), (200, 136, 1000)])
@pytest.mark.parametrize("aligned", [True, False])
def test_f32_edge_shapes(torch, M, N, K, aligned):
    pad = 4 if aligned else 3
    lda = ((K + 3) // 4) * 4 + (0 if aligned else 1)
    ldb = ((N + 3) // 4) * 4 + (0 if aligned else 1)
    ldc = ((N + 3) // 4) * 4 + (0 if aligned else pad)
    A = inputs.pad_rows(inputs.uniform_f32(M * 7 + K, (M, K)), lda)
    B = inputs.pad_rows(inputs.uniform_f32(N * 3 + K, (K, N)), ldb)
    C0 = inputs.pad_rows(inputs.uniform_f32(M + N, (M, N)), ldc)
    w = dict(M=M, N=N, K=K, alpha=np.float32(0.75), beta=np.float32(-1.25), A=A, lda=lda, B=B,
             ldb=ldb, C0=C0, ldc=ldc)
    C, ref, den = check_f32_full(torch, w)
    assert_f32_close(C, ref, den, f"sgemm {M}x{N}x{K} aligned={aligned}")


def test_f32_alpha_zero_and_k_zero(torch):
    M, N, K = 33, 65, 17
    A = inputs.uniform_f32(1, (M, K))
    B = inputs.uniform_f32(2, (K, N))
    C0 = inputs.uniform_f32(3, (M, N))
    C = run_f32(torch, M, N, K, 0.0, A, K, B, N, 0.5, C0, N).reshape(M, N)
    assert np.array_equal(C, (np.float32(0.5) * C0))
    C = run_f32(torch, M, N, 0, 1.0, A, K, B, N, -2.0, C0, N).reshape(M, N)
    assert np.array_equal(C, (np.float32(-2.0) * C0))
    # beta = 0: NaN in C is not read
    C = run_f32(torch, M, N, K, 1.0, A, K, B, N, 0.0, None, N).reshape(M, N)
    assert np.all(np.isfinite(C))


def test_f32_no_tf32_substitution(torch):
    # A = 1 + r * 2^-12 (r in 1..7), B = 1, K = 64: every partial sum is a multiple of 2^-12
    # below 128, so FP32 accumulation is exact and the result must match bit for bit.  A
    # TF32 (10-bit mantissa) operand would round r * 2^-12 away, an error of about
    # 2.4e-4 * D, 24 times the FP32 bound.
    M, N, K = 128, 128, 64
    r = np.random.Generator(np.random.PCG64(5)).integers(1, 8, size=(M, K))
    A = (1.0 + r * 2.0 ** -12).astype(np.float32)
    B = np.ones((K, N), dtype=np.float32)
    C = run_f32(torch, M, N, K, 1.0, A, K, B, N, 0.0, None, N).reshape(M, N)
    ref, den = oracle.gemm(M, N, K, 1.0, A, K, B, N, absden=True)
    assert np.array_equal(C.astype(np.float64), ref[0])
    tf32_like = oracle.gemm(M, N, K, 1.0, np.ones_like(A), K, B, N)[0]  # r * 2^-12 rounded away
    assert not oracle.check_f32(tf32_like, ref[0], den[0])[0]


@pytest.mark.parametrize("op_b", [dg.DG_OP_N, dg.DG_OP_T])
def test_f32_strided_batched(torch, op_b):
    batch, M, N, K = 3, 130, 70, 45
    lda, ldc = 48, 72
    ldb = 72 if op_b == dg.DG_OP_N else 48
    brows = K if op_b == dg.DG_OP_N else N
    sA, sB, sC = M * lda + 8, brows * ldb + 4, M * ldc + 12
    A = inputs.uniform_f32(10, (batch * sA,))
    B = inputs.uniform_f32(11, (batch * sB,))
    C0 = inputs.uniform_f32(12, (batch * sC,))
    dA, dB, dC = dev_f32(A), dev_f32(B), dev_f32(C0)
    dg.gemm_f32_strided_batched(M, N, K, 1.5, dA, lda, sA, dB, ldb, sB, op_b, 0.25, dC, ldc, sC,
                                batch)
    sync(torch)
    C = host_f32(dC)
    ref, den = oracle.gemm(M, N, K, 1.5, A, lda, B, ldb, 0.25, C0, ldc, op_b=op_b, batch=batch,
                           strideA=sA, strideB=sB, strideC=sC, absden=True)
    for b in range(batch):
        Cb = C[b * sC:b * sC + M * ldc].reshape(M, ldc)[:, :N]
        assert_f32_close(Cb, ref[b], den[b], f"batched f32 b={b}")


def test_f32_4096_whole_matrix(torch):
    # The headline configuration (4096^3, alpha = 1, beta = 0.5), every element of C against
    # the oracle: the split tail (the last partial wave's tiles cut along K) included.
    w = inputs.sgemm_4096()
    M, N, K = w["M"], w["N"], w["K"]
    dA, dB, dC = dev_f32(w["A"]), dev_f32(w["B"]), dev_f32(w["C0"])
    dg.gemm_f32(M, N, K, float(w["alpha"]), dA, K, dB, N, float(w["beta"]), dC, N)
    sync(torch)
    C = host_f32(dC).reshape(M, N)
    ref, den = oracle.gemm(M, N, K, w["alpha"], w["A"], K, w["B"], N, w["beta"], w["C0"], N,
                           absden=True)
    assert_f32_close(C, ref[0], den[0], "sgemm 4096^3 (whole matrix)")


# ------------------------------------------------------------------------- BF16 path

@pytest.fixture(params=["pair", "single"])
def tile_mode(request, monkeypatch):
    """Runs a BF16 tile-kernel test on CTA pairs (the default for M > 128) and on single
    CTAs (DG_TC_PAIR=0, read by the planner at each call)."""
    if request.param == "single":
        monkeypatch.setenv("DG_TC_PAIR", "0")
    else:
        monkeypatch.delenv("DG_TC_PAIR", raising=False)
    return request.param


def run_bf16(torch, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, out_f32=False):
    dA, dB = dev_bf16(A), dev_bf16(B)
    if out_f32:
        dC = dev_f32(C0) if C0 is not None else torch.full((M * ldc,), float("nan"), device="cuda")
    else:
        dC = dev_bf16(C0) if C0 is not None else torch.full((M * ldc,), float("nan"), device="cuda",
                                                             dtype=torch.bfloat16)
    dg.gemm_bf16(M, N, K, float(alpha), dA, lda, dB, ldb, float(beta), dC, ldc,
                 dg.DG_OUT_F32 if out_f32 else dg.DG_OUT_BF16)
    sync(torch)
    if out_f32:
        return host_f32(dC).reshape(M, ldc)[:, :N]
    return host_bf16_bits(dC).reshape(M, ldc)[:, :N]


@pytest.mark.parametrize("M,N,K", [(256, 384, 320), (1, 256, 128), (16, 12288, 4096),
                                   (40, 520, 136)])
def test_bf16_integer_bit_exact(torch, tile_mode, M, N, K):
    A = inputs.f32_to_bf16_bits(inputs.integer_f32(M + K, (M, K)))
    B = inputs.f32_to_bf16_bits(inputs.integer_f32(N + K, (K, N)))
    C = run_bf16(torch, M, N, K, 1.0, A, K, B, N, 0.0, None, N)
    ref = oracle.gemm(M, N, K, 1.0, A, K, B, N)[0]
    assert np.array_equal(C, oracle.round_bf16(ref))


def test_bf16_ffn_reduced_full_compare(torch, tile_mode):
    w = inputs.ffn_bf16(M=512, K=1024, N=2048)
    M, N, K = w["M"], w["N"], w["K"]
    C = run_bf16(torch, M, N, K, w["alpha"], w["A"], K, w["B"], N, 0.0, None, N)
    ref, den = oracle.gemm(M, N, K, w["alpha"], w["A"], K, w["B"], N, absden=True)
    assert_bf16_close(C, ref[0], den[0], "ffn-shaped 512x2048x1024")


# Shapes whose tiles overfill the last wave (152 CTAs, or 76 pairs): the tail tiles run
# stream-K first (K split 4 ways) before the whole-wave tiles.
@pytest.mark.parametrize("M,N,K,ldc,beta,out_f32", [
    (1280, 4096, 6144, 4096, 0.0, False),     # whole-wave tiles stored with TMA
    (1280, 4096, 6144, 4096, 0.0, True),
    (1200, 4000, 6104, 4003, -0.75, False),   # ragged tiles and K block, beta, direct stores
    (1200, 4000, 6104, 4003, -0.75, True)])
def test_bf16_stream_k_tail(torch, tile_mode, M, N, K, ldc, beta, out_f32):
    plan = dg.dg_plan_gemm(1, M, N, K, c_type=dg.DG_OUT_F32 if out_f32 else dg.DG_OUT_BF16,
                           num_sms=152)
    assert plan["kernel"] in (dg.DG_KERNEL_TC_BF16, dg.DG_KERNEL_TC2_BF16)
    assert plan["tail_tiles"] > 0
    A = inputs.f32_to_bf16_bits(inputs.normal_f32(M + 7, (M, K)))
    B = inputs.f32_to_bf16_bits(inputs.normal_f32(N + 8, (K, N), 0.1))
    c0 = inputs.normal_f32(M + N + 1, (M, N))
    C0 = None
    if beta != 0.0:
        C0 = inputs.pad_rows(c0 if out_f32 else inputs.f32_to_bf16_bits(c0), ldc, 0)
    alpha = np.float32(0.5)
    C = run_bf16(torch, M, N, K, alpha, A, K, B, N, np.float32(beta), C0, ldc, out_f32)
    ref, den = oracle.gemm(M, N, K, alpha, A, K, B, N, np.float32(beta), C0, ldc, absden=True)
    if out_f32:
        assert_f32_close(C, ref[0], den[0], f"stream-K tail {M}x{N}x{K}")
    else:
        assert_bf16_close(C, ref[0], den[0], f"stream-K tail {M}x{N}x{K}")


def test_bf16_stream_k_tail_deterministic(torch, tile_mode):
    M, N, K = 1280, 4096, 6144
    A = dev_bf16(inputs.f32_to_bf16_bits(inputs.normal_f32(M + 7, (M, K))))
    B = dev_bf16(inputs.f32_to_bf16_bits(inputs.normal_f32(N + 8, (K, N), 0.1)))
    outs = []
    for _ in range(3):
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        dg.gemm_bf16(M, N, K, 1.0, A, K, B, N, 0.0, dC, N, c_type=dg.DG_OUT_F32)
        sync(torch)
        outs.append(host_f32(dC).view(np.uint32))
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


@pytest.mark.parametrize("M,N,K", [(129, 264, 72), (300, 1000, 200), (200, 136, 8), (33, 8, 16),
                                   (128, 256, 64), (255, 520, 4104)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_bf16_edge_shapes(torch, tile_mode, M, N, K, out_f32):
    lda = ((K + 7) // 8) * 8
    ldb = ((N + 7) // 8) * 8 + 8
    ldc = N + 3
    A = inputs.pad_rows(inputs.f32_to_bf16_bits(inputs.normal_f32(M + 1, (M, K))), lda, 0)
    B = inputs.pad_rows(inputs.f32_to_bf16_bits(inputs.normal_f32(N + 2, (K, N), 0.1)), ldb, 0)
    c0 = inputs.normal_f32(M + N, (M, N))
    C0 = inputs.pad_rows(c0 if out_f32 else inputs.f32_to_bf16_bits(c0), ldc, 0)
    alpha, beta = np.float32(0.5), np.float32(-0.75)
    C = run_bf16(torch, M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, out_f32)
    ref, den = oracle.gemm(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, absden=True)
    if out_f32:
        assert_f32_close(C, ref[0], den[0], f"bf16->f32 {M}x{N}x{K}")
    else:
        assert_bf16_close(C, ref[0], den[0], f"bf16 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(129, 264, 72), (300, 1000, 200), (33, 8, 16), (255, 520, 4104),
                                   (1000, 136, 64)])
@pytest.mark.parametrize("out_f32", [False, True])
def test_bf16_beta_zero_edge_shapes(torch, tile_mode, M, N, K, out_f32):
    # beta = 0 with 16-byte aligned C rows: the epilogue's TMA-store path (edge tiles clipped
    # by the tensor map); the NaN-filled C checks that nothing outside M x N is written.
    lda = ((K + 7) // 8) * 8
    A = inputs.pad_rows(inputs.f32_to_bf16_bits(inputs.normal_f32(M + 5, (M, K))), lda, 0)
    B = inputs.f32_to_bf16_bits(inputs.normal_f32(N + 6, (K, N), 0.1))
    ldc = N + 8
    C = run_bf16(torch, M, N, K, 0.75, A, lda, B, N, 0.0, None, ldc, out_f32)
    ref, den = oracle.gemm(M, N, K, 0.75, A, lda, B, N, absden=True)
    if out_f32:
        assert_f32_close(C, ref[0], den[0], f"bf16->f32 beta=0 {M}x{N}x{K}")
    else:
        assert_bf16_close(C, ref[0], den[0], f"bf16 beta=0 {M}x{N}x{K}")


def test_bf16_tma_store_leaves_padding_untouched(torch, tile_mode):
    M, N, K, ldc = 200, 264, 128, 272
    A = inputs.f32_to_bf16_bits(inputs.normal_f32(50, (M, K)))
    B = inputs.f32_to_bf16_bits(inputs.normal_f32(51, (K, N)))
    dA, dB = dev_bf16(A), dev_bf16(B)
    dC = torch.full((M + 3, ldc), float("nan"), dtype=torch.float32, device="cuda")
    dg.gemm_bf16(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, ldc, dg.DG_OUT_F32)
    sync(torch)
    C = host_f32(dC)
    assert np.all(np.isnan(C[:, N:])) and np.all(np.isnan(C[M:, :]))
    assert np.all(np.isfinite(C[:M, :N]))


@pytest.mark.parametrize("M", [1, 4, 16, 17, 32])
def test_bf16_decode_full_size(torch, M):
    W = inputs.ffn_weight()
    w = inputs.decode_bf16(M, W=W)
    N, K = w["N"], w["K"]
    C = run_bf16(torch, M, N, K, 1.0, w["A"], K, W, N, 0.0, None, N)
    ref, den = oracle.gemm(M, N, K, 1.0, w["A"], K, W, N, absden=True)
    assert_bf16_close(C, ref[0], den[0], f"decode M={M}")


@pytest.mark.parametrize("M,N,K", [(1, 8, 8), (3, 136, 200), (16, 1000, 4104), (5, 128, 64),
                                   (9, 4096, 64), (32, 264, 2056), (16, 19456, 64),
                                   (7, 19400, 128), (32, 12200, 136), (2, 3000, 4096)])
def test_bf16_thin_ragged(torch, M, N, K):
    # On 152 SMs: (16, 19456, 64) and (7, 19400, 128) give every CTA one whole tile of one
    # or two K blocks; (32, 12200, 136) three K blocks per tile (a ragged last one) shared by
    # neighbouring CTAs; (2, 3000, 4096) ranges shorter than a tile, so some tiles hold the
    # ends of two ranges.
    lda = ((K + 7) // 8) * 8
    ldb = ((N + 7) // 8) * 8
    A = inputs.pad_rows(inputs.f32_to_bf16_bits(inputs.normal_f32(K + M, (M, K))), lda, 0)
    B = inputs.pad_rows(inputs.f32_to_bf16_bits(inputs.normal_f32(N + K, (K, N), 0.05)), ldb, 0)
    c0 = inputs.f32_to_bf16_bits(inputs.normal_f32(7, (M, N)))
    C = run_bf16(torch, M, N, K, 1.25, A, lda, B, ldb, 0.5, c0, N)
    ref, den = oracle.gemm(M, N, K, 1.25, A, lda, B, ldb, 0.5, c0, N, absden=True)
    assert_bf16_close(C, ref[0], den[0], f"thin {M}x{N}x{K}")


@pytest.mark.parametrize("op_b", [dg.DG_OP_N, dg.DG_OP_T])
@pytest.mark.parametrize("M", [1, 16, 32])
def test_bf16_decode_w_layouts(torch, op_b, M):
    # Decode with W as K x N (N-major) and as N x K, the nn.Linear layout (K-major); N = 3000
    # leaves a ragged last 128-column tile.
    N, K = 3000, 4096
    brows, bcols = (K, N) if op_b == dg.DG_OP_N else (N, K)
    X = inputs.f32_to_bf16_bits(inputs.normal_f32(M + 40, (M, K)))
    W = inputs.f32_to_bf16_bits(inputs.normal_f32(M + 41, (brows, bcols), 0.05))
    plan = dg.dg_plan_gemm(1, M, N, K, op_b=op_b, num_sms=152)
    assert plan["kernel"] == dg.DG_KERNEL_THIN_BF16 and plan["tile_n"] == 128
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    dg.gemm_bf16_strided_batched(M, N, K, 1.0, dev_bf16(X), K, 0, dev_bf16(W), bcols, 0, op_b,
                                 0.0, dC, N, 0, 1, dg.DG_OUT_F32)
    sync(torch)
    ref, den = oracle.gemm(M, N, K, 1.0, X, K, W, bcols, op_b=op_b, absden=True)
    assert_f32_close(host_f32(dC), ref[0], den[0], f"decode M={M} op_b={op_b}")


@pytest.mark.parametrize("M", [1, 6, 16])
def test_bf16_decode_deterministic(torch, M):
    # FP32 output shows any change in the order the split-K parts are added.  Which CTA
    # combines a tile depends on arrival timing; the sum order must not.
    W = inputs.ffn_weight()
    w = inputs.decode_bf16(M, W=W)
    dA, dB = dev_bf16(w["A"]), dev_bf16(W)
    outs = []
    for _ in range(4):
        dC = torch.empty((M, 12288), dtype=torch.float32, device="cuda")
        dg.gemm_bf16(M, 12288, 4096, 1.0, dA, 4096, dB, 12288, 0.0, dC, 12288, c_type=dg.DG_OUT_F32)
        sync(torch)
        outs.append(host_f32(dC).view(np.uint32))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)
    ref, den = oracle.gemm(M, 12288, 4096, 1.0, w["A"], 4096, W, 12288, 0.0, None, 12288,
                           absden=True)
    assert_f32_close(outs[0].view(np.float32), ref[0], den[0], f"decode M={M}, FP32 out")


def test_bf16_decode_graph_replay(torch):
    # A captured call replays its kernel parameters unchanged, split-K workspace included;
    # every replay must still combine only the parts it wrote.  X changes between replays.
    M, N, K = 16, 12288, 4096
    W = inputs.ffn_weight()
    dB = dev_bf16(W)
    x0 = inputs.f32_to_bf16_bits(inputs.normal_f32(inputs.BASE_SEED + 900, (M, K)))
    dX = dev_bf16(x0)
    dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first call on this stream sets up its workspace
        dg.gemm_bf16(M, N, K, 1.0, dX, K, dB, N, 0.0, dC, N, c_type=dg.DG_OUT_F32)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dg.gemm_bf16(M, N, K, 1.0, dX, K, dB, N, 0.0, dC, N, c_type=dg.DG_OUT_F32)
    for seed in (901, 902, 903):
        x = inputs.f32_to_bf16_bits(inputs.normal_f32(inputs.BASE_SEED + seed, (M, K)))
        dX.copy_(dev_bf16(x))
        g.replay()
        sync(torch)
        ref, den = oracle.gemm(M, N, K, 1.0, x, K, W, N, 0.0, None, N, absden=True)
        assert_f32_close(host_f32(dC), ref[0], den[0], f"graph replay, X seed {seed}")
    assert dg.dg_device_status() == dg.DG_OK


def test_bf16_ffn_full_size_whole_matrix(torch, tile_mode):
    # The FFN projection 1024 x 12288 x 4096, every element against the oracle (the stream-K
    # tail tiles included), on CTA pairs (the default) and on single CTAs.
    w = inputs.ffn_bf16()
    M, N, K = w["M"], w["N"], w["K"]
    dA, dB = dev_bf16(w["A"]), dev_bf16(w["B"])
    dC = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    dg.gemm_bf16(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
    sync(torch)
    ref, den = ffn_reference(w)
    assert_bf16_close(host_bf16_bits(dC), ref, den, "FFN 1024x12288x4096 (whole matrix)")


_FFN_REF = {}


def ffn_reference(w):
    """Oracle result and error scale of the FFN projection, computed once per session."""
    if "ffn" not in _FFN_REF:
        M, N, K = w["M"], w["N"], w["K"]
        ref, den = oracle.gemm(M, N, K, 1.0, w["A"], K, w["B"], N, absden=True)
        _FFN_REF["ffn"] = (ref[0], den[0])
    return _FFN_REF["ffn"]


def test_bf16_square_4096_whole_matrix(torch):
    w = inputs.bf16_square(4096)
    n = 4096
    dA, dB = dev_bf16(w["A"]), dev_bf16(w["B"])
    dC = torch.full((n, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    dg.gemm_bf16(n, n, n, 1.0, dA, n, dB, n, 0.0, dC, n)
    sync(torch)
    ref, den = oracle.gemm(n, n, n, 1.0, w["A"], n, w["B"], n, absden=True)
    assert_bf16_close(host_bf16_bits(dC), ref[0], den[0], "BF16 4096^3 (whole matrix)")


@pytest.mark.parametrize("path", ["f32", "bf16"])
def test_outputs_past_2_31_elements(torch, path):
    # C of 65536 x 32800 = 2,149,580,800 elements (> 2^31): the element and byte offsets of
    # the last rows overflow 32-bit integers, so every index on the store path must be 64-bit.
    # N leaves a 32-column last tile; K = 64 keeps the call short.  Sampled entries, the
    # corners and the last row's tail are gathered on the device and checked against the
    # oracle's single entries.
    M, N, K = 65536, 32800, 64
    assert M * N > 2 ** 31
    rows, cols = sample_indices(71, 2000, M, N)
    tail = np.arange(N - 80, N)
    rows = np.concatenate([rows, np.full(tail.size, M - 1), np.full(tail.size, M - 129)])
    cols = np.concatenate([cols, tail, tail])
    ri = torch.from_numpy(rows).cuda()
    ci = torch.from_numpy(cols).cuda()
    if path == "f32":
        A = inputs.uniform_f32(72, (M, K))
        B = inputs.uniform_f32(73, (K, N))
        dC = torch.empty((M, N), dtype=torch.float32, device="cuda")
        dg.gemm_f32(M, N, K, 1.0, dev_f32(A), K, dev_f32(B), N, 0.0, dC, N)
        sync(torch)
        got = host_f32(dC[ri, ci])
        ref, den = oracle.gemm_entries(M, N, K, 1.0, A, K, B, N, 0.0, None, N, rows, cols)
        assert_f32_close(got, ref, den, "FP32 C past 2^31 elements (sampled)")
    else:
        A = inputs.f32_to_bf16_bits(inputs.normal_f32(74, (M, K)))
        B = inputs.f32_to_bf16_bits(inputs.normal_f32(75, (K, N), 0.125))
        dC = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        dg.gemm_bf16(M, N, K, 1.0, dev_bf16(A), K, dev_bf16(B), N, 0.0, dC, N)
        sync(torch)
        got = host_bf16_bits(dC[ri, ci])
        ref, den = oracle.gemm_entries(M, N, K, 1.0, A, K, B, N, 0.0, None, N, rows, cols)
        assert_bf16_close(got, ref, den, "BF16 C past 2^31 elements (sampled)")
    del dC
    torch.cuda.empty_cache()


def run_qk(torch, w):
    batch, S, D = w["batch"], w["M"], w["K"]
    dQ, dK = dev_bf16(w["A"]), dev_bf16(w["B"])
    dC = torch.empty((batch, S, S), dtype=torch.float32, device="cuda")
    dg.gemm_bf16_strided_batched(S, S, D, float(w["alpha"]), dQ, D, S * D, dK, D, S * D,
                                 dg.DG_OP_T, 0.0, dC, S, S * S, batch, dg.DG_OUT_F32)
    sync(torch)
    return dC


def test_bf16_batched_qk_reduced_full_compare(torch):
    w = inputs.qk_batched(batch=3, S=384, D=128)
    batch, S, D = w["batch"], w["M"], w["K"]
    C = host_f32(run_qk(torch, w))
    ref, den = oracle.gemm(S, S, D, w["alpha"], w["A"], D, w["B"], D, op_b=1, batch=batch,
                           strideA=S * D, strideB=S * D, absden=True)
    for b in range(batch):
        assert_f32_close(C[b], ref[b], den[b], f"QK^T batch {b}")


# Heads compared whole at full size: the first and last of each sequence (batch = 2 sequences
# x 32 heads) and two in the middle.
QK_WHOLE_HEADS = (0, 1, 17, 31, 32, 33, 50, 63)


def test_bf16_batched_qk_full_size(torch):
    w = inputs.qk_batched()
    batch, S, D = w["batch"], w["M"], w["K"]
    C = host_f32(run_qk(torch, w))
    A = w["A"].reshape(batch, S * D)
    B = w["B"].reshape(batch, S * D)
    for b in QK_WHOLE_HEADS:
        ref, den = oracle.gemm(S, S, D, w["alpha"], A[b], D, B[b], D, op_b=1, absden=True)
        assert_f32_close(C[b], ref[0], den[0], f"QK^T 64x2048x2048x128, head {b} (whole)")
    # every other head on sampled entries
    bidx, rows, cols = sample_indices(44, 4000, batch, S, S)
    ref, den = oracle.gemm_entries(S, S, D, w["alpha"], w["A"], D, w["B"], D, 0.0, None, S, rows,
                                   cols, op_b=1, bidx=bidx, strideA=S * D, strideB=S * D,
                                   strideC=S * S)
    assert_f32_close(C[bidx, rows, cols], ref, den, "QK^T 64x2048x2048x128 (sampled)")


@pytest.mark.parametrize("op_b", [dg.DG_OP_N, dg.DG_OP_T])
def test_bf16_strided_batched_bf16_out(torch, op_b):
    batch, M, N, K = 5, 200, 264, 136
    brows, bcols = (K, N) if op_b == dg.DG_OP_N else (N, K)
    sA, sB, sC = M * K + 64, brows * bcols + 8, M * N + 40
    A = inputs.f32_to_bf16_bits(inputs.normal_f32(30, (batch * sA,)))
    B = inputs.f32_to_bf16_bits(inputs.normal_f32(31, (batch * sB,), 0.1))
    C0 = inputs.f32_to_bf16_bits(inputs.normal_f32(32, (batch * sC,)))
    dA, dB, dC = dev_bf16(A), dev_bf16(B), dev_bf16(C0)
    dg.gemm_bf16_strided_batched(M, N, K, 0.5, dA, K, sA, dB, bcols, sB, op_b, 2.0, dC, N, sC,
                                 batch, dg.DG_OUT_BF16)
    sync(torch)
    C = host_bf16_bits(dC)
    ref, den = oracle.gemm(M, N, K, 0.5, A, K, B, bcols, 2.0, C0, N, op_b=op_b, batch=batch,
                           strideA=sA, strideB=sB, strideC=sC, absden=True)
    for b in range(batch):
        Cb = C[b * sC:b * sC + M * N].reshape(M, N)
        assert_bf16_close(Cb, ref[b], den[b], f"batched bf16 op_b={op_b} b={b}")


def test_bf16_tile_kernel_deterministic(torch, tile_mode):
    w = inputs.ffn_bf16(M=384, K=2048, N=1536)
    dA, dB = dev_bf16(w["A"]), dev_bf16(w["B"])
    outs = []
    for _ in range(2):
        dC = torch.empty((384, 1536), dtype=torch.bfloat16, device="cuda")
        dg.gemm_bf16(384, 1536, 2048, 1.0, dA, 2048, dB, 1536, 0.0, dC, 1536)
        sync(torch)
        outs.append(host_bf16_bits(dC))
    assert np.array_equal(outs[0], outs[1])


def test_bf16_argument_errors(torch):
    A = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    st = dg.gemm_bf16(64, 64, 60, 1.0, A, 60, A, 64, 0.0, C, 64, check=False)
    assert st == dg.DG_ERR_MISALIGNED                              # lda % 8 != 0
    st = dg.gemm_bf16(64, 64, 64, 1.0, A.data_ptr() + 2, 64, A, 64, 0.0, C, 64, check=False)
    assert st == dg.DG_ERR_MISALIGNED                              # base not 16-byte aligned
    assert dg.gemm_bf16(-1, 64, 64, 1.0, A, 64, A, 64, 0.0, C, 64, check=False) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16(64, 64, 64, 1.0, A, 32, A, 64, 0.0, C, 64, check=False) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16(64, 64, 64, 1.0, A, 64, A, 64, 0.0, C, 64, c_type=7,
                        check=False) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16(0, 64, 64, 1.0, None, 64, None, 64, 0.0, None, 64, check=False) == dg.DG_OK
    sync(torch)
