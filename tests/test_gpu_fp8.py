"""GPU parity of the FP8 E4M3 path against the CPU oracle.

  * quantize_rows_e4m3: codes and scales bit-exact (both sides take the rounding decision
    in IEEE float32, the kernel's precision);
  * gemm_fp8_e4m3 on oracle-quantised codes: FP32 output within 1e-5 * D, BF16 output
    within 2e-4 * D + ulp_bf16, D = |s_a s_b| sum_k |qa qb|; bit-exact where the sums are
    exact (small-integer codes, unit scales, FP32 output).
"""
import numpy as np
import pytest

import oracle
import dense_gemm_sm_gb300 as dg
from dense_gemm_sm_gb300 import inputs

from .helpers import dev_bf16, host_bf16_bits, host_f32, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    dg.load()
    return t


@pytest.fixture(params=["pair", "single"])
def tile_mode(request, monkeypatch):
    if request.param == "single":
        monkeypatch.setenv("DG_TC_PAIR", "0")
    else:
        monkeypatch.delenv("DG_TC_PAIR", raising=False)
    return request.param


def sync(torch):
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK


def dev_u8(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_f32(a, torch):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def quantize_gpu(torch, rows, cols, X, ldx, ldq):
    dQ = torch.full((rows * ldq,), 0xA5, dtype=torch.uint8, device="cuda")
    ds = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    dg.quantize_rows_e4m3(rows, cols, dev_bf16(X), ldx, dQ, ldq, ds)
    sync(torch)
    return dQ.cpu().numpy().reshape(rows, ldq), ds.cpu().numpy()


@pytest.mark.parametrize("rows,cols,ldx,ldq", [(300, 1000, 1000, 1008), (7, 33, 35, 33),
                                               (1024, 4096, 4096, 4096), (3, 8, 8, 16),
                                               (5, 12301, 12304, 12304)])
def test_quantize_rows_bit_exact(torch, rows, cols, ldx, ldq):
    rng = np.random.default_rng(51)
    X = inputs.f32_to_bf16_bits((rng.standard_normal((rows, ldx)) *
                                 np.exp(rng.normal(0, 2, (rows, 1)))).astype(np.float32))
    X[rows // 2] = 0                                  # an all-zero row
    Q, s = quantize_gpu(torch, rows, cols, X, ldx, ldq)
    q_ref, s_ref = oracle.quantize_rows_e4m3(rows, cols, X, ldx)
    assert np.array_equal(Q[:, :cols], q_ref), f"{np.mean(Q[:, :cols] != q_ref):.2e} of codes differ"
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))
    assert np.all(Q[:, cols:] == 0xA5)                # padding untouched


def quantized_operands(M, N, K, lda, ldb, seed):
    """Oracle-quantised codes (padded to the leading dimensions) and scales of FFN-like data."""
    rng = np.random.default_rng(seed)
    X = inputs.f32_to_bf16_bits(rng.normal(0, 1, (M, K)).astype(np.float32))
    W = inputs.f32_to_bf16_bits(rng.normal(0, 1 / np.sqrt(K), (N, K)).astype(np.float32))
    qa, sa = oracle.quantize_rows_e4m3(M, K, X, K)
    qb, sb = oracle.quantize_rows_e4m3(N, K, W, K)
    A = np.zeros((M, lda), np.uint8); A[:, :K] = qa
    B = np.zeros((N, ldb), np.uint8); B[:, :K] = qb
    return A, sa, B, sb


def run_fp8(torch, M, N, K, A, lda, sa, B, ldb, sb, ldc, c_type):
    dt = torch.float32 if c_type == dg.DG_OUT_F32 else torch.bfloat16
    dC = torch.full((M * ldc,), float("nan"), dtype=dt, device="cuda")
    dg.gemm_fp8_e4m3(M, N, K, dev_u8(A, torch), lda, dev_f32(sa, torch), dev_u8(B, torch), ldb,
                     dev_f32(sb, torch), dC, ldc, c_type)
    sync(torch)
    C = host_f32(dC) if c_type == dg.DG_OUT_F32 else host_bf16_bits(dC)
    return C.reshape(M, ldc)


@pytest.mark.parametrize("M,N,K,lda,ldb", [(512, 2048, 1024, 1024, 1024), (300, 1000, 1000, 1008, 1024),
                                           (128, 128, 256, 256, 256), (1280, 2048, 6144, 6144, 6144),
                                           (256, 520, 200, 208, 224), (512, 8960, 256, 256, 256)])
@pytest.mark.parametrize("c_type", [dg.DG_OUT_BF16, dg.DG_OUT_F32])
def test_fp8_gemm_parity(torch, tile_mode, M, N, K, lda, ldb, c_type):
    # Pairs take 224-column tiles on every shape here but 512 x 8960 x 256, whose 2 x 35
    # tiles of 256 fill one wave where 2 x 40 tiles of 224 would need two.
    A, sa, B, sb = quantized_operands(M, N, K, lda, ldb, seed=M + N + K)
    ldc = N + 3 if M == 300 else N   # one case with unaligned C rows (direct stores)
    C = run_fp8(torch, M, N, K, A, lda, sa, B, ldb, sb, ldc, c_type)
    ref, D = oracle.gemm_fp8(M, N, K, A, lda, sa, B, ldb, sb)
    if c_type == dg.DG_OUT_F32:
        ok, worst = oracle.check_f32(C[:, :N], ref, D)
    else:
        ok, worst = oracle.check_bf16(C[:, :N], ref, D)
    assert ok, f"fp8 {M}x{N}x{K}: error {worst:.3g} of the bound"
    if ldc > N:
        assert np.all(np.isnan(C[:, N:].astype(np.float64) if c_type == dg.DG_OUT_F32 else
                               oracle.bf16_to_f64(C[:, N:])))


def test_fp8_gemm_integer_codes_bit_exact(torch, tile_mode):
    # Small-integer codes with unit scales: every partial sum is exact in FP32.
    M, N, K = 384, 768, 512
    rng = np.random.default_rng(52)
    A = oracle.round_e4m3(rng.integers(-8, 9, (M, K)).astype(np.float32))
    B = oracle.round_e4m3(rng.integers(-8, 9, (N, K)).astype(np.float32))
    one_a, one_b = np.ones(M, np.float32), np.ones(N, np.float32)
    C = run_fp8(torch, M, N, K, A, K, one_a, B, K, one_b, N, dg.DG_OUT_F32)
    ref, _ = oracle.gemm_fp8(M, N, K, A, K, one_a, B, K, one_b)
    assert np.array_equal(C.astype(np.float64), ref)


def test_fp8_ffn_full_size_whole_matrix(torch):
    # The FFN shape on FP8: M = 1024, N = 12288, K = 4096, GPU-quantised operands checked
    # bit-exact against the oracle's codes, then every output against the oracle GEMM.
    w = inputs.fp8_gemm()
    M, N, K = w["M"], w["N"], w["K"]
    qa, sa = quantize_gpu(torch, M, K, w["X"], K, K)
    qb, sb = quantize_gpu(torch, N, K, w["W"], K, K)
    qa_ref, sa_ref = oracle.quantize_rows_e4m3(M, K, w["X"], K)
    assert np.array_equal(qa, qa_ref) and np.array_equal(sa, sa_ref)
    qb_ref, sb_ref = oracle.quantize_rows_e4m3(N, K, w["W"], K)
    assert np.array_equal(qb, qb_ref) and np.array_equal(sb, sb_ref)
    C = run_fp8(torch, M, N, K, qa_ref, K, sa_ref, qb_ref, K, sb_ref, N, dg.DG_OUT_BF16)
    ref, D = oracle.gemm_fp8(M, N, K, qa_ref, K, sa_ref, qb_ref, K, sb_ref)
    ok, worst = oracle.check_bf16(C, ref, D)
    assert ok, f"fp8 FFN (whole matrix): {worst:.3g} of the bound"


def test_fp8_pair224_streamk_whole_matrix(torch):
    # 224-column pair tiles with a stream-K tail: FFN widths with K = 6144 give 4 x 55 tiles,
    # 2 whole waves of 76 pairs and 68 tail tiles spread over the pairs.  Random codes (no
    # NaN codes) and scales; every FP32 output against the oracle, and a repeat bit for bit
    # (the tail tiles' parts are added in a fixed order).
    M, N, K = 1024, 12288, 6144
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = dg.dg_plan_gemm(2, M, N, K, num_sms=sms)
    if sms == 152:
        assert plan["tile_n"] == 224 and plan["tail_tiles"] == 68
    rng = np.random.default_rng(61)

    def codes(r, c):
        q = rng.integers(0, 256, (r, c), dtype=np.uint8)
        q[(q & 0x7F) == 0x7F] = 0
        return q

    A, B = codes(M, K), codes(N, K)
    sa = (rng.uniform(0.5, 2.0, M) / 448).astype(np.float32)
    sb = (rng.uniform(0.5, 2.0, N) / 448).astype(np.float32)
    C = run_fp8(torch, M, N, K, A, K, sa, B, K, sb, N, dg.DG_OUT_F32)
    again = run_fp8(torch, M, N, K, A, K, sa, B, K, sb, N, dg.DG_OUT_F32)
    assert np.array_equal(C.view(np.uint32), again.view(np.uint32))
    ref, D = oracle.gemm_fp8(M, N, K, A, K, sa, B, K, sb)
    ok, worst = oracle.check_f32(C, ref, D)
    assert ok, f"fp8 224-wide pairs with stream-K (whole matrix): {worst:.3g} of the bound"


def test_fp8_deterministic(torch):
    A, sa, B, sb = quantized_operands(1280, 2048, 6144, 6144, 6144, seed=7)
    outs = [run_fp8(torch, 1280, 2048, 6144, A, 6144, sa, B, 6144, sb, 2048, dg.DG_OUT_F32)
            for _ in range(3)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_fp8_edges_and_errors(torch):
    u8 = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    f = torch.ones(64, dtype=torch.float32, device="cuda")
    C = torch.full((64 * 64,), 3.0, dtype=torch.float32, device="cuda")
    assert dg.gemm_fp8_e4m3(64, 64, 0, u8, 64, f, u8, 64, f, C, 64, dg.DG_OUT_F32) == dg.DG_OK
    sync(torch)
    assert torch.count_nonzero(C).item() == 0                         # K = 0: C = 0
    assert dg.gemm_fp8_e4m3(0, 64, 64, u8, 64, f, u8, 64, f, C, 64, dg.DG_OUT_F32) == dg.DG_OK
    kw = dict(check=False)
    assert dg.gemm_fp8_e4m3(64, 64, 64, u8, 32, f, u8, 64, f, C, 64, dg.DG_OUT_F32, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_fp8_e4m3(64, 64, 64, u8, 64, None, u8, 64, f, C, 64, dg.DG_OUT_F32, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_fp8_e4m3(64, 64, 64, u8, 64, f, u8, 64, f, C, 64, 7, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_fp8_e4m3(64, 64, 56, u8, 56, f, u8, 64, f, C, 64, dg.DG_OUT_F32, **kw) == dg.DG_ERR_MISALIGNED
    assert dg.gemm_fp8_e4m3(64, 64, 64, u8.data_ptr() + 8, 64, f, u8, 64, f, C, 64, dg.DG_OUT_F32,
                            **kw) == dg.DG_ERR_MISALIGNED
    assert dg.gemm_fp8_e4m3(64, 64, 64, u8, 64, f, u8, 64, f.data_ptr() + 4, C, 64, dg.DG_OUT_F32,
                            **kw) == dg.DG_ERR_MISALIGNED
    x = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    assert dg.quantize_rows_e4m3(-1, 64, x, 64, u8, 64, f, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.quantize_rows_e4m3(4, 64, x, 32, u8, 64, f, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.quantize_rows_e4m3(0, 64, x, 64, u8, 64, f) == dg.DG_OK
