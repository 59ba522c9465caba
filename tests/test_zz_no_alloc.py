"""gemm_bf16_decode_noalloc: the decode-shaped BF16 GEMM for callers that cannot allocate.

Some callers cannot let the library call cudaMalloc (a framework whose allocator already
holds the device memory, or a decode loop that cannot take cudaMalloc's device-wide
synchronisation).  This entry point runs the split-K decode kernel with a fixed scratch
array inside the library instead of an allocated workspace.  These tests call it through
the C ABI several times in a row and check every result against the oracle, within the
bound the other tests use (BF16 output 2e-4 * D + one bf16 ulp, FP32 output 1e-5 * D), and
bit for bit against gemm_bf16 on the same inputs: where the GPU has at most 160 SMs both
run the same kernel on the same split, so stale scratch (a partial or counter left by the
previous call) would show as a difference.  The file is named so that pytest collects it
last.
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


def bits_of(t, f32):
    return host_f32(t).view(np.uint32) if f32 else host_bf16_bits(t)


def same_split_as_gemm_bf16(torch):
    # gemm_bf16 splits decode shapes over min(units, SMs) CTAs, this entry point over
    # min(units, SMs, 160): the same split, and so the same bits, up to 160 SMs.
    return torch.cuda.get_device_properties(0).multi_processor_count <= 160


def check_against_oracle(got, f32, M, N, K, alpha, x, w, beta=0.0, c0=None, what=""):
    ref, den = oracle.gemm(M, N, K, alpha, x, K, w, N, beta, c0, N, absden=True)
    if f32:
        ok, worst = oracle.check_f32(host_f32(got), ref[0], den[0])
    else:
        ok, worst = oracle.check_bf16(host_bf16_bits(got), ref[0], den[0])
    assert ok, f"{what}: error reaches {worst:.3g} x the bound"


@pytest.mark.parametrize("f32", [False, True])
def test_noalloc_calls_in_a_row_match_the_oracle_and_gemm_bf16(torch, f32):
    # The FFN weight (N = 12288, K = 4096) and a ragged N = 12200 (a last tile of 40 columns)
    # at M = 16, then M = 5 and M = 1: calls back to back on one stream sharing the scratch.
    K = 4096
    W = inputs.ffn_weight(K, 12288)
    W2 = np.ascontiguousarray(W.reshape(K, 12288)[:, :12200])   # K x 12200, row-major
    weights = {12288: (W, dev_bf16(W)), 12200: (W2, dev_bf16(W2))}
    cases = [(16, 12288, 101), (16, 12200, 102), (5, 12288, 103), (1, 12288, 104)]
    dtype = torch.float32 if f32 else torch.bfloat16
    c_type = dg.DG_OUT_F32 if f32 else dg.DG_OUT_BF16
    xs = [inputs.f32_to_bf16_bits(inputs.normal_f32(seed, (M, K))) for M, _, seed in cases]
    dxs = [dev_bf16(x) for x in xs]
    outs = [torch.full((M, N), float("nan"), dtype=dtype, device="cuda") for M, N, _ in cases]
    for (M, N, _), dx, out in zip(cases, dxs, outs):      # back to back, one stream
        dg.gemm_bf16_decode_noalloc(M, N, K, 1.0, dx, K, weights[N][1], N, 0.0, out, N, c_type)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    for (M, N, _), x, dx, out in zip(cases, xs, dxs, outs):
        Wn, dWn = weights[N]
        check_against_oracle(out, f32, M, N, K, 1.0, x, Wn, what=f"no-alloc M={M} N={N}")
        ref_dev = torch.full((M, N), float("nan"), dtype=dtype, device="cuda")
        dg.gemm_bf16(M, N, K, 1.0, dx, K, dWn, N, 0.0, ref_dev, N, c_type)
        torch.cuda.synchronize()
        assert dg.dg_device_status() == dg.DG_OK
        if same_split_as_gemm_bf16(torch):
            assert np.array_equal(bits_of(out, f32), bits_of(ref_dev, f32)), f"M={M} N={N}"


def test_noalloc_same_call_repeated(torch):
    # The same call four times in a row with FP32 output: each result equals the first bit for
    # bit (the arrival counters are back at zero after every call) and the oracle's.
    M, N, K = 16, 12288, 4096
    W = inputs.ffn_weight(K, N)
    x = inputs.f32_to_bf16_bits(inputs.normal_f32(110, (M, K)))
    dx, dW = dev_bf16(x), dev_bf16(W)
    outs = []
    for _ in range(4):
        out = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        dg.gemm_bf16_decode_noalloc(M, N, K, 1.0, dx, K, dW, N, 0.0, out, N, dg.DG_OUT_F32)
        outs.append(out)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    first = host_f32(outs[0]).view(np.uint32)
    for o in outs[1:]:
        assert np.array_equal(host_f32(o).view(np.uint32), first)
    check_against_oracle(outs[0], True, M, N, K, 1.0, x, W, what="repeated no-alloc call")


def test_noalloc_alpha_beta_and_ragged(torch):
    M, N, K = 3, 1000, 520
    x = inputs.f32_to_bf16_bits(inputs.normal_f32(103, (M, K)))
    w = inputs.f32_to_bf16_bits(inputs.normal_f32(104, (K, N), 0.05))
    c0 = inputs.f32_to_bf16_bits(inputs.normal_f32(105, (M, N)))
    dx, dw = dev_bf16(x), dev_bf16(w)
    a = dev_bf16(c0)
    b = dev_bf16(c0)
    dg.gemm_bf16_decode_noalloc(M, N, K, 0.5, dx, K, dw, N, -1.5, a, N)
    dg.gemm_bf16(M, N, K, 0.5, dx, K, dw, N, -1.5, b, N)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    check_against_oracle(a, False, M, N, K, 0.5, x, w, -1.5, c0, what="no-alloc alpha/beta")
    if same_split_as_gemm_bf16(torch):
        assert np.array_equal(host_bf16_bits(a), host_bf16_bits(b))


def test_noalloc_rejects_sizes_beyond_its_scratch(torch):
    z = torch.zeros(17 * 4096, dtype=torch.bfloat16, device="cuda")
    st = dg.gemm_bf16_decode_noalloc(17, 128, 64, 1.0, z, 64, z, 128, 0.0, z, 128, check=False)
    assert st == dg.DG_ERR_UNSUPPORTED
    big_n = 8192 * 128 + 8
    st = dg.gemm_bf16_decode_noalloc(1, big_n, 64, 1.0, z, 64, z, big_n, 0.0, z, big_n, check=False)
    assert st == dg.DG_ERR_UNSUPPORTED
