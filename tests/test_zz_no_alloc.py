"""gemm_bf16_decode_noalloc: the decode-shaped BF16 GEMM for callers that cannot allocate.

Some callers cannot let the library call cudaMalloc (a framework whose allocator already
holds the device memory, or a decode loop that cannot take cudaMalloc's device-wide
synchronisation).  This entry point runs the split-K decode kernel with a fixed scratch
array inside the library instead of an allocated workspace.  These tests call it through
the C ABI twice in a row and check each result against gemm_bf16 on the same inputs,
within the BF16 bound the other tests use (2e-4 * D + one bf16 ulp).  The file is named so
that pytest collects it last.
"""
import numpy as np
import pytest

import oracle
import dense_gemm_sm_gb300 as dg
from dense_gemm_sm_gb300 import inputs

from .helpers import dev_bf16, host_bf16_bits, torch_mod

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = torch_mod()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    dg.load()
    return t


def test_noalloc_matches_gemm_bf16_on_two_calls_in_a_row(torch):
    K, N = 4096, 12288
    W = inputs.ffn_weight(K, N)
    dW = dev_bf16(W)
    cases = [(16, 101), (5, 102)]
    xs = [inputs.f32_to_bf16_bits(inputs.normal_f32(seed, (M, K))) for M, seed in cases]
    dxs = [dev_bf16(x) for x in xs]
    outs = [torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda") for M, _ in cases]
    # two calls of the new entry point back to back, sharing its scratch
    for (M, _), dx, out in zip(cases, dxs, outs):
        dg.gemm_bf16_decode_noalloc(M, N, K, 1.0, dx, K, dW, N, 0.0, out, N)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    for (M, _), x, dx, out in zip(cases, xs, dxs, outs):
        ref_dev = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        dg.gemm_bf16(M, N, K, 1.0, dx, K, dW, N, 0.0, ref_dev, N)
        torch.cuda.synchronize()
        assert dg.dg_device_status() == dg.DG_OK
        got = host_bf16_bits(out)
        ref = oracle.bf16_to_f64(host_bf16_bits(ref_dev))
        _, den = oracle.gemm(M, N, K, 1.0, x, K, W, N, absden=True)
        ok, worst = oracle.check_bf16(got, ref, den[0])
        assert ok, f"M={M}: no-alloc result differs from gemm_bf16 by {worst:.3g} x the bound"


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
    _, den = oracle.gemm(M, N, K, 0.5, x, K, w, N, -1.5, c0, N, absden=True)
    ok, worst = oracle.check_bf16(host_bf16_bits(a), oracle.bf16_to_f64(host_bf16_bits(b)), den[0])
    assert ok, worst


def test_noalloc_rejects_sizes_beyond_its_scratch(torch):
    z = torch.zeros(17 * 4096, dtype=torch.bfloat16, device="cuda")
    st = dg.gemm_bf16_decode_noalloc(17, 128, 64, 1.0, z, 64, z, 128, 0.0, z, 128, check=False)
    assert st == dg.DG_ERR_UNSUPPORTED
    big_n = 8192 * 128 + 8
    st = dg.gemm_bf16_decode_noalloc(1, big_n, 64, 1.0, z, 64, z, big_n, 0.0, z, big_n, check=False)
    assert st == dg.DG_ERR_UNSUPPORTED
