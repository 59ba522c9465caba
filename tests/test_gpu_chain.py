"""GPU tests of the persistent decode chain (gemm_bf16_decode_chain).

  * against the oracle chain, layer by layer, within the BF16 GEMM bound plus the
    propagated effect of the previous layer's rounding;
  * against the same layers run as separate gemm_bf16 calls: bit for bit when every layer
    has at least as many W blocks as the GPU has SMs (same partition and combine order);
  * repeated calls and CUDA-graph replay give identical results (the device-side epoch).
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


def sync(torch):
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK


def setup(torch, w):
    M, dims = w["M"], w["dims"]
    dX = dev_bf16(w["X"])
    dW = [dev_bf16(W) for W in w["Ws"]]
    dY = [torch.full((M * dims[l + 1],), float("nan"), dtype=torch.bfloat16, device="cuda")
          for l in range(len(dW))]
    return dX, dW, dY


def run_chain(torch, w, dX, dW, dY):
    dims = w["dims"]
    dg.gemm_bf16_decode_chain(w["M"], dims, dX, dims[0], dW, dims[1:], dY)
    sync(torch)
    return [host_bf16_bits(y).reshape(w["M"], -1) for y in dY]


@pytest.mark.parametrize("M,dims", [(16, (4096, 12288, 4096)), (3, (520, 1000, 776, 3000)),
                                    (1, (4096, 12288, 4096, 12288, 4096)), (7, (64, 128, 64, 8, 200))])
def test_chain_oracle_parity(torch, M, dims):
    w = inputs.decode_chain(M, dims)
    Ys = run_chain(torch, w, *setup(torch, w))
    ref = oracle.decode_chain(M, list(dims), w["X"], dims[0], w["Ws"], list(dims[1:]))
    for l, (y, _, bound) in enumerate(ref):
        ok, worst = oracle.check_chain_layer(Ys[l], y, bound)
        assert ok, f"chain M={M} dims={dims}: layer {l} error {worst:.3g} of the bound"


@pytest.mark.parametrize("M", [1, 5, 16])
def test_chain_equals_separate_calls_bitwise(torch, M):
    w = inputs.decode_chain(M)
    dX, dW, dY = setup(torch, w)
    Ys = run_chain(torch, w, dX, dW, dY)
    dims = w["dims"]
    x, ldx = dX, dims[0]
    for l in range(len(dW)):
        out = torch.empty(M * dims[l + 1], dtype=torch.bfloat16, device="cuda")
        dg.gemm_bf16(M, dims[l + 1], dims[l], 1.0, x, ldx, dW[l], dims[l + 1], 0.0, out, dims[l + 1],
                     dg.DG_OUT_BF16)
        sync(torch)
        assert np.array_equal(host_bf16_bits(out).reshape(M, -1), Ys[l]), f"layer {l} differs"
        x, ldx = out, dims[l + 1]


def test_chain_repeats_and_graph_replay(torch):
    w = inputs.decode_chain(4)
    dX, dW, dY = setup(torch, w)
    first = run_chain(torch, w, dX, dW, dY)
    for _ in range(4):
        again = run_chain(torch, w, dX, dW, dY)
        assert all(np.array_equal(a, b) for a, b in zip(first, again))
    dims = w["dims"]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        dg.gemm_bf16_decode_chain(w["M"], dims, dX, dims[0], dW, dims[1:], dY, stream=side)
    side.synchronize()
    for y in dY:
        y.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for _ in range(3):
            dg.gemm_bf16_decode_chain(w["M"], dims, dX, dims[0], dW, dims[1:], dY, stream=side)
    for _ in range(2):
        graph.replay()
    sync(torch)
    assert all(np.array_equal(a, host_bf16_bits(y).reshape(w["M"], -1)) for a, y in zip(first, dY))


def test_chain_errors(torch):
    t = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    kw = dict(check=False)
    assert dg.gemm_bf16_decode_chain(0, [64, 64], t, 64, [t], [64], [t]) == dg.DG_OK
    assert dg.gemm_bf16_decode_chain(17, [64, 64], t, 64, [t], [64], [t], **kw) == dg.DG_ERR_UNSUPPORTED
    assert dg.gemm_bf16_decode_chain(1, [64, 0], t, 64, [t], [64], [t], **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_decode_chain(1, [64, 64], t, 32, [t], [64], [t], **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_decode_chain(1, [64] * 10, t, 64, [t] * 9, [64] * 9, [t] * 9, **kw) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_decode_chain(1, [64, 60, 64], t, 64, [t, t], [64, 64], [t, t], **kw) == dg.DG_ERR_MISALIGNED
    assert dg.gemm_bf16_decode_chain(1, [64, 64], t.data_ptr() + 2, 64, [t], [64], [t], **kw) == dg.DG_ERR_MISALIGNED
