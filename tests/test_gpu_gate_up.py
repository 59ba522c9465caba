"""GPU parity of the fused FFN gate/up projections (gemm_bf16_gate_up_silu) against the
CPU oracle: Z = bf16(SiLU(bf16(X W_g)) * bf16(X W_u)).

Acceptance (oracle.check_gate_up): every element within the bound derived from the BF16
GEMM bound of G and U, SiLU's slope and Z's own rounding; and at least 99 % of the
elements equal, bit for bit, the BF16 rounding of the oracle's z (only G or U values at a
BF16 rounding boundary may round differently on the GPU, which accumulates in FP32).
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


@pytest.fixture(params=["pair", "single"])
def tile_mode(request, monkeypatch):
    if request.param == "single":
        monkeypatch.setenv("DG_TC_PAIR", "0")
    else:
        monkeypatch.delenv("DG_TC_PAIR", raising=False)
    return request.param


def run(torch, M, N, K, X, ldx, Wg, ldwg, Wu, ldwu, ldz):
    dZ = torch.full((M * ldz,), float("nan"), device="cuda", dtype=torch.bfloat16)
    dg.gemm_bf16_gate_up_silu(M, N, K, dev_bf16(X), ldx, dev_bf16(Wg), ldwg, dev_bf16(Wu), ldwu,
                              dZ, ldz)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    return host_bf16_bits(dZ).reshape(M, ldz)


def check(Z, M, N, K, X, ldx, Wg, ldwg, Wu, ldwu, what):
    z, gb, ub, Dg, Du = oracle.gate_up_silu(M, N, K, X, ldx, Wg, ldwg, Wu, ldwu)
    ok, worst, same = oracle.check_gate_up(Z[:, :N], z, gb, ub, Dg, Du)
    assert ok, f"{what}: error reaches {worst:.3g} x the bound"
    assert same >= 0.99, f"{what}: only {same:.4f} of Z equals bf16(z)"
    return same


@pytest.mark.parametrize("M,N,K", [(512, 2048, 1024), (300, 1000, 1000), (128, 640, 512),
                                   (1280, 2048, 6144)])
def test_gate_up_parity(torch, tile_mode, M, N, K):
    # (300, 1000, 1000): ragged M, N and K tiles; (128, 640, 512): one 128-row tile row;
    # (1280, 2048, 6144): the tail tiles run stream-K before the whole waves.
    w = inputs.ffn_gate_up(M, K, N)
    Z = run(torch, M, N, K, w["X"], K, w["Wg"], N, w["Wu"], N, N)
    check(Z, M, N, K, w["X"], K, w["Wg"], N, w["Wu"], N, f"gate/up {M}x{N}x{K}")


def test_gate_up_padded_rows(torch, tile_mode):
    # Leading dimensions beyond the row lengths; Z rows not 16-byte aligned (direct stores);
    # the padding of Z is left untouched.
    M, N, K = 256, 520, 264
    ldx, ldw, ldz = K + 8, N + 8, N + 3
    rng = np.random.default_rng(11)
    X = inputs.pad_rows(inputs.f32_to_bf16_bits(rng.normal(0, 1, (M, K)).astype(np.float32)), ldx, 0)
    Wg = inputs.pad_rows(inputs.f32_to_bf16_bits(rng.normal(0, 0.06, (K, N)).astype(np.float32)), ldw, 0)
    Wu = inputs.pad_rows(inputs.f32_to_bf16_bits(rng.normal(0, 0.06, (K, N)).astype(np.float32)), ldw, 0)
    Z = run(torch, M, N, K, X, ldx, Wg, ldw, Wu, ldw, ldz)
    check(Z, M, N, K, X, ldx, Wg, ldw, Wu, ldw, "gate/up padded")
    pad = Z[:, N:]
    assert np.all((pad & 0x7FFF) > 0x7F80), "padding of Z was written"   # still NaN


def test_gate_up_ffn_full_size(torch):
    # The FFN shape of the pages' running example, compared in full.
    w = inputs.ffn_gate_up()
    M, N, K = w["M"], w["N"], w["K"]
    Z = run(torch, M, N, K, w["X"], K, w["Wg"], N, w["Wu"], N, N)
    check(Z, M, N, K, w["X"], K, w["Wg"], N, w["Wu"], N, "gate/up FFN 1024x12288x4096")


def test_gate_up_integer_data(torch, tile_mode):
    # Small integers: G and U are exact in FP32 and BF16, so only SiLU's FP32 evaluation
    # can move a value across a BF16 rounding boundary.
    M, N, K = 256, 512, 128
    rng = np.random.default_rng(12)
    X = inputs.f32_to_bf16_bits(rng.integers(-2, 3, (M, K)).astype(np.float32))
    Wg = inputs.f32_to_bf16_bits(rng.integers(-1, 2, (K, N)).astype(np.float32))
    Wu = inputs.f32_to_bf16_bits(rng.integers(-1, 2, (K, N)).astype(np.float32))
    Z = run(torch, M, N, K, X, K, Wg, N, Wu, N, N)
    check(Z, M, N, K, X, K, Wg, N, Wu, N, "gate/up integer")
    # Every element whose BF16 rounding differs from the oracle's must be a rounding decided
    # at FP32 precision: z within a few FP32 ulps of the midpoint between the two BF16
    # neighbours (e.g. SiLU(g) = g in FP32 for g >= 17, so g * u lands on a tie).
    z, _, _, _, _ = oracle.gate_up_silu(M, N, K, X, K, Wg, N, Wu, N)
    ref = oracle.round_bf16(z)
    diff = Z[:, :N] != ref
    zg = oracle.bf16_to_f64(Z[:, :N][diff])
    zr = oracle.bf16_to_f64(ref[diff])
    mid = 0.5 * (zg + zr)
    assert np.all(np.abs(zg - zr) <= oracle.ulp_bf16(np.abs(zr)) * 1.0 + 0.0)
    assert np.all(np.abs(z[diff] - mid) <= 2.0 ** -20 * np.abs(mid)), "a non-tie rounds differently"


def test_gate_up_deterministic(torch):
    w = inputs.ffn_gate_up(1280, 6144, 2048)   # stream-K tail active
    outs = [run(torch, 1280, 2048, 6144, w["X"], 6144, w["Wg"], 2048, w["Wu"], 2048, 2048)
            for _ in range(3)]
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[1], outs[2])


def test_gate_up_edges_and_errors(torch):
    X = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(64 * 64, dtype=torch.bfloat16, device="cuda")
    Z = torch.full((64 * 64,), 3.0, dtype=torch.bfloat16, device="cuda")
    assert dg.gemm_bf16_gate_up_silu(0, 64, 64, X, 64, W, 64, W, 64, Z, 64) == dg.DG_OK
    assert dg.gemm_bf16_gate_up_silu(64, 64, 0, X, 64, W, 64, W, 64, Z, 64) == dg.DG_OK
    torch.cuda.synchronize()
    assert torch.count_nonzero(Z).item() == 0                      # K = 0: Z = SiLU(0) * 0
    f = dict(check=False)
    assert dg.gemm_bf16_gate_up_silu(-1, 64, 64, X, 64, W, 64, W, 64, Z, 64, **f) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_gate_up_silu(64, 64, 64, X, 32, W, 64, W, 64, Z, 64, **f) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_gate_up_silu(64, 64, 64, X, 64, W, 64, W, 64, Z, 60, **f) == dg.DG_ERR_INVALID_ARG
    assert dg.gemm_bf16_gate_up_silu(64, 64, 60, X, 60, W, 64, W, 64, Z, 64, **f) == dg.DG_ERR_MISALIGNED
    assert dg.gemm_bf16_gate_up_silu(64, 64, 64, X, 64, W.data_ptr() + 2, 64, W, 64, Z, 64,
                                     **f) == dg.DG_ERR_MISALIGNED
