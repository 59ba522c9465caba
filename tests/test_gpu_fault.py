"""Bounded waits: a kernel that cannot make progress reports DG_ERR_TIMEOUT and exits.

dg_set_fault_injection(1) makes the tile kernel's MMA issuer skip its shared-memory stage
releases, so the TMA producer's wait for a free stage can never succeed.  Every wait in the
kernel is bounded (about one second): the CTAs record the timeout in the device status
word, wait for their own copies and MMAs, free TMEM and return -- no hang, no fault.  The
context stays usable: a normal GEMM afterwards is correct.
"""
import numpy as np
import pytest

import oracle
import dense_gemm_sm_gb300 as dg
from dense_gemm_sm_gb300 import inputs

from .helpers import dev_bf16, host_bf16_bits, torch_mod

pytestmark = pytest.mark.gpu


def test_bounded_wait_expiry_is_reported_and_context_survives():
    torch = torch_mod()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    M, N, K = 256, 512, 1024  # 4 tiles, 16 K blocks each: more K blocks than ring stages
    w = inputs.ffn_bf16(M=M, K=K, N=N)
    dA, dB = dev_bf16(w["A"]), dev_bf16(w["B"])
    dC = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert dg.dg_device_status() == dg.DG_OK
    dg.dg_set_fault_injection(1)
    try:
        dg.gemm_bf16(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
        torch.cuda.synchronize()
    finally:
        dg.dg_set_fault_injection(0)
    assert dg.dg_device_status() == dg.DG_ERR_TIMEOUT
    assert dg.dg_device_status() == dg.DG_OK  # read-and-clear
    dg.gemm_bf16(M, N, K, 1.0, dA, K, dB, N, 0.0, dC, N)
    torch.cuda.synchronize()
    assert dg.dg_device_status() == dg.DG_OK
    ref, den = oracle.gemm(M, N, K, 1.0, w["A"], K, w["B"], N, absden=True)
    ok, worst = oracle.check_bf16(host_bf16_bits(dC), ref[0], den[0])
    assert ok, worst
