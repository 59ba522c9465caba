"""Shared test helpers: moving seeded host arrays to the GPU and comparing with the oracle."""
from __future__ import annotations

import numpy as np

import oracle


def torch_mod():
    import torch
    return torch


def dev_f32(x: np.ndarray):
    torch = torch_mod()
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def dev_bf16(bits: np.ndarray):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def host_bf16_bits(t) -> np.ndarray:
    torch = torch_mod()
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def host_f32(t) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def sample_indices(seed: int, n: int, *dims):
    """n random index tuples over the given dimension sizes, plus the corners."""
    r = np.random.Generator(np.random.PCG64(seed))
    cols = [r.integers(0, d, size=n) for d in dims]
    corners = np.array(np.meshgrid(*[[0, d - 1] for d in dims], indexing="ij")).reshape(len(dims), -1)
    return [np.concatenate([c, corners[i]]) for i, c in enumerate(cols)]


def assert_f32_close(C, ref, den, what=""):
    ok, worst = oracle.check_f32(C, ref, den)
    assert ok, f"{what}: FP32 normalised error {worst:.3g} exceeds {oracle.FP32_REL}"
    return worst


def assert_bf16_close(C_bits, ref, den, what=""):
    ok, worst = oracle.check_bf16(C_bits, ref, den)
    assert ok, f"{what}: BF16 error reaches {worst:.3g} x the bound (2e-4*D + ulp)"
    return worst
