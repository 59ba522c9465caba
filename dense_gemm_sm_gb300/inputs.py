"""Seeded synthetic inputs for the GEMM workloads.

This module is shared by the tests, the bench and the smoke check; it feeds the
same host arrays to the CUDA path and to the oracle.  It holds none of the
GEMM arithmetic: only random draws (numpy PCG64), the float32 -> bfloat16
input conversion, and padding to a leading dimension.

Workloads (shapes and distributions from the FFN running example of
"Operator & Runtime", section 5.2.1, and the SGEMM tutorial's square problems):

  sgemm_256      FP32 256^3, U[-1,1] (and an integer-valued copy in [-4,4])
  sgemm_4096     FP32 4096^3, alpha=1, beta=0.5, A, B, C0 ~ U[-1,1]
  sgemm_ragged   FP32 1000x3000x777, lda=780, ldb=ldc=3000, alpha=1, beta=0.5
  ffn_bf16       X[1024,4096] ~ N(0,1), W[4096,12288] ~ N(0,1/4096), BF16
  decode_bf16    X[M,4096] ~ N(0,1), same W, M in {1,4,16}
  bf16_square    BF16 4096^3 with the same operand distributions
  qk_batched     64 x (Q[2048,128] . K[2048,128]^T), alpha=fp32(1/sqrt(128)), FP32 out
  ffn_gate_up    X[1024,4096] ~ N(0,1), W_g, W_u [4096,12288] ~ N(0,1/4096), BF16
  attention      Q, K, V [batch, L, 128] ~ N(0,1) BF16, scale fp32(1/sqrt(128)); the batched
                 shape (64 heads x 2048) and one causal head of 8192 ("Operator & Runtime",
                 section 5.3.3)
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def uniform_f32(seed: int, shape, lo=-1.0, hi=1.0) -> np.ndarray:
    return rng(seed).uniform(lo, hi, size=shape).astype(np.float32)


def integer_f32(seed: int, shape, lo=-4, hi=4) -> np.ndarray:
    """Integer values in [lo, hi] stored as float32 (exact)."""
    return rng(seed).integers(lo, hi + 1, size=shape).astype(np.float32)


def normal_f32(seed: int, shape, std=1.0) -> np.ndarray:
    return (rng(seed).standard_normal(size=shape, dtype=np.float32) * np.float32(std)).astype(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 input data to bfloat16 (nearest, ties to even); finite inputs only.

    Returns the raw 16-bit patterns (uint16), the form both the CUDA path
    (as torch.bfloat16 storage) and the oracle consume.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not np.all(np.isfinite(x)):
        raise ValueError("synthetic inputs must be finite")
    bits = x.view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((bits >> np.uint64(16)) & np.uint64(1))
    return ((bits + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float32 (for display / sanity)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def pad_rows(x: np.ndarray, ld: int, fill=np.nan) -> np.ndarray:
    """Copy a 2-D array into a (rows, ld) buffer; columns beyond x.shape[1] get `fill`."""
    rows, cols = x.shape
    if ld < cols:
        raise ValueError("leading dimension smaller than the row length")
    out = np.full((rows, ld), fill, dtype=x.dtype)
    out[:, :cols] = x
    return out


# --------------------------------------------------------------------------
# The named workloads.  Each returns a dict of host arrays and scalars.
# --------------------------------------------------------------------------

def sgemm_256(integer: bool = False) -> dict:
    s = BASE_SEED + 0
    M = N = K = 256
    if integer:
        A, B = integer_f32(s, (M, K)), integer_f32(s + 100, (K, N))
    else:
        A, B = uniform_f32(s, (M, K)), uniform_f32(s + 100, (K, N))
    return dict(M=M, N=N, K=K, alpha=np.float32(1.0), beta=np.float32(0.0), A=A, lda=K, B=B,
                ldb=N, C0=None, ldc=N)


def sgemm_4096(M=4096, N=4096, K=4096) -> dict:
    s = BASE_SEED + 1
    return dict(M=M, N=N, K=K, alpha=np.float32(1.0), beta=np.float32(0.5),
                A=uniform_f32(s, (M, K)), lda=K, B=uniform_f32(s + 100, (K, N)), ldb=N,
                C0=uniform_f32(s + 200, (M, N)), ldc=N)


def sgemm_ragged() -> dict:
    s = BASE_SEED + 1
    M, N, K = 1000, 3000, 777
    lda, ldb, ldc = 780, 3000, 3000
    A = pad_rows(uniform_f32(s + 300, (M, K)), lda)
    B = pad_rows(uniform_f32(s + 400, (K, N)), ldb)
    C0 = pad_rows(uniform_f32(s + 500, (M, N)), ldc)
    return dict(M=M, N=N, K=K, alpha=np.float32(1.0), beta=np.float32(0.5), A=A, lda=lda,
                B=B, ldb=ldb, C0=C0, ldc=ldc)


def ffn_weight(K=4096, N=12288) -> np.ndarray:
    """W[K,N] ~ N(0, 1/K) rounded to bf16 bits."""
    return f32_to_bf16_bits(normal_f32(BASE_SEED + 2 + 100, (K, N), std=1.0 / np.sqrt(K)))


def ffn_bf16(M=1024, K=4096, N=12288, W=None) -> dict:
    s = BASE_SEED + 2
    X = f32_to_bf16_bits(normal_f32(s, (M, K)))
    if W is None:
        W = ffn_weight(K, N)
    return dict(M=M, N=N, K=K, alpha=np.float32(1.0), beta=np.float32(0.0), A=X, lda=K, B=W,
                ldb=N, C0=None, ldc=N)


def ffn_gate_up(M=1024, K=4096, N=12288) -> dict:
    """FFN gate and up projections: X [M,K] ~ N(0,1), W_g and W_u [K,N] ~ N(0, 1/K), BF16."""
    s = BASE_SEED + 7
    X = f32_to_bf16_bits(normal_f32(s, (M, K)))
    Wg = f32_to_bf16_bits(normal_f32(s + 1, (K, N), std=1.0 / np.sqrt(K)))
    Wu = f32_to_bf16_bits(normal_f32(s + 2, (K, N), std=1.0 / np.sqrt(K)))
    return dict(M=M, N=N, K=K, X=X, ldx=K, Wg=Wg, ldwg=N, Wu=Wu, ldwu=N, ldz=N)


def bf16_square(n=4096) -> dict:
    """BF16 n^3 GEMM with the FFN operand distributions (the "4096-class" square shape)."""
    s = BASE_SEED + 5
    X = f32_to_bf16_bits(normal_f32(s, (n, n)))
    W = f32_to_bf16_bits(normal_f32(s + 100, (n, n), std=1.0 / np.sqrt(n)))
    return dict(M=n, N=n, K=n, alpha=np.float32(1.0), beta=np.float32(0.0), A=X, lda=n, B=W,
                ldb=n, C0=None, ldc=n)


def decode_bf16(M: int, K=4096, N=12288, W=None) -> dict:
    s = BASE_SEED + 3
    X = f32_to_bf16_bits(normal_f32(s + M, (M, K)))
    if W is None:
        W = ffn_weight(K, N)
    return dict(M=M, N=N, K=K, alpha=np.float32(1.0), beta=np.float32(0.0), A=X, lda=K, B=W,
                ldb=N, C0=None, ldc=N)


def qk_batched(batch=64, S=2048, D=128) -> dict:
    s = BASE_SEED + 4
    Q = f32_to_bf16_bits(normal_f32(s, (batch, S, D)))
    Kt = f32_to_bf16_bits(normal_f32(s + 100, (batch, S, D)))
    return dict(M=S, N=S, K=D, batch=batch, alpha=np.float32(1.0 / np.sqrt(np.float32(D))),
                beta=np.float32(0.0), A=Q, lda=D, strideA=S * D, B=Kt, ldb=D, strideB=S * D,
                op_b=1, C0=None, ldc=S, strideC=S * S)


def attention(batch=64, L=2048, d=128, causal=False, Lkv=None, std_q=1.0) -> dict:
    """Q [batch, L, d], K and V [batch, Lkv, d] ~ N(0,1) BF16 (Q scaled by std_q), contiguous."""
    s = BASE_SEED + 8 + (1 if causal else 0)
    Lkv = L if Lkv is None else Lkv
    Q = f32_to_bf16_bits(normal_f32(s, (batch, L, d), std=std_q))
    K = f32_to_bf16_bits(normal_f32(s + 100, (batch, Lkv, d)))
    V = f32_to_bf16_bits(normal_f32(s + 200, (batch, Lkv, d)))
    return dict(batch=batch, Lq=L, Lkv=Lkv, d=d, causal=causal,
                scale=np.float32(1.0 / np.sqrt(np.float32(d))), Q=Q, ldq=d, sQ=L * d, K=K, ldk=d,
                sK=Lkv * d, V=V, ldv=d, sV=Lkv * d, ldo=d, sO=L * d)


def fp8_gemm(M=1024, N=12288, K=4096) -> dict:
    """BF16 activations X [M, K] ~ N(0,1) and weights W [N, K] ~ N(0, 1/K) (stored by output
    column), to be quantised per row to FP8 E4M3."""
    s = BASE_SEED + 10
    X = f32_to_bf16_bits(normal_f32(s, (M, K)))
    W = f32_to_bf16_bits(normal_f32(s + 1, (N, K), std=1.0 / np.sqrt(K)))
    return dict(M=M, N=N, K=K, X=X, W=W)


def decode_chain(M=1, dims=(4096, 12288, 4096, 12288, 4096)) -> dict:
    """X [M, dims[0]] ~ N(0,1) and layer weights W_l [dims[l], dims[l+1]] ~ N(0, 1/dims[l])
    (so activations keep unit scale), BF16: FFN-shaped up/down layers."""
    s = BASE_SEED + 11
    X = f32_to_bf16_bits(normal_f32(s + M, (M, dims[0])))
    Ws = [f32_to_bf16_bits(normal_f32(s + 100 + l, (dims[l], dims[l + 1]), std=1.0 / np.sqrt(dims[l])))
          for l in range(len(dims) - 1)]
    return dict(M=M, dims=list(dims), X=X, Ws=Ws)
