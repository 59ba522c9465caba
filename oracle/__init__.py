"""CPU FP64 oracle for the dense GEMM hot path -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
the two share no code: the oracle is plain C (``oracle.c``) built with gcc,
loaded here with ctypes.

Definition followed (see the header of ``oracle.c`` for the passages):
``C[b,i,j] = alpha * sum_k A[b,i,k] * opB[b,k,j] + beta * C0[b,i,j]`` in IEEE
double, with exact widening of float32 / bfloat16 inputs, and one
round-to-nearest-even to bfloat16 afterwards where the output is BF16
("Operator & Runtime", sections 5.4.2-5.4.3: round once after the full K
accumulation).

Every function is pinned by tests/test_oracle_pins.py against values fixed by
the pages or by mathematics (hand products, identities, closed forms,
numpy's float64 matmul on integer data, IEEE rounding cases).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, BF16, F64 = 0, 1, 2

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, no CUDA)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        # -O2 without -ffast-math: IEEE double arithmetic, no reassociation.
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
               "-ffp-contract=off", "-pthread", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        gemm_args = [i64, i64, i64, i64, dbl,
                     vp, ci, i64, i64,
                     vp, ci, i64, i64, ci,
                     dbl, vp, ci, i64, i64,
                     vp, i64, i64, ci]
        lib.oracle_gemm.argtypes = gemm_args
        lib.oracle_gemm.restype = ci
        lib.oracle_gemm_absden.argtypes = gemm_args
        lib.oracle_gemm_absden.restype = ci
        lib.oracle_gemm_entries.argtypes = [i64, i64, i64, dbl,
                                            vp, ci, i64, i64,
                                            vp, ci, i64, i64, ci,
                                            dbl, vp, ci, i64, i64,
                                            i64, vp, vp, vp, vp, vp]
        lib.oracle_gemm_entries.restype = ci
        lib.oracle_round_bf16.argtypes = [vp, vp, i64]
        lib.oracle_round_bf16.restype = None
        lib.oracle_bf16_to_double.argtypes = [vp, vp, i64]
        lib.oracle_bf16_to_double.restype = None
        lib.oracle_ulp_bf16_array.argtypes = [vp, vp, i64]
        lib.oracle_ulp_bf16_array.restype = None
        lib.oracle_ulp_bf16.argtypes = [dbl]
        lib.oracle_ulp_bf16.restype = dbl
        lib.oracle_gemm_flops.argtypes = [i64, i64, i64, i64]
        lib.oracle_gemm_flops.restype = dbl
        _lib = lib
        return lib


def _typed(arr: np.ndarray):
    """(contiguous array, type code) for a float32 / bf16-bits (uint16) / float64 array."""
    arr = np.ascontiguousarray(arr)
    if arr.dtype == np.float32:
        return arr, F32
    if arr.dtype == np.uint16:
        return arr, BF16
    if arr.dtype == np.float64:
        return arr, F64
    raise TypeError(f"oracle inputs are float32, float64 or uint16 (bf16 bits), got {arr.dtype}")


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def gemm(M, N, K, alpha, A, lda, B, ldb, beta=0.0, C0=None, ldc=None, *, op_b=0,
         batch=1, strideA=0, strideB=0, strideC=0, nthreads=None, absden=False):
    """Full result (batch, M, N) in float64 (and the error scale D if absden).

    ``A``, ``B``, ``C0`` are flat (or any-shape, contiguous) arrays indexed with
    the given leading dimensions and batch strides, exactly as the GPU sees them.
    ``alpha`` and ``beta`` should be the float32 values passed to the GPU.
    """
    lib = _load()
    A, at = _typed(A)
    B, bt = _typed(B)
    if C0 is not None:
        C0, ct = _typed(C0)
    else:
        ct = F64
    if ldc is None:
        ldc = N
    nthreads = nthreads or default_threads()
    out = np.empty((batch, M, N), dtype=np.float64)
    rc = lib.oracle_gemm(batch, M, N, K, float(alpha), _ptr(A), at, lda, strideA,
                         _ptr(B), bt, ldb, strideB, op_b, float(beta), _ptr(C0), ct, ldc,
                         strideC, _ptr(out), N, M * N, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm failed ({rc})")
    if not absden:
        return out
    den = np.empty((batch, M, N), dtype=np.float64)
    rc = lib.oracle_gemm_absden(batch, M, N, K, float(alpha), _ptr(A), at, lda, strideA,
                                _ptr(B), bt, ldb, strideB, op_b, float(beta), _ptr(C0), ct,
                                ldc, strideC, _ptr(den), N, M * N, nthreads)
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_absden failed ({rc})")
    return out, den


def gemm_entries(M, N, K, alpha, A, lda, B, ldb, beta, C0, ldc, rows, cols, *, op_b=0,
                 bidx=None, strideA=0, strideB=0, strideC=0):
    """Selected outputs (values, error scales) computed one dot product each."""
    lib = _load()
    A, at = _typed(A)
    B, bt = _typed(B)
    if C0 is not None:
        C0, ct = _typed(C0)
    else:
        ct = F64
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    if bidx is not None:
        bidx = np.ascontiguousarray(bidx, dtype=np.int64)
    out = np.empty(n, dtype=np.float64)
    den = np.empty(n, dtype=np.float64)
    rc = lib.oracle_gemm_entries(M, N, K, float(alpha), _ptr(A), at, lda, strideA,
                                 _ptr(B), bt, ldb, strideB, op_b, float(beta), _ptr(C0), ct,
                                 ldc if ldc is not None else N, strideC, n, _ptr(bidx),
                                 _ptr(rows), _ptr(cols), _ptr(out), _ptr(den))
    if rc != 0:
        raise RuntimeError(f"oracle_gemm_entries failed ({rc})")
    return out, den


def round_bf16(x) -> np.ndarray:
    """Round-to-nearest-even of float64 values to bfloat16 bit patterns (uint16)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.oracle_round_bf16(_ptr(x), _ptr(out), x.size)
    return out


def bf16_to_f64(bits) -> np.ndarray:
    """Exact widening of bfloat16 bit patterns to float64."""
    lib = _load()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    lib.oracle_bf16_to_double(_ptr(bits), _ptr(out), bits.size)
    return out


def ulp_bf16(x) -> np.ndarray:
    """Spacing of bfloat16 values at |x|."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    lib.oracle_ulp_bf16_array(_ptr(x), _ptr(out), x.size)
    return out


def flops(batch, M, N, K) -> float:
    return _load().oracle_gemm_flops(batch, M, N, K)


# ---------------------------------------------------------------------------
# Acceptance bounds (the tolerance stated for this path):
#   FP32 output: |C - C_ref| <= 1e-5 * D
#   BF16 output: |C - C_ref| <= 2e-4 * D + ulp_bf16(|C_ref|)
# with D = sum_k |alpha a b| + |beta c0| (the error scale from gemm(absden=True)).
# Where D == 0 the result must equal C_ref exactly.
# ---------------------------------------------------------------------------
FP32_REL = 1e-5
BF16_REL = 2e-4


def check_f32(C, ref, den):
    """(ok, worst normalised error) for FP32 output."""
    C = np.asarray(C, dtype=np.float64)
    err = np.abs(C - ref)
    bound = FP32_REL * den
    ok = bool(np.all((err <= bound) | ((den == 0) & (err == 0))) and np.all(np.isfinite(C)))
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(den > 0, err / np.where(den > 0, den, 1.0), np.where(err == 0, 0.0, np.inf))
    return ok, float(ratio.max()) if ratio.size else 0.0


def check_bf16(C_bits, ref, den):
    """(ok, worst error / bound) for BF16 output given as uint16 bit patterns."""
    C = bf16_to_f64(C_bits)
    err = np.abs(C - ref)
    bound = BF16_REL * den + ulp_bf16(np.abs(ref))
    ok = bool(np.all(err <= bound) and np.all(np.isfinite(C)))
    ratio = err / bound
    return ok, float(ratio.max()) if ratio.size else 0.0


# ---------------------------------------------------------------------------
# FFN gate/up activation chain ("Operator & Runtime", section 5.3.1: G = X W_g,
# U = X W_u, Z = SiLU(G) (.) U; section 5.4.3: the FP32 accumulation is rounded
# to BF16 before the activation, as the unfused program stores G and U as BF16).
# Steps in the pages' order: the two GEMMs (the oracle's own FP64 GEMM above),
# round each to BF16, SiLU(x) = x / (1 + e^-x) and the product in FP64.  The
# result is returned before Z's own rounding to BF16.
# ---------------------------------------------------------------------------
SILU_SLOPE_MAX = 1.0999  # >= max |d/dx SiLU(x)| = 1.09984 (at x ~ 2.40), for the error bound


def silu(x):
    """SiLU(x) = x / (1 + e^-x) in float64 (the limit 0 for x -> -inf)."""
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore"):
        return x / (1.0 + np.exp(-x))


def gate_up_silu(M, N, K, X, ldx, Wg, ldwg, Wu, ldwu, nthreads=None):
    """(z, gb, ub, Dg, Du) for Z = SiLU(bf16(X Wg)) * bf16(X Wu): z before Z's rounding, the
    BF16-rounded G and U as float64, and the error scales sum_k |x w| of G and U."""
    G, Dg = gemm(M, N, K, 1.0, X, ldx, Wg, ldwg, absden=True, nthreads=nthreads)
    U, Du = gemm(M, N, K, 1.0, X, ldx, Wu, ldwu, absden=True, nthreads=nthreads)
    gb = bf16_to_f64(round_bf16(G[0]))
    ub = bf16_to_f64(round_bf16(U[0]))
    return silu(gb) * ub, gb, ub, Dg[0], Du[0]


def check_gate_up(Z_bits, z, gb, ub, Dg, Du):
    """(ok, worst error / bound, fraction bit-equal to bf16(z)) for the GPU's BF16 Z.

    Bound: the GPU's bf16(G) lies within dg = BF16_REL*Dg + ulp_bf16(|G|) of G (the BF16
    GEMM bound) and the oracle's within half an ulp, so the two differ by at most
    Dg' = dg + ulp/2 (likewise U).  SiLU is SILU_SLOPE_MAX-Lipschitz, so
    |z_gpu - z| <= L*Dg'*(|ub| + Du') + |SiLU(gb)|*Du', plus the GPU's FP32 evaluation
    (a few float32 ulps, 1e-6 relative) and Z's rounding (one BF16 ulp)."""
    dgp = BF16_REL * Dg + 1.5 * ulp_bf16(np.abs(gb))
    dup = BF16_REL * Du + 1.5 * ulp_bf16(np.abs(ub))
    bound = (SILU_SLOPE_MAX * dgp * (np.abs(ub) + dup) + np.abs(silu(gb)) * dup +
             1e-6 * np.abs(z) + ulp_bf16(np.abs(z)))
    Zv = bf16_to_f64(Z_bits)
    err = np.abs(Zv - z)
    ok = bool(np.all(err <= bound) and np.all(np.isfinite(Zv)))
    same = float(np.mean(Z_bits == round_bf16(z))) if z.size else 1.0
    return ok, float((err / bound).max()) if z.size else 0.0, same


# ---------------------------------------------------------------------------
# Attention ("Operator & Runtime", section 5.3.3): S = Q K^T / sqrt(d), P = softmax(S)
# row by row, O = P V.  The fused method (tiling + online softmax) reaches this same
# result up to rounding, so the oracle is the definition written out in float64, with
# numpy's float64 matmul as the product step and the row maximum subtracted before the
# exponential (which leaves softmax unchanged).  Causal: key j is visible to query i
# iff j <= i (the pages' causal experiment; queries and keys of one sequence).
# online_softmax is the pages' block recurrence for one query row, kept beside it.
# ---------------------------------------------------------------------------
def attention_f64(Q, K, V, scale, causal=False, rows=None):
    """One head in float64: Q [Lq, d], K [Lkv, d], V [Lkv, dv] (any float arrays).

    Returns (O, PVabs, Ds) for the query rows `rows` (all by default):
      O     = softmax(scale * Q K^T) V                   [r, dv]
      PVabs = P |V|, the error scale of O                [r, dv]
      Ds    = max_j scale * sum_d |q_id k_jd| over visible keys, the error scale of S   [r]
    """
    Q = np.asarray(Q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    qi = np.arange(Q.shape[0]) if rows is None else np.asarray(rows, dtype=np.int64)
    S = float(scale) * (Q[qi] @ K.T)
    Sabs = abs(float(scale)) * (np.abs(Q[qi]) @ np.abs(K).T)
    if causal:
        hidden = np.arange(K.shape[0])[None, :] > qi[:, None]
        S[hidden] = -np.inf
        Sabs[hidden] = 0.0
    m = S.max(axis=1, keepdims=True)
    E = np.exp(S - m)
    P = E / E.sum(axis=1, keepdims=True)
    return P @ V, P @ np.abs(V), Sabs.max(axis=1)


def online_softmax(scores, values, block):
    """The pages' recurrence for one query row, `block` keys at a time:
    m' = max(m, max s), r = exp(m - m'), p_j = exp(s_j - m'), l' = r l + sum p_j,
    u' = r u + sum p_j v_j; the output is u / l.  Returns (u / l, [(m, l, u) after each
    block])."""
    s = np.asarray(scores, dtype=np.float64)
    v = np.asarray(values, dtype=np.float64)
    m, l = -np.inf, 0.0
    u = np.zeros(v.shape[1:], dtype=np.float64)
    states = []
    for b0 in range(0, s.shape[0], block):
        sb, vb = s[b0:b0 + block], v[b0:b0 + block]
        m_new = max(m, float(sb.max()))
        r = np.exp(m - m_new)
        pj = np.exp(sb - m_new)
        l = r * l + pj.sum()
        u = r * u + np.tensordot(pj, vb, axes=(0, 0))
        m = m_new
        states.append((m, l, u.copy()))
    return u / l, states


def _bf16_view(bits, batch, L, ld, stride, d):
    """[batch, L, d] float64 view of a strided BF16 array (elements b*stride + i*ld + c)."""
    x = bf16_to_f64(np.asarray(bits).reshape(-1))
    out = np.empty((batch, L, d), dtype=np.float64)
    for b in range(batch):
        base = b * stride
        out[b] = x[base: base + (L - 1) * ld + d].reshape(-1)[
            (np.arange(L)[:, None] * ld + np.arange(d)[None, :])]
    return out


def attention(batch, Lq, Lkv, d, scale, causal, Q, ldq, sQ, K, ldk, sK, V, ldv, sV,
              rows=None):
    """attention_f64 over a strided batch of BF16 (uint16 bit pattern) heads.  `rows`
    (optional) lists the query rows to compute in every batch.  Returns (O, PVabs, Ds)
    stacked over the batch."""
    q = _bf16_view(Q, batch, Lq, ldq, sQ, d)
    k = _bf16_view(K, batch, Lkv, ldk, sK, d)
    v = _bf16_view(V, batch, Lkv, ldv, sV, d)
    res = [attention_f64(q[b], k[b], v[b], scale, causal, rows) for b in range(batch)]
    return tuple(np.stack([r[i] for r in res]) for i in range(3))


# Acceptance bound for BF16 attention output (derived; the pages state none):
#   |O - O_ref| <= (2^-9 + BF16_REL + 1e-5 + 2 * FP32_REL * Ds) * (P|V|) + ulp_bf16(|O_ref|)
# 2^-9: P rounded to BF16 before the P V product (relative half-ulp per weight, the
# normaliser summed from the unrounded weights); BF16_REL: FP32 accumulation of P V and
# of the normaliser over the keys (the figure of the BF16 GEMM bound); 1e-5: the FP32
# exponential and its argument; 2 * FP32_REL * Ds: an error e in the scores moves every
# normalised weight by at most a factor e^(2e); one BF16 ulp for the rounding of O.
ATTN_P_REL = 2.0 ** -9


def check_attention(O_bits, O_ref, PVabs, Ds):
    """(ok, worst error / bound) for BF16 attention output (uint16 bit patterns)."""
    O = bf16_to_f64(O_bits)
    rel = ATTN_P_REL + BF16_REL + 1e-5 + 2.0 * FP32_REL * np.asarray(Ds)[..., None]
    bound = rel * PVabs + ulp_bf16(np.abs(O_ref))
    err = np.abs(O - O_ref)
    ok = bool(np.all(err <= bound) and np.all(np.isfinite(O)))
    return ok, float((err / bound).max()) if err.size else 0.0


# ---------------------------------------------------------------------------
# FP8 E4M3 with per-row scales ("Operator & Runtime", section 5.4.3, Example 5-7, and
# section 5.4.4, Example 5-8).  E4M3FN: 1 sign, 4 exponent (bias 7) and 3 mantissa bits,
# no infinities, largest finite value 448.  A row is quantised with the scale of its
# absolute maximum over the whole row: x -> round(x * 448 / amax), dequantised as
# q * amax / 448.  The quantised code is an integer decided by floating point, so the
# oracle takes that decision in the kernel's precision: amax, 448 / amax and the product
# x * (448 / amax) in IEEE float32, then round-to-nearest-even of that float32 value to
# E4M3, values beyond 448 saturating to +-448.  The GEMM on the codes is the definition
# C[i, j] = s_a[i] * s_b[j] * sum_k qa[i, k] qb[j, k] in float64 (B stored [N, K], so the
# per-output-column scale of B is the scale of its row).
# ---------------------------------------------------------------------------
E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of every E4M3FN code 0..255 (NaN for the two NaN codes), from the format."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e, m = (code >> 3) & 0xF, code & 0x7
        if e == 0xF and m == 0x7:
            vals[code] = np.nan
        elif e == 0:
            vals[code] = sign * (m / 8.0) * 2.0 ** -6          # subnormal
        else:
            vals[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return vals


_E4M3 = None


def e4m3_to_f64(codes) -> np.ndarray:
    global _E4M3
    if _E4M3 is None:
        _E4M3 = e4m3_values()
    return _E4M3[np.asarray(codes, dtype=np.uint8)]


def round_e4m3(y) -> np.ndarray:
    """Round-to-nearest-even of (float32-valued) y to E4M3FN codes, saturating to +-448;
    NaN gives the NaN code 0x7F."""
    y = np.asarray(y, dtype=np.float64)
    pos = e4m3_values()[:127]                 # codes 0..126: 0 .. 448, increasing
    a = np.minimum(np.abs(y), E4M3_MAX)
    hi = np.clip(np.searchsorted(pos, a, side="left"), 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    d_lo, d_hi = a - pos[lo], pos[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))   # ties: even mantissa
    code = np.where(pick_hi, hi, lo).astype(np.uint8)
    code = np.where(a == pos[hi], hi, code).astype(np.uint8)     # exact values
    code = np.where((y < 0) & (code != 0), code | 0x80, code).astype(np.uint8)
    code = np.where(np.signbit(y) & (code == 0), np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(y), np.uint8(0x7F), code).astype(np.uint8)


def quantize_rows_e4m3(rows, cols, X, ldx):
    """(codes [rows, cols] uint8, scales [rows] float32) of BF16 (bits) or float32 X.
    Per row: amax = max |x|, multiplier 448 / amax and scale amax / 448 in float32; an
    all-zero row has codes 0 and scale 0."""
    X = np.asarray(X).reshape(-1)
    x = (bf16_to_f64(X) if X.dtype == np.uint16 else X.astype(np.float64)).astype(np.float32)
    idx = np.arange(rows)[:, None] * ldx + np.arange(cols)[None, :]
    xr = x[idx]
    amax = np.abs(xr).max(axis=1).astype(np.float32) if cols > 0 else np.zeros(rows, np.float32)
    with np.errstate(divide="ignore"):
        mult = np.where(amax > 0, np.float32(E4M3_MAX) / amax, np.float32(0)).astype(np.float32)
    y = (xr * mult[:, None]).astype(np.float32)                   # float32 product (RNE)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return round_e4m3(y), scale


def quantize_rows_e4m3_f64(rows, cols, X, ldx):
    """The same per-row quantisation with every decision in float64: amax, y = x * 448 / amax
    and the scale amax / 448 in double, then round-to-nearest-even of y to E4M3.  Kept beside
    the float32 form above to show how many codes depend on the precision of the decision."""
    X = np.asarray(X).reshape(-1)
    x = bf16_to_f64(X) if X.dtype == np.uint16 else X.astype(np.float64)
    idx = np.arange(rows)[:, None] * ldx + np.arange(cols)[None, :]
    xr = x[idx]
    amax = np.abs(xr).max(axis=1) if cols > 0 else np.zeros(rows)
    safe = np.where(amax > 0, amax, 1.0)
    y = np.where(amax[:, None] > 0, xr * E4M3_MAX / safe[:, None], 0.0)
    return round_e4m3(y), amax / E4M3_MAX


def gemm_fp8(M, N, K, QA, lda, sa, QB, ldb, sb, nthreads=None):
    """(C, D): C[i, j] = sa[i] * sb[j] * sum_k qa[i, k] qb[j, k] and its error scale
    D = |sa[i] sb[j]| sum_k |qa qb|, float64, for E4M3 codes QA [M, lda] and QB [N, ldb]."""
    a = e4m3_to_f64(np.asarray(QA).reshape(-1))
    b = e4m3_to_f64(np.asarray(QB).reshape(-1))
    P, D = gemm(M, N, K, 1.0, a, lda, b, ldb, op_b=1, absden=True, nthreads=nthreads)
    s = np.asarray(sa, np.float64)[:, None] * np.asarray(sb, np.float64)[None, :]
    return P[0] * s, D[0] * np.abs(s)


# ---------------------------------------------------------------------------
# A chain of decode GEMMs ("Operator & Runtime", sections 5.5.2 and 5.5.4): y_0 = X,
# y_{l+1} = bf16(y_l W_l) -- each layer the BF16 GEMM above, its output rounded once and
# fed to the next.  The acceptance bound of layer l adds to the BF16 GEMM bound the effect
# of the input's difference: the GPU's input (its rounded y_l) and the oracle's (its own
# rounded y_l) differ by at most b_{l-1} + ulp/2 <= 2 b_{l-1} elementwise, which moves
# each output by at most (2 b_{l-1}) |W_l|.
# ---------------------------------------------------------------------------
def decode_chain(M, dims, X, ldx, Ws, ldws, nthreads=None):
    """[(y_l float64 before rounding, y_l BF16 bits, bound_l)] for layers l = 0 .. L-1."""
    out = []
    x, ld, b_prev = X, ldx, None
    for l, (W, ldw) in enumerate(zip(Ws, ldws)):
        K, N = dims[l], dims[l + 1]
        y, D = gemm(M, N, K, 1.0, x, ld, W, ldw, absden=True, nthreads=nthreads)
        y, D = y[0], D[0]
        bound = BF16_REL * D + ulp_bf16(np.abs(y))
        if b_prev is not None:
            w = np.abs(bf16_to_f64(np.asarray(W).reshape(-1)[: (K - 1) * ldw + N]))
            wk = w[(np.arange(K)[:, None] * ldw + np.arange(N)[None, :])]
            bound = bound + (2.0 * b_prev) @ wk
        bits = round_bf16(y)
        out.append((y, bits, bound))
        x, ld, b_prev = bits, N, bound
    return out


def check_chain_layer(Y_bits, y, bound):
    """(ok, worst error / bound) of one layer's BF16 output."""
    Yv = bf16_to_f64(Y_bits)
    err = np.abs(Yv - y)
    ok = bool(np.all(err <= bound) and np.all(np.isfinite(Yv)))
    return ok, float((err / bound).max()) if err.size else 0.0
