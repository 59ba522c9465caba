"""Pins for the CPU oracle: values fixed by the pages or by mathematics.

None of these re-type the oracle's own loop.  Each case is chosen so that a
plausible slip in the oracle (a dropped alpha/beta term, a sign, a swapped
index or a transposed operand, a wrong rounding rule) fails at least one test:

* hand products (tests/golden/hand_*.txt) with non-symmetric operands and
  alpha/beta not in {0, 1}: catch transposition, A.B vs B.A, beta dropped;
* identity / permutation matrices: exact data movement, index mapping;
* the rank-1 closed form (u v^T)(w z^T) = (v.w) u z^T;
* numpy's float64 matmul on integer-valued data (exact in double);
* IEEE round-to-nearest-even cases for bfloat16 and its ulp;
* the FLOP count printed by "Operator & Runtime" section 5.2.1.
"""
import os

import numpy as np
import pytest

import oracle
from dense_gemm_sm_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def read_golden(name):
    vals = {}
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            try:
                float(parts[0])
                rows.append([float(p) for p in parts])
            except ValueError:
                key = parts[0]
                nums = [float(p) for p in parts[1:]]
                vals[key] = nums if len(nums) > 1 else nums[0]
    return vals, rows


def test_hand_2x2():
    g, _ = read_golden("hand_2x2.txt")
    A = np.array(g["A"], dtype=np.float32)
    B = np.array(g["B"], dtype=np.float32)
    C = oracle.gemm(2, 2, 2, g["alpha"], A, 2, B, 2)[0]
    assert C.ravel().tolist() == g["C"]


@pytest.mark.parametrize("op_b", [0, 1])
def test_hand_3x3_alpha_beta(op_b):
    g, _ = read_golden("hand_3x3.txt")
    A = np.array(g["A"], dtype=np.float32)
    B = np.array(g["B"], dtype=np.float32).reshape(3, 3)
    Bstore = B if op_b == 0 else np.ascontiguousarray(B.T)  # op(B)[k][j] = B[j][k]
    C0 = np.array(g["C0"], dtype=np.float32)
    C = oracle.gemm(3, 3, 3, g["alpha"], A, 3, Bstore.ravel(), 3, g["beta"], C0, 3, op_b=op_b)[0]
    assert C.ravel().tolist() == g["C"]
    AB = oracle.gemm(3, 3, 3, 1.0, A, 3, Bstore.ravel(), 3, op_b=op_b)[0]
    assert AB.ravel().tolist() == g["AB"]


def test_identity_and_zero():
    A = inputs.uniform_f32(1, (37, 23))
    I = np.eye(23, dtype=np.float32)
    C = oracle.gemm(37, 23, 23, 1.0, A, 23, I, 23)[0]
    assert np.array_equal(C, A.astype(np.float64))
    I2 = np.eye(37, dtype=np.float32)
    C2 = oracle.gemm(37, 23, 37, 1.0, I2, 37, A, 23)[0]
    assert np.array_equal(C2, A.astype(np.float64))
    Z = np.zeros((23, 11), dtype=np.float32)
    assert np.all(oracle.gemm(37, 11, 23, 1.0, A, 23, Z, 11)[0] == 0)


def test_permutations():
    r = inputs.rng(7)
    A = inputs.uniform_f32(2, (9, 13))
    p_rows = r.permutation(9)
    P = np.zeros((9, 9), dtype=np.float32)
    P[np.arange(9), p_rows] = 1.0          # (P A)[i] = A[p_rows[i]]
    C = oracle.gemm(9, 13, 9, 1.0, P, 9, A, 13)[0]
    assert np.array_equal(C, A[p_rows].astype(np.float64))
    p_cols = r.permutation(13)
    Q = np.zeros((13, 13), dtype=np.float32)
    Q[p_cols, np.arange(13)] = 1.0         # (A Q)[:, j] = A[:, p_cols[j]]
    C = oracle.gemm(9, 13, 13, 1.0, A, 13, Q, 13)[0]
    assert np.array_equal(C, A[:, p_cols].astype(np.float64))


def test_rank1_closed_form():
    M, K, N = 17, 29, 11
    u = inputs.uniform_f32(3, M).astype(np.float64)
    v = inputs.uniform_f32(4, K).astype(np.float64)
    w = inputs.uniform_f32(5, K).astype(np.float64)
    z = inputs.uniform_f32(6, N).astype(np.float64)
    A = np.outer(u, v)
    B = np.outer(w, z)
    C = oracle.gemm(M, N, K, 1.0, A, K, B, N)[0]
    expect = float(v @ w) * np.outer(u, z)
    assert np.max(np.abs(C - expect)) <= 1e-12 * np.max(np.abs(expect))


def test_alpha_beta_special_cases():
    M, N, K = 6, 5, 4
    A = inputs.uniform_f32(8, (M, K))
    B = inputs.uniform_f32(9, (K, N))
    C0 = inputs.uniform_f32(10, (M, N))
    # alpha = 0: C = beta * C0 exactly
    C = oracle.gemm(M, N, K, 0.0, A, K, B, N, 0.75, C0, N)[0]
    assert np.array_equal(C, 0.75 * C0.astype(np.float64))
    # beta = 0: C0 is never read (NaN does not propagate)
    nan_c0 = np.full((M, N), np.nan, dtype=np.float32)
    C = oracle.gemm(M, N, K, 1.0, A, K, B, N, 0.0, nan_c0, N)[0]
    assert np.all(np.isfinite(C))
    # B = 0, alpha = beta = 1: C = C0
    C = oracle.gemm(M, N, K, 1.0, A, K, np.zeros((K, N), np.float32), N, 1.0, C0, N)[0]
    assert np.array_equal(C, C0.astype(np.float64))
    # K = 0: C = beta * C0
    C = oracle.gemm(M, N, 0, 1.0, A, K, B, N, -2.0, C0, N)[0]
    assert np.array_equal(C, -2.0 * C0.astype(np.float64))


@pytest.mark.parametrize("op_b", [0, 1])
def test_integer_data_matches_numpy_exactly(op_b):
    M, N, K = 37, 53, 29
    A = inputs.integer_f32(11, (M, K))
    B = inputs.integer_f32(12, (K, N))
    Bstore = B if op_b == 0 else np.ascontiguousarray(B.T)
    C = oracle.gemm(M, N, K, 1.0, A, K, Bstore, N if op_b == 0 else K, op_b=op_b)[0]
    assert np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64))


def test_leading_dimension_padding_not_read():
    M, N, K = 7, 9, 5
    A = inputs.integer_f32(13, (M, K))
    B = inputs.integer_f32(14, (K, N))
    C0 = inputs.integer_f32(15, (M, N))
    Ap = inputs.pad_rows(A, 8)
    Bp = inputs.pad_rows(B, 12)
    C0p = inputs.pad_rows(C0, 10)
    C = oracle.gemm(M, N, K, 1.0, Ap, 8, Bp, 12, 1.0, C0p, 10)[0]
    assert np.array_equal(C, A.astype(np.float64) @ B.astype(np.float64) + C0)


def test_batched_strides():
    batch, M, N, K = 3, 5, 4, 6
    sA, sB, sC = M * K + 3, K * N + 1, M * N + 2
    A = inputs.integer_f32(16, (batch * sA,))
    B = inputs.integer_f32(17, (batch * sB,))
    C0 = inputs.integer_f32(18, (batch * sC,))
    C = oracle.gemm(M, N, K, 2.0, A, K, B, N, -1.0, C0, N, batch=batch, strideA=sA, strideB=sB,
                    strideC=sC)
    for b in range(batch):
        Ab = A[b * sA:b * sA + M * K].reshape(M, K).astype(np.float64)
        Bb = B[b * sB:b * sB + K * N].reshape(K, N).astype(np.float64)
        C0b = C0[b * sC:b * sC + M * N].reshape(M, N).astype(np.float64)
        assert np.array_equal(C[b], 2.0 * (Ab @ Bb) - C0b)


def test_bf16_inputs_widen_exactly():
    vals = np.array([1.0, -1.5, 0.0078125, 3.0e38, -2.0 ** -130], dtype=np.float32)
    bits = inputs.f32_to_bf16_bits(vals[:4])
    assert bits.tolist() == [0x3F80, 0xBFC0, 0x3C00, 0x7F62]
    w = oracle.bf16_to_f64(bits)
    assert w[:3].tolist() == [1.0, -1.5, 0.0078125]
    # bf16 GEMM == GEMM of the widened values
    X = inputs.f32_to_bf16_bits(inputs.normal_f32(19, (8, 16)))
    W = inputs.f32_to_bf16_bits(inputs.normal_f32(20, (16, 12)))
    C1 = oracle.gemm(8, 12, 16, 1.0, X, 16, W, 12)[0]
    C2 = oracle.gemm(8, 12, 16, 1.0, oracle.bf16_to_f64(X), 16, oracle.bf16_to_f64(W), 12)[0]
    assert np.array_equal(C1, C2)


def test_round_bf16_ieee_cases():
    one = 1.0
    cases = [
        (1.0, 0x3F80),
        (-2.0, 0xC000),
        (one + 2.0 ** -8, 0x3F80),             # exact tie -> even (down)
        (one + 3 * 2.0 ** -8, 0x3F82),         # exact tie -> even (up)
        (one + 2.0 ** -8 + 2.0 ** -30, 0x3F81),  # just above the tie -> up
        (one + 2.0 ** -9, 0x3F80),             # below half -> down
        (0.0, 0x0000),
        (-0.0, 0x8000),
        (2.0 ** -133, 0x0001),                 # smallest subnormal
        (2.0 ** -134, 0x0000),                 # tie between 0 and 2^-133 -> even (0)
        (3 * 2.0 ** -134, 0x0002),             # tie between 1 and 2 quanta -> 2
        ((2 - 2.0 ** -7) * 2.0 ** 127, 0x7F7F),  # largest finite
        ((2 - 2.0 ** -8) * 2.0 ** 127, 0x7F80),  # tie at the top rounds to infinity
        (float("inf"), 0x7F80),
        (-float("inf"), 0xFF80),
        (3.140625, 0x4049),                    # exactly representable
        (0.1, 0x3DCD),                         # 0.1 = 0x3DCCCCCD (f32) -> 0x3DCD
    ]
    xs = np.array([c[0] for c in cases], dtype=np.float64)
    got = oracle.round_bf16(xs)
    assert got.tolist() == [c[1] for c in cases]
    nan = oracle.round_bf16(np.array([np.nan]))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_round_bf16_agrees_with_float32_path_on_f32_values():
    # For values that are already float32, rounding the double directly and the
    # integer-rounding of the float32 bits (the input converter) must agree.
    x = inputs.normal_f32(21, 20000) * np.float32(1000)
    assert np.array_equal(oracle.round_bf16(x.astype(np.float64)), inputs.f32_to_bf16_bits(x))


def test_ulp_bf16():
    got = oracle.ulp_bf16(np.array([1.0, 1.99, 2.0, 0.75, -3.0, 0.0, 2.0 ** -140]))
    assert got.tolist() == [2.0 ** -7, 2.0 ** -7, 2.0 ** -6, 2.0 ** -8, 2.0 ** -6, 2.0 ** -133,
                            2.0 ** -133]


def test_entries_and_error_scale():
    g, _ = read_golden("hand_3x3.txt")
    A = np.array(g["A"], dtype=np.float32)
    B = np.array(g["B"], dtype=np.float32)
    C0 = np.array(g["C0"], dtype=np.float32)
    rows = np.array([0, 1, 2, 2])
    cols = np.array([0, 1, 2, 0])
    out, den = oracle.gemm_entries(3, 3, 3, g["alpha"], A, 3, B, 3, g["beta"], C0, 3, rows, cols)
    C = np.array(g["C"]).reshape(3, 3)
    assert out.tolist() == [C[r, c] for r, c in zip(rows, cols)]
    # error scale by hand: D_00 = 2*(|1*2|+|2*1|+|3*0|) + |-1*1| = 9
    assert den[0] == 9.0
    full, D = oracle.gemm(3, 3, 3, g["alpha"], A, 3, B, 3, g["beta"], C0, 3, absden=True)
    assert D[0, 0, 0] == 9.0
    assert den.tolist() == [D[0, r, c] for r, c in zip(rows, cols)]


def test_flop_count_of_ffn_example():
    g, _ = read_golden("ffn_counts.txt")
    f = oracle.flops(1, int(g["M"]), int(g["N"]), int(g["K"]))
    assert f == 103_079_215_104
    assert round(f / 1e9) == g["F_gemm_GFLOP_approx"]
    e = g["bytes_per_element"]
    mib = 2 ** 20
    M, K, N = g["M"], g["K"], g["N"]
    assert (e * M * K / mib, e * K * N / mib, e * M * N / mib) == (g["X_MiB"], g["W_MiB"], g["C_MiB"])
    assert e * (M * K + K * N + M * N) / mib == g["V_once_MiB"]


def test_fp32_order_example_from_pages():
    g, _ = read_golden("fp32_order.txt")
    one, t = np.float32(1.0), np.float32(2.0 ** -24)
    assert float((one + t) + t) == g["left_to_right"]
    assert float(one + (t + t)) == g["small_first"]


def test_acceptance_checkers():
    ref = np.array([1.0, -2.0, 0.0])
    den = np.array([10.0, 10.0, 0.0])
    ok, worst = oracle.check_f32(np.array([1.0 + 0.5e-4, -2.0 - 0.9e-4, 0.0]), ref, den)
    assert ok and worst <= 1e-5
    ok, _ = oracle.check_f32(np.array([1.0 + 1.5e-4, -2.0, 0.0]), ref, den)
    assert not ok
    ok, _ = oracle.check_f32(np.array([1.0, -2.0, 1e-30]), ref, den)
    assert not ok  # D == 0 demands exact equality
    bits = oracle.round_bf16(ref)
    ok, worst = oracle.check_bf16(bits, ref, den)
    assert ok and worst == 0.0


# BF16 output bound |C - C_ref| <= 2e-4 * D + ulp_bf16(|C_ref|): GPU values are BF16 numbers,
# so each case fixes a BF16 value c and puts the reference just inside (0.99 x the bound) or
# just outside (1.01 x) of it, in three binades whose ulps differ (2^-7 at 1.5, 2 at 384 and
# 2^-14 at 3 * 2^-8) and with D chosen so that both terms matter (2e-4 * D is 20% to 50% of the
# bound).  The references stay in c's binade, so the ulp term is that binade's spacing.  A
# relative figure typed as 2e-3, a doubled or dropped ulp term, or an error measured from the
# wrong operand moves at least one case to the other side.
BF16_BOUND_CASES = [  # (c, D, ulp of the binade)
    (1.5, 10.0, 2.0 ** -7),
    (384.0, 1000.0, 2.0),
    (3.0 * 2.0 ** -8, 0.1, 2.0 ** -14),
]


@pytest.mark.parametrize("c,D,ulp", BF16_BOUND_CASES)
@pytest.mark.parametrize("side", [-1.0, 1.0])
def test_check_bf16_accepts_inside_and_rejects_outside_the_bound(c, D, ulp, side):
    bound = 2e-4 * D + ulp
    bits = oracle.round_bf16(np.array([c]))
    assert oracle.bf16_to_f64(bits)[0] == c                      # c is a BF16 number
    for factor, expect in ((0.99, True), (1.01, False)):
        ref = np.array([c - side * factor * bound])
        assert oracle.ulp_bf16(np.abs(ref))[0] == ulp            # same binade as c
        ok, worst = oracle.check_bf16(bits, ref, np.array([D]))
        assert ok == expect, (c, D, factor, side)
        assert abs(worst - factor) < 1e-9


def test_check_bf16_needs_every_element_and_finite_values():
    c = np.array([1.5, 384.0])
    bits = oracle.round_bf16(c)
    den = np.array([10.0, 1000.0])
    inside = c - 0.99 * (2e-4 * den + np.array([2.0 ** -7, 2.0]))
    ok, _ = oracle.check_bf16(bits, inside, den)
    assert ok
    one_out = inside.copy()
    one_out[1] = 384.0 - 1.01 * (2e-4 * 1000.0 + 2.0)            # only the second one fails
    ok, worst = oracle.check_bf16(bits, one_out, den)
    assert not ok and abs(worst - 1.01) < 1e-9
    nan_bits = bits.copy()
    nan_bits[0] = 0x7FC0                                          # a NaN output never passes
    assert not oracle.check_bf16(nan_bits, c, den)[0]
    inf_bits = bits.copy()
    inf_bits[1] = 0x7F80                                          # nor does an infinity
    assert not oracle.check_bf16(inf_bits, c, den)[0]


# --------------------------------------------------------------------------- FFN gate/up
def test_silu_values_printed_by_the_pages():
    g, _ = read_golden("silu_chain.txt")
    assert oracle.silu(0.0) == g["silu_0"]
    assert round(float(oracle.silu(1.0) + oracle.silu(-1.0)), 4) == g["silu_1_plus_silu_m1"]


def test_silu_closed_forms():
    x = np.random.default_rng(5).normal(0, 6, 1000)
    # sigma(x) + sigma(-x) = 1  =>  SiLU(x) - SiLU(-x) = x
    assert np.allclose(oracle.silu(x) - oracle.silu(-x), x, rtol=1e-12, atol=1e-12)
    assert np.all(oracle.silu(np.array([-1000.0])) == 0.0)           # e^-x overflows: limit 0
    assert oracle.silu(np.array([1000.0]))[0] == 1000.0
    assert abs(oracle.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-15
    # sigma(ln 3) = 3/4 exactly, so SiLU(ln 3) = (3/4) ln 3
    assert abs(oracle.silu(np.log(3.0)) - 0.75 * np.log(3.0)) < 1e-15
    # The checker's Lipschitz constant: the steepest slope of SiLU (near x = 2.4) is just
    # below SILU_SLOPE_MAX, and nowhere steeper.
    t = np.linspace(-20, 20, 400001)
    slope = np.abs(np.diff(oracle.silu(t)) / np.diff(t))
    assert 1.0995 < slope.max() <= oracle.SILU_SLOPE_MAX


def _bits(a):
    from dense_gemm_sm_gb300 import inputs
    return inputs.f32_to_bf16_bits(np.asarray(a, np.float32))


def test_gate_up_rounds_g_before_the_activation():
    g, _ = read_golden("silu_chain.txt")
    X = _bits([[1.0, 1.0]])
    Wg = _bits([[1.0], [2.0 ** -9]])      # G = 1 + 2^-9, exact in float64, not in BF16
    Wu = _bits([[1.0], [0.0]])            # U = 1
    z, gb, ub, _, _ = oracle.gate_up_silu(1, 1, 2, X, 2, Wg, 1, Wu, 1)
    assert gb[0, 0] == 1.0 and ub[0, 0] == 1.0
    assert oracle.bf16_to_f64(oracle.round_bf16(z))[0, 0] == g["z_rounded_g"]
    unrounded = oracle.silu(1.0 + 2.0 ** -9)
    assert oracle.bf16_to_f64(oracle.round_bf16(np.array([unrounded])))[0] == g["z_unrounded_g"]


def test_gate_up_special_cases_and_numpy():
    rng = np.random.default_rng(6)
    M, N, K = 5, 7, 11
    X = _bits(rng.integers(-3, 4, (M, K)))
    Wg = _bits(rng.integers(-3, 4, (K, N)))
    Wu = _bits(rng.integers(-3, 4, (K, N)))
    zero = _bits(np.zeros((K, N)))
    z, _, _, _, _ = oracle.gate_up_silu(M, N, K, X, K, Wg, N, zero, N)
    assert np.all(z == 0.0)                                          # U = 0
    z, _, _, _, _ = oracle.gate_up_silu(M, N, K, X, K, zero, N, Wu, N)
    assert np.all(z == 0.0)                                          # G = 0, SiLU(0) = 0
    # Integer data: G and U are small integers, exact in BF16; check against numpy's
    # float64 matmul and the logistic written out.
    z, gb, ub, _, _ = oracle.gate_up_silu(M, N, K, X, K, Wg, N, Wu, N)
    x = oracle.bf16_to_f64(X).reshape(M, K)
    G = x @ oracle.bf16_to_f64(Wg).reshape(K, N)
    U = x @ oracle.bf16_to_f64(Wu).reshape(K, N)
    assert np.array_equal(gb, G) and np.array_equal(ub, U)
    assert np.allclose(z, G * (1.0 / (1.0 + np.exp(-G))) * U, rtol=1e-14, atol=0)


def test_gate_up_check_catches_a_missing_rounding():
    # The checker must reject a result computed without rounding G and U to BF16 first
    # (a plausible epilogue mistake): FFN-like data, where the rounding changes most Z.
    rng = np.random.default_rng(7)
    M, N, K = 16, 64, 512
    X = _bits(rng.normal(0, 1, (M, K)))
    Wg = _bits(rng.normal(0, 1 / 16, (K, N)))
    Wu = _bits(rng.normal(0, 1 / 16, (K, N)))
    z, gb, ub, Dg, Du = oracle.gate_up_silu(M, N, K, X, K, Wg, N, Wu, N)
    ok, _, same = oracle.check_gate_up(oracle.round_bf16(z), z, gb, ub, Dg, Du)
    assert ok and same == 1.0
    G = oracle.gemm(M, N, K, 1.0, X, K, Wg, N)[0]
    U = oracle.gemm(M, N, K, 1.0, X, K, Wu, N)[0]
    wrong = oracle.round_bf16(oracle.silu(G) * U)
    _, _, same_wrong = oracle.check_gate_up(wrong, z, gb, ub, Dg, Du)
    assert same_wrong < 0.95


# --------------------------------------------------------------------------- attention
def test_online_softmax_example_5_6():
    g, _ = read_golden("online_softmax.txt")
    out, states = oracle.online_softmax([0.0, np.log(2.0)], [[1.0], [3.0]], 1)
    (m1, l1, u1), (m2, l2, u2) = states
    assert (m1, l1, u1[0]) == (g["block1_m"], g["block1_l"], g["block1_u"])
    assert np.isclose(np.exp(m1 - m2), g["block2_r"], rtol=1e-15)
    assert np.isclose(l2, g["block2_l"], rtol=1e-15) and np.isclose(u2[0], g["block2_u"], rtol=1e-15)
    assert np.isclose(out[0], g["output"], rtol=1e-15)
    # The definition gives the same 7/3: one query with q . k_j equal to the scores.
    O, _, _ = oracle.attention_f64([[1.0]], [[0.0], [np.log(2.0)]], [[1.0], [3.0]], 1.0)
    assert np.isclose(O[0, 0], g["output"], rtol=1e-15)


def test_attention_uniform_scores_closed_forms():
    # Q = 0: every visible key has the same weight.  Non-causal: O = mean of V; causal:
    # row i is the mean of V[0..i] (catches a mask that drops or adds the diagonal).
    rng = np.random.default_rng(21)
    L, d = 37, 5
    V = rng.normal(0, 1, (L, d))
    O, _, _ = oracle.attention_f64(np.zeros((L, d)), rng.normal(0, 1, (L, d)), V, 0.3)
    assert np.allclose(O, V.mean(axis=0)[None, :], rtol=0, atol=1e-14)
    O, _, _ = oracle.attention_f64(np.zeros((L, d)), rng.normal(0, 1, (L, d)), V, 0.3, causal=True)
    prefix = np.cumsum(V, axis=0) / np.arange(1, L + 1)[:, None]
    assert np.allclose(O, prefix, rtol=0, atol=1e-14)
    assert np.array_equal(O[0], V[0])


def test_attention_dominant_key_and_invariants():
    rng = np.random.default_rng(22)
    Lq, Lkv, d = 6, 50, 8
    Q = rng.normal(0, 1, (Lq, d))
    K = rng.normal(0, 0.1, (Lkv, d))
    V = rng.normal(0, 1, (Lkv, d))
    # One key aligned with every query and far larger: its weight is 1 to within e^-60.
    K2 = K.copy()
    K2[17] = 1000.0 * Q.sum(axis=0) / np.linalg.norm(Q.sum(axis=0))
    Qpos = np.abs(Q) * np.sign(Q.sum(axis=0))   # every query has a positive dot with key 17
    O, _, _ = oracle.attention_f64(Qpos, K2, V, 1.0)
    assert np.allclose(O, V[17][None, :], atol=1e-12)
    # Permuting the keys with their values leaves O unchanged; constant V gives O = V.
    perm = rng.permutation(Lkv)
    O1, _, _ = oracle.attention_f64(Q, K, V, 0.7)
    O2, _, _ = oracle.attention_f64(Q, K[perm], V[perm], 0.7)
    assert np.allclose(O1, O2, rtol=1e-13, atol=1e-14)
    O3, _, _ = oracle.attention_f64(Q, K, np.full((Lkv, d), 2.5), 0.7)
    assert np.allclose(O3, 2.5, rtol=1e-14)
    # O is a convex combination of the rows of V.
    assert np.all(O1 <= V.max(axis=0) + 1e-12) and np.all(O1 >= V.min(axis=0) - 1e-12)


def test_attention_definition_matches_the_block_recurrence():
    # The pages' block recurrence (any block size) against the definition, per query row.
    rng = np.random.default_rng(23)
    Lq, Lkv, d = 4, 300, 16
    Q, K, V = rng.normal(0, 2, (Lq, d)), rng.normal(0, 2, (Lkv, d)), rng.normal(0, 1, (Lkv, d))
    scale = 1.0 / np.sqrt(d)
    O, _, _ = oracle.attention_f64(Q, K, V, scale)
    for blk in (1, 7, 128):
        for i in range(Lq):
            o, _ = oracle.online_softmax(scale * (K @ Q[i]), V, blk)
            assert np.allclose(o, O[i], rtol=1e-12, atol=1e-13)


def test_attention_strided_bf16_view():
    # The strided BF16 entry equals attention_f64 on the widened, de-strided heads.
    from dense_gemm_sm_gb300 import inputs
    rng = np.random.default_rng(24)
    batch, L, d, ld = 2, 9, 8, 16
    stride = L * ld + 8
    raw = [inputs.f32_to_bf16_bits(rng.normal(0, 1, batch * stride).astype(np.float32))
           for _ in range(3)]
    O, PV, Ds = oracle.attention(batch, L, L, d, 0.5, True, raw[0], ld, stride, raw[1], ld, stride,
                                 raw[2], ld, stride)
    for b in range(batch):
        heads = [oracle.bf16_to_f64(r[b * stride: b * stride + L * ld]).reshape(L, ld)[:, :d]
                 for r in raw]
        o, pv, ds = oracle.attention_f64(*heads, 0.5, causal=True)
        assert np.array_equal(O[b], o) and np.array_equal(PV[b], pv) and np.array_equal(Ds[b], ds)


def test_attention_check_catches_planted_mistakes():
    # Each plausible kernel mistake, planted here in oracle-side arithmetic, must fail the
    # acceptance check: scale 1/d instead of 1/sqrt(d), a causal mask that hides the
    # diagonal, and blocks combined without rescaling by r.
    from dense_gemm_sm_gb300 import inputs
    rng = np.random.default_rng(25)
    L, d = 256, 128
    bits = [inputs.f32_to_bf16_bits(rng.normal(0, 1, (L, d)).astype(np.float32)) for _ in range(3)]
    Q, K, V = (oracle.bf16_to_f64(b) for b in bits)
    scale = 1.0 / np.sqrt(d)
    O, PV, Ds = oracle.attention_f64(Q, K, V, scale, causal=True)
    ok, worst = oracle.check_attention(oracle.round_bf16(O), O, PV, Ds)
    assert ok and worst <= 0.51
    wrong_scale, _, _ = oracle.attention_f64(Q, K, V, 1.0 / d, causal=True)
    assert not oracle.check_attention(oracle.round_bf16(wrong_scale), O, PV, Ds)[0]
    strict = np.array([oracle.attention_f64(Q[i:i + 1], K[:i], V[:i], scale)[0][0]
                       if i > 0 else V[0] for i in range(L)])
    assert not oracle.check_attention(oracle.round_bf16(strict), O, PV, Ds)[0]
    no_rescale = np.empty_like(O)
    for i in range(L):
        s = scale * (K[:i + 1] @ Q[i])
        l, u = 0.0, np.zeros(d)
        for b0 in range(0, i + 1, 128):       # per block: own maximum, no r
            pj = np.exp(s[b0:b0 + 128] - s[b0:b0 + 128].max())
            l, u = l + pj.sum(), u + pj @ V[b0:b0 + pj.size]
        no_rescale[i] = u / l
    assert not oracle.check_attention(oracle.round_bf16(no_rescale), O, PV, Ds)[0]


# --------------------------------------------------------------------------- FP8 E4M3
def test_e4m3_format_values():
    g, _ = read_golden("fp8_e4m3.txt")
    v = oracle.e4m3_values()
    pos = v[:127]
    assert pos[126] == g["e4m3_max"] and np.all(np.diff(pos) > 0)         # 0 .. 448, increasing
    assert pos[1] == 2.0 ** -9 and pos[8] == 2.0 ** -6                    # subnormal, normal
    assert np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert np.array_equal(v[128:255], -pos) and np.signbit(v[128])
    # Spacing: 3 mantissa bits, so 8 values per binade from 2^-6 up.
    assert pos[120] == 256.0 and pos[121] == 288.0 and pos[112] == 128.0


def test_e4m3_rounding_ties_and_saturation():
    r = oracle.round_e4m3
    assert oracle.e4m3_to_f64(r([17.0, 19.0, 2.0 ** -10, 3 * 2.0 ** -11, 460.0, 470.0, 1e9]))\
        .tolist() == [16.0, 20.0, 0.0, 2.0 ** -9, 448.0, 448.0, 448.0]
    assert r([-44.8])[0] == (r([44.8])[0] | 0x80) and r([np.nan])[0] == 0x7F


def test_e4m3_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this torch")
    x = np.random.default_rng(41).normal(0, 60, 200000).astype(np.float32)
    x = np.concatenate([np.clip(x, -448, 448), np.float32(2.0) ** np.arange(-12, 9, 0.25).astype(np.float32)])
    t = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.round_e4m3(x), t)


def test_quantize_decision_precision_float32_against_float64():
    # The codes are integers decided by floating point; the oracle takes the decision in
    # float32 (the kernel's precision).  The float64 decision is kept beside it: on the FFN
    # activations X [1024, 4096] and the first 1024 rows of W [12288, 4096] (stored [N, K]),
    # the two agree except where y = x * 448 / amax lies within float32 rounding of a
    # midpoint between two E4M3 values; there they differ by one code step, the scales by at
    # most one float32 rounding.  The counts are stated in the design notes.
    w = inputs.fp8_gemm()
    K = w["K"]
    for name, X, rows in (("X", w["X"], 1024), ("W", w["W"], 1024)):
        q32, s32 = oracle.quantize_rows_e4m3(rows, K, X, K)
        q64, s64 = oracle.quantize_rows_e4m3_f64(rows, K, X, K)
        diff = q32 != q64
        n = int(diff.sum())
        assert n <= rows * K // 2000, (name, n)
        v32 = oracle.e4m3_to_f64(q32[diff])
        v64 = oracle.e4m3_to_f64(q64[diff])
        # one code step apart: no E4M3 value strictly between the two
        pos = oracle.e4m3_values()[:127]
        lo, hi = np.minimum(np.abs(v32), np.abs(v64)), np.maximum(np.abs(v32), np.abs(v64))
        between = np.searchsorted(pos, hi, side="left") - np.searchsorted(pos, lo, side="right")
        assert np.all(between == 0) and np.all(np.sign(v32) == np.sign(v64))
        assert np.all(np.abs(s32.astype(np.float64) - s64) <= np.abs(s64) * 2.0 ** -24)
        print(f"{name}: {n} of {rows * K} codes differ between float32 and float64 decisions")


def test_quantize_example_5_7():
    g, _ = read_golden("fp8_e4m3.txt")
    row = np.zeros(256, np.float32)
    row[0], row[128] = 1.0, 10.0
    q, s = oracle.quantize_rows_e4m3(1, 256, row, 256)
    assert np.isclose(np.float32(448) / np.float32(10), g["scaled_first"], rtol=1e-7)
    assert oracle.e4m3_to_f64(q[0, 0]) == g["rounded_first"]
    # Dequantised exactly (q * amax / 448) the code gives 55/56; the stored float32 scale is
    # amax / 448 rounded once.
    assert oracle.e4m3_to_f64(q[0, 0]) * 10.0 / 448.0 == g["dequant_row_scale"]
    assert s[0] == np.float32(10.0) / np.float32(448.0)
    assert np.isclose(oracle.e4m3_to_f64(q[0, 0]) * float(s[0]), g["dequant_row_scale"], rtol=1e-7)
    qb, sb = oracle.quantize_rows_e4m3(1, 128, row, 128)              # first block alone
    assert oracle.e4m3_to_f64(qb[0, 0]) == g["e4m3_max"]
    assert oracle.e4m3_to_f64(qb[0, 0]) * 1.0 / 448.0 == g["dequant_block_scale"]
    assert np.isclose(g["dequant_block_scale"] - g["dequant_row_scale"], g["difference"], rtol=1e-12)
    assert oracle.e4m3_to_f64(q[0, 128]) == 448.0                        # the maximum maps to 448


def test_quantize_rows_special_cases():
    from dense_gemm_sm_gb300 import inputs
    rng = np.random.default_rng(42)
    X = rng.normal(0, 3, (5, 40)).astype(np.float32)
    X[2] = 0.0
    bits = inputs.f32_to_bf16_bits(X)
    q, s = oracle.quantize_rows_e4m3(5, 40, bits, 40)
    assert np.all(q[2] == 0) and s[2] == 0.0                              # all-zero row
    xb = oracle.bf16_to_f64(bits)
    for i in (0, 1, 3, 4):
        j = np.argmax(np.abs(xb[i]))
        assert oracle.e4m3_to_f64(q[i, j]) == 448.0 * np.sign(xb[i, j])   # the maximum maps to 448
        assert s[i] == np.float32(np.abs(xb[i]).max()) / np.float32(448)
    qn, sn = oracle.quantize_rows_e4m3(5, 40, inputs.f32_to_bf16_bits(-X), 40)
    assert np.array_equal(qn[[0, 1, 3, 4]], q[[0, 1, 3, 4]] ^ 0x80) and np.array_equal(sn, s)
    # Dequantised values are within half an E4M3 spacing (relative 1/16) of the input.
    deq = oracle.e4m3_to_f64(q) * s[:, None].astype(np.float64)
    big = np.abs(xb) >= 2.0 ** -6 * s[:, None]
    assert np.all(np.abs(deq - xb)[big] <= np.abs(xb)[big] / 16 + 1e-12)


def test_gemm_fp8_closed_forms():
    # Codes of small integers (exact in E4M3) with unit scales: the integer matmul; then
    # row and column scales multiply the rows and columns.
    rng = np.random.default_rng(43)
    M, N, K = 7, 5, 33
    A = rng.integers(-8, 9, (M, K)).astype(np.float32)
    B = rng.integers(-8, 9, (N, K)).astype(np.float32)
    qa, qb = oracle.round_e4m3(A), oracle.round_e4m3(B)
    assert np.array_equal(oracle.e4m3_to_f64(qa), A)
    C, D = oracle.gemm_fp8(M, N, K, qa, K, np.ones(M, np.float32), qb, K, np.ones(N, np.float32))
    assert np.array_equal(C, A.astype(np.float64) @ B.T.astype(np.float64))
    assert np.array_equal(D, np.abs(A).astype(np.float64) @ np.abs(B).T.astype(np.float64))
    sa = np.float32(2.0) ** rng.integers(-3, 4, M).astype(np.float32)
    sb = rng.uniform(0.1, 2.0, N).astype(np.float32)
    C2, _ = oracle.gemm_fp8(M, N, K, qa, K, sa, qb, K, sb)
    assert np.allclose(C2, C * sa[:, None].astype(np.float64) * sb[None, :].astype(np.float64),
                       rtol=1e-15, atol=0)


# --------------------------------------------------------------------------- decode chain
def test_decode_chain_structure():
    from dense_gemm_sm_gb300 import inputs
    rng = np.random.default_rng(61)
    M, d = 3, 24
    X = inputs.f32_to_bf16_bits(rng.normal(0, 1, (M, d)).astype(np.float32))
    eye = inputs.f32_to_bf16_bits(np.eye(d, dtype=np.float32))
    perm = rng.permutation(d)
    P = inputs.f32_to_bf16_bits(np.eye(d, dtype=np.float32)[:, perm])
    # Identity and permutation layers move values exactly.
    res = oracle.decode_chain(M, [d, d, d], X, d, [eye, P], [d, d])
    assert np.array_equal(res[0][1], X.reshape(M, d))
    assert np.array_equal(res[1][1], X.reshape(M, d)[:, perm])
    # One layer is the BF16 GEMM rounded once; layer 2 takes layer 1's rounded output.
    W1 = inputs.f32_to_bf16_bits(rng.normal(0, 0.3, (d, 40)).astype(np.float32))
    W2 = inputs.f32_to_bf16_bits(rng.normal(0, 0.3, (40, 16)).astype(np.float32))
    res = oracle.decode_chain(M, [d, 40, 16], X, d, [W1, W2], [40, 16])
    x = oracle.bf16_to_f64(X).reshape(M, d)
    y1 = x @ oracle.bf16_to_f64(W1).reshape(d, 40)
    assert np.allclose(res[0][0], y1, rtol=1e-14, atol=1e-14)
    y2 = oracle.bf16_to_f64(oracle.round_bf16(y1)) @ oracle.bf16_to_f64(W2).reshape(40, 16)
    assert np.allclose(res[1][0], y2, rtol=1e-14, atol=1e-14)
    # The second layer's bound includes the propagated first-layer bound.
    assert np.all(res[1][2] > oracle.BF16_REL * 0 + oracle.ulp_bf16(np.abs(res[1][0])))


def test_decode_chain_check_catches_a_dropped_k_block():
    # A layer that drops its last 64 K rows (a plausible split-K mistake) fails the check.
    from dense_gemm_sm_gb300 import inputs
    rng = np.random.default_rng(62)
    M, dims = 4, [256, 384, 256]
    X = inputs.f32_to_bf16_bits(rng.normal(0, 1, (M, 256)).astype(np.float32))
    Ws = [inputs.f32_to_bf16_bits(rng.normal(0, 1 / 16, (dims[l], dims[l + 1])).astype(np.float32))
          for l in range(2)]
    res = oracle.decode_chain(M, dims, X, 256, Ws, [384, 256])
    ok, _ = oracle.check_chain_layer(res[0][1], res[0][0], res[0][2])
    assert ok
    x = oracle.bf16_to_f64(X).reshape(M, 256)
    w = oracle.bf16_to_f64(Ws[0]).reshape(256, 384)
    wrong = oracle.round_bf16(x[:, :192] @ w[:192])
    assert not oracle.check_chain_layer(wrong, res[0][0], res[0][2])[0]
