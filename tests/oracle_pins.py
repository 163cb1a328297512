"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each pin takes an ``oracle.OracleLib`` and raises AssertionError on a mismatch.
They check the oracle against hand-computed golden products, closed forms
(identity, all-ones), exact integer and exact rational arithmetic, the plain
i-j-k triple loop written out in Python, and the Freivalds matrix-vector
invariant.  ``test_oracle.py`` runs them on the real oracle; the mutation test
runs them on deliberately broken copies of the oracle source and requires every
copy to fail at least one pin.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np

from conftest import load_golden
from workloads import make_operands


def _np(t):
    return t.numpy() if hasattr(t, "numpy") else np.asarray(t)


def pin_golden_hand_cases(o):
    for case in load_golden("hand_cases.txt"):
        A = case["A"].astype(np.float32)
        B = case["B"].astype(np.float32)
        C, bound = o.gemm_f64(A, B)
        assert C.shape == (case["M"], case["N"]), case["name"]
        assert np.array_equal(C, case["C"]), (case["name"], C, case["C"])
        if case.get("BOUND") is not None:
            assert np.array_equal(bound, case["BOUND"]), (case["name"], bound, case["BOUND"])
        elif (A >= 0).all() and (B >= 0).all():
            assert np.array_equal(bound, case["C"]), case["name"]


def pin_identity(o):
    A, B = make_operands(37, 53, 29, "uniform", 11)
    A, B = _np(A), _np(B)
    C, _ = o.gemm_f64(A, np.eye(29, dtype=np.float32))
    assert np.array_equal(C, A.astype(np.float64))
    C, _ = o.gemm_f64(np.eye(29, dtype=np.float32), B)
    assert np.array_equal(C, B.astype(np.float64))


def pin_all_ones(o):
    for (M, N, K) in [(5, 7, 16384), (129, 131, 1027), (1, 1, 1)]:
        C, bound = o.gemm_f64(np.ones((M, K), np.float32), np.ones((K, N), np.float32))
        assert np.all(C == K), (M, N, K)
        assert np.all(bound == K), (M, N, K)


def pin_integer_exact(o):
    A, B = make_operands(64, 48, 40, "int", 7)
    A, B = _np(A), _np(B)
    ref = A.astype(np.int64) @ B.astype(np.int64)  # exact integer arithmetic
    C, bound = o.gemm_f64(A, B)
    assert np.array_equal(C, ref.astype(np.float64))
    assert np.array_equal(bound, (np.abs(A).astype(np.int64) @ np.abs(B).astype(np.int64)).astype(np.float64))
    # tiny case with Python integers and an explicit triple loop
    a, b = make_operands(6, 5, 7, "int", 8)
    a, b = _np(a), _np(b)
    C, _ = o.gemm_f64(a, b)
    for i in range(6):
        for j in range(5):
            s = 0
            for k in range(7):
                s += int(a[i, k]) * int(b[k, j])
            assert C[i, j] == s


def pin_fraction_bruteforce(o):
    """Exact rational sums on tiny float32 inputs: error within K * 2^-53 * bound."""
    for seed, (M, N, K) in enumerate([(1, 1, 8), (3, 4, 5), (8, 8, 8), (2, 7, 3)]):
        A, B = make_operands(M, N, K, "normal", 100 + seed)
        A, B = _np(A), _np(B)
        C, bound = o.gemm_f64(A, B)
        for i in range(M):
            for j in range(N):
                exact = sum(Fraction(float(A[i, k])) * Fraction(float(B[k, j])) for k in range(K))
                ebound = sum(abs(Fraction(float(A[i, k])) * Fraction(float(B[k, j]))) for k in range(K))
                tol = Fraction(K) * Fraction(1, 2**53) * ebound
                assert abs(Fraction(C[i, j]) - exact) <= tol, (i, j)
                assert abs(Fraction(bound[i, j]) - ebound) <= tol, (i, j)


def pin_loop_order(o):
    """Bit-identical to the plain i-j-k triple loop with a double accumulator."""
    A, B = make_operands(9, 11, 13, "uniform", 21)
    A, B = _np(A), _np(B)
    C, bound = o.gemm_f64(A, B)
    for i in range(9):
        for j in range(11):
            s = 0.0
            sb = 0.0
            for k in range(13):
                p = float(A[i, k]) * float(B[k, j])
                s += p
                sb += abs(float(A[i, k])) * abs(float(B[k, j]))
            assert C[i, j] == s, (i, j, C[i, j], s)
            assert bound[i, j] == sb, (i, j)


def pin_empty(o):
    C, bound = o.gemm_f64(np.ones((3, 0), np.float32), np.ones((0, 4), np.float32))
    assert C.shape == (3, 4) and np.all(C == 0) and np.all(bound == 0)
    C, _ = o.gemm_f64(np.ones((0, 5), np.float32), np.ones((5, 4), np.float32))
    assert C.shape == (0, 4)
    C, _ = o.gemm_f64(np.ones((3, 5), np.float32), np.ones((5, 0), np.float32))
    assert C.shape == (3, 0)


def pin_leading_dims(o):
    """Padded rows (NaN in the padding) give the compact result, bit for bit."""
    A, B = make_operands(19, 23, 17, "uniform", 5)
    Ap, Bp = make_operands(19, 23, 17, "uniform", 5, lda=21, ldb=30)
    C0, b0 = o.gemm_f64(_np(A), _np(B))
    C1, b1 = o.gemm_f64(_np(Ap), _np(Bp))
    assert np.isfinite(C1).all()
    assert np.array_equal(C0, C1) and np.array_equal(b0, b1)


def pin_freivalds(o):
    """C x == A (B x) for a random x, within the double rounding of both sides."""
    A, B = make_operands(300, 200, 500, "normal", 9)
    A, B = _np(A).astype(np.float64), _np(B).astype(np.float64)
    C, bound = o.gemm_f64(A.astype(np.float32), B.astype(np.float32))
    x = np.random.default_rng(3).standard_normal(200)
    lhs = C @ x
    rhs = A @ (B @ x)
    scale = (np.abs(A) @ (np.abs(B) @ np.abs(x)))
    assert np.all(np.abs(lhs - rhs) <= 1e-12 * scale + 1e-300)
    assert np.all(bound >= np.abs(C))


def pin_bound_dominates(o):
    A, B = make_operands(33, 17, 40, "normal", 2)
    C, bound = o.gemm_f64(_np(A), _np(B))
    assert np.all(bound >= np.abs(C))
    An, Bn = np.abs(_np(A)), np.abs(_np(B))
    C2, bound2 = o.gemm_f64(An, Bn)
    assert np.array_equal(C2, bound2)
    assert np.array_equal(bound, bound2)


def pin_sampling_entry_points(o):
    """Row and single-entry entry points agree bit for bit with the full product."""
    A, B = make_operands(41, 37, 29, "normal", 4)
    A, B = _np(A), _np(B)
    C, bound = o.gemm_f64(A, B)
    rows = [0, 40, 17, 17]
    Cr, br = o.gemm_rows_f64(A, B, rows)
    assert np.array_equal(Cr, C[rows]) and np.array_equal(br, bound[rows])
    ii, jj = [0, 40, 5, 39], [0, 36, 7, 1]
    ce, be = o.gemm_entries_f64(A, B, ii, jj)
    assert np.array_equal(ce, C[ii, jj]) and np.array_equal(be, bound[ii, jj])


def pin_thread_invariance(o):
    A, B = make_operands(57, 31, 44, "normal", 6)
    C1, b1 = o.gemm_f64(_np(A), _np(B), threads=1)
    C7, b7 = o.gemm_f64(_np(A), _np(B), threads=7)
    assert np.array_equal(C1, C7) and np.array_equal(b1, b7)


# ---------------------------------------------------------------- general form

def pin_general_hand_cases(o):
    for case in load_golden("general_cases.txt"):
        op = case["opts"]
        A = case["A"].astype(np.float32)
        B = case["B"].astype(np.float32)
        Cin = case.get("CIN")
        Cin = None if Cin is None else Cin.astype(np.float32)
        C, bound = o.gemm_general_f64(A, B, Cin, alpha=op["alpha"], beta=op["beta"], transa=op["transa"],
                                      transb=op["transb"])
        assert C.shape == (case["M"], case["N"]), case["name"]
        assert np.array_equal(C, case["C"]), (case["name"], C, case["C"])
        assert np.array_equal(bound, case["BOUND"]), (case["name"], bound, case["BOUND"])


def pin_general_transposed_storage(o):
    """Transposed storage gives the plain product of the explicitly transposed
    copies, bit for bit (alpha 1, beta 0), also with padded rows."""
    M, N, K = 23, 19, 31
    A, B = make_operands(M, N, K, "normal", 61)
    A, B = _np(A), _np(B)
    ref, rbound = o.gemm_f64(A, B)
    At = np.full((K, M + 5), np.nan, np.float32)
    At[:, :M] = A.T
    Bt = np.full((N, K + 3), np.nan, np.float32)
    Bt[:, :K] = B.T
    for ta, tb in [(0, 0), (1, 0), (0, 1), (1, 1)]:
        C, bound = o.gemm_general_f64(At[:, :M] if ta else A, Bt[:, :K] if tb else B, transa=ta, transb=tb)
        assert np.array_equal(C, ref), (ta, tb)
        assert np.array_equal(bound, rbound), (ta, tb)


def pin_general_scaling(o):
    """alpha = 0 leaves beta * C_in exactly; beta = 0 ignores C_in (NaN there
    has no effect) and a power-of-two alpha scales the product exactly."""
    A, B = make_operands(17, 13, 29, "uniform", 62)
    A, B = _np(A), _np(B)
    Cin = _np(make_operands(17, 1, 13, "uniform", 63)[0])
    ref, rbound = o.gemm_f64(A, B)
    C, bound = o.gemm_general_f64(A, B, Cin, alpha=0.0, beta=3.0)
    assert np.array_equal(C, 3.0 * Cin.astype(np.float64))
    assert np.array_equal(bound, 3.0 * np.abs(Cin).astype(np.float64))
    nan = np.full((17, 13), np.nan, np.float32)
    C, bound = o.gemm_general_f64(A, B, nan, alpha=-4.0, beta=0.0)
    assert np.array_equal(C, -4.0 * ref) and np.array_equal(bound, 4.0 * rbound)
    C, bound = o.gemm_general_f64(A, B, Cin, alpha=1.0, beta=1.0)
    assert np.all(np.abs(C - (ref + Cin)) <= 2.0**-52 * np.abs(ref + Cin))


def pin_general_integer_bruteforce(o):
    """Integer inputs and integer alpha, beta: equal to Python-integer
    arithmetic with the transposed indexing written out."""
    M, N, K = 5, 4, 6
    for ta, tb in [(0, 0), (1, 0), (0, 1), (1, 1)]:
        a, b = make_operands(M, N, K, "int", 70 + 2 * ta + tb)
        a, b = _np(a), _np(b)
        cin = _np(make_operands(M, 1, N, "int", 80 + 2 * ta + tb)[0])
        As = np.ascontiguousarray(a.T) if ta else a
        Bs = np.ascontiguousarray(b.T) if tb else b
        alpha, beta = 3, -2
        C, _ = o.gemm_general_f64(As, Bs, cin, alpha=alpha, beta=beta, transa=ta, transb=tb)
        for i in range(M):
            for j in range(N):
                s = 0
                for k in range(K):
                    aik = int(As[k, i]) if ta else int(As[i, k])
                    bkj = int(Bs[j, k]) if tb else int(Bs[k, j])
                    s += aik * bkj
                assert C[i, j] == alpha * s + beta * int(cin[i, j]), (ta, tb, i, j)


def pin_general_fraction(o):
    """Exact rationals with non-trivial alpha, beta and transposed A: error
    within (K + 2) * 2^-53 * bound."""
    M, N, K = 3, 4, 5
    a, b = make_operands(M, N, K, "normal", 64)
    a, b = _np(a), _np(b)
    cin = _np(make_operands(M, 1, N, "normal", 65)[0])
    alpha, beta = float(np.float32(0.7)), float(np.float32(-1.3))
    At = np.ascontiguousarray(a.T)
    C, bound = o.gemm_general_f64(At, b, cin, alpha=alpha, beta=beta, transa=1)
    for i in range(M):
        for j in range(N):
            prods = [Fraction(float(a[i, k])) * Fraction(float(b[k, j])) for k in range(K)]
            exact = Fraction(alpha) * sum(prods) + Fraction(beta) * Fraction(float(cin[i, j]))
            ebound = abs(Fraction(alpha)) * sum(abs(p) for p in prods) + abs(Fraction(beta)) * abs(
                Fraction(float(cin[i, j])))
            tol = Fraction(K + 2) * Fraction(1, 2**53) * ebound
            assert abs(Fraction(C[i, j]) - exact) <= tol, (i, j)
            assert abs(Fraction(bound[i, j]) - ebound) <= tol, (i, j)


def pin_general_sampled_rows(o):
    """The row-sampled general form equals the matching rows of the full one."""
    A, B = make_operands(21, 9, 14, "normal", 66)
    A, B = _np(A), _np(B)
    Cin = _np(make_operands(21, 1, 9, "normal", 67)[0])
    At = np.ascontiguousarray(A.T)
    full, fb = o.gemm_general_f64(At, B, Cin, alpha=1.5, beta=-0.25, transa=1)
    rows = np.array([0, 20, 7, 7, 13])
    part, pb = o.gemm_general_f64(At, B, Cin, alpha=1.5, beta=-0.25, transa=1, rows=rows)
    assert np.array_equal(part, full[rows]) and np.array_equal(pb, fb[rows])


ALL_PINS = [
    pin_golden_hand_cases,
    pin_identity,
    pin_all_ones,
    pin_integer_exact,
    pin_fraction_bruteforce,
    pin_loop_order,
    pin_empty,
    pin_leading_dims,
    pin_freivalds,
    pin_bound_dominates,
    pin_sampling_entry_points,
    pin_thread_invariance,
    pin_general_hand_cases,
    pin_general_transposed_storage,
    pin_general_scaling,
    pin_general_integer_bruteforce,
    pin_general_fraction,
    pin_general_sampled_rows,
]
