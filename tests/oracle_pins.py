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
]
