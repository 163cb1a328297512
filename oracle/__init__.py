"""CPU oracle for C = A x B (float32 inputs, float64 result).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the benchmark's CPU-baseline leg may import this package.  The product library
(``dense_fp32_gemm_f32_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle_gemm.c`` (plain C, double accumulation, the
textbook definition C[i][j] = sum_k A[i][k] * B[k][j] of "Hardware acceleration:
optimising the memory access pattern of CUDA kernels for matrix multiply",
section "computational characteristics of matrix multiplication").  This module
compiles it with gcc on first use and marshals numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_gemm.c")
_LIB = os.path.join(_HERE, "liboracle_gemm.so")
# No fused multiply-add contraction, no fast-math reassociation: the sums are
# evaluated exactly in the order the C source writes them.
CFLAGS = ["-O2", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared", "-pthread"]

_lock = threading.Lock()
_default = None


def compile_source(src: str, out: str) -> str:
    """Compile a C source file with the oracle's flags into shared library ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", *CFLAGS, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc) if it is missing or stale."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        compile_source(_SRC, _LIB)
    return _LIB


def default_threads() -> int:
    if hasattr(os, "sched_getaffinity"):
        return max(1, len(os.sched_getaffinity(0)))
    return max(1, os.cpu_count() or 1)


def _as_f32_rows(X, name):
    """Accept a 2-D float32 array whose last dimension is contiguous (any row stride)."""
    X = np.asarray(X)
    if X.dtype != np.float32 or X.ndim != 2:
        raise TypeError(f"{name} must be a 2-D float32 array")
    if X.shape[0] > 0 and X.shape[1] > 1 and X.strides[1] != 4:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    if X.shape[0] > 1:
        if X.strides[0] % 4 or X.strides[0] < 4 * X.shape[1]:
            raise ValueError(f"{name} row stride must be a whole number of floats >= the row width")
        ld = X.strides[0] // 4
    else:
        ld = X.shape[1]
    return X, ld


def _ptr(X):
    return ctypes.c_void_p(X.ctypes.data) if X is not None and X.size else ctypes.c_void_p(0)


class OracleLib:
    """ctypes view of one compiled copy of ``oracle_gemm.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_sgemm_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p, i64, ctypes.c_int]
        lib.oracle_sgemm_rows_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, i64, p, p, ctypes.c_int]
        lib.oracle_sgemm_entries_f64.argtypes = [i64, i64, i64, p, i64, p, i64, p, p, i64, p, p]
        f32, i32 = ctypes.c_float, ctypes.c_int
        lib.oracle_gemm_general_f64.argtypes = [i32, i32, i64, i64, i64, f32, p, i64, p, i64, f32, p, i64, p, i64,
                                                p, i64, p, i64, i32]
        for f in (lib.oracle_sgemm_f64, lib.oracle_sgemm_rows_f64, lib.oracle_sgemm_entries_f64,
                  lib.oracle_gemm_general_f64):
            f.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    @staticmethod
    def _operands(A, B):
        A, lda = _as_f32_rows(A, "A")
        B, ldb = _as_f32_rows(B, "B")
        if A.shape[1] != B.shape[0]:
            raise ValueError(f"inner dimensions differ: A is {A.shape}, B is {B.shape}")
        return A, lda, B, ldb, A.shape[0], B.shape[1], A.shape[1]

    def gemm_f64(self, A, B, *, with_bound: bool = True, threads: int | None = None):
        """Full product in float64 and (optionally) bound[i][j] = sum_k |A_ik||B_kj|.

        A: (M, K) float32, B: (K, N) float32, row-major with any row stride.
        Returns (C, bound) as float64 (M, N) arrays; bound is None if not requested.
        """
        A, lda, B, ldb, M, N, K = self._operands(A, B)
        C = np.empty((M, N), dtype=np.float64)
        bound = np.empty((M, N), dtype=np.float64) if with_bound else None
        rc = self.lib.oracle_sgemm_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(C), max(N, 1),
                                       _ptr(bound), max(N, 1), threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_sgemm_f64 failed with {rc}")
        return C, bound

    def gemm_rows_f64(self, A, B, rows, *, threads: int | None = None):
        """Rows ``rows`` of the product (float64) and of the bound."""
        A, lda, B, ldb, M, N, K = self._operands(A, B)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        C = np.empty((rows.size, N), dtype=np.float64)
        bound = np.empty((rows.size, N), dtype=np.float64)
        rc = self.lib.oracle_sgemm_rows_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(rows), rows.size,
                                            _ptr(C), _ptr(bound), threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_sgemm_rows_f64 failed with {rc}")
        return C, bound

    def gemm_entries_f64(self, A, B, ii, jj):
        """Entries C[ii[t], jj[t]] computed one by one (float64), with their bounds."""
        A, lda, B, ldb, M, N, K = self._operands(A, B)
        ii = np.ascontiguousarray(ii, dtype=np.int64)
        jj = np.ascontiguousarray(jj, dtype=np.int64)
        if ii.shape != jj.shape:
            raise ValueError("ii and jj must have the same shape")
        c = np.empty(ii.size, dtype=np.float64)
        bound = np.empty(ii.size, dtype=np.float64)
        rc = self.lib.oracle_sgemm_entries_f64(M, N, K, _ptr(A), lda, _ptr(B), ldb, _ptr(ii), _ptr(jj),
                                               ii.size, _ptr(c), _ptr(bound))
        if rc != 0:
            raise RuntimeError(f"oracle_sgemm_entries_f64 failed with {rc}")
        return c, bound


    def gemm_general_f64(self, A, B, C=None, *, alpha=1.0, beta=0.0, transa=False, transb=False, rows=None,
                         with_bound: bool = True, threads: int | None = None):
        """C_out = alpha * op(A) op(B) + beta * C in float64, with its bound
        |alpha| sum_k |a||b| + |beta||c|.

        A and B are the stored operands (float32, row-major, any row stride):
        A is (M, K), or (K, M) when ``transa``; B is (K, N), or (N, K) when
        ``transb``.  C is (M, N) float32, needed only when beta != 0.  With
        ``rows``, only those output rows are computed.  Returns (C_out, bound)
        as float64 arrays (bound None if not requested).
        """
        A, lda = _as_f32_rows(A, "A")
        B, ldb = _as_f32_rows(B, "B")
        M, K = (A.shape[1], A.shape[0]) if transa else A.shape
        KB, N = (B.shape[1], B.shape[0]) if transb else B.shape
        if K != KB:
            raise ValueError(f"inner dimensions differ: op(A) is {(M, K)}, op(B) is {(KB, N)}")
        ldcin = 0
        if beta != 0 and C is None:
            raise ValueError("beta != 0 needs C")
        if C is not None:  # passed even when beta == 0, which must leave it unread
            C, ldcin = _as_f32_rows(C, "C")
            if C.shape != (M, N):
                raise ValueError(f"C must be {(M, N)}, got {C.shape}")
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        nrows = M if rows_arr is None else rows_arr.size
        out = np.empty((nrows, N), dtype=np.float64)
        bound = np.empty((nrows, N), dtype=np.float64) if with_bound else None
        rc = self.lib.oracle_gemm_general_f64(int(bool(transa)), int(bool(transb)), M, N, K, float(alpha), _ptr(A),
                                              lda, _ptr(B), ldb, float(beta),
                                              _ptr(C) if C is not None else ctypes.c_void_p(0), ldcin,
                                              _ptr(rows_arr) if rows_arr is not None else ctypes.c_void_p(0), nrows,
                                              _ptr(out), max(N, 1), _ptr(bound), max(N, 1),
                                              threads or default_threads())
        if rc != 0:
            raise RuntimeError(f"oracle_gemm_general_f64 failed with {rc}")
        return out, bound


def default() -> OracleLib:
    global _default
    with _lock:
        if _default is None:
            _default = OracleLib(build())
    return _default


def gemm_f64(A, B, **kw):
    return default().gemm_f64(A, B, **kw)


def gemm_rows_f64(A, B, rows, **kw):
    return default().gemm_rows_f64(A, B, rows, **kw)


def gemm_entries_f64(A, B, ii, jj):
    return default().gemm_entries_f64(A, B, ii, jj)


def gemm_general_f64(A, B, C=None, **kw):
    return default().gemm_general_f64(A, B, C, **kw)
