"""Helpers shared by the GPU parity tests: device placement and the acceptance
rule against the CPU oracle.

Acceptance rule (per element): |C - C_oracle| <= TOL * sum_k |A_ik||B_kj| on
real-valued inputs, with TOL = 5e-5; where that bound is 0 the result must be
exactly 0; on integer-valued inputs the result must equal the oracle exactly.
"""
from __future__ import annotations

import functools

import numpy as np
import torch

TOL = 5e-5


def to_device(X: torch.Tensor, ld: int | None = None, device="cuda", offset: int = 0, fill=float("nan")):
    """Copy a CPU matrix to the device with row stride ``ld`` (padding filled
    with NaN) after ``offset`` floats of NaN.  With ld == cols the matrix ends
    exactly at the end of its allocation, so any read past it would fault or
    pick up NaN."""
    rows, cols = X.shape
    ld = cols if ld is None else ld
    store = torch.full((offset + rows * ld,), fill, dtype=torch.float32, device=device)
    if rows == 0 or cols == 0:
        return torch.empty((rows, cols), dtype=torch.float32, device=device)
    view = store[offset:].view(rows, ld)
    view[:, :cols] = X.to(device)
    return view[:, :cols]


def check(C_gpu, C64, bound, *, exact: bool, tol: float = TOL, what: str = ""):
    """Assert the acceptance rule; return the worst |err| / bound."""
    C = np.asarray(C_gpu, dtype=np.float32).astype(np.float64)
    assert C.shape == C64.shape, (what, C.shape, C64.shape)
    assert np.isfinite(C).all(), f"{what}: non-finite output"
    if exact:
        bad = C != C64
        if bad.any():
            i, j = np.argwhere(bad)[0]
            raise AssertionError(f"{what}: {bad.sum()} entries differ from the exact result, first at ({i},{j}): "
                                 f"{C[i, j]!r} vs {C64[i, j]!r}")
        return 0.0
    err = np.abs(C - C64)
    zero = bound == 0
    assert np.all(C[zero] == 0), f"{what}: non-zero result where every product is zero"
    lim = tol * bound
    bad = err > lim
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} entries outside {tol}*bound, first at ({i},{j}): "
                             f"gpu {C[i, j]!r} oracle {C64[i, j]!r} bound {bound[i, j]!r}")
    rel = np.where(zero, 0.0, err / np.where(zero, 1.0, bound))
    return float(rel.max()) if rel.size else 0.0


def sample_rows(M: int, n_random: int = 16, seed: int = 0, tile: int = 128):
    """Rows on the edges of the output tiles plus a few random ones."""
    rows = {0, 1, M - 1, M - 2, M // 2}
    for t in range(tile, M, tile):
        if t % (tile * 8) == 0 or t == tile:
            rows.update({t - 1, t})
    rows.update({M - tile, M - tile - 1})
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, M, size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < M), dtype=np.int64)


@functools.lru_cache(maxsize=4)
def oracle_named(name: str):
    """The oracle's full result (C64, bound) for a named problem (or its
    ``_int`` twin), computed once per test process: at 4096^3 it takes a few
    seconds on the host cores, and several test files compare against it."""
    import oracle
    from workloads import PROBLEMS, problem_operands

    p = PROBLEMS[name[:-4]].int_variant() if name.endswith("_int") and name not in PROBLEMS else PROBLEMS[name]
    A, B = problem_operands(p)
    return oracle.gemm_f64(A.numpy(), B.numpy())
