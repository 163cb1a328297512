"""Seeded synthetic inputs and the named problem shapes.

This module holds no arithmetic of the matrix product: it only draws the
operands.  It is the one module shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.

Generator reading.  The pages draw their inputs with ``srand(42)`` and
``(rand() % 100) / 100.0f`` ("[infra] 03: writing CUDA kernels, from vector add
to matrix multiply", host set-up of experiments 2-4) and name no generator for
anything else.  Here every problem draws from a freshly seeded
``torch.Generator('cpu')``: A first, then B, from the same generator.

* ``uniform``: float32 i.i.d. in [-1, 1): ``rand * 2 - 1`` (an exact affine map
  of torch's [0, 1) float32 draw).
* ``normal``: float32 standard normal (``randn``).
* ``int``: integers uniform in {-8, ..., 8}, stored as float32.  Every product
  is at most 64 in magnitude and every partial sum an integer below 2^24 for
  K <= 2^18, so any summation order gives the same exact float32 result.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

INT_LO, INT_HI = -8, 8  # inclusive range of the integer-valued variant


@dataclass(frozen=True)
class Problem:
    name: str
    M: int
    N: int
    K: int
    dist: str  # "uniform" | "normal" | "int"
    seed: int

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def min_bytes(self) -> int:
        """Algorithmic minimum traffic: A and B read once, C written once."""
        return 4 * (self.M * self.K + self.K * self.N + self.M * self.N)

    def int_variant(self) -> "Problem":
        return Problem(self.name + "_int", self.M, self.N, self.K, "int", self.seed + 100)


# The named synthetic workloads: shapes, distributions and seeds.
PROBLEMS = {
    p.name: p
    for p in [
        Problem("square_256", 256, 256, 256, "uniform", 0),
        Problem("ragged_1023x1025x1027", 1023, 1025, 1027, "uniform", 1),
        Problem("square_1024", 1024, 1024, 1024, "uniform", 2),
        Problem("square_2048", 2048, 2048, 2048, "uniform", 2),
        Problem("square_4096", 4096, 4096, 4096, "normal", 3),
        Problem("square_8192", 8192, 8192, 8192, "normal", 3),
        Problem("skinny_8192x128x8192", 8192, 128, 8192, "uniform", 4),
        Problem("skinny_128x8192x16384", 128, 8192, 16384, "uniform", 4),
        Problem("flat_4096x4096x256", 4096, 4096, 256, "uniform", 4),
    ]
}
# The integer-valued twin of the 256^3 problem (the pages' bit-exact check).
PROBLEMS["square_256_int"] = PROBLEMS["square_256"].int_variant()


def _draw(shape, dist: str, g: torch.Generator) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=g, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=g, dtype=torch.float32)
    if dist == "int":
        return torch.randint(INT_LO, INT_HI + 1, shape, generator=g, dtype=torch.int32).to(torch.float32)
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(f"unknown distribution {dist!r}")


def make_operands(M: int, N: int, K: int, dist: str = "uniform", seed: int = 0,
                  lda: int | None = None, ldb: int | None = None):
    """Return CPU float32 tensors (A, B) of logical shapes (M, K), (K, N).

    If ``lda``/``ldb`` exceed the row width the tensors are views into wider
    row-major storage whose padding columns hold NaN, so a read outside the
    logical matrix poisons the result instead of passing silently.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    A = _draw((M, K), dist, g)
    B = _draw((K, N), dist, g)
    if lda is not None and lda > K:
        store = torch.full((M, lda), float("nan"), dtype=torch.float32)
        store[:, :K] = A
        A = store[:, :K]
    if ldb is not None and ldb > N:
        store = torch.full((K, ldb), float("nan"), dtype=torch.float32)
        store[:, :N] = B
        B = store[:, :N]
    return A, B


def problem_operands(p: Problem):
    return make_operands(p.M, p.N, p.K, p.dist, p.seed)
