"""Randomised parity: random shapes (biased to tile edges), strides, offsets,
value distributions and forced variants of sgemm_f32_ex, and random storage
orders and scalars of sgemm_f32_gemm, each against the oracle.  A variant the
shape does not allow must be refused with an error, never run."""
import numpy as np
import pytest
import torch

import dense_fp32_gemm_f32_gb300 as g
import oracle
from parity import check, to_device
from workloads import make_operands

pytestmark = pytest.mark.gpu

OPTIONS = [
    {}, dict(producer=1), dict(producer=2), dict(producer=3), dict(producer=5), dict(producer=4),
    dict(stream_k=2), dict(stream_k=1), dict(split_k=2), dict(split_k=3), dict(tile_n=256), dict(tile_n=64),
    dict(a_layout=2), dict(a_layout=1), dict(repack=2), dict(math=1), dict(stages=3),
    dict(group_m=1), dict(group_m=3), dict(producer=5, stream_k=2), dict(a_layout=2, stream_k=2), dict(tile_n=256, stream_k=2), dict(producer=6),
    dict(producer=8), dict(producer=8, stages=3), dict(producer=8, split_k=2), dict(repack=1), dict(l2_hint=4),
    dict(edge=1),
]


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert g.check_status() == 0, "a kernel reported a timeout"


def _dim(rng):
    """1..700, half the time within one of a multiple of 32 or 128."""
    if rng.random() < 0.5:
        base = int(rng.choice([32, 128, 256, 384, 512])) * int(rng.integers(1, 3))
        return max(1, base + int(rng.integers(-1, 2)))
    return int(rng.integers(1, 701))


@pytest.mark.parametrize("case", range(64))
def test_fuzz_sgemm_f32_ex(case):
    rng = np.random.default_rng(1000 + case)
    M, N, K = _dim(rng), _dim(rng), _dim(rng)
    dist = "int" if rng.random() < 0.3 else ("normal" if rng.random() < 0.5 else "uniform")
    lda = K + int(rng.choice([0, 0, 1, 4, 7]))
    ldb = N + int(rng.choice([0, 0, 3, 4]))
    oa, ob = int(rng.choice([0, 0, 1])), int(rng.choice([0, 0, 2]))
    opt = OPTIONS[int(rng.integers(len(OPTIONS)))]
    A, B = make_operands(M, N, K, dist, 2000 + case)
    dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
    dC = torch.full((M, N), float("nan"), device="cuda")
    try:
        g.sgemm_f32_ex(dA, dB, dC, **opt)
    except g._lib.SgemmError as e:
        assert e.status in (1, 2), f"{opt} on {M}x{N}x{K}: {e}"  # refused, not failed
        return
    torch.cuda.synchronize()
    exact = dist == "int"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=not exact)
    check(dC.cpu().numpy(), C64, bound, exact=exact, what=f"{opt} {M}x{N}x{K} {dist} lda{lda} ldb{ldb}")


@pytest.mark.parametrize("case", range(24))
def test_fuzz_sgemm_f32_gemm(case):
    rng = np.random.default_rng(3000 + case)
    M, N, K = _dim(rng), _dim(rng), _dim(rng)
    ta, tb = int(rng.integers(2)), int(rng.integers(2))
    exact = rng.random() < 0.3
    dist = "int" if exact else "uniform"
    if exact:
        alpha, beta = float(rng.integers(-3, 4)), float(rng.integers(-2, 3))
    else:
        alpha, beta = float(rng.uniform(-2, 2)), float(rng.choice([0.0, float(rng.uniform(-2, 2))]))
    a, b = (x.numpy() for x in make_operands(M, N, K, dist, 4000 + case))
    cin = make_operands(M, 1, N, dist, 5000 + case)[0].numpy()
    A = np.ascontiguousarray(a.T) if ta else a
    B = np.ascontiguousarray(b.T) if tb else b
    dA = to_device(torch.from_numpy(A), A.shape[1] + int(rng.choice([0, 1, 4])))
    dB = to_device(torch.from_numpy(B), B.shape[1] + int(rng.choice([0, 2])))
    dC = to_device(torch.from_numpy(cin))
    g.sgemm_f32_gemm(dA, dB, dC, alpha=alpha, beta=beta, transa=bool(ta), transb=bool(tb))
    torch.cuda.synchronize()
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=alpha, beta=beta, transa=ta, transb=tb,
                                         with_bound=not exact)
    check(dC.cpu().numpy(), ref, bound, exact=exact,
          what=f"t{ta}{tb} a{alpha:.3f} b{beta:.3f} {M}x{N}x{K} {dist}")
