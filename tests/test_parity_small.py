"""GPU parity of the small-problem kernel (one 8-warp CTA per 32 x 32 tile of
C, K split across the warps in 32-deep chunks, the partials summed in warp
order) against the oracle: every element, on shapes ragged against the 32 x
32 tiles and the 32-deep chunks, with several chunks per warp, padded and
misaligned operands, integer inputs (exact), and through the general entry
(A stored transposed, alpha and beta)."""
import numpy as np
import pytest
import torch

import dense_fp32_gemm_f32_gb300 as g
import oracle
from parity import check, to_device
from workloads import make_operands

pytestmark = pytest.mark.gpu

SMALL = dict(producer=6)


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert g.check_status() == 0, "a kernel reported a timeout"


def run(A, B, *, lda=None, ldb=None, oa=0, ob=0):
    dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
    dC = torch.full((A.shape[0], B.shape[1]), float("nan"), device="cuda")
    g.sgemm_f32_ex(dA, dB, dC, **SMALL)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


# K spans: under one chunk, exactly 8 chunks (one per warp), 8 chunks + 1
# element (warp 0 takes two, the second holding one k), many chunks per warp.
@pytest.mark.parametrize("shape", [(1, 1, 1), (31, 33, 17), (32, 32, 256), (33, 65, 257), (96, 80, 3000),
                                   (257, 31, 1025), (5, 700, 64), (700, 5, 64), (100, 3000, 50), (1, 1, 10000)])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_small_kernel_shapes(shape, dist):
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 300)
    C = run(A, B)
    exact = dist == "int"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=not exact)
    check(C, C64, bound, exact=exact, what=f"small {shape} {dist}")


@pytest.mark.parametrize("pads", [(3, 1, 1, 2), (0, 0, 3, 0), (7, 4, 2, 1)])
def test_small_kernel_padded_and_misaligned(pads):
    """Row pitches and bases with no 16-byte alignment: the kernel reads with
    4-byte loads, so any layout is taken as it is (NaN in the padding would
    show up in C if it were read)."""
    pa, pb, oa, ob = pads
    M, N, K = 150, 170, 190
    A, B = make_operands(M, N, K, "normal", 301)
    C = run(A, B, lda=K + pa, ldb=N + pb, oa=oa, ob=ob)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=f"small pads {pads}")


def test_small_kernel_output_pitch_and_guards():
    """C with padded rows inside a sentinel-filled store: the padding and the
    floats around C are never written."""
    M, N, K, ldc, guard = 70, 90, 50, 97, 64
    A, B = make_operands(M, N, K, "uniform", 302)
    sentinel = -3.5
    store = torch.full((guard + M * ldc + guard,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    g.sgemm_f32_ex(to_device(A), to_device(B), dC, **SMALL)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what="small ldc")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[-guard:] == sentinel)
    assert np.all(store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy() == sentinel)


def test_small_kernel_tall_grid():
    """ceil(M / 32) = 2188 rows of CTAs (grid y)."""
    M, N, K = 70000, 40, 36
    A, B = make_operands(M, N, K, "int", 303)
    C = run(A, B)
    C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
    check(C, C64, None, exact=True, what="small tall")


def test_small_kernel_deterministic():
    """The partials are summed in a fixed order: repeated calls agree bit for bit."""
    A, B = make_operands(200, 300, 2500, "normal", 304)
    C1, C2 = run(A, B), run(A, B)
    assert np.array_equal(C1.view(np.uint32), C2.view(np.uint32))


def test_small_kernel_is_the_automatic_choice():
    M, N, K = 256, 256, 256
    A, B = make_operands(M, N, K, "uniform", 305)
    dA, dB = to_device(A), to_device(B)
    assert g.describe(dA, dB) == "small/t32/w8"
    for fn in (g.sgemm_f32, g.sgemm_f32_noalloc):
        dC = torch.full((M, N), float("nan"), device="cuda")
        fn(dA, dB, dC)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
        check(dC.cpu().numpy(), C64, bound, exact=False, what=fn.__name__)


@pytest.mark.parametrize("other", [dict(split_k=2), dict(stream_k=2), dict(stages=2), dict(math=2),
                                   dict(tile_n=128), dict(repack=2), dict(a_layout=2), dict(multicast=1),
                                   dict(tail_split=2), dict(debug_skip_stage=1)])
def test_small_kernel_refuses_other_forced_fields(other):
    dA = torch.zeros((64, 64), device="cuda")
    dB = torch.zeros((64, 64), device="cuda")
    with pytest.raises(g._lib.SgemmError) as e:
        g.sgemm_f32_ex(dA, dB, **SMALL, **other)
    assert e.value.status == 1


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (-0.5, 1.5), (2.0, 0.0)])
def test_small_kernel_general_entry(ta, tb, alpha, beta):
    """sgemm_f32_gemm on a small product: A stored transposed is read in
    place (K x M), B stored transposed is copied first; C = alpha A B + beta C
    (beta == 0: C holds NaN and is not read)."""
    M, N, K = 90, 130, 300
    a, b = (x.numpy() for x in make_operands(M, N, K, "uniform", 306))
    A = np.ascontiguousarray(a.T) if ta else a
    B = np.ascontiguousarray(b.T) if tb else b
    cin = make_operands(M, 1, N, "uniform", 307)[0].numpy()
    dC = torch.from_numpy(cin).cuda() if beta else torch.full((M, N), float("nan"), device="cuda")
    g.sgemm_f32_gemm(to_device(torch.from_numpy(A), A.shape[1] + 1), to_device(torch.from_numpy(B)), dC,
                     alpha=alpha, beta=beta, transa=bool(ta), transb=bool(tb))
    torch.cuda.synchronize()
    ref, bound = oracle.gemm_general_f64(A, B, cin if beta else None, alpha=alpha, beta=beta, transa=ta, transb=tb)
    check(dC.cpu().numpy(), ref, bound, exact=False, what=f"small general t{ta}{tb} a{alpha} b{beta}")
