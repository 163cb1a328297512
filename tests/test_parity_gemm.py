"""GPU parity of the general entry sgemm_f32_gemm against the oracle's
general form: C = alpha * op(A) op(B) + beta * C with transposed storage.

Contract: |C - C_oracle| <= 5e-5 * (|alpha| sum_k |a||b| + |beta||c|) per
element on real-valued inputs; exact equality on integer-valued inputs with
integer alpha and beta.
"""
import numpy as np
import pytest
import torch

import dense_fp32_gemm_f32_gb300 as g
import oracle
from parity import check, to_device
from workloads import make_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert g.check_status() == 0, "a kernel reported a timeout"


def stored(a, b, ta, tb):
    """The stored operands for op(A) = a, op(B) = b."""
    A = np.ascontiguousarray(a.T) if ta else a
    B = np.ascontiguousarray(b.T) if tb else b
    return A, B


def run(A, B, Cin, *, alpha, beta, ta, tb, lda=None, ldb=None, ldc=None):
    dA = to_device(torch.from_numpy(A), lda)
    dB = to_device(torch.from_numpy(B), ldb)
    M = A.shape[1] if ta else A.shape[0]
    N = B.shape[0] if tb else B.shape[1]
    dC = to_device(torch.from_numpy(Cin) if Cin is not None else torch.full((M, N), float("nan")), ldc)
    g.sgemm_f32_gemm(dA, dB, dC, alpha=alpha, beta=beta, transa=ta, transb=tb)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


TRANS = [(0, 0), (1, 0), (0, 1), (1, 1)]
SCALES = [(1.0, 0.0), (2.0, -1.0), (0.5, 2.0), (-1.0, 0.5), (1.0, 1.0)]


# 300 x 500 x 700 runs on the small-problem kernel (32 x 32 tiles); 700 x 900
# x 500 (48 tiles of 128 x 128) on the FFMA kernels with the scaled epilogue.
# Both are ragged against their tiles, with several tiles per axis.
SHAPES = [(300, 500, 700), (700, 900, 500)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("ta,tb", TRANS)
@pytest.mark.parametrize("alpha,beta", SCALES)
def test_general_form(ta, tb, alpha, beta, shape):
    M, N, K = shape
    a, b = (x.numpy() for x in make_operands(M, N, K, "uniform", 201))
    cin = make_operands(M, 1, N, "uniform", 202)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=alpha, beta=beta, ta=ta, tb=tb)
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=alpha, beta=beta, transa=ta, transb=tb)
    check(C, ref, bound, exact=False, what=f"t{ta}{tb} a{alpha} b{beta}")


@pytest.mark.parametrize("shape", [(257, 190, 333), (700, 900, 333)])
@pytest.mark.parametrize("ta,tb", TRANS)
def test_general_form_integer_exact(ta, tb, shape):
    M, N, K = shape
    a, b = (x.numpy() for x in make_operands(M, N, K, "int", 203))
    cin = make_operands(M, 1, N, "int", 204)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=3.0, beta=-2.0, ta=ta, tb=tb)
    ref, _ = oracle.gemm_general_f64(A, B, cin, alpha=3.0, beta=-2.0, transa=ta, transb=tb, with_bound=False)
    check(C, ref, None, exact=True, what=f"int t{ta}{tb}")


@pytest.mark.parametrize("shape", [(130, 140, 150), (700, 900, 150)])
def test_beta_zero_does_not_read_c(shape):
    a, b = (x.numpy() for x in make_operands(*shape, "uniform", 205))
    C = run(a, b, None, alpha=1.5, beta=0.0, ta=0, tb=0)  # C holds NaN
    ref, bound = oracle.gemm_general_f64(a, b, alpha=1.5, beta=0.0)
    assert np.isfinite(C).all()
    check(C, ref, bound, exact=False, what="beta 0")


@pytest.mark.parametrize("K", [0, 64])
def test_alpha_zero_or_empty_sum_scales_c(K):
    """alpha == 0 (or K == 0): C = beta * C and A, B are not read (NaN there)."""
    M, N = 70, 90
    A = np.full((M, K), np.nan, np.float32)
    B = np.full((K, N), np.nan, np.float32)
    cin = make_operands(M, 1, N, "uniform", 206)[0].numpy()
    for alpha, beta in ((0.0, 2.0), (0.0, 0.0)) if K else ((1.0, -3.0), (2.0, 0.0)):
        C = run(A, B, cin.copy(), alpha=alpha, beta=beta, ta=0, tb=0)
        assert np.array_equal(C, (np.float32(beta) * cin) if beta else np.zeros_like(cin)), (alpha, beta)


@pytest.mark.parametrize("shape", [(200, 152, 96), (1100, 700, 96)])
@pytest.mark.parametrize("ta,tb", TRANS)
def test_general_padded_and_odd_pitches(ta, tb, shape):
    """Odd leading dimensions (no 16-byte rows) in every storage order."""
    M, N, K = shape
    a, b = (x.numpy() for x in make_operands(M, N, K, "uniform", 207))
    cin = make_operands(M, 1, N, "uniform", 208)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=0.75, beta=-1.25, ta=ta, tb=tb, lda=A.shape[1] + 3, ldb=B.shape[1] + 1,
            ldc=N + 5)
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=0.75, beta=-1.25, transa=ta, transb=tb)
    check(C, ref, bound, exact=False, what=f"padded t{ta}{tb}")


@pytest.mark.parametrize("ta,tb", [(1, 0), (0, 1), (1, 1)])
def test_general_split_k_shapes(ta, tb):
    """Small output, long K: cluster split-K, with the scaled epilogue on rank 0."""
    M, N, K = 256, 256, 8192
    a, b = (x.numpy() for x in make_operands(M, N, K, "normal", 209))
    cin = make_operands(M, 1, N, "normal", 210)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=-0.5, beta=1.5, ta=ta, tb=tb)
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=-0.5, beta=1.5, transa=ta, transb=tb)
    check(C, ref, bound, exact=False, what=f"split-K t{ta}{tb}")


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_general_4096_every_element(ta, tb):
    """4096^3 (stream-K schedule, finishing CTAs apply the epilogue) in every
    storage order: every element against the oracle."""
    M = N = K = 4096
    a, b = (x.numpy() for x in make_operands(M, N, K, "normal", 211))
    cin = make_operands(M, 1, N, "normal", 212)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=1.25, beta=0.75, ta=ta, tb=tb)
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=1.25, beta=0.75, transa=ta, transb=tb)
    check(C, ref, bound, exact=False, what=f"4096 t{ta}{tb}")


@pytest.mark.parametrize("ta,tb", [(0, 1), (1, 1)])
def test_general_4096_integer_exact(ta, tb):
    """Transposed B at 4096^3 on integer inputs, alpha = 2, beta = -1: exact."""
    M = N = K = 4096
    a, b = (x.numpy() for x in make_operands(M, N, K, "int", 214))
    cin = make_operands(M, 1, N, "int", 215)[0].numpy()
    A, B = stored(a, b, ta, tb)
    C = run(A, B, cin, alpha=2.0, beta=-1.0, ta=ta, tb=tb)
    ref, _ = oracle.gemm_general_f64(A, B, cin, alpha=2.0, beta=-1.0, transa=ta, transb=tb, with_bound=False)
    check(C, ref, None, exact=True, what=f"4096 int t{ta}{tb}")


def test_general_rejects_bad_arguments():
    lib = g._lib.load()
    A = torch.zeros((64, 32), device="cuda")  # stored K x M for transa: K = 64, M = 32
    B = torch.zeros((64, 48), device="cuda")
    C = torch.zeros((32, 48), device="cuda")
    pa, pb, pc = A.data_ptr(), B.data_ptr(), C.data_ptr()
    assert lib.sgemm_f32_gemm(1, 0, 32, 48, 64, 1.0, pa, 32, pb, 48, 0.0, pc, 48, None) == 0
    torch.cuda.synchronize()
    assert lib.sgemm_f32_gemm(1, 0, 32, 48, 64, 1.0, pa, 31, pb, 48, 0.0, pc, 48, None) == 1  # lda < M
    assert lib.sgemm_f32_gemm(0, 1, 32, 48, 64, 1.0, pa, 64, pb, 63, 0.0, pc, 48, None) == 1  # ldb < K
    assert lib.sgemm_f32_gemm(2, 0, 32, 48, 64, 1.0, pa, 32, pb, 48, 0.0, pc, 48, None) == 1  # bad flag
    assert lib.sgemm_f32_gemm(1, 0, 32, 48, 64, 1.0, pa, 32, pb, 48, 0.0, pa, 48, None) == 1  # C overlaps A
    with pytest.raises(ValueError):
        g.sgemm_f32_gemm(A, B, C)  # op(A) is 64 x 32: does not multiply 64 x 48
    with pytest.raises(ValueError):
        g.sgemm_f32_gemm(A, B, None, beta=1.0, transa=True)  # beta != 0 needs C


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("pad_a,pad_b", [(0, 4), (3, 0), (3, 8)])
def test_transposed_b_read_in_place(ta, pad_a, pad_b):
    """op(B) = B^T with 16-byte B rows is read in place (a producer warp
    transposes its slices in shared memory), also with padded B rows and
    with an A whose odd pitch makes the library copy it first; ragged against
    the 128 x 128 tiles in M, N and K."""
    M, N, K = 650, 900, 1000
    a, b = (x.numpy() for x in make_operands(M, N, K, "uniform", 216))
    cin = make_operands(M, 1, N, "uniform", 217)[0].numpy()
    A, B = stored(a, b, ta, 1)
    C = run(A, B, cin, alpha=-0.75, beta=0.5, ta=ta, tb=1, lda=A.shape[1] + pad_a, ldb=B.shape[1] + pad_b)
    ref, bound = oracle.gemm_general_f64(A, B, cin, alpha=-0.75, beta=0.5, transa=ta, transb=1)
    check(C, ref, bound, exact=False, what=f"t{ta}1 pads {pad_a},{pad_b}")
    C1 = run(A, B, None, alpha=1.0, beta=0.0, ta=ta, tb=1, ldb=B.shape[1] + pad_b)  # plain epilogue
    ref1, bound1 = oracle.gemm_general_f64(A, B, alpha=1.0, beta=0.0, transa=ta, transb=1)
    check(C1, ref1, bound1, exact=False, what=f"t{ta}1 plain")


@pytest.mark.parametrize("ta", [0, 1])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_transposed_b_skinny_every_element(ta, dist):
    """128 x 8192 x 16384 with op(B) = B^T (one row of 64 tiles, stream-K over
    512 K slices each): every element; integer inputs exactly."""
    M, N, K = 128, 8192, 16384
    a, b = (x.numpy() for x in make_operands(M, N, K, dist, 218))
    A, B = stored(a, b, ta, 1)
    C = run(A, B, None, alpha=1.0, beta=0.0, ta=ta, tb=1)
    ref, bound = oracle.gemm_general_f64(A, B, alpha=1.0, beta=0.0, transa=ta, transb=1, with_bound=dist != "int")
    check(C, ref, None if dist == "int" else bound, exact=dist == "int", what=f"skinny t{ta}1 {dist}")


@pytest.mark.parametrize("dist", ["uniform", "int"])
@pytest.mark.parametrize("offsets", [(0, 0, 0), (1, 3, 2)])
def test_general_misaligned_rows_on_class_maps(dist, offsets):
    """The ragged named shape in the stored order (rows of 1027 and 1025
    floats, bases off the 16-byte grid by `offsets` floats): A and B read in
    place through the residue-class maps with the scaled epilogue; integer
    inputs with integer alpha and beta exactly."""
    M, N, K = 1023, 1025, 1027
    a, b = (x.numpy() for x in make_operands(M, N, K, dist, 211))
    cin = make_operands(M, 1, N, dist, 212)[0].numpy()
    alpha, beta = (2.0, -1.0) if dist == "int" else (0.75, -1.25)
    oa, ob, oc = offsets
    dA = to_device(torch.from_numpy(a), K, offset=oa)
    dB = to_device(torch.from_numpy(b), N, offset=ob)
    dC = to_device(torch.from_numpy(cin), N, offset=oc)
    g.sgemm_f32_gemm(dA, dB, dC, alpha=alpha, beta=beta)
    torch.cuda.synchronize()
    ref, bound = oracle.gemm_general_f64(a, b, cin, alpha=alpha, beta=beta, transa=0, transb=0)
    check(dC.cpu().numpy(), ref, bound, exact=(dist == "int"), what=f"class maps, scaled, {offsets} {dist}")
