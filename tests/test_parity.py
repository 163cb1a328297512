"""GPU parity: the CUDA library against the CPU oracle, element by element.

Every test goes through the C ABI (via the thin binding) and compares with
``oracle`` on the same seeded inputs from ``workloads``.  Real-valued inputs
must satisfy |C - C_oracle| <= 5e-5 * sum_k |A_ik||B_kj| for every element;
integer-valued inputs must match exactly.
"""
import numpy as np
import pytest
import torch

import dense_fp32_gemm_f32_gb300 as g
import oracle
from parity import check, oracle_named, sample_rows, to_device
from workloads import PROBLEMS, make_operands, problem_operands

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def cuda_device():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    yield
    assert g.check_status() == 0, "a kernel reported a timeout"


def run(A, B, *, lda=None, ldb=None, ldc=None, fn=None, **opt):
    dA = to_device(A, lda)
    dB = to_device(B, ldb)
    M, N = A.shape[0], B.shape[1]
    dC = to_device(torch.full((M, N), float("nan")), ldc)
    if fn is not None:
        fn(dA, dB, dC)
    elif opt:
        g.sgemm_f32_ex(dA, dB, dC, **opt)
    else:
        g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


# ---------------------------------------------------------------- named problems, every element

FULL = ["square_256", "ragged_1023x1025x1027", "square_1024", "square_2048", "flat_4096x4096x256",
        "skinny_8192x128x8192", "skinny_128x8192x16384"]


@pytest.mark.parametrize("name", FULL)
def test_named_problem_every_element(name):
    p = PROBLEMS[name]
    A, B = problem_operands(p)
    C = run(A, B)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    worst = check(C, C64, bound, exact=False, what=name)
    print(f"{name}: worst |err|/bound = {worst:.3e}")


@pytest.mark.parametrize("name", ["square_256"] + FULL[1:])
def test_named_problem_integer_exact(name):
    p = PROBLEMS[name].int_variant()
    A, B = problem_operands(p)
    C = run(A, B)
    C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
    check(C, C64, None, exact=True, what=p.name)


@pytest.mark.parametrize("dist", ["real", "int"])
def test_named_problem_4096_every_element(dist):
    """The benchmark's workload, in the launch the benchmark times: every
    element against the oracle (real inputs within the bound, integer inputs
    exactly)."""
    p = PROBLEMS["square_4096"] if dist == "real" else PROBLEMS["square_4096"].int_variant()
    A, B = problem_operands(p)
    C = run(A, B)
    C64, bound = oracle_named(p.name)
    worst = check(C, C64, None if dist == "int" else bound, exact=(dist == "int"), what=p.name)
    print(f"{p.name}: worst |err|/bound = {worst:.3e}")


@pytest.mark.parametrize("dist", ["real", "int"])
def test_named_problem_8192_sampled_rows(dist):
    """8192^3 (the full oracle would take over half a minute on the host):
    whole rows on every tile edge plus random rows, and single entries on the
    tile-edge columns of those rows."""
    p = PROBLEMS["square_8192"] if dist == "real" else PROBLEMS["square_8192"].int_variant()
    A, B = problem_operands(p)
    C = run(A, B)
    rows = sample_rows(p.M, n_random=8, seed=p.seed)
    C64, bound = oracle.gemm_rows_f64(A.numpy(), B.numpy(), rows)
    check(C[rows], C64, bound, exact=(dist == "int"), what=f"{p.name} rows")
    ii = np.repeat(rows, 4)
    jj = np.tile(np.array([0, 127, 128, p.N - 1]), rows.size)
    ce, be = oracle.gemm_entries_f64(A.numpy(), B.numpy(), ii, jj)
    check(C[ii, jj][None, :], ce[None, :], be[None, :], exact=(dist == "int"), what=f"{p.name} entries")


# ---------------------------------------------------------------- every forced variant

VARIANTS = (
    [dict(producer=1, math=m, stages=s, split_k=1, multicast=1) for m in (1, 2) for s in (1, 2, 3, 4, 5, 6)]
    + [dict(producer=pr, math=m, split_k=s, multicast=1) for pr in (1, 2) for m in (1, 2) for s in (2, 3, 4, 8)]
    + [dict(producer=2, math=m, stages=s, split_k=1) for m in (1, 2) for s in (2, 4)]
    + [dict(producer=pr, math=m, stream_k=2) for pr in (1, 2) for m in (1, 2)]
    + [dict(stream_k=2, stages=s) for s in (2, 6)]
    # tile order: row by row, and groups of 2 rows of tiles (the last group short)
    + [dict(group_m=gm) for gm in (1, 2)]
    + [dict(group_m=2, stream_k=2), dict(group_m=2, split_k=2), dict(group_m=2, producer=4),
       dict(group_m=2, tile_n=256, split_k=1)]
    # 16-deep K slices (the transposing producer): stages, schedules
    + [dict(tile_k=16, stages=s) for s in (2, 3, 4, 6)]
    + [dict(tile_k=16, split_k=2), dict(tile_k=16, stream_k=1, split_k=1), dict(tile_k=16, stream_k=2),
       dict(tile_k=16, group_m=1)]
    # loader warps (operands of any alignment; here aligned)
    + [dict(producer=7, stages=s) for s in (2, 3, 4)]
    + [dict(producer=7, split_k=2), dict(producer=7, stream_k=1, split_k=1), dict(producer=7, group_m=1)]
    # residue-class tensor maps (operands of any alignment; here aligned)
    + [dict(producer=8, stages=s) for s in (2, 3, 4)]
    + [dict(producer=8, split_k=2), dict(producer=8, stream_k=1, split_k=1), dict(producer=8, group_m=1)]
    # A's slices with the L2 evict-last policy
    + [dict(l2_hint=h) for h in (1, 2, 3, 4)] + [dict(l2_hint=2, group_m=2, stream_k=2), dict(l2_hint=3, producer=1)]
    # producer warpgroup with the setmaxnreg register split
    + [dict(producer=3, math=m, stages=s, split_k=1, multicast=1) for m in (1, 2) for s in (1, 4, 6)]
    + [dict(producer=3, math=2, split_k=s, multicast=1) for s in (2, 4)]
    + [dict(producer=3, math=m, stream_k=2) for m in (1, 2)]
    # 128 x 256 tiles (8 x 16 accumulators per thread)
    + [dict(tile_n=256, math=m, stages=s, split_k=1) for m in (1, 2) for s in (2, 3, 4)]
    + [dict(tile_n=256, split_k=s) for s in (2, 4)]
    + [dict(tile_n=256, stream_k=2, math=m) for m in (1, 2)]
    # fused producer: 4-warp CTAs on 128 x 64 tiles, two per SM
    + [dict(producer=4, math=m, stages=s, split_k=1) for m in (1, 2) for s in (2, 3, 4)]
    + [dict(tile_n=64, stream_k=2, math=m) for m in (1, 2)]
    + [dict(tile_n=64, stream_k=2, stages=2)]
    # A transposed in shared memory by a second producer warp
    + [dict(producer=5, math=m, stages=s, split_k=1) for m in (1, 2) for s in (2, 3, 4)]
    + [dict(producer=5, stream_k=2), dict(producer=5, split_k=3)]
)


def _vid(v):
    return "-".join(f"{k}{v[k]}" for k in sorted(v))


@pytest.mark.parametrize("opt", VARIANTS, ids=_vid)
def test_forced_variant(opt):
    # 300 x 500 x 700: ragged against every tile size, several tiles per axis,
    # 22 K slices (uneven over every split), 16-byte aligned rows (TMA allowed).
    A, B = make_operands(300, 500, 700, "uniform", 31)
    C = run(A, B, **opt)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=_vid(opt))
    Ai, Bi = make_operands(300, 500, 700, "int", 32)
    Ci = run(Ai, Bi, **opt)
    check(Ci, oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None, exact=True, what=_vid(opt) + " int")


@pytest.mark.parametrize("tail", [2, 3, 4, 8])
def test_tail_split(tail):
    """169 output tiles (13 x 13) on 152 SMs: one full wave plus 17 tiles that
    run as a second launch split along K; K = 1040 is ragged (33 K slices)."""
    M = N = 1664
    K = 1040
    A, B = make_operands(M, N, K, "uniform", 41)
    dA, dB = to_device(A), to_device(B)
    C = g.sgemm_f32_ex(dA, dB, tail_split=tail).cpu().numpy()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=f"tail {tail}")
    Ai, Bi = make_operands(M, N, K, "int", 42)
    Ci = g.sgemm_f32_ex(to_device(Ai), to_device(Bi), tail_split=tail).cpu().numpy()
    check(Ci, oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None, exact=True, what=f"tail {tail} int")


@pytest.mark.parametrize("tile_n", [128, 64])
@pytest.mark.parametrize("name", ["square_2048", "ragged_1023x1025x1027", "flat_4096x4096x256",
                                  "skinny_8192x128x8192"])
def test_stream_k_every_element(name, tile_n):
    """Stream-K: one CTA per SM (two with the fused producer's 128 x 64
    tiles), tiles shared between CTAs finished through the workspace; every
    element against the oracle, and bitwise repeatable."""
    p = PROBLEMS[name]
    A, B = problem_operands(p)
    opt = dict(stream_k=2, tile_n=tile_n)
    if tile_n == 64:
        opt["repack"] = 2  # the fused producer needs tensor-map-readable operands
    C = run(A, B, **opt)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=f"{name} stream-K n{tile_n}")
    assert np.array_equal(C, run(A, B, **opt))
    Ai, Bi = problem_operands(p.int_variant())
    check(run(Ai, Bi, **opt), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None,
          exact=True, what=f"{name} stream-K n{tile_n} int")


@pytest.mark.parametrize("dist", ["real", "int"])
def test_stream_k_sampled_rows_4096(dist):
    p = PROBLEMS["square_4096"] if dist == "real" else PROBLEMS["square_4096"].int_variant()
    A, B = problem_operands(p)
    C = run(A, B, stream_k=2)
    rows = sample_rows(p.M, n_random=8, seed=p.seed)
    C64, bound = oracle.gemm_rows_f64(A.numpy(), B.numpy(), rows)
    check(C[rows], C64, bound, exact=(dist == "int"), what=f"{p.name} stream-K rows")


@pytest.mark.parametrize("group_m", [1, 5, 7, 16, 24, 100])
def test_tile_order_every_element(group_m):
    # 3000 x 2500: 24 x 20 tiles of 128 x 128, two whole data-parallel waves of
    # 152 CTAs then stream-K units; groups of 5 and 7 rows leave a short last
    # group, 24 and 100 make one group.  Every output tile must be computed
    # once, whatever the order.
    A, B = make_operands(3000, 2500, 256, "uniform", 41)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, group_m=group_m), C64, bound, exact=False, what=f"group_m={group_m}")
    Ai, Bi = make_operands(3000, 2500, 256, "int", 42)
    check(run(Ai, Bi, group_m=group_m), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None,
          exact=True, what=f"group_m={group_m} int")


@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (1000, 1001, 1000), (640, 768, 2000), (4096, 4096, 4096)])
def test_sixteen_deep_slices_every_element(shape):
    """tile_k = 16 (64-byte swizzled A slices, 16 k per stage) against the
    oracle on square, ragged (K = 1000: a last slice of 8 k) and stream-K
    shapes; integer inputs exactly."""
    M, N, K = shape
    A, B = make_operands(M, N, K, "uniform", 43)
    ldb = (N + 3) // 4 * 4  # 16-byte rows of B: the tensor-map kernels
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, ldb=ldb, tile_k=16), C64, bound, exact=False, what=f"tile_k=16 {shape}")
    Ai, Bi = make_operands(M, N, K, "int", 44)
    check(run(Ai, Bi, ldb=ldb, tile_k=16), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None,
          exact=True, what=f"tile_k=16 {shape} int")


def test_sixteen_deep_slices_refusals():
    A, B = make_operands(512, 512, 512, "uniform", 45)
    for bad in (dict(tile_k=8), dict(tile_k=64), dict(tile_k=16, producer=1), dict(tile_k=16, stages=5),
                dict(tile_k=16, tile_n=256)):
        with pytest.raises(g.SgemmError) as e:
            run(A, B, **bad)
        assert e.value.status == 1, bad


def test_forced_tma_rejects_unaligned_rows():
    A, B = make_operands(64, 64, 63, "uniform", 1)
    with pytest.raises(g.SgemmError) as e:
        run(A, B, producer=1)
    assert e.value.status == 1


def test_multicast_form_is_not_built():
    # The cluster-multicast form of the operand loads is not in the library:
    # asking for it is refused before any launch, for every tile width.
    A, B = make_operands(512, 512, 256, "uniform", 2)
    for extra in (dict(), dict(tile_n=256), dict(producer=3)):
        with pytest.raises(g.SgemmError) as e:
            run(A, B, multicast=2, split_k=1, **extra)
        assert e.value.status == 5
    # 0 and 1 both mean "off"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, multicast=1), C64, bound, exact=False, what="multicast=1")


# ---------------------------------------------------------------- ragged shapes, edges, layouts

# Small shapes run on the small-problem kernel when nothing is forced;
# a_layout = 1 (A as stored) keeps the automatic choice among the 128 x 128
# FFMA kernels, so that their edge handling is covered at the same shapes.
AUTO_FORMS = [dict(), dict(a_layout=1)]


@pytest.mark.parametrize("opt", AUTO_FORMS, ids=["auto", "ffma128"])
def test_ragged_shapes_sweep(opt):
    rng = np.random.default_rng(1234)
    for t in range(24):
        M, N, K = (int(x) for x in rng.integers(1, 301, size=3))
        A, B = make_operands(M, N, K, "normal", 500 + t)
        C = run(A, B, **opt)
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
        check(C, C64, bound, exact=False, what=f"{M}x{N}x{K} {opt}")


@pytest.mark.parametrize("opt", AUTO_FORMS + [dict(producer=6)], ids=["auto", "ffma128", "small"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (1, 1, 10000), (1, 300, 7), (300, 1, 7), (129, 127, 1), (5, 3, 2),
                                   (128, 128, 32), (129, 129, 33), (256, 256, 8192)])
def test_small_and_degenerate_shapes(shape, opt):
    M, N, K = shape
    A, B = make_operands(M, N, K, "uniform", 77)
    C = run(A, B, **opt)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=f"{shape} {opt}")


@pytest.mark.parametrize("opt", AUTO_FORMS + [dict(producer=6)], ids=["auto", "ffma128", "small"])
def test_k_zero_writes_zeros(opt):
    A = torch.empty((37, 0))
    B = torch.empty((0, 45))
    C = run(A, B, **opt)
    assert np.array_equal(C, np.zeros((37, 45), np.float32))


@pytest.mark.parametrize("shape", [(0, 5, 3), (5, 0, 3), (0, 0, 0)])
def test_empty_output_leaves_memory_untouched(shape):
    M, N, K = shape
    dA = torch.ones((M, K), device="cuda")
    dB = torch.ones((K, N), device="cuda")
    guard = torch.full((16,), 7.0, device="cuda")
    dC = guard[:0].view(M, N) if M * N == 0 else None
    g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    assert torch.all(guard == 7.0)


def test_leading_dimensions_and_guard_bands():
    """Padded rows hold NaN (never read); C's row padding and the floats around
    C hold a sentinel (never written)."""
    M, N, K = 200, 150, 90
    A, B = make_operands(M, N, K, "uniform", 8)
    lda, ldb, ldc = 96, 156, 160
    dA, dB = to_device(A, lda), to_device(B, ldb)
    sentinel = -12345.0
    guard = 64
    store = torch.full((guard + M * ldc + guard,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what="padded")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[-guard:] == sentinel)
    pad = store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy()
    assert np.all(pad == sentinel)


@pytest.mark.parametrize("opt", [dict(), dict(producer=5, stages=3), dict(producer=5, stream_k=1, split_k=1),
                                 dict(producer=5, split_k=2), dict(producer=5, stages=4), dict(l2_hint=1),
                                 dict(producer=8), dict(producer=8, stages=3), dict(producer=8, stages=4)],
                         ids=["auto", "stages3", "plain-grid", "split2", "stages4-no-staging", "no-policy",
                              "res", "res-stages3", "res-stages4-no-staging"])
@pytest.mark.parametrize("c_offset,N", [(0, 1004), (0, 1001), (1, 1004)])
def test_tensor_map_stores_of_c_and_guard_bands(opt, c_offset, N):
    """The 128 x 128 kernels that write finished tiles of C through a staging
    tile and tensor-map stores (K of 128 slices or more, C 16-byte aligned,
    ldc % 4 == 0 and N % 4 == 0; with N = 1001, or c_offset = 1 making C's
    base misaligned, the same kernels store directly): outputs of 600 rows
    ragged against the tiles in both directions; C's row padding and the
    floats around C hold a sentinel that must survive."""
    M, K = 600, 4096
    A, B = make_operands(M, N, K, "uniform", 17)
    ldc, guard = 1012, 64 + c_offset
    sentinel = -12345.0
    store = torch.full((guard + M * ldc + 64,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    dA, dB = to_device(A), to_device(B, 1004)  # 16-byte rows of B: the tensor-map kernels
    if opt:
        g.sgemm_f32_ex(dA, dB, dC, **opt)
    else:
        assert g.describe(dA, dB, dC).startswith("tmax/")
        g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what=f"tma-store {opt} offset {c_offset}")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[guard + M * ldc:] == sentinel)
    pad = store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy()
    assert np.all(pad == sentinel)


@pytest.mark.parametrize("offsets", [(1, 0), (0, 3), (2, 1)])
@pytest.mark.parametrize("shape", [(190, 170, 260), (700, 900, 260)])
def test_unaligned_bases(offsets, shape):
    """Bases that are not 16-byte aligned: the small-problem kernel (plain
    loads) or, above its range, the residue-class tensor maps."""
    oa, ob = offsets
    M, N, K = shape
    A, B = make_operands(M, N, K, "uniform", 9)
    dA, dB = to_device(A, offset=oa), to_device(B, offset=ob)
    d = g.describe(dA, dB)
    assert d.startswith("small") if M < 256 else d.endswith("/res/ec4")
    C = g.sgemm_f32(dA, dB)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.cpu().numpy(), C64, bound, exact=False, what=f"offsets {offsets}")


def test_unaligned_output():
    M, N, K = 70, 90, 50
    A, B = make_operands(M, N, K, "uniform", 10)
    store = torch.full((1 + M * N,), float("nan"), device="cuda")
    dC = store[1:].view(M, N)
    g.sgemm_f32(to_device(A), to_device(B), dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what="unaligned C")


def test_split_k_is_deterministic():
    A, B = make_operands(256, 256, 8192, "normal", 11)
    dA, dB = to_device(A), to_device(B)
    outs = []
    for _ in range(3):
        C = g.sgemm_f32_ex(dA, dB, split_k=4)
        torch.cuda.synchronize()
        outs.append(C.cpu().numpy())
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_side_streams():
    A, B = make_operands(384, 320, 448, "uniform", 12)
    dA, dB = to_device(A), to_device(B)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    C1 = torch.empty((384, 320), device="cuda")
    C2 = torch.empty((384, 320), device="cuda")
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    g.sgemm_f32(dA, dB, C1, stream=s1)
    g.sgemm_f32_ex(dA, dB, C2, stream=s2, split_k=2)
    s1.synchronize()
    s2.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C1.cpu().numpy(), C64, bound, exact=False, what="stream 1")
    check(C2.cpu().numpy(), C64, bound, exact=False, what="stream 2")


def test_host_buffer_entry():
    A, B = make_operands(130, 260, 390, "uniform", 13)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.numpy(), C64, bound, exact=False, what="host buffers")


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_host_buffer_entry_row_blocks(dist):
    """2048 x 1536 x 2048 (2^34 flop): four K chunks, the last in four row
    blocks, whose copies overlap the products; every element."""
    A, B = make_operands(2048, 1536, 2048, dist, 14)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C.numpy(), C64, bound, exact=(dist == "int"), what=f"host row blocks {dist}")


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_host_buffer_entry_ragged_chunks(dist):
    """1500 x 1300 x 2500: K chunks of 64, 320, 864 and 1252, the last in row
    blocks of 896, 256, 128, 128 and 92 rows (the last one ragged against
    the 128-row tiles); every element."""
    A, B = make_operands(1500, 1300, 2500, dist, 16)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C.numpy(), C64, bound, exact=(dist == "int"), what=f"host ragged chunks {dist}")


def test_host_buffer_entry_4096_every_element():
    """The end-to-end leg of the benchmark (4096^3 through the host-buffer
    entry on pinned buffers): every element against the oracle."""
    p = PROBLEMS["square_4096"]
    A, B = problem_operands(p)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle_named(p.name)
    check(C.numpy(), C64, bound, exact=False, what="host 4096")


@pytest.mark.parametrize("dist", ["int", "uniform"])
def test_host_buffer_entry_tall_pipelined(dist):
    """262144 x 256 x 512 (2^36 flop) through the host-buffer entry: K chunks
    of 64, 192 and 256 columns (the 1/32 boundary rounds down to nothing and
    drops out), the last in row blocks of 163840, 49152, 32768 and 16384
    rows; every element, integer inputs exactly."""
    M, N, K = 1 << 18, 256, 512
    A, B = make_operands(M, N, K, dist, 63)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C.numpy(), C64, bound, exact=(dist == "int"), what=f"host tall {dist}")


def test_host_buffer_entry_pitched_and_pageable():
    """Padded host rows (odd pitches) and pageable (not pinned) memory on the
    row-block path; the padding of C is left untouched."""
    M, N, K = 1300, 700, 2400
    A, B = make_operands(M, N, K, "uniform", 15, lda=K + 3, ldb=N + 1)
    store = torch.full((M, N + 5), -7.0)
    out = store[:, :N]
    C = g.sgemm_f32_host(A, B, out)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.numpy(), C64, bound, exact=False, what="host pitched")
    assert torch.all(store[:, N:] == -7.0)


def test_variant_choice():
    def desc(M, N, K):
        return g.describe(torch.empty((M, K), device="cuda"), torch.empty((K, N), device="cuda"))

    # A transposed in shared memory by the transposing producer warps, at
    # every size (the copy of A transposed in HBM only when forced)
    assert desc(4096, 4096, 4096).startswith("tmax/") and desc(2048, 2048, 2048).startswith("tmax/")
    assert desc(8192, 128, 8192).startswith("tmax/") and desc(1024, 1024, 1024).startswith("tmax/")
    assert desc(8192, 8192, 8192).startswith("tmax/") and "/at" not in desc(8192, 8192, 8192)
    assert "/s1/" in desc(4096, 4096, 4096) and "/sk" in desc(4096, 4096, 4096)  # stream-K
    assert "/tail" not in desc(4096, 4096, 4096)  # the tail split is opt-in
    assert "/sk" in desc(8192, 128, 8192) and "/sk" in desc(128, 8192, 16384)
    # small products (2MNK <= 2^28, 128 x 128 tiles at most a quarter of the
    # SMs): the 32 x 32-tile kernel
    assert desc(256, 256, 256) == "small/t32/w8" and desc(512, 512, 512) == "small/t32/w8"
    assert desc(300, 500, 701) == "small/t32/w8" and desc(64, 64, 64) == "small/t32/w8"
    assert desc(640, 640, 640).startswith("tmax/") and desc(1024, 1024, 128).startswith("tmax/")
    # 1027-float rows are not 16-byte multiples: below 2MNK = 2^35 the
    # residue-class tensor maps read the rows in place; larger products
    # repack them into pitched rows first
    # (and N mod 128 = 1 .. 4 columns past the last full column of tiles are
    # computed with that column: "/ec<columns>")
    assert desc(1023, 1025, 1027).startswith("tmax/") and desc(1023, 1025, 1027).endswith("/res/ec1")
    assert desc(700, 900, 701).startswith("tmax/") and desc(700, 900, 701).endswith("/res/ec4")
    assert desc(2048, 2049, 2048).endswith("/res/ec1") and desc(700, 901, 701).endswith("/res")
    assert desc(4096, 4097, 4096).endswith("/repackB/ec1") and desc(8192, 8193, 8192).endswith("/repackB/ec1")
    assert "/ec" not in desc(4096, 4096, 4096) and "/ec" not in desc(127, 129, 4096)


# ---------------------------------------------------------------- A's layout

@pytest.mark.parametrize("shape", [(300, 500, 700), (257, 190, 333), (129, 130, 4), (1, 700, 64), (513, 64, 1000)])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_forced_transposed_a(shape, dist):
    """a_layout = 2: A copied transposed (pitch M rounded up to 4) and read by
    the transposed-A kernel, whose threads own rows 16*(i/4) + 4*tm + i%4."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 95)
    C = run(A, B, a_layout=2)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C, C64, bound, exact=(dist == "int"), what=f"a_layout 2 {shape} {dist}")


@pytest.mark.parametrize("opt", [dict(a_layout=2, stream_k=2), dict(a_layout=2, stream_k=1, split_k=1),
                                 dict(a_layout=2, split_k=3), dict(a_layout=1), dict(a_layout=2, tile_n=256),
                                 dict(a_layout=2, tile_n=256, stream_k=2)])
def test_transposed_a_schedules(opt):
    """The transposed-A kernel under each schedule (stream-K, plain grid,
    cluster split-K), and a_layout = 1 (A as stored) on a size that would
    otherwise be transposed."""
    A, B = make_operands(700, 900, 1100, "uniform", 96)
    C = run(A, B, **opt)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C, C64, bound, exact=False, what=str(opt))


def test_transposed_a_rejects_forced_kernel_choices():
    A, B = make_operands(128, 128, 64, "uniform", 97)
    dA, dB = to_device(A), to_device(B)
    for bad in (dict(a_layout=2, producer=2), dict(a_layout=2, tile_n=64), dict(a_layout=3)):
        with pytest.raises(g._lib.SgemmError):
            g.sgemm_f32_ex(dA, dB, **bad)


# ---------------------------------------------------------------- repacking

@pytest.mark.parametrize("case", [
    # (M, N, K, lda, ldb, offset A, offset B): misaligned A only, B only, both,
    # and misaligned bases with aligned pitches
    (300, 500, 701, 701, 500, 0, 0),
    (300, 501, 700, 700, 501, 0, 0),
    (257, 333, 385, 387, 335, 0, 0),
    (200, 256, 260, 260, 256, 1, 2),
])
def test_forced_repack(case):
    M, N, K, lda, ldb, oa, ob = case
    for dist, seed in (("uniform", 91), ("int", 92)):
        A, B = make_operands(M, N, K, dist, seed)
        dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
        C = g.sgemm_f32_ex(dA, dB, repack=2)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"repack {case} {dist}")


def test_ragged_problem_cp_async():
    """The ragged problem on the cp.async producer (forced): 4-byte copies of
    the misaligned rows."""
    p = PROBLEMS["ragged_1023x1025x1027"]
    A, B = problem_operands(p)
    dA, dB = to_device(A), to_device(B)
    C = g.sgemm_f32_ex(dA, dB, producer=2)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.cpu().numpy(), C64, bound, exact=False, what="ragged, cp.async")
    Ai, Bi = problem_operands(p.int_variant())
    Ci = g.sgemm_f32_ex(to_device(Ai), to_device(Bi), producer=2)
    torch.cuda.synchronize()
    check(Ci.cpu().numpy(), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None, exact=True,
          what="ragged int, cp.async")


def test_repacked_large_ragged_sampled_rows():
    """2047 x 2049 x 2051 with both operands repacked (forced): sampled full
    rows against the oracle."""
    M, N, K = 2047, 2049, 2051
    A, B = make_operands(M, N, K, "uniform", 93)
    dA, dB = to_device(A), to_device(B)
    C = g.sgemm_f32_ex(dA, dB, repack=2)
    torch.cuda.synchronize()
    rows = sample_rows(M, n_random=8, seed=93)
    C64, bound = oracle.gemm_rows_f64(A.numpy(), B.numpy(), rows)
    check(C.cpu().numpy()[rows], C64, bound, exact=False, what="2047x2049x2051 rows")


# ---------------------------------------------------------------- bounded waits

def test_timeout_is_reported_and_recovers():
    """The producer of one CTA skips a K slice; its consumers' bounded wait
    expires, the kernel returns, and the status word says so.  The next call is
    unaffected."""
    A, B = make_operands(128, 256, 256, "uniform", 14)
    dA, dB = to_device(A), to_device(B)
    assert g.check_status() == 0
    for producer in (1, 2, 4, 5, 7):
        g.sgemm_f32_ex(dA, dB, producer=producer, split_k=1, debug_skip_stage=3, timeout_ns=20_000_000)
        assert g.check_status() == 4
        g.sgemm_f32_ex(dA, dB, producer=producer, stream_k=2, debug_skip_stage=1, timeout_ns=20_000_000)
        assert g.check_status() == 4
    C = g.sgemm_f32(dA, dB)
    assert g.check_status() == 0
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.cpu().numpy(), C64, bound, exact=False, what="after timeout")


# ---------------------------------------------------------------- CUDA graphs

def test_cuda_graph_capture_and_replay():
    """The entries enqueue only stream-ordered work (pool allocation and free,
    a memset, kernels), so a call can be captured in a CUDA graph and
    replayed; each replay recomputes from the current inputs."""
    M, N, K = 1024, 768, 1536  # stream-K: the workspace and flags are captured too
    A, B = make_operands(M, N, K, "uniform", 16)
    dA, dB = to_device(A), to_device(B)
    dC = torch.empty((M, N), device="cuda")
    dG = torch.empty((M, N), device="cuda")
    g.sgemm_f32(dA, dB, dC)  # first call on the device outside the capture (one-time set-up)
    g.sgemm_f32_gemm(dA, dB, dG, alpha=2.0, beta=0.0)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    dN = torch.empty((M, N), device="cuda")
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.sgemm_f32(dA, dB, dC, stream=s)
            g.sgemm_f32_gemm(dA, dB, dG, alpha=2.0, beta=0.0, stream=s)
            g.sgemm_f32_noalloc(dA, dB, dN, stream=s)
    # Eager calls on the same stream between replays take the stream's own
    # stream-K scratch (sequence-numbered flags); the graph's calls keep the
    # workspaces and memsets recorded with them.
    E1, E2 = make_operands(M, N, K, "int", 19)
    dE1, dE2 = to_device(E1), to_device(E2)
    dE, dEn = torch.empty((M, N), device="cuda"), torch.empty((M, N), device="cuda")
    E64, _ = oracle.gemm_f64(E1.numpy(), E2.numpy(), with_bound=False)
    for seed in (17, 18, 20):
        A2, B2 = make_operands(M, N, K, "uniform", seed)
        dA.copy_(A2)
        dB.copy_(B2)
        for X in (dC, dG, dN, dE, dEn):
            X.fill_(float("nan"))
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            g.sgemm_f32(dE1, dE2, dE, stream=s)
            graph.replay()
            g.sgemm_f32_noalloc(dE1, dE2, dEn, stream=s)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A2.numpy(), B2.numpy())
        check(dC.cpu().numpy(), C64, bound, exact=False, what=f"graph replay {seed}")
        check(dG.cpu().numpy(), 2.0 * C64, 2.0 * bound, exact=False, what=f"graph replay gemm {seed}")
        check(dN.cpu().numpy(), C64, bound, exact=False, what=f"graph replay noalloc {seed}")
        check(dE.cpu().numpy(), E64, None, exact=True, what=f"eager between replays {seed}")
        check(dEn.cpu().numpy(), E64, None, exact=True, what=f"eager noalloc between replays {seed}")
    assert g.check_status() == 0


# ---------------------------------------------------------------- stream-K scratch kept per stream

# Shapes on the stream-K schedule with different CTA runs (so that different
# CTAs publish partial tiles from one call to the next).
STREAM_K_SHAPES = [(700, 900, 1100), (1024, 768, 1536), (640, 1300, 900), (1500, 300, 2000)]


@pytest.mark.parametrize("fn", ["sgemm_f32", "sgemm_f32_noalloc"])
def test_stream_k_scratch_back_to_back(fn):
    """Calls on one stream reuse the same stream-K flags without zeroing them:
    each call waits for its own sequence number, so flags left by an earlier
    call (another schedule, other inputs) never match.  Integer inputs, all
    calls enqueued back to back before one synchronisation, every result
    exact."""
    call = getattr(g, fn)
    cases = []
    for t, (M, N, K) in enumerate(STREAM_K_SHAPES * 2):
        A, B = make_operands(M, N, K, "int", 600 + t)
        dA, dB = to_device(A), to_device(B)
        assert "/sk" in g.describe(dA, dB)
        cases.append((A, B, dA, dB, torch.full((M, N), float("nan"), device="cuda")))
    torch.cuda.synchronize()
    for _, _, dA, dB, dC in cases:
        call(dA, dB, dC)
    torch.cuda.synchronize()
    for A, B, _, _, dC in cases:
        C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
        check(dC.cpu().numpy(), C64, None, exact=True, what=f"{fn} back to back {tuple(dC.shape)}")


def test_stream_k_scratch_from_many_host_threads():
    """8 host threads, each with a stream of its own, 4 stream-K calls each,
    all at once: the library's per-device table of stream-K scratch is shared
    by the threads (under its lock), and each stream's calls use its own
    scratch with their own sequence numbers."""
    import threading

    M, N, K = 512, 640, 700
    cases = []
    for t in range(8):
        row = []
        for i in range(4):
            A, B = make_operands(M, N, K, "int", 800 + 4 * t + i)
            row.append((A, B, to_device(A), to_device(B), torch.full((M, N), float("nan"), device="cuda")))
        cases.append(row)
    assert "/sk" in g.describe(cases[0][0][2], cases[0][0][3])
    torch.cuda.synchronize()
    errors = []

    def work(t):
        try:
            s = torch.cuda.Stream()
            for _, _, dA, dB, dC in cases[t]:
                g.sgemm_f32(dA, dB, dC, stream=s)
            s.synchronize()
        except Exception as e:  # reported below, in the test's own thread
            errors.append(e)

    threads = [threading.Thread(target=work, args=(t,)) for t in range(len(cases))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    for row in cases:
        for A, B, _, _, dC in row:
            C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
            check(dC.cpu().numpy(), C64, None, exact=True, what="host threads")
    assert g.check_status() == 0


def test_stream_k_scratch_more_streams_than_entries():
    """20 streams, two calls each, all in flight together: the library keeps
    stream-K scratch for 16 streams, so entries move to new streams (whose
    work first waits for the entry's last call on its old stream)."""
    M, N, K = 512, 640, 700
    streams = [torch.cuda.Stream() for _ in range(20)]
    cases = []
    for t in range(2 * len(streams)):
        A, B = make_operands(M, N, K, "int", 700 + t)
        cases.append((A, B, to_device(A), to_device(B), torch.full((M, N), float("nan"), device="cuda")))
    assert "/sk" in g.describe(cases[0][2], cases[0][3])
    torch.cuda.synchronize()
    for t, (_, _, dA, dB, dC) in enumerate(cases):
        g.sgemm_f32(dA, dB, dC, stream=streams[t % len(streams)])
    torch.cuda.synchronize()
    for A, B, _, _, dC in cases:
        C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
        check(dC.cpu().numpy(), C64, None, exact=True, what="many streams")
    assert g.check_status() == 0


# ---------------------------------------------------------------- loader warps

@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (700, 900, 701), (1500, 1300, 2000)])
def test_loader_warps_match_tensor_map_kernel_bitwise(shape):
    """Aligned operands: the loader warps feed the consumers the same slices
    as the tensor maps, so the result equals the transposing-producer
    kernel's bit for bit (same schedule, same order of multiply-adds; the
    loader warps have no thin-edge form, so N = 900 runs both with a column
    of tiles for its last 4 columns)."""
    M, N, K = shape
    A, B = make_operands(M, N, K, "normal", 47)
    ldb = (N + 3) // 4 * 4
    lda = (K + 3) // 4 * 4
    C_ldg = run(A, B, lda=lda, ldb=ldb, producer=7)
    C_tma = run(A, B, lda=lda, ldb=ldb, producer=5, edge=1)
    assert np.array_equal(C_ldg, C_tma)


@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 2), (3, 1), (2, 3)])
@pytest.mark.parametrize("pads", [(0, 0), (1, 3), (5, 2)])
def test_loader_warps_any_alignment_every_element(offsets, pads):
    """Bases 0-3 floats off a 16-byte boundary and rows of any length (pads
    added to K and N): every element against the oracle, integer inputs
    exactly; M, N, K ragged against the tiles and slices."""
    M, N, K = 777, 1153, 611
    oa, ob = offsets
    lda, ldb = K + pads[0], N + pads[1]
    for dist in ("uniform", "int"):
        A, B = make_operands(M, N, K, dist, 48)
        dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
        C = g.sgemm_f32_ex(dA, dB, producer=7)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"ldg {offsets} {pads} {dist}")



# ---------------------------------------------------------------- residue-class tensor maps

@pytest.mark.parametrize("shape", [(1024, 1024, 1024), (700, 900, 701), (1500, 1300, 2000)])
def test_residue_maps_match_tensor_map_kernel_bitwise(shape):
    """Aligned operands: the four class maps per operand bring the same
    slices as one map, so the result equals the transposing-producer
    kernel's bit for bit (same schedule, same order of multiply-adds)."""
    M, N, K = shape
    A, B = make_operands(M, N, K, "normal", 49)
    ldb = (N + 3) // 4 * 4
    lda = (K + 3) // 4 * 4
    C_res = run(A, B, lda=lda, ldb=ldb, producer=8)
    C_tma = run(A, B, lda=lda, ldb=ldb, producer=5)
    assert np.array_equal(C_res, C_tma)


@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 2), (3, 1), (2, 3)])
@pytest.mark.parametrize("pads", [(0, 0), (1, 3), (5, 2), (2, 0)])
def test_residue_maps_any_alignment_every_element(offsets, pads):
    """Bases 0-3 floats off a 16-byte boundary and rows of any length (pads
    added to K and N, so that the four classes' offsets are all different,
    pairwise equal or all equal): every element against the oracle, integer
    inputs exactly; M, N, K ragged against the tiles and slices."""
    M, N, K = 777, 1153, 611
    oa, ob = offsets
    lda, ldb = K + pads[0], N + pads[1]
    for dist in ("uniform", "int"):
        A, B = make_operands(M, N, K, dist, 50)
        dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
        C = g.sgemm_f32_ex(dA, dB, producer=8)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"res {offsets} {pads} {dist}")


@pytest.mark.parametrize("shape", [(4, 1, 4), (5, 3, 7), (7, 130, 5), (4, 129, 33), (131, 257, 4), (6, 6, 97)])
@pytest.mark.parametrize("opt", [dict(producer=8), dict(producer=8, stream_k=1, split_k=1)])
def test_residue_maps_smallest_classes(shape, opt):
    """The fewest rows the classes allow (M, K = 4: one row of A and of B per
    class), classes of unequal length (M, K not multiples of 4), N below one
    16-byte block, K below one slice; pitches K + 1 and N + 1, bases off by
    one float."""
    M, N, K = shape
    for dist in ("uniform", "int"):
        A, B = make_operands(M, N, K, dist, 51)
        dA, dB = to_device(A, K + 1, offset=1), to_device(B, N + 1, offset=1)
        C = g.sgemm_f32_ex(dA, dB, **opt)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"res {shape} {opt} {dist}")


@pytest.mark.parametrize("name", ["ragged_1023x1025x1027", "square_1024"])
def test_residue_maps_named_problem_every_element(name):
    """The ragged problem (rows of 1027 and 1025 floats) read in place by the
    class maps, and an aligned one forced onto them; integer twins exactly."""
    p = PROBLEMS[name]
    for q in (p, p.int_variant()):
        A, B = problem_operands(q)
        C = run(A, B, producer=8)
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(q is p))
        check(C, C64, bound, exact=(q is not p), what=f"res {q.name}")


def test_residue_maps_rejections():
    """Classes need a row of A and of B each (M, K >= 4); the kernels have
    128 x 128 tiles, 32-deep slices, paired FMA, 2 to 4 stages; a forced copy
    contradicts the in-place read."""
    A, B = make_operands(8, 8, 8, "uniform", 52)
    dA, dB = to_device(A), to_device(B)
    for bad in (dict(stages=5), dict(math=1), dict(tile_n=256), dict(tile_k=16), dict(repack=2)):
        with pytest.raises(g._lib.SgemmError):
            g.sgemm_f32_ex(dA, dB, producer=8, **bad)
    for M, K in ((3, 8), (8, 3)):
        A, B = make_operands(M, 8, K, "uniform", 53)
        with pytest.raises(g._lib.SgemmError):
            g.sgemm_f32_ex(to_device(A), to_device(B), producer=8)


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_residue_maps_with_tensor_map_stores(dist):
    """Misaligned A (rows of 4097 floats) and B (rows of 1005) read in place by
    the class maps, with a K loop long enough (129 slices) for the finished
    tiles to go out by tensor-map stores into a 16-byte aligned C with padded
    rows; C's padding and the floats around it keep a sentinel."""
    M, N, K = 600, 1004, 4100
    A, B = make_operands(M, N, K, dist, 54)
    dA, dB = to_device(A, 4101, offset=3), to_device(B, 1005, offset=2)
    ldc, guard, sentinel = 1012, 64, -12345.0
    store = torch.full((guard + M * ldc + guard,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    assert g.describe(dA, dB, dC).endswith("/res")
    g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(dC.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"res + tma store {dist}")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[-guard:] == sentinel)
    assert np.all(store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy() == sentinel)


def test_cuda_graph_capture_on_residue_class_maps():
    """A call on misaligned rows (the residue-class maps: four tensor maps per
    operand, encoded at capture with the operands' addresses) captured in a
    CUDA graph; each replay recomputes from the current contents."""
    M, N, K = 1023, 1025, 1027
    A, B = make_operands(M, N, K, "uniform", 57)
    dA, dB = to_device(A, offset=1), to_device(B, offset=2)
    dC = torch.empty((M, N), device="cuda")
    assert g.describe(dA, dB, dC).endswith("/res/ec1")  # (the edge's partial sums in the capture's workspace)
    g.sgemm_f32(dA, dB, dC)  # outside the capture first
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            g.sgemm_f32(dA, dB, dC, stream=s)
    for seed in (58, 59):
        A2, B2 = make_operands(M, N, K, "uniform", seed)
        dA.copy_(A2)
        dB.copy_(B2)
        dC.fill_(float("nan"))
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            graph.replay()
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A2.numpy(), B2.numpy())
        check(dC.cpu().numpy(), C64, bound, exact=False, what=f"graph replay on class maps {seed}")


# ---------------------------------------------------------------- thin column edge

@pytest.mark.parametrize("dist", ["uniform", "int"])
@pytest.mark.parametrize("b_rows", ["exact", "padded"])
@pytest.mark.parametrize("shape", [(1023, 1025, 1027), (2000, 130, 700), (3201, 515, 96), (1000, 644, 333),
                                   (128, 2050, 4096), (300, 516, 4096), (4, 1025, 65536), (129, 257, 8192)])
def test_thin_column_edge(shape, b_rows, dist):
    """N mod 128 = 1 .. 4 columns past the last full column of tiles,
    computed by the CTAs working on that column (B's edge values copied per
    slice by a transposing warp, the sums exchanged with the stream-K partial
    tiles): B's rows of N floats or padded to a 16-byte multiple (the
    residue-class maps wherever a row of A or B is not a 16-byte multiple,
    else the plain tensor maps); one column of tiles (N = 130), a last row of
    tiles holding one row and K of 3 slices (3201 x 515 x 96), one row of
    tiles with K = 4096, N = 516 with the tensor-map stores of C, four rows
    with K = 65536 (each edge tile's slices shared by every CTA) and two rows
    of tiles, the second holding one row, on two columns of tiles; every
    element, integer inputs exactly."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 64)
    ldb = N if b_rows == "exact" else (N + 3) // 4 * 4
    dA, dB = to_device(A), to_device(B, ldb)
    dC = to_device(torch.full((M, N), float("nan")))
    d = g.describe(dA, dB, dC)
    assert d.endswith(f"/ec{N % 128}") and ("/res" in d) == (ldb % 4 != 0 or K % 4 != 0), d
    g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(dC.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"edge {shape} ldb {ldb} {dist}")


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_thin_column_edge_with_whole_tiles(dist):
    """4096 x 1281 x 256: 32 x 10 tiles, two waves, so that the first 152
    tiles run whole (their edge sums stored directly) and the rest are dealt
    out as K-slice units (edge sums exchanged); every element."""
    M, N, K = 4096, 1281, 256
    A, B = make_operands(M, N, K, dist, 65)
    C = run(A, B)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C, C64, bound, exact=(dist == "int"), what=f"edge with whole tiles {dist}")


@pytest.mark.parametrize("c_offset", [0, 1])
def test_thin_column_edge_guard_bands(c_offset):
    """The edge columns' stores stop at N: C's rows padded to 1040 floats
    (and, with c_offset = 1, a misaligned base: the staged row stores) hold a
    sentinel past N = 1027 and around C that must survive."""
    M, N, K = 700, 1027, 900
    A, B = make_operands(M, N, K, "uniform", 66)
    ldc, guard, sentinel = 1040, 64 + c_offset, -12345.0
    store = torch.full((guard + M * ldc + 64,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    dA, dB = to_device(A), to_device(B)
    assert g.describe(dA, dB, dC).endswith("/ec3")
    g.sgemm_f32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what=f"edge guard bands {c_offset}")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[guard + M * ldc:] == sentinel)
    assert np.all(store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy() == sentinel)


@pytest.mark.parametrize("opt", [dict(edge=1), dict(edge=1, producer=8), dict(stages=3), dict(stages=4),
                                 dict(producer=8, stages=3), dict(repack=2), dict(math=1, repack=2), dict(group_m=1),
                                 dict(stream_k=1, split_k=1), dict(split_k=2), dict(tile_n=64, repack=2),
                                 dict(producer=2)])
def test_thin_column_edge_forced_choices(opt):
    """The edge fold under the other stage counts, repacked operands and
    row-by-row tile order; switched off (edge = 1: a ninth column of tiles)
    and not taken with scalar FFMA or without stream-K or the transposing
    producer (plain grid, cluster split-K, 128 x 64 tiles, cp.async)."""
    M, N, K = 1023, 1025, 1027
    A, B = make_operands(M, N, K, "int", 67)
    C = run(A, B, **opt)
    C64, _ = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)
    check(C, C64, None, exact=True, what=f"edge forced {opt}")


def test_thin_column_edge_option_is_checked():
    A, B = make_operands(300, 257, 300, "uniform", 68)
    with pytest.raises(g._lib.SgemmError):
        g.sgemm_f32_ex(to_device(A), to_device(B), edge=2)
    with pytest.raises(g._lib.SgemmError):
        g.sgemm_f32_ex(to_device(A), to_device(B), edge=-1)


@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_host_buffer_entry_thin_column_edge(dist):
    """4096 x 1025 x 2048 through the host-buffer entry (K chunks, the
    first a plain product of 256 x 2 units that computes the edge column with
    the last column of tiles, the later ones accumulating); every element."""
    A, B = make_operands(4096, 1025, 2048, dist, 69)
    C = g.sgemm_f32_host(A.pin_memory(), B.pin_memory())
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C.numpy(), C64, bound, exact=(dist == "int"), what=f"host edge {dist}")


# ---------------------------------------------------------------- extreme shapes

@pytest.mark.parametrize("shape,dist", [((1 << 20, 8, 64), "int"), ((8, 1 << 20, 64), "int"),
                                        ((1 << 20, 8, 64), "uniform"), ((128, 128, 1 << 20), "uniform")])
def test_extreme_shapes_every_element(shape, dist):
    """A million rows (8192 rows of tiles), a million columns (8192 columns
    of tiles, one tile row) and a million-deep K on one output tile (every
    SM's stream-K share of 32768 slices, one finishing CTA adding 151 partial
    tiles): every element against the oracle, integer inputs exactly."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 60)
    C = run(A, B)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C, C64, bound, exact=(dist == "int"), what=f"{shape} {dist}")


@pytest.mark.parametrize("dist", ["int", "uniform"])
def test_extreme_shape_on_residue_class_maps(dist):
    """A million rows of 63 floats times rows of 9 floats (neither a 16-byte
    multiple): the residue-class maps over 8192 rows of tiles."""
    M, N, K = 1 << 20, 9, 63
    A, B = make_operands(M, N, K, dist, 61)
    dA, dB = to_device(A), to_device(B)
    assert g.describe(dA, dB).endswith("/res")
    C = g.sgemm_f32(dA, dB)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"res extreme {dist}")
