"""GPU parity of the tensor-core entry (sgemm_3xtf32) against the CPU oracle.

Same contract as sgemm_f32: |C - C_oracle| <= 5e-5 * sum_k |A_ik||B_kj| for
every element on real-valued inputs, exact equality on integer-valued inputs.
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


# 0 = the automatic choice of sgemm_3xtf32; 1 = split-tile kernel; 2 =
# direct-A kernel; 3 = split-tile kernel on 128 x 256 tiles, K-slices of 16;
# 4 = the same with B's TF32 parts split and transposed in HBM first.
VARIANTS = [0, 1, 2, 3, 4]


def run(A, B, *, lda=None, ldb=None, ldc=None, variant=0, split_k=0):
    dA = to_device(A, lda)
    dB = to_device(B, ldb)
    dC = to_device(torch.full((A.shape[0], B.shape[1]), float("nan")), ldc)
    if variant or split_k:
        g.sgemm_3xtf32_ex(dA, dB, dC, variant=variant, split_k=split_k)
    else:
        g.sgemm_3xtf32(dA, dB, dC)
    torch.cuda.synchronize()
    return dC.cpu().numpy()


@pytest.mark.parametrize("variant", VARIANTS)
def test_one_tile_first(variant):
    """One output tile, one K slice: the smallest launch of each kernel."""
    A, B = make_operands(128, 128, 32, "uniform", 50)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, variant=variant), C64, bound, exact=False, what="128x128x32")
    Ai, Bi = make_operands(128, 128, 32, "int", 51)
    check(run(Ai, Bi, variant=variant), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None,
          exact=True, what="128x128x32 int")


FULL = ["square_256", "square_1024", "square_2048", "flat_4096x4096x256", "skinny_8192x128x8192",
        "skinny_128x8192x16384"]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", FULL)
def test_named_problem_every_element(name, variant):
    p = PROBLEMS[name]
    A, B = problem_operands(p)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    worst = check(run(A, B, variant=variant), C64, bound, exact=False, what=name)
    print(f"{name} variant {variant}: worst |err|/bound = {worst:.3e}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("name", FULL)
def test_named_problem_integer_exact(name, variant):
    p = PROBLEMS[name].int_variant()
    A, B = problem_operands(p)
    check(run(A, B, variant=variant), oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=False)[0], None, exact=True,
          what=p.name)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dist", ["real", "int"])
def test_named_problem_4096_every_element(dist, variant):
    p = PROBLEMS["square_4096"] if dist == "real" else PROBLEMS["square_4096"].int_variant()
    A, B = problem_operands(p)
    C64, bound = oracle_named(p.name)
    check(run(A, B, variant=variant), C64, None if dist == "int" else bound, exact=(dist == "int"), what=p.name)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("dist", ["real", "int"])
def test_named_problem_8192_sampled_rows(dist, variant):
    p = PROBLEMS["square_8192"] if dist == "real" else PROBLEMS["square_8192"].int_variant()
    A, B = problem_operands(p)
    C = run(A, B, variant=variant)
    rows = sample_rows(p.M, n_random=8, seed=p.seed)
    C64, bound = oracle.gemm_rows_f64(A.numpy(), B.numpy(), rows)
    check(C[rows], C64, bound, exact=(dist == "int"), what=f"{p.name} rows")


@pytest.mark.parametrize("variant", VARIANTS)
def test_ragged_problem_misaligned_rows(variant):
    """1023 x 1025 x 1027: rows of 1027 floats are not 16-byte multiples.  The
    automatic choice and variant 1 read them in place through residue-class
    tensor maps; variants 2-4 repack the operands into pitched rows first."""
    p = PROBLEMS["ragged_1023x1025x1027"]
    A, B = problem_operands(p)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, variant=variant), C64, bound, exact=False, what=p.name)
    Ai, Bi = problem_operands(p.int_variant())
    check(run(Ai, Bi, variant=variant), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0], None,
          exact=True, what=p.name + " int")


def test_small_misaligned_on_class_maps_or_ffma():
    """Small products with misaligned rows run the split-tile kernel on
    residue-class maps; with fewer than 4 rows of A (a class without a row)
    the FFMA kernels, under the same contract."""
    for M, N, K in ((200, 301, 333), (3, 301, 333), (200, 301, 3)):
        A, B = make_operands(M, N, K, "uniform", 94)
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
        check(run(A, B), C64, bound, exact=False, what=f"{M}x{N}x{K}")


@pytest.mark.parametrize("offsets", [(0, 0), (1, 0), (0, 2), (3, 1), (2, 3)])
@pytest.mark.parametrize("pads", [(0, 0), (1, 3), (5, 2), (2, 0)])
def test_residue_maps_any_alignment_every_element(offsets, pads):
    """Bases 0-3 floats off a 16-byte boundary and rows of any length: the
    split-tile kernel on residue-class maps (automatic below 2^30 flop, and
    with its K split over 2 CTAs: 700 x 900 x 611 has 48 tiles); every element
    against the oracle, integer inputs exactly."""
    M, N, K = 700, 900, 611
    oa, ob = offsets
    lda, ldb = K + pads[0], N + pads[1]
    for dist in ("uniform", "int"):
        A, B = make_operands(M, N, K, dist, 55)
        dA, dB = to_device(A, lda, offset=oa), to_device(B, ldb, offset=ob)
        C = g.sgemm_3xtf32(dA, dB)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"3xtf32 res {offsets} {pads} {dist}")


@pytest.mark.parametrize("split_k", [1, 2, 3, 4])
@pytest.mark.parametrize("shape", [(4, 5, 4), (7, 130, 33), (131, 257, 1027), (1023, 1025, 4099)])
def test_residue_maps_forced_splits_and_smallest_classes(split_k, shape):
    """Variant 1 on residue-class maps with the K split forced (1 = none, 2-4
    parts), from the fewest rows the classes allow (M, K = 4) to a product
    above 2^30 flop (forced variant 1 keeps the class maps there); pitches
    K + 1 and N + 3, bases off by one and two floats."""
    M, N, K = shape
    if split_k > (K + 31) // 32:
        pytest.skip("fewer K slices than parts")
    for dist in ("uniform", "int"):
        A, B = make_operands(M, N, K, dist, 56)
        dA, dB = to_device(A, K + 1, offset=1), to_device(B, N + 3, offset=2)
        C = g.sgemm_3xtf32_ex(dA, dB, variant=1, split_k=split_k)
        torch.cuda.synchronize()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
        check(C.cpu().numpy(), C64, bound, exact=(dist == "int"), what=f"3xtf32 res {shape} s{split_k} {dist}")


@pytest.mark.parametrize("variant", VARIANTS)
def test_ragged_shapes_sweep(variant):
    rng = np.random.default_rng(4321)
    for t in range(24):
        M, N = (int(x) for x in rng.integers(1, 301, size=2))
        K = 4 * int(rng.integers(1, 76))  # rows of A stay 16-byte multiples
        N4 = 4 * ((N + 3) // 4)
        A, B = make_operands(M, N4, K, "normal", 600 + t)
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
        check(run(A, B, variant=variant), C64, bound, exact=False, what=f"{M}x{N4}x{K}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(1, 4, 4), (1, 128, 10000), (129, 132, 36), (300, 4, 8), (256, 256, 8192),
                                   (130, 260, 100)])
def test_small_and_degenerate_shapes(shape, variant):
    M, N, K = shape
    A, B = make_operands(M, N, K, "uniform", 78)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, variant=variant), C64, bound, exact=False, what=str(shape))


@pytest.mark.parametrize("variant", VARIANTS)
def test_padded_rows_and_unaligned_output(variant):
    M, N, K = 200, 152, 96
    A, B = make_operands(M, N, K, "uniform", 79)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, lda=100, ldb=160, ldc=157, variant=variant), C64, bound, exact=False, what="padded")


def test_k_zero_writes_zeros():
    C = run(torch.empty((40, 0)), torch.empty((0, 36)))
    assert np.array_equal(C, np.zeros((40, 36), np.float32))


@pytest.mark.parametrize("variant", [3, 4])
@pytest.mark.parametrize("shape,split_k", [((1200, 4000, 1040), 2), ((1200, 3852, 1100), 2), ((1300, 4100, 1025), 2),
                                           ((1200, 4000, 2080), 0), ((1200, 4000, 300), 0)])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_wide_tiles_with_split_tail(shape, split_k, dist, variant):
    """Variants 3 and 4 with more 128 x 256 tiles than SMs: whole waves of
    wide tiles, then the last partial wave's tiles in a second launch with
    their K slices split between two CTAs, the second halves added into C
    afterwards (1200 x 4000: 160 wide tiles, the last wide column 160 floats
    wide; 1200 x 3852: the second half of each last wide tile lies wholly
    beyond N; K = 1040 / 1100 / 1025 ragged against the 16-deep slices, split
    32 + 33, 34 + 35 and 32 + 33 when forced (split_k = 2); K = 2080: split by
    the automatic rule; K = 300: below the rule's threshold, one launch of
    four waves)."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 81)
    exact = dist == "int"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=not exact)
    check(run(A, B, variant=variant, split_k=split_k), C64, bound, exact=exact,
          what=f"wide tail v{variant} {shape} {dist}")


@pytest.mark.parametrize("shape", [(256, 256, 2500), (128, 1024, 4096), (1000, 700, 2100), (300, 500, 1000),
                                   (300, 500, 500), (1023, 1025, 3001), (1024, 1024, 1024)])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_variant1_k_split(shape, dist):
    """Variant 1 with at most half as many tiles as SMs: each tile's nk K
    slices split among s CTAs when that takes 7 + 2 (s - 1) slices off each,
    the CTA of a tile that finishes last adding the parts (256 x 256 x
    2500: 4 tiles, s = 4, 79 slices in parts of 19 and 20; 128 x 1024 x 4096:
    s = 4; 1000 x 700 x 2100: 48 tiles, s = 3; 300 x 500 x 1000: 12 tiles,
    s = 4; 300 x 500 x 500: 16 slices, too few, no split; 1023 x 1025 x 3001:
    72 tiles on repacked operands, s = 2; 1024 x 1024 x 1024: s = 2), the
    later parts added into C in order."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 82)
    exact = dist == "int"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=not exact)
    check(run(A, B, variant=1), C64, bound, exact=exact, what=f"v1 split {shape} {dist}")


@pytest.mark.parametrize("shape,s", [((1000, 700, 300), 2), ((257, 516, 100), 4), ((256, 256, 1000), 3),
                                     ((129, 132, 64), 2), ((300, 260, 36), 2), ((1024, 1024, 1024), 1),
                                     ((2048, 2048, 512), 4)])
@pytest.mark.parametrize("dist", ["uniform", "int"])
def test_variant1_forced_k_split(shape, s, dist):
    """split_k forces the CTAs per tile along K (1 = none), down to one
    32-deep slice per CTA (257 x 516 x 100: 4 slices in 4 parts; 300 x 260 x
    36: a full slice and a 4-deep one), also with more CTAs than SMs (2048 x
    2048 x 512: 256 tiles x 4).  Row pitches are multiples of 16 bytes, so the
    tensor maps read the operands in place."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 83)
    exact = dist == "int"
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=not exact)
    check(run(A, B, variant=1, split_k=s), C64, bound, exact=exact, what=f"v1 split_k={s} {shape} {dist}")


@pytest.mark.parametrize("M,N,K,s,ldc", [(256, 384, 1000, 3, None), (200, 300, 700, 2, 301), (130, 260, 2048, 4, None)])
def test_k_split_sums_parts_in_order(M, N, K, s, ldc):
    """The K-split result is the float32 sum, in part order, of the parts'
    own products: part q covers the 32-deep slices [floor(nk q / s),
    floor(nk (q + 1) / s)), and its product, computed alone by the unsplit
    kernel on that K range (the same MMAs in the same order), is bit-identical
    to the part's partial tile.  So C must equal ((P_0 + P_1) + ...) exactly,
    whichever CTA of a tile finishes last and adds the parts, on the
    vector path and (ldc = 301) the element path with ragged edge tiles."""
    A, B = make_operands(M, N, K, "normal", 85)
    dA, dB = to_device(A), to_device(B)
    nk = -(-K // 32)
    parts = []
    for q in range(s):
        k0, k1 = 32 * (nk * q // s), min(K, 32 * (nk * (q + 1) // s))
        parts.append(g.sgemm_3xtf32_ex(dA[:, k0:k1], dB[k0:k1, :], variant=1, split_k=1))
    torch.cuda.synchronize()
    expect = parts[0].cpu().numpy()
    for P in parts[1:]:
        expect = expect + P.cpu().numpy()
    for _ in range(3):
        dC = to_device(torch.full((M, N), float("nan")), ldc)
        g.sgemm_3xtf32_ex(dA, dB, dC, variant=1, split_k=s)
        torch.cuda.synchronize()
        assert np.array_equal(dC.cpu().numpy().view(np.uint32), expect.view(np.uint32))
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(expect, C64, bound, exact=False, what=f"split parts {M}x{N}x{K}")


@pytest.mark.parametrize("variant", [0, 3, 4])
def test_wide_tiles_without_split_tail(variant):
    """split_k = 1 on the 128 x 256 tiles: the last partial wave runs whole."""
    M, N, K = 1200, 4000, 1040
    A, B = make_operands(M, N, K, "uniform", 84)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, variant=variant, split_k=1), C64, bound, exact=False, what=f"v{variant} split_k=1")


@pytest.mark.parametrize("variant", [3, 4])
@pytest.mark.parametrize("K", [48, 300, 700])
def test_wide_tiles_forced_split_tail_short_k(variant, K):
    """split_k = 2 on the 128 x 256 tiles splits the last partial wave along
    K below the automatic threshold too (1200 x 4000: 160 wide tiles, 8 in
    the last wave; K = 48: three 16-deep slices, split 1 + 2)."""
    A, B = make_operands(1200, 4000, K, "uniform", 85)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(run(A, B, variant=variant, split_k=2), C64, bound, exact=False, what=f"v{variant} K={K} split_k=2")
    Ai, Bi = make_operands(1200, 4000, K, "int", 86)
    check(run(Ai, Bi, variant=variant, split_k=2), oracle.gemm_f64(Ai.numpy(), Bi.numpy(), with_bound=False)[0],
          None, exact=True, what=f"v{variant} K={K} split_k=2 int")


@pytest.mark.parametrize("kw,K", [(dict(split_k=5), 256), (dict(split_k=-1), 256), (dict(variant=3, split_k=3), 256),
                                  (dict(variant=2, split_k=2), 256), (dict(variant=4, split_k=4), 256),
                                  (dict(variant=1, split_k=3), 64), (dict(split_k=3), 4096)])
def test_forced_k_split_refusals(kw, K):
    """Refused before any launch: split_k out of 0..4, a K split on the
    direct-A kernel, more than two parts on the wide-tile kernels (also when
    the automatic choice is a wide one: 2048 x 2048 tiles fill half the SMs),
    more parts than 32-deep slices."""
    M = N = 2048 if K == 4096 else 256
    dA = torch.zeros((M, K), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    with pytest.raises(g._lib.SgemmError) as e:
        g.sgemm_3xtf32_ex(dA, dB, **kw)
    assert e.value.status == 1


@pytest.mark.parametrize("variant,split_k", [(1, 0), (1, 4), (2, 0), (3, 0), (4, 0)])
def test_timeout_is_reported_and_recovers(variant, split_k):
    """CTA 0's producer skips its second K slice (with split_k = 4 CTA 0 takes
    the first two of the tile's 8 slices): its split warps' bounded wait
    expires, the MMA issuer and the epilogue give up in turn, tensor memory is
    freed, and the status word says so.  The next call is unaffected."""
    A, B = make_operands(128, 256, 256, "uniform", 80)
    dA, dB = to_device(A), to_device(B)
    assert g.check_status() == 0
    g.sgemm_3xtf32_ex(dA, dB, variant=variant, split_k=split_k, debug_skip_stage=2, timeout_ns=20_000_000)
    assert g.check_status() == 4
    C = g.sgemm_3xtf32(dA, dB)
    assert g.check_status() == 0
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(C.cpu().numpy(), C64, bound, exact=False, what="after timeout")


@pytest.mark.parametrize("variant,split_k", [(0, 0), (1, 1), (1, 2), (3, 0), (4, 0), (4, 2)])
@pytest.mark.parametrize("c_offset", [0, 1])
def test_unaligned_output_guard_bands(variant, split_k, c_offset):
    """C with rows of 1029 floats (and, with c_offset = 1, a base off the
    16-byte grid) written by the epilogue's shared-memory patches (or the K
    split's finishing CTA): every element against the oracle, and the row
    padding and the floats around C keep their sentinel."""
    M, N, K = 700, 1025, 600
    A, B = make_operands(M, N, K, "uniform", 81)
    ldc, guard, sentinel = 1029, 64 + c_offset, -12345.0
    store = torch.full((guard + M * ldc + 64,), sentinel, device="cuda")
    dC = store[guard:guard + M * ldc].view(M, ldc)[:, :N]
    dA, dB = to_device(A), to_device(B, 1028)
    if variant or split_k:
        g.sgemm_3xtf32_ex(dA, dB, dC, variant=variant, split_k=split_k)
    else:
        g.sgemm_3xtf32(dA, dB, dC)
    torch.cuda.synchronize()
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
    check(dC.cpu().numpy(), C64, bound, exact=False, what=f"3xtf32 v{variant} s{split_k} c+{c_offset}")
    s = store.cpu().numpy()
    assert np.all(s[:guard] == sentinel) and np.all(s[guard + M * ldc:] == sentinel)
    assert np.all(store[guard:guard + M * ldc].view(M, ldc)[:, N:].cpu().numpy() == sentinel)


@pytest.mark.parametrize("shape,dist", [((1 << 20, 8, 64), "int"), ((128, 128, 1 << 20), "uniform"),
                                        ((1 << 20, 9, 63), "int")])
def test_extreme_shapes_every_element(shape, dist):
    """A million rows (aligned, and with rows of 63 and 9 floats on the
    residue-class maps) and a million-deep K on one tile (its K split into
    four parts): every element against the oracle, integer inputs exactly."""
    M, N, K = shape
    A, B = make_operands(M, N, K, dist, 62)
    C = run(A, B)
    C64, bound = oracle.gemm_f64(A.numpy(), B.numpy(), with_bound=(dist != "int"))
    check(C, C64, bound, exact=(dist == "int"), what=f"3xtf32 {shape} {dist}")
