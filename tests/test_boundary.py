"""The C ABI boundary on the host: the library loads, exports every declared
symbol, and rejects bad arguments before touching a GPU (no GPU needed)."""
import ctypes
import os
import re

import pytest

from dense_fp32_gemm_f32_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        # function declarations: "<type> name(" at statement start
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_headers_declare_the_abi():
    names = declared_functions()
    for required in ("sgemm_f32", "sgemm_3xtf32", "sgemm_f32_ex", "sgemm_check_status", "sgemm_status_string"):
        assert required in names
    assert set(names) == set(_lib.SIGNATURES), "binding signatures and headers disagree"


def test_options_struct_matches_the_header():
    """The binding's struct sgemm_options has the header's fields, in the
    header's order, with the header's types (int, uint64_t), so that a field
    added on one side only cannot shift the others."""
    text = open(os.path.join(ROOT, "include", "sgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    body = re.search(r"typedef\s+struct\s+sgemm_options\s*\{(.*?)\}\s*sgemm_options\s*;", text, re.S).group(1)
    fields = re.findall(r"(int|uint64_t)\s+(\w+)\s*;", body)
    assert fields, "no fields parsed"
    ctypes_of = {"int": ctypes.c_int, "uint64_t": ctypes.c_uint64}
    assert [(n, ctypes_of[t]) for t, n in fields] == list(_lib.Options._fields_)


def test_library_exports_every_declared_symbol():
    lib = _lib.load()
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_status_strings():
    lib = _lib.load()
    assert lib.sgemm_status_string(0) == b"ok"
    assert lib.sgemm_status_string(_lib.ERR_INVALID_ARG) == b"invalid argument"
    assert lib.sgemm_status_string(_lib.ERR_TIMEOUT) == b"kernel wait timed out"
    assert lib.sgemm_status_string(12345) == b"unknown status"


FAKE_A, FAKE_B, FAKE_C = 0x10000000, 0x20000000, 0x30000000  # never dereferenced


@pytest.mark.parametrize("fn", ["sgemm_f32", "sgemm_3xtf32"])
@pytest.mark.parametrize(
    "args",
    [
        (-1, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4),  # negative M
        (4, -1, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4),  # negative N
        (4, 4, -1, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4),  # negative K
        (4, 4, 8, FAKE_A, 7, FAKE_B, 4, FAKE_C, 4),  # lda < K
        (4, 8, 4, FAKE_A, 4, FAKE_B, 7, FAKE_C, 8),  # ldb < N
        (4, 8, 4, FAKE_A, 4, FAKE_B, 8, FAKE_C, 7),  # ldc < N
        (4, 4, 4, 0, 4, FAKE_B, 4, FAKE_C, 4),  # A NULL
        (4, 4, 4, FAKE_A, 4, 0, 4, FAKE_C, 4),  # B NULL
        (4, 4, 4, FAKE_A, 4, FAKE_B, 4, 0, 4),  # C NULL
        (4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_A + 32, 4),  # C overlaps A
        (4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_B - 16, 4),  # C overlaps B
        (4, 4, 4, FAKE_A + 2, 4, FAKE_B, 4, FAKE_C, 4),  # A not float-aligned
        (4, 4, 4, FAKE_A, 4, FAKE_B + 1, 4, FAKE_C, 4),  # B not float-aligned
        (4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C + 3, 4),  # C not float-aligned
        (2**31 - 1, 65536 * 128, 4, FAKE_A, 4, FAKE_B, 65536 * 128, 0x7000000000, 65536 * 128),  # tile count beyond int
    ],
)
def test_invalid_arguments_rejected_on_host(fn, args):
    lib = _lib.load()
    assert getattr(lib, fn)(*args, None) == _lib.ERR_INVALID_ARG


def test_empty_output_is_a_noop_without_device():
    lib = _lib.load()
    # M == 0 or N == 0: nothing to do, returns OK without any CUDA call
    assert lib.sgemm_f32(0, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None) == _lib.OK
    assert lib.sgemm_f32(4, 0, 4, FAKE_A, 4, FAKE_B, 0, FAKE_C, 0, None) == _lib.OK
    # NULL operands are fine when they are empty
    assert lib.sgemm_f32(0, 0, 0, 0, 0, 0, 0, 0, 0, None) == _lib.OK


def test_bad_options_rejected():
    lib = _lib.load()
    opt = _lib.Options(0, 0, 0, 0, 0, -1, 0, 0, 0)  # negative debug_skip_stage
    assert lib.sgemm_f32_ex(4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None, ctypes.byref(opt)) == _lib.ERR_INVALID_ARG


@pytest.mark.parametrize("split_k", [-1, 5, 9])
def test_tensor_core_split_count_rejected_on_host(split_k):
    """sgemm_3xtf32_ex takes 0..4 CTAs per tile along K; anything else is
    refused before any device call."""
    lib = _lib.load()
    opt = _lib.Options(0, split_k, 0, 0, 0, 0, 0, 0, 0)
    assert lib.sgemm_3xtf32_ex(4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None, ctypes.byref(opt)) == \
        _lib.ERR_INVALID_ARG


def test_no_cpu_fallback_without_gpu():
    """Without a usable GPU a valid call fails loudly instead of computing on the host."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    lib = _lib.load()
    rc = lib.sgemm_f32(4, 4, 4, FAKE_A, 4, FAKE_B, 4, FAKE_C, 4, None)
    assert rc in (_lib.ERR_CUDA, _lib.ERR_UNSUPPORTED)


def test_binding_rejects_cpu_tensors():
    import torch

    import dense_fp32_gemm_f32_gb300 as g

    with pytest.raises(TypeError):
        g.sgemm_f32(torch.ones(2, 2), torch.ones(2, 2))


@pytest.mark.parametrize(
    "args",
    [
        # transa, transb, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc
        (2, 0, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.0, FAKE_C, 4),  # bad flag
        (0, -1, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.0, FAKE_C, 4),  # bad flag
        (1, 0, 8, 4, 4, 1.0, FAKE_A, 7, FAKE_B, 4, 0.0, FAKE_C, 4),  # transposed A: lda < M
        (0, 1, 4, 4, 8, 1.0, FAKE_A, 8, FAKE_B, 7, 0.0, FAKE_C, 4),  # transposed B: ldb < K
        (0, 0, 4, 8, 4, 1.0, FAKE_A, 4, FAKE_B, 8, 0.0, FAKE_C, 7),  # ldc < N
        (1, 1, 4, 4, 4, 1.0, 0, 4, FAKE_B, 4, 0.0, FAKE_C, 4),  # A NULL
        (0, 0, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 1.0, 0, 4),  # C NULL
        (1, 0, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.0, FAKE_A + 32, 4),  # C overlaps (transposed) A
        (1, 1, 4, 4, 4, 1.0, FAKE_A + 2, 4, FAKE_B, 4, 0.0, FAKE_C, 4),  # A not float-aligned
        (0, 1, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B + 1, 4, 0.0, FAKE_C, 4),  # B not float-aligned
        (0, 0, 4, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.5, FAKE_C + 2, 4),  # C not float-aligned
    ],
)
def test_general_entry_invalid_arguments_rejected_on_host(args):
    lib = _lib.load()
    assert lib.sgemm_f32_gemm(*args, None) == _lib.ERR_INVALID_ARG


def test_general_entry_empty_and_unread_operands():
    import torch

    lib = _lib.load()
    assert lib.sgemm_f32_gemm(0, 0, 0, 4, 4, 1.0, FAKE_A, 4, FAKE_B, 4, 0.0, FAKE_C, 4, None) == _lib.OK
    if torch.cuda.is_available():
        return  # the call below would write C at a fake address
    # alpha == 0: A and B are not read, so NULL passes validation; C = beta C
    # needs a device, and without one the call fails loudly
    rc = lib.sgemm_f32_gemm(0, 0, 4, 4, 4, 0.0, 0, 4, 0, 4, 2.0, FAKE_C, 4, None)
    assert rc in (_lib.ERR_CUDA, _lib.ERR_UNSUPPORTED)


def test_no_cluster_multicast_load_in_library_or_bench():
    # The library runs on every rank of a multi-GPU bench; no cluster-multicast
    # bulk copy may be compiled into it.
    offenders = []
    for d in (os.path.join(ROOT, "dense_fp32_gemm_f32_gb300", "csrc"), ROOT):
        for f in sorted(os.listdir(d)):
            if f.endswith((".cu", ".cuh", ".h", ".py")):
                if "multicast::cluster" in open(os.path.join(d, f)).read():
                    offenders.append(f)
    assert offenders == []


def _header_list(tag):
    text = open(os.path.join(ROOT, "include", "sgemm.h")).read()
    m = re.search(r"^\s*\*\s*" + re.escape(tag) + r":\s*([\w ]+)$", text, flags=re.M)
    assert m, f"sgemm.h has no '{tag}:' line"
    return m.group(1).split()


def test_header_states_which_entry_points_allocate():
    # Every entry point of sgemm.h is listed exactly once as allocating device
    # memory or not.
    alloc, none = _header_list("ALLOCATING"), _header_list("NON-ALLOCATING")
    text = open(os.path.join(ROOT, "include", "sgemm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    declared = set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(sgemm_\w+)\s*\(", text, flags=re.M))
    assert sorted(alloc + none) == sorted(declared)
    assert not set(alloc) & set(none)


def _function_body(src, name):
    """Code of the function `name` (comments removed)."""
    src = re.sub(r"//[^\n]*", "", re.sub(r"/\*.*?\*/", "", src, flags=re.S))
    i = src.index(name + "(")
    i = src.index("{", i)
    depth, j = 0, i
    while True:
        depth += {"{": 1, "}": -1}.get(src[j], 0)
        j += 1
        if depth == 0:
            return src[i:j]


def test_non_allocating_entries_reach_no_allocation_in_source():
    # The host code behind the entries listed as non-allocating names no
    # allocating call, pool, per-stream scratch or repack buffer.
    csrc = os.path.join(ROOT, "dense_fp32_gemm_f32_gb300", "csrc")
    banned = ("cudaMalloc", "cudaFree", "MallocFromPool", "workspace_pool", "sk_lease", "Repacked", "malloc(",
              "cudaStreamCreate", "cudaEventCreate", "at::", "torch")
    bodies = {
        "run_ffma_noalloc": _function_body(open(os.path.join(csrc, "api_ffma.cu")).read(), "int run_ffma_noalloc"),
        "sgemm_check_status": _function_body(open(os.path.join(csrc, "sgemm_api.cu")).read(),
                                             "int sgemm_check_status"),
        "sgemm_status_string": _function_body(open(os.path.join(csrc, "sgemm_api.cu")).read(),
                                              "const char* sgemm_status_string"),
        "sgemm_describe": _function_body(open(os.path.join(csrc, "sgemm_api.cu")).read(),
                                         "const char* sgemm_describe"),
    }
    for name, body in bodies.items():
        for b in banned:
            assert b not in body, f"{name} names {b}"
    # the small-problem launch and the plan it shares with sgemm_f32 allocate nothing either
    plan = _function_body("int f(){" + open(os.path.join(csrc, "api_plan.cu")).read() + "}", "int f")
    for b in banned:
        assert b not in plan, f"api_plan.cu names {b}"
    launch_small = _function_body(open(os.path.join(csrc, "api_ffma.cu")).read(), "int launch_small")
    for b in banned:
        assert b not in launch_small, f"launch_small names {b}"
