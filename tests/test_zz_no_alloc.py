"""sgemm_f32_noalloc: the allocation-free entry point, through the C ABI.

It serves callers that may not allocate device memory during a call (a fixed
memory footprint, or all device memory handed to their own allocator up
front): its stream-K scratch lives in a fixed device array in the library
instead of a per-call pool allocation.  This file runs after every other
test file (pytest collects it last) and also passes alone in a fresh process.
Two calls in a row, of different shapes and producers, are each checked
against the existing entry point sgemm_f32 with the tolerance every parity
test uses, 5e-5 * sum_k |A_ik||B_kj|, and against the CPU oracle.
"""
import ctypes

import numpy as np
import pytest
import torch

import dense_fp32_gemm_f32_gb300 as g
import oracle
from dense_fp32_gemm_f32_gb300 import _lib
from parity import TOL, check, to_device
from workloads import make_operands

pytestmark = pytest.mark.gpu


def _noalloc_c_abi(dA, dB, dC):
    lib = _lib.load()
    M, K = dA.shape
    N = dB.shape[1]
    rc = lib.sgemm_f32_noalloc(M, N, K, ctypes.c_void_p(dA.data_ptr()), dA.stride(0),
                               ctypes.c_void_p(dB.data_ptr()), dB.stride(0), ctypes.c_void_p(dC.data_ptr()),
                               dC.stride(0), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, lib.sgemm_status_string(rc)


@pytest.mark.parametrize("shapes", [((1024, 1536, 1200, 0), (1023, 1025, 1027, 3))])
def test_noalloc_matches_sgemm_f32_on_two_calls_in_a_row(shapes):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    for call, (M, N, K, a_offset) in enumerate(shapes):
        # The second call has unaligned rows (read in place through the
        # residue-class tensor maps) and a different shape: nothing of the
        # first call's scratch may leak in.
        A, B = make_operands(M, N, K, "normal", 900 + call)
        dA, dB = to_device(A, offset=a_offset), to_device(B)
        C_noalloc = torch.full((M, N), float("nan"), device="cuda")
        _noalloc_c_abi(dA, dB, C_noalloc)
        C_ref = g.sgemm_f32(dA, dB)
        torch.cuda.synchronize()
        assert g.check_status() == 0
        cn, cr = C_noalloc.cpu().numpy(), C_ref.cpu().numpy()
        C64, bound = oracle.gemm_f64(A.numpy(), B.numpy())
        assert np.isfinite(cn).all()
        assert np.all(np.abs(cn.astype(np.float64) - cr.astype(np.float64)) <= TOL * bound), f"call {call}"
        check(cn, C64, bound, exact=False, what=f"noalloc call {call}")


_FOOTPRINT_SCRIPT = r"""
import ctypes, json, sys
import torch
sys.path.insert(0, sys.argv[1])
from dense_fp32_gemm_f32_gb300 import _lib
from workloads import make_operands

lib = _lib.load()
torch.cuda.set_device(0)
shapes = [(1024, 1536, 1200, 0), (1023, 1025, 1027, 3)]
ops = []
for i, (M, N, K, off) in enumerate(shapes):
    A, B = make_operands(M, N, K, "normal", 950 + i)
    store = torch.empty(off + M * K, device="cuda")
    dA = store[off:].view(M, K)
    dA.copy_(A)
    dB = B.cuda()
    dC = torch.empty((M, N), device="cuda")
    ops.append((M, N, K, dA, dB, dC))
streams = [torch.cuda.Stream() for _ in range(4)]

def call(op, stream):
    M, N, K, dA, dB, dC = op
    rc = lib.sgemm_f32_noalloc(M, N, K, ctypes.c_void_p(dA.data_ptr()), K, ctypes.c_void_p(dB.data_ptr()), N,
                               ctypes.c_void_p(dC.data_ptr()), N, ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0, lib.sgemm_status_string(rc)

# First calls: the library's one-time set-up and the loading of both kernels.
for op in ops:
    call(op, torch.cuda.current_stream())
torch.cuda.synchronize()
free0 = torch.cuda.mem_get_info()[0]
# Calls on streams the library has not seen (sgemm_f32 would give each of
# them its own stream-K scratch), also on the misaligned shape.
for s in streams:
    for op in ops:
        call(op, s)
        s.synchronize()
torch.cuda.synchronize()
free1 = torch.cuda.mem_get_info()[0]
assert lib.sgemm_check_status(None) == 0
print(json.dumps({"free0": free0, "free1": free1}))
"""


def test_noalloc_calls_take_no_device_memory():
    """The property the entry point exists for: after the first calls (the
    one-time set-up and kernel loading), further calls, on new streams and on
    a shape with misaligned rows, leave the device's free memory
    unchanged.  Run in a fresh process, so that no earlier test's pool cache
    or scratch can hide an allocation."""
    import json
    import os
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "-c", _FOOTPRINT_SCRIPT, root], capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    rec = json.loads(r.stdout.strip().splitlines()[-1])
    assert rec["free1"] == rec["free0"], rec
