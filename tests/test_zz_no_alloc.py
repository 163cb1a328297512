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
        # The second call has unaligned rows (cp.async producer) and a
        # different shape: nothing of the first call's scratch may leak in.
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
