"""GB300 (sm_103a) single-precision matrix multiply, C = A x B.

Thin Python binding over the C ABI in ``include/sgemm.h``: it checks tensor
types, reads sizes and strides, passes raw device pointers and the current
CUDA stream, and raises on a non-zero status.  All arithmetic runs in the
library's CUDA kernels; there is no other path.
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import Options, SgemmError

__all__ = [
    "sgemm_f32",
    "sgemm_f32_ex",
    "sgemm_f32_noalloc",
    "sgemm_f32_gemm",
    "sgemm_3xtf32",
    "sgemm_3xtf32_ex",
    "sgemm_f32_host",
    "check_status",
    "describe",
    "Options",
    "SgemmError",
]


def _stream_ptr(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(s.cuda_stream)


def _row_stride(X: torch.Tensor, name: str) -> int:
    if X.dim() != 2:
        raise ValueError(f"{name} must be 2-D, got shape {tuple(X.shape)}")
    rows, cols = X.shape
    if cols > 1 and X.stride(1) != 1:
        raise ValueError(f"{name} must be row-major with unit column stride")
    ld = X.stride(0) if rows > 1 else cols
    return max(ld, cols)


def _operands(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None):
    for name, X in (("A", A), ("B", B)):
        if not isinstance(X, torch.Tensor) or X.dtype != torch.float32 or not X.is_cuda:
            raise TypeError(f"{name} must be a CUDA float32 tensor")
    if A.dim() != 2 or B.dim() != 2 or A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes do not multiply: {tuple(A.shape)} x {tuple(B.shape)}")
    if A.device != B.device:
        raise ValueError("A and B are on different devices")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif out.dtype != torch.float32 or out.device != A.device or tuple(out.shape) != (M, N):
        raise ValueError("out must be a float32 (M, N) tensor on A's device")
    return A, B, out, M, N, K, _row_stride(A, "A"), _row_stride(B, "B"), _row_stride(out, "out")


def _call(fn_name, A, B, out, stream, opt=None):
    A, B, out, M, N, K, lda, ldb, ldc = _operands(A, B, out)
    lib = _lib.load()
    with torch.cuda.device(A.device):
        s = _stream_ptr(stream)
        args = [M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc, s]
        if opt is not None:
            args.append(ctypes.byref(opt))
        _lib.check(getattr(lib, fn_name)(*args), fn_name)
    return out


def sgemm_f32(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """C = A @ B on the CUDA cores (float32 FFMA kernels), enqueued on ``stream``."""
    return _call("sgemm_f32", A, B, out, stream)


def sgemm_f32_noalloc(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, *, stream=None) -> torch.Tensor:
    """sgemm_f32 without any device allocation in the call: the stream-K
    scratch comes from a fixed array inside the library (shared by all calls
    on the device: calls that overlap on the GPU race).  ``out`` is required,
    so this wrapper allocates nothing either."""
    if out is None:
        raise ValueError("sgemm_f32_noalloc needs a preallocated `out`")
    return _call("sgemm_f32_noalloc", A, B, out, stream)


def sgemm_f32_gemm(A: torch.Tensor, B: torch.Tensor, C: torch.Tensor | None = None, *, alpha: float = 1.0,
                   beta: float = 0.0, transa: bool = False, transb: bool = False, stream=None) -> torch.Tensor:
    """C = alpha * op(A) @ op(B) + beta * C (float32 FFMA kernels).

    ``A`` and ``B`` are the stored operands: A is (M, K), or (K, M) with
    ``transa`` (op(A) = A.T); B is (K, N), or (N, K) with ``transb``.  ``C``
    is (M, N); it is required when beta != 0 and not read when beta == 0.
    """
    for name, X in (("A", A), ("B", B)):
        if not isinstance(X, torch.Tensor) or X.dtype != torch.float32 or not X.is_cuda or X.dim() != 2:
            raise TypeError(f"{name} must be a 2-D CUDA float32 tensor")
    M, K = (A.shape[1], A.shape[0]) if transa else tuple(A.shape)
    KB, N = (B.shape[1], B.shape[0]) if transb else tuple(B.shape)
    if K != KB:
        raise ValueError(f"shapes do not multiply: op(A) {(M, K)} x op(B) {(KB, N)}")
    if A.device != B.device:
        raise ValueError("A and B are on different devices")
    if C is None:
        if beta != 0:
            raise ValueError("beta != 0 needs C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif C.dtype != torch.float32 or C.device != A.device or tuple(C.shape) != (M, N):
        raise ValueError("C must be a float32 (M, N) tensor on A's device")
    lib = _lib.load()
    with torch.cuda.device(A.device):
        rc = lib.sgemm_f32_gemm(int(bool(transa)), int(bool(transb)), M, N, K, float(alpha), A.data_ptr(),
                                _row_stride(A, "A"), B.data_ptr(), _row_stride(B, "B"), float(beta), C.data_ptr(),
                                _row_stride(C, "C"), _stream_ptr(stream))
        _lib.check(rc, "sgemm_f32_gemm")
    return C


def sgemm_3xtf32(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, *, stream=None) -> torch.Tensor:
    """C = A @ B on the tensor cores with the three-product TF32 split."""
    return _call("sgemm_3xtf32", A, B, out, stream)


def sgemm_f32_ex(A, B, out=None, *, stream=None, producer=0, split_k=0, multicast=0, math=0, stages=0,
                 debug_skip_stage=0, timeout_ns=0, tail_split=0, stream_k=0, tile_n=0, repack=0,
                 a_layout=0, group_m=0, l2_hint=0, tile_k=0, edge=0) -> torch.Tensor:
    """sgemm_f32 with forced variant choices (see struct sgemm_options)."""
    opt = Options(producer, split_k, multicast, math, stages, debug_skip_stage, timeout_ns, tail_split, stream_k,
                  tile_n, repack, a_layout, group_m, l2_hint, tile_k, edge)
    return _call("sgemm_f32_ex", A, B, out, stream, opt)


def sgemm_3xtf32_ex(A, B, out=None, *, stream=None, variant=0, split_k=0, debug_skip_stage=0,
                    timeout_ns=0) -> torch.Tensor:
    """sgemm_3xtf32 with forced choices: ``variant`` 1 = split-tile kernel,
    2 = direct-A kernel, 3 = split-tile kernel on 128 x 256 tiles with
    K-slices of 16, 4 = variant 3 with B's TF32 parts pre-split in HBM
    (0 = automatic); ``split_k`` 1 = no K split, 2..4 = each tile's K slices
    split among that many CTAs (variant 1; 0 = automatic)."""
    opt = Options(0, split_k, 0, variant, 0, debug_skip_stage, timeout_ns, 0, 0, 0, 0, 0)
    return _call("sgemm_3xtf32_ex", A, B, out, stream, opt)


def sgemm_f32_host(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None, *,
                   device: int | torch.device = 0, stream=None) -> torch.Tensor:
    """Host-buffer form (the C entry sgemm_f32_host): A, B and ``out`` are CPU
    float32 tensors (pinned memory lets the copies overlap the product); the
    library copies them to and from ``device`` itself.  Returns ``out`` once
    the result is in it."""
    dev = torch.device("cuda", device) if isinstance(device, int) else torch.device(device)
    for name, X in (("A", A), ("B", B)):
        if not isinstance(X, torch.Tensor) or X.dtype != torch.float32 or X.is_cuda or X.dim() != 2:
            raise TypeError(f"{name} must be a 2-D CPU float32 tensor")
    if A.shape[1] != B.shape[0]:
        raise ValueError(f"shapes do not multiply: {tuple(A.shape)} x {tuple(B.shape)}")
    M, K = A.shape
    N = B.shape[1]
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, pin_memory=True)
    elif out.dtype != torch.float32 or out.is_cuda or tuple(out.shape) != (M, N):
        raise ValueError("out must be a CPU float32 (M, N) tensor")
    lib = _lib.load()
    with torch.cuda.device(dev):
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = lib.sgemm_f32_host(M, N, K, A.data_ptr(), _row_stride(A, "A"), B.data_ptr(), _row_stride(B, "B"),
                                out.data_ptr(), _row_stride(out, "out"), _stream_ptr(s))
        _lib.check(rc, "sgemm_f32_host")
        s.synchronize()
    return out


def check_status(stream=None) -> int:
    """Synchronise and return/clear the device status word (0 or ERR_TIMEOUT)."""
    lib = _lib.load()
    return lib.sgemm_check_status(_stream_ptr(stream))


def describe(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor | None = None) -> str:
    """Name of the variant sgemm_f32 would launch for these operands."""
    A, B, out, M, N, K, lda, ldb, ldc = _operands(A, B, out)
    lib = _lib.load()
    with torch.cuda.device(A.device):
        return lib.sgemm_describe(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, out.data_ptr(), ldc).decode()
