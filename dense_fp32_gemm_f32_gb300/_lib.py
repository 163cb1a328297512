"""ctypes view of the C ABI declared in include/sgemm.h and include/sgemm_bench.h.

Loading never falls back to anything: if the shared library is missing it is
built (nvcc), and if that fails the import error propagates.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

# Status codes (enum sgemm_status).
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_TIMEOUT = 4
ERR_NOT_IMPLEMENTED = 5

PRODUCER_AUTO, PRODUCER_TMA, PRODUCER_CPASYNC, PRODUCER_TMA_WG, PRODUCER_FUSED, PRODUCER_TMA_X, PRODUCER_SMALL = 0, 1, 2, 3, 4, 5, 6

# Every symbol the headers declare, with its ctypes signature.
_i, _p, _u64, _d = ctypes.c_int, ctypes.c_void_p, ctypes.c_uint64, ctypes.c_double


class Options(ctypes.Structure):
    """struct sgemm_options."""

    _fields_ = [
        ("producer", _i),
        ("split_k", _i),
        ("multicast", _i),
        ("math", _i),
        ("stages", _i),
        ("debug_skip_stage", _i),
        ("timeout_ns", _u64),
        ("tail_split", _i),
        ("stream_k", _i),
        ("tile_n", _i),
        ("repack", _i),
        ("a_layout", _i),
        ("group_m", _i),
        ("l2_hint", _i),
        ("tile_k", _i),
        ("edge", _i),
    ]


_GEMM_ARGS = [_i, _i, _i, _p, _i, _p, _i, _p, _i, _p]
SIGNATURES = {
    "sgemm_f32": (_i, _GEMM_ARGS),
    "sgemm_f32_noalloc": (_i, _GEMM_ARGS),
    "sgemm_f32_host": (_i, _GEMM_ARGS),
    "sgemm_3xtf32": (_i, _GEMM_ARGS),
    "sgemm_f32_ex": (_i, _GEMM_ARGS + [ctypes.POINTER(Options)]),
    "sgemm_3xtf32_ex": (_i, _GEMM_ARGS + [ctypes.POINTER(Options)]),
    "sgemm_f32_gemm": (_i, [_i, _i, _i, _i, _i, ctypes.c_float, _p, _i, _p, _i, ctypes.c_float, _p, _i, _p]),
    "sgemm_check_status": (_i, [_p]),
    "sgemm_status_string": (ctypes.c_char_p, [_i]),
    "sgemm_describe": (ctypes.c_char_p, [_i, _i, _i, _p, _i, _p, _i, _p, _i]),
    "sgemm_bench_fma_peak": (_i, [_i, _i, _i, _p, _p, ctypes.POINTER(_d)]),
    "sgemm_bench_copy": (_i, [_p, _p, ctypes.c_longlong, _i, _p]),
}


def library_path() -> str:
    return _build.lib_path()


def load() -> ctypes.CDLL:
    """Load (building first if needed) the CUDA library and bind its symbols."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            lib = ctypes.CDLL(path, mode=ctypes.RTLD_LOCAL)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(lib, name)
                f.restype = res
                f.argtypes = args
            _lib = lib
    return _lib


class SgemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = load().sgemm_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")
        self.status = status


def check(status: int, where: str) -> None:
    if status != OK:
        raise SgemmError(status, where)


def loaded_path() -> str | None:
    return os.path.abspath(_lib._name) if _lib is not None else None
