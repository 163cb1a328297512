"""Builds the CUDA library in-tree: ``_build/libgb300_sgemm.so`` (sm_103a only).

Every translation unit is compiled by nvcc in parallel, then linked into one
shared library with the CUDA runtime linked statically.  ``-Xptxas -v``
register/spill reports go to ``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import re
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libgb300_sgemm.so"
SOURCES = ["sgemm_api.cu", "api_device.cu", "api_plan.cu", "api_ffma.cu", "api_tf32.cu", "api_host.cu", "sgemm_ffma_tma.cu", "sgemm_ffma_tma_wg.cu", "sgemm_ffma_tma_wide.cu", "sgemm_ffma_tma_fused.cu", "sgemm_ffma_tma_x.cu", "sgemm_ffma_tma_x16.cu",
           "sgemm_ffma_cpasync.cu", "sgemm_ffma_scaled.cu", "sgemm_ffma_bt.cu", "sgemm_ffma_ldg.cu", "sgemm_ffma_res.cu", "sgemm_small.cu", "sgemm_3xtf32.cu", "sgemm_3xtf32_direct.cu", "pack.cu", "peak.cu"]
# Kernels that split registers between warpgroups with setmaxnreg must be
# built with exactly this many registers per thread (the split's total).
REGSPLIT_SOURCES = ("sgemm_ffma_tma_wg.cu", "sgemm_ffma_tma_wide.cu")
REGSPLIT_LAUNCH_REGS = 168
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return path


def lib_path() -> str:
    return os.path.join(OUT_DIR, LIB_NAME)


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files += [os.path.join(HERE, "..", "include", f) for f in os.listdir(os.path.join(HERE, "..", "include"))]
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    lib = lib_path()
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _compile(src: str) -> tuple[str, str]:
    obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def check_regsplit(src: str, log: str) -> None:
    """The register-split kernels' ptxas report: every entry uses exactly
    REGSPLIT_LAUNCH_REGS registers, and ptxas kept the setmaxnreg instructions
    (it says so when it drops them)."""
    used = re.findall(r"Compiling entry function '([^']+)'.*?Used (\d+) registers", log, re.S)
    if not used:
        raise RuntimeError(f"{src}: no kernel entries in the ptxas report")
    bad = [(name, n) for name, n in used if int(n) != REGSPLIT_LAUNCH_REGS]
    if bad:
        raise RuntimeError(f"{src}: kernels not at {REGSPLIT_LAUNCH_REGS} registers: {bad}")
    if "setmaxnreg" in log:
        raise RuntimeError(f"{src}: ptxas reported on setmaxnreg:\n{log}")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of the shared library."""
    if not force and up_to_date():
        return lib_path()
    os.makedirs(OUT_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(_compile, SOURCES))
    objs = [o for o, _ in results]
    with open(os.path.join(OUT_DIR, "ptxas.log"), "w") as f:
        for (o, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    logs = dict(zip(SOURCES, (log for _, log in results)))
    for src in REGSPLIT_SOURCES:
        check_regsplit(src, logs[src])
    tmp = lib_path() + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path())
    if verbose:
        print(f"built {lib_path()}", file=sys.stderr)
    return lib_path()


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
