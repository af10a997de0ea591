"""Compile the CUDA library (libfa_mha.so) in-tree for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel to an object file
under _build/, then linked into one shared library exporting the C ABI of
include/fa_mha.h. The CUDA runtime is linked statically; the driver's
tensor-map encoder is resolved at run time, so loading the library needs no
GPU and no libcuda.

The debug variant (``build(variant="debug")``, ``_build/debug/libfa_mha_debug.so``)
compiles the same sources with FA_TRACE=1: the prefill kernel records an
event trace into a caller buffer and checks its run-time indexes with bounds
guards that set a status bit instead of trapping.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libfa_mha.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
DEBUG_DIR = os.path.join(BUILD_DIR, "debug")
DEBUG_LIB_PATH = os.path.join(DEBUG_DIR, "libfa_mha_debug.so")
VARIANTS = {"default": (BUILD_DIR, LIB_PATH, []),
            "debug": (DEBUG_DIR, DEBUG_LIB_PATH, ["-DFA_TRACE=1"])}
HEADER = os.path.join(ROOT, "include", "fa_mha.h")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    cuda_home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(cuda_home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs() -> list[str]:
    deps = [HEADER, os.path.abspath(__file__)]
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    return deps


def up_to_date(variant: str = "default") -> bool:
    lib = VARIANTS[variant][1]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          variant: str = "default") -> str:
    """Build the library variant ("default": libfa_mha.so, "debug":
    libfa_mha_debug.so) if any source is newer than it; return its path."""
    build_dir, lib_path, defines = VARIANTS[variant]
    if not force and up_to_date(variant):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH_FLAGS, *COMMON_FLAGS, *defines, "-c", src, "-o", obj]
        if ptxas_info:
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    failed = []
    for src, pr in procs:
        outp, _ = pr.communicate()
        if pr.returncode != 0 or (verbose and outp) or ptxas_info:
            sys.stderr.write(outp)
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run([nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                variant="debug" if "--debug" in sys.argv else "default"))
