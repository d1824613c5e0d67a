"""In-tree build of libqsa.so (nvcc, sm_103a only)."""
from __future__ import annotations

import glob
import os
import subprocess

_HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(_HERE, "csrc")
LIB_PATH = os.path.join(_HERE, "libqsa.so")
INCLUDE = os.path.join(os.path.dirname(_HERE), "include")

NVCC_FLAGS = [
    "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
    "-Xptxas", "-v", "-shared", "-Xcompiler", "-fPIC", "-I", INCLUDE,
]


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + [os.path.join(INCLUDE, "qsa.h")]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu under csrc/ into libqsa.so next to this file, then
    the CPython entry points of the per-step calls (build_fastcall)."""
    _build_lib(force, verbose)
    build_fastcall(force)
    return LIB_PATH


def _build_lib(force: bool, verbose: bool) -> str:
    newest = max(os.path.getmtime(p) for p in _deps())
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= newest:
        return LIB_PATH
    nvcc = os.environ.get("NVCC", "nvcc")
    if not os.path.exists(nvcc) and os.path.exists("/usr/local/cuda/bin/nvcc"):
        nvcc = "/usr/local/cuda/bin/nvcc"
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [nvcc, *NVCC_FLAGS, "-o", tmp, *_sources()]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed ({r.returncode}):\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(r.stderr)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


FASTCALL_SRC = os.path.join(_HERE, "_fastcall.c")


def fastcall_path() -> str:
    import sysconfig
    return os.path.join(_HERE, "_fastcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def build_fastcall(force: bool = False) -> str | None:
    """Compile the CPython entry points of the per-step calls (_fastcall.c)
    against libqsa.so; None where the Python headers or a C compiler are
    missing (the ctypes path is used then)."""
    import shutil
    import sysconfig
    out = fastcall_path()
    inc = sysconfig.get_paths().get("include", "")
    cc = os.environ.get("CC", "gcc")
    if not inc or not os.path.exists(os.path.join(inc, "Python.h")) or shutil.which(cc) is None:
        return None
    deps = [FASTCALL_SRC, os.path.join(INCLUDE, "qsa.h"), LIB_PATH]
    if not force and os.path.exists(out) and os.path.getmtime(out) >= max(os.path.getmtime(p) for p in deps):
        return out
    tmp = out + f".{os.getpid()}.tmp"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-I", inc, "-I", INCLUDE, FASTCALL_SRC, "-o", tmp, "-L", _HERE,
           "-l:libqsa.so", "-Wl,-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return None
    os.replace(tmp, out)
    return out
