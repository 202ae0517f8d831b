"""Build libattn.so in-tree with nvcc for sm_103a (no cmake, no torch), and
the CPython extension `_calls` (csrc/pycalls.c) with the host C compiler.

Each .cu under csrc/ compiles to an object in parallel; the objects link into
attention_attn_prefill_causal_gb300/libattn.so with the CUDA runtime linked
statically, so the library loads on a machine without a GPU driver (the
driver is only needed when a call reaches the device).  `_calls` is not
linked against libattn.so: the package hands it the library's function
addresses at import.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys
import sysconfig

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")
ROOT = os.path.dirname(PKG)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn")


PYCALLS_SRC = os.path.join(CSRC, "pycalls.c")
PYCALLS = os.path.join(PKG, "_calls" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))


def _deps_mtime() -> float:
    files = [f for f in glob.glob(os.path.join(CSRC, "*")) if f != PYCALLS_SRC]
    files.append(os.path.join(ROOT, "include", "attn.h"))
    return max(os.path.getmtime(f) for f in files)


def _host_cc() -> str:
    for c in (os.environ.get("CC"), shutil.which("gcc"), shutil.which("cc")):
        if c and (os.path.exists(c) or shutil.which(c)):
            return c
    raise RuntimeError("no host C compiler (gcc) found: it builds the _calls extension")


def build_pycalls(force: bool = False) -> str:
    """Compile the _calls extension if its source or the header is newer."""
    hdr = os.path.join(ROOT, "include", "attn.h")
    if (not force and os.path.exists(PYCALLS)
            and os.path.getmtime(PYCALLS) >= max(os.path.getmtime(PYCALLS_SRC),
                                                 os.path.getmtime(hdr))):
        return PYCALLS
    inc = sysconfig.get_paths()["include"]
    if not os.path.exists(os.path.join(inc, "Python.h")):
        raise RuntimeError(f"Python.h not found in {inc}: it builds the _calls extension")
    tmp = PYCALLS + f".tmp{os.getpid()}"
    cmd = [_host_cc(), "-O2", "-shared", "-fPIC", "-Wall", "-I", inc, PYCALLS_SRC,
           "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building _calls failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, PYCALLS)
    return PYCALLS


def _compile(src: str, verbose: bool) -> tuple[str, str]:
    obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
    cmd = [_nvcc(), *ARCH, *FLAGS, "-Xptxas", "-v", "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = r.stdout + r.stderr
    with open(obj + ".log", "w") as f:
        f.write(" ".join(cmd) + "\n" + log)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{log[-4000:]}")
    if verbose:
        print(log, file=sys.stderr)
    return obj, log


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libattn.so if any source is newer than it, and the
    _calls extension likewise."""
    os.makedirs(BUILD, exist_ok=True)
    build_pycalls(force)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = [o for o, _ in ex.map(lambda s: _compile(s, verbose), srcs)]
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", *objs,
           "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
