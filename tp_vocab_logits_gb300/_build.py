"""Build of libhg.so: the CUDA kernels and the C ABI, for sm_103a only.

Each .cu file under csrc/ is compiled by nvcc in parallel, then linked into
tp_vocab_logits_gb300/libhg.so (static CUDA runtime, so the library needs
nothing beyond the CUDA driver at run time). ptxas resource usage (registers,
spills, shared memory) of the last build is kept in _build/ptxas.log.

Alongside, csrc/hg_pycall.c is compiled with the host C compiler into the
CPython extension _hgcall (the Python binding's direct-call object).
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
import sysconfig

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libhg.so")
PYCALL_SRC = os.path.join(CSRC, "hg_pycall.c")
PYCALL = os.path.join(PKG, "_hgcall" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libhg.so")
    return exe


def sources() -> list:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(PYCALL):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(PYCALL))
    return any(os.path.getmtime(p) > t for p in _deps() + [PYCALL_SRC, __file__])


def _pycall_cmd(out: str) -> list:
    cc = shutil.which("gcc") or shutil.which("cc")
    if not cc:
        raise RuntimeError("a C compiler (gcc) is required to build the _hgcall extension")
    inc = sysconfig.get_paths()["include"]
    if not os.path.exists(os.path.join(inc, "Python.h")):
        raise RuntimeError(f"Python.h not found under {inc}: the _hgcall extension needs it")
    return [cc, "-O2", "-shared", "-fPIC", "-Wall", f"-I{inc}", PYCALL_SRC, "-o", out]


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libhg.so if it is missing or older than its sources."""
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    exe = nvcc()
    procs = []
    objs = []
    pycall_tmp = PYCALL + f".{os.getpid()}.tmp"
    procs.append((PYCALL_SRC, subprocess.Popen(_pycall_cmd(pycall_tmp), stdout=subprocess.PIPE,
                                               stderr=subprocess.STDOUT, text=True)))
    for src in sources():
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [exe, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    logs = []
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        logs.append(f"== {os.path.basename(src)}\n{out}")
        if p.returncode != 0:
            failed.append(src)
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        f.write("\n".join(logs))
    if failed:
        sys.stderr.write("\n".join(logs))
        raise RuntimeError(f"nvcc failed on {', '.join(os.path.basename(s) for s in failed)}")
    tmp = LIB + f".{os.getpid()}.tmp"
    subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIB)
    os.replace(pycall_tmp, PYCALL)
    if verbose:
        print("\n".join(logs))
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
