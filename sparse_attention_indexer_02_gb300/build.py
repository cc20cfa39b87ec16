"""Builds libqsa.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu in csrc/ compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically, so the library loads
without any particular libcudart on the search path.  ptxas register/spill
reports go to _build/ptxas_<unit>.log.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import json
import os
import resource
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqsa.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-Xptxas", "-v", f"-I{INCLUDE}"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqsa.so")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def _raise_stack_limit():
    # the compiler recurses deeply on large unrolled kernels: give it the hard stack limit
    soft, hard = resource.getrlimit(resource.RLIMIT_STACK)
    try:
        resource.setrlimit(resource.RLIMIT_STACK, (hard, hard))
    except (ValueError, OSError):
        pass


O0_RECORD = os.path.join(BUILD, "ptxas_O0_units.json")


def _compile(src: str):
    unit = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(BUILD, unit + ".o")
    cmd = [nvcc(), *ARCH, *FLAGS, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True, preexec_fn=_raise_stack_limit)
    o0 = False
    if res.returncode in (139, -11) or "Segmentation fault" in res.stderr:
        # the compiler itself crashed (seen with ptxas 13.0 on aarch64 hosts):
        # rebuild this unit without ptxas optimisation rather than fail the build
        sys.stderr.write(f"WARNING: the CUDA compiler crashed on {unit}.cu; rebuilding it with "
                         f"-Xptxas -O0 (correct but slower code)\n")
        res = subprocess.run(cmd[:-3] + ["-Xptxas", "-O0"] + cmd[-3:], capture_output=True, text=True,
                             preexec_fn=_raise_stack_limit)
        o0 = True
    with open(os.path.join(BUILD, f"ptxas_{unit}.log"), "w") as f:
        f.write(res.stdout + res.stderr)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {unit}.cu:\n{res.stderr[-4000:]}")
    return obj, (unit if o0 else None)


def o0_units() -> list:
    """Units of the current libqsa.so that build() compiled with -Xptxas -O0
    because the optimising compiler crashed (normally none)."""
    try:
        with open(O0_RECORD) as f:
            return list(json.load(f))
    except (OSError, ValueError):
        return []


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        done = list(ex.map(_compile, srcs))
    objs = [o for o, _ in done]
    with open(O0_RECORD, "w") as f:
        json.dump(sorted(u for _, u in done if u), f)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link of libqsa.so failed:\n{res.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        print(f"built {LIB}")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
