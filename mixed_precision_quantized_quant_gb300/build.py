"""Builds libkvq.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu under csrc/ is compiled to an object in parallel, then linked into
mixed_precision_quantized_quant_gb300/libkvq.so.  Objects go to _build/ at the
repository root; both are git-ignored.  Rebuilds only what changed.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libkvq.so")
# debug variant: every kernel checks its computed accesses against the buffers
# it was given and records kErrBadAddress instead of touching memory outside them
DEBUG_BUILD = os.path.join(ROOT, "_build", "debug")
DEBUG_LIB = os.path.join(PKG, "libkvq_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs.append(os.path.join(ROOT, "include", "kvq.h"))
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, verbose: bool, defines=()) -> str:
    cmd = [nvcc(), *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}\n{res.stderr}")
    return res.stderr


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Builds libkvq.so, or with debug=True libkvq_debug.so (compiled with
    KVQ_DEBUG: device-side range checks of computed accesses)."""
    bdir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug else (BUILD, LIB)
    defines = ("-DKVQ_DEBUG",) if debug else ()
    os.makedirs(bdir, exist_ok=True)
    srcs = _sources()
    hdrs = _headers()
    objs = [os.path.join(bdir, os.path.basename(s)[:-3] + ".o") for s in srcs]
    todo = [(s, o) for s, o in zip(srcs, objs) if force or _stale(o, [s, *hdrs])]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=min(len(todo), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(lambda so: _compile(so[0], so[1], verbose, defines), todo))
        if verbose:
            for (s, _), log in zip(todo, logs):
                print(f"== {os.path.basename(s)}\n{log}", file=sys.stderr)
    if force or todo or _stale(lib, objs):
        cmd = [nvcc(), *ARCH, "-shared", "-o", lib, *objs, "-lcudart"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))
