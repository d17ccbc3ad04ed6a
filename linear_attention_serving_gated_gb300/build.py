"""Builds libkda.so in-tree from csrc/*.cu for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library next to this file.  Rebuilds only when a source is newer than the
library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import tempfile

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libkda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = srcs + sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")))
    deps.append(os.path.join(os.path.dirname(HERE), "include", "kda.h"))
    return srcs, deps


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    _, deps = _sources()
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    nvcc = _nvcc()
    srcs, _ = _sources()
    with tempfile.TemporaryDirectory(prefix="kda_build_") as tmp:
        procs, objs = [], []
        for s in srcs:
            obj = os.path.join(tmp, os.path.basename(s)[:-3] + ".o")
            objs.append(obj)
            cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", s, "-o", obj]
            if verbose:
                print(" ".join(cmd))
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        failed = []
        for cmd, p in procs:
            out, _ = p.communicate()
            if p.returncode != 0:
                failed.append((cmd, out.decode(errors="replace")))
        if failed:
            raise RuntimeError("nvcc failed:\n" + "\n".join(" ".join(c) + "\n" + o for c, o in failed))
        tmp_lib = os.path.join(tmp, "libkda.so")
        subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp_lib, *objs])
        os.replace(tmp_lib, LIB) if os.path.dirname(tmp_lib) == os.path.dirname(LIB) else shutil.move(tmp_lib, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
