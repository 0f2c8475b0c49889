"""Build ``libmoira.so`` in-tree with nvcc for sm_103a (GB300).

Each .cu file is compiled in parallel; the objects are linked into a shared
library against the shared CUDA runtime (the same libcudart PyTorch loads, so
streams and graphs from PyTorch can be passed straight through).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
SOURCES = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
HEADERS = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
LIB = os.path.join(HERE, "libmoira.so")
# The load-balance build: the same library with per-block attention timings
# (include/moira_cta_times.h); the translation units that differ are rebuilt
# with MOIRA_CTA_TIMES and linked with the others.
LIB_CTA_TIMES = os.path.join(HERE, "libmoira_cta_times.so")
CTA_TIMES_SOURCES = ("api.cu", "attend.cu", "fused.cu")
BUILD_DIR = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MOIRA CUDA library cannot be built")


def _stale() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(LIB_CTA_TIMES):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(LIB_CTA_TIMES))
    deps = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    deps.append(os.path.join(ROOT, "include", "moira.h"))
    deps.append(os.path.join(ROOT, "include", "moira_cta_times.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile (if stale) libmoira.so and its load-balance build; return the
    path of libmoira.so."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    objs_cta = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        if src in CTA_TIMES_SOURCES:
            obj_cta = os.path.join(BUILD_DIR, src.replace(".cu", "_cta_times.o"))
            objs_cta.append(obj_cta)
            cmd = [cc] + flags + ["-DMOIRA_CTA_TIMES", "-c", os.path.join(CSRC, src), "-o", obj_cta]
            procs.append((src + " (cta times)",
                          subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        else:
            objs_cta.append(obj)
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append((src, text))
        elif verbose or ptxas_info:
            sys.stdout.write(text)
    if failed:
        msg = "\n".join(f"--- {s} ---\n{t}" for s, t in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    for lib, obj_list in ((LIB, objs), (LIB_CTA_TIMES, objs_cta)):
        tmp = lib + ".tmp"
        subprocess.run([cc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + obj_list, check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv))
