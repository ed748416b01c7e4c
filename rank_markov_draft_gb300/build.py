"""Build libdspark.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each .cu translation unit is compiled in parallel, then linked into one shared
library (CUDA runtime linked statically, no libcuda link: the TMA descriptor
encoder is fetched through the runtime's driver entry-point query).

The same build links libdspark_debug.so: the draft kernel compiled with
DSPARK_DEVICE_CHECKS (device-side checks of its TMEM and shared-memory
offsets, reported as DSPARK_ERR_DEVICE_OOB), the other units shared.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdspark.so")
LIB_DEBUG = os.path.join(BUILD, "libdspark_debug.so")
CHECKED = "draft.cu"  # the unit that holds the checks
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "draft.cu", "gate.cu", "selector.cu", "confidence.cu", "noalloc.cu", "verify.cu",
           "schedule.cu", "label.cu", "calibrate.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdspark")
    return path


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "dspark.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not os.path.exists(LIB_DEBUG):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(LIB_DEBUG))
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-diag-suppress", "1160", "-I", INCLUDE]

    def compile_one(job):
        src, checked = job
        stem = os.path.splitext(src)[0] + ("_checked" if checked else "")
        obj = os.path.join(BUILD, stem + ".o")
        flags = ["-DDSPARK_DEVICE_CHECKS=1"] if checked else []
        cmd = [cc] + common + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    jobs = [(CHECKED, True)] + [(src, False) for src in SOURCES]  # the longest unit first
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    checked_obj, objs = objs[0], objs[1:]
    plain = [o for o, src in zip(objs, SOURCES) if src != CHECKED]
    release = objs
    debug = plain + [checked_obj]
    for lib, parts in ((LIB, release), (LIB_DEBUG, debug)):
        tmp = lib + f".{os.getpid()}.tmp"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + parts + ["-cudart", "static"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
