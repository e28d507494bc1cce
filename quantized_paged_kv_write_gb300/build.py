"""Build libkvq.so in-tree with nvcc for sm_103a (GB300).

Each .cu translation unit compiles in parallel to an object file; the objects
are linked into ``libkvq.so`` next to this file.  No cmake, no torch
extension machinery: the library is plain C ABI (include/kvq.h).

Rebuilds are decided by content, not by file times: every object records the
hash of what it was compiled from (its source, every header, the flags), and
the library embeds the hash of all sources (``kvq_build_id()``), so a library
or object left from other sources is never reused.
"""
from __future__ import annotations

import concurrent.futures
import hashlib
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libkvq.so")
HEADER = os.path.join(ROOT, "include", "kvq.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _all_inputs():
    """Every file the library is built from: csrc/* and include/kvq.h."""
    files = sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                   if f.endswith((".cu", ".cuh", ".h")))
    return files + [HEADER]


def _digest(paths, extra=()) -> str:
    h = hashlib.sha256()
    for p in paths:
        h.update(os.path.relpath(p, ROOT).encode())
        with open(p, "rb") as f:
            h.update(f.read())
    for x in extra:
        h.update(x.encode())
    return h.hexdigest()[:16]


def source_hash() -> str:
    """The build id: a hash over every kernel source, header and the build flags."""
    return _digest(_all_inputs(), ARCH + FLAGS)


def _read(path: str) -> str:
    try:
        with open(path) as f:
            return f.read().strip()
    except OSError:
        return ""


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs]
    heads = [p for p in _all_inputs() if not p.endswith(".cu")]
    bid = source_hash()

    def compile_one(pair):
        src, obj = pair
        extra = ["-DKVQ_BUILD_ID=\"%s\"" % bid] if os.path.basename(src) == "kvq_api.cu" else []
        want = _digest([src] + heads, ARCH + FLAGS + extra)
        stamp = obj + ".hash"
        if not ptxas_info and os.path.exists(obj) and _read(stamp) == want:
            return ""
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        if ptxas_info:
            cmd += ["-Xptxas", "-v"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{res.stderr}")
        with open(stamp, "w") as f:
            f.write(want)
        return res.stderr

    jobs = min(len(srcs), os.cpu_count() or 4)
    with concurrent.futures.ThreadPoolExecutor(jobs) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    if verbose or ptxas_info:
        for s, lg in zip(srcs, logs):
            if lg:
                print(f"== {os.path.basename(s)}\n{lg}", file=sys.stderr)
    lib_stamp = os.path.join(BUILD, "libkvq.so.hash")
    if not os.path.exists(LIB) or _read(lib_stamp) != bid:
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stderr}")
        os.replace(LIB + ".tmp", LIB)
        with open(lib_stamp, "w") as f:
            f.write(bid)
    return LIB


if __name__ == "__main__":
    build(verbose=True, ptxas_info="--ptxas" in sys.argv)
    print(LIB)
