"""Build libmla_decode.so in-tree with nvcc for sm_103a (no cmake, no torch).

Each .cu file compiles to an object in parallel; the objects link into one
shared library with the CUDA runtime linked statically, so the library loads
on a machine without a GPU driver (the exported symbols can be inspected
there; calling them needs a GPU).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmla_decode.so")
SOURCES = ["mla_api.cu", "kv_write.cu", "plan_merge.cu", "decode_sm103.cu", "uv_project.cu", "selftest.cu"]
HEADERS = ["ptx.cuh", "mla_internal.h", "trace.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _deps():
    inc = os.path.join(os.path.dirname(HERE), "include", "mla_decode.h")
    return [os.path.join(CSRC, h) for h in HEADERS] + [inc, os.path.abspath(__file__)]


def _stale(target, inputs):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(i) > t for i in inputs)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, defines=(),
          lib_path: str = LIB, build_dir: str = BUILD) -> str:
    """Compile every kernel file and link libmla_decode.so (only what is stale).
    `defines` (e.g. ["-DMLA_TRACE"] for the event-traced build) go with
    their own lib_path and build_dir."""
    os.makedirs(build_dir, exist_ok=True)
    deps = _deps()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "--expt-relaxed-constexpr", *defines]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or ptxas_info or _stale(o, [s] + deps):
            jobs.append([nvcc(), *flags, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4) or 1) as ex:
        for log in ex.map(run, jobs):
            if verbose and log:
                print(log)
    if force or jobs or _stale(lib_path, objs):
        tmp = lib_path + ".tmp.%d" % os.getpid()
        run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
