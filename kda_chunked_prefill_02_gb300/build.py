"""Build the KDA CUDA library in-tree for sm_103a.

    python -m kda_chunked_prefill_02_gb300.build [--force]

Compiles csrc/*.cu (one nvcc per translation unit, in parallel) and links
  libkda.so          the product library (C ABI of include/kda.h)
  libkda_selftest.so test-only checks of the tcgen05 / TMA building blocks
next to this file.  Objects go to _build/ (git-ignored).
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
ROOT = os.path.dirname(HERE)
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "-I" + os.path.join(ROOT, "include"), "-diag-suppress", "1160"]

LIB_SOURCES = ["kda_api.cu", "kda_prep.cu", "kda_state.cu", "kda_state_head.cu", "kda_verify.cu",
               "kda_verify_wy.cu", "kda_noalloc.cu", "kda_host.cu"]
SELFTEST_SOURCES = ["selftest.cu"]
HEADERS = ["sm103.cuh", "kda_internal.h", "tmap.h"]

LIB = os.path.join(HERE, "libkda.so")
SELFTEST_LIB = os.path.join(HERE, "libkda_selftest.so")


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_input(srcs):
    files = [os.path.join(CSRC, s) for s in srcs + HEADERS] + [
        os.path.join(ROOT, "include", "kda.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def _compile(src):
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
    cmd = [_nvcc()] + ARCH + FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return obj


def _link(objs, out):
    tmp = out + ".tmp.%d" % os.getpid()
    cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed for %s:\n%s\n%s" % (out, r.stdout, r.stderr))
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    todo = []
    for out, srcs in ((LIB, LIB_SOURCES), (SELFTEST_LIB, SELFTEST_SOURCES)):
        if force or not os.path.exists(out) or os.path.getmtime(out) < _newest_input(srcs):
            todo.append((out, srcs))
    if not todo:
        return LIB
    all_srcs = sorted({s for _, srcs in todo for s in srcs})
    with cf.ThreadPoolExecutor(max_workers=min(8, len(all_srcs))) as ex:
        objs = dict(zip(all_srcs, ex.map(_compile, all_srcs)))
    for out, srcs in todo:
        _link([objs[s] for s in srcs], out)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
