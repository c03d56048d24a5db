"""Builds libmoe.so, the sm_103a CUDA library behind include/moe.h, in-tree.

Each .cu file is compiled to an object in parallel, then linked.  Only
`-gencode arch=compute_103a,code=sm_103a` is emitted: the library runs on
GB300 and nowhere else.
"""
import concurrent.futures as cf
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
SO = os.path.join(HERE, "libmoe.so")
ROOT = os.path.dirname(HERE)
SOURCES = ["router.cu", "dispatch.cu", "gemv.cu", "ggemm_tc.cu", "misc.cu", "moe_api.cu",
           "route_trace.cu", "decode_tc.cu"]
HEADERS = ["moe_internal.cuh", "ptx.cuh", "tc.cuh"]

NVCC_FLAGS = ["-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
              "-Xptxas", "-warn-spills", "-I", os.path.join(ROOT, "include")]


def nvcc():
    return os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(force=False, verbose=False, extra_flags=()):
    os.makedirs(BUILD, exist_ok=True)
    deps = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "moe.h")]
    dep_t = _newest(deps)
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        objs.append(o)
        if force or not os.path.exists(o) or os.path.getmtime(o) < max(dep_t, os.path.getmtime(s)):
            jobs.append([nvcc(), *NVCC_FLAGS, *extra_flags, "-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
            if verbose or res.returncode != 0:
                print(" ".join(cmd))
                print(res.stdout + res.stderr)
            if res.returncode != 0:
                raise RuntimeError("nvcc failed for %s" % cmd[-3])
    if jobs or not os.path.exists(SO) or os.path.getmtime(SO) < _newest(objs):
        subprocess.check_call([nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-cudart", "static", "-o", SO, *objs])
    return SO


if __name__ == "__main__":
    import sys
    build(force=True, verbose="-v" in sys.argv)
