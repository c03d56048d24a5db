"""Builds the generator's two small libraries in-tree.

libsynth.so      host fills (gcc, plain C; -ffp-contract=off keeps the gs64
                 scale's two separate roundings)
libsynth_dev.so  device fills for sm_103a (nvcc), for weights too large to
                 generate on the host and upload
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_SO = os.path.join(HERE, "libsynth.so")
DEV_SO = os.path.join(HERE, "libsynth_dev.so")


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(s) > t for s in srcs)


def build_host(force=False):
    srcs = [os.path.join(HERE, "synth_host.c"), os.path.join(HERE, "synth.h")]
    if force or _stale(HOST_SO, srcs):
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-ffp-contract=off", "-fvisibility=hidden",
                               "-o", HOST_SO, srcs[0], "-lm"])
    return HOST_SO


def build_dev(force=False):
    srcs = [os.path.join(HERE, "synth_dev.cu"), os.path.join(HERE, "synth.h")]
    if force or _stale(DEV_SO, srcs):
        nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
        subprocess.check_call([nvcc, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
                               "-Xcompiler", "-fvisibility=hidden",
                               "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
                               "-cudart", "static", "-o", DEV_SO, srcs[0]])
    return DEV_SO


def build(force=False):
    build_host(force)
    build_dev(force)


if __name__ == "__main__":
    build(force=True)
