"""Builds the synthetic-input generator: a host library (gcc) and a device
library (nvcc, sm_103a). Both compile gen.h with floating-point contraction
disabled so their outputs agree bit for bit."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
HOST_LIB = os.path.join(HERE, "libnvfp4gen_host.so")
CUDA_LIB = os.path.join(HERE, "libnvfp4gen_cuda.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")


def _stale(lib, srcs):
    return not os.path.exists(lib) or any(os.path.getmtime(lib) < os.path.getmtime(s) for s in srcs)


def build_host(force: bool = False) -> str:
    srcs = [os.path.join(HERE, "gen_host.c"), os.path.join(HERE, "gen.h")]
    if force or _stale(HOST_LIB, srcs):
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-fno-math-errno", "-fopenmp", "-o", HOST_LIB + ".tmp", srcs[0], "-lm"],
                       check=True)
        os.replace(HOST_LIB + ".tmp", HOST_LIB)
    return HOST_LIB


def build_cuda(force: bool = False) -> str:
    srcs = [os.path.join(HERE, "gen_cuda.cu"), os.path.join(HERE, "gen.h")]
    if force or _stale(CUDA_LIB, srcs):
        subprocess.run([NVCC, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-fmad=false",
                        "-Xcompiler", "-fPIC", "-shared", "-o", CUDA_LIB + ".tmp", srcs[0]],
                       check=True)
        os.replace(CUDA_LIB + ".tmp", CUDA_LIB)
    return CUDA_LIB


def build(force: bool = False):
    return build_host(force), build_cuda(force)


if __name__ == "__main__":
    print(build(force=True))
