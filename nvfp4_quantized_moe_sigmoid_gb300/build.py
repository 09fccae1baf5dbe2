"""In-tree build of libnvfp4moe.so (the C-ABI CUDA library) for sm_103a."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libnvfp4moe.so")
SRC_DIR = os.path.join(HERE, "csrc")
MAIN = os.path.join(SRC_DIR, "nvfp4moe.cu")
HEADER = os.path.join(ROOT, "include", "nvfp4moe.h")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return [os.path.join(SRC_DIR, f) for f in sorted(os.listdir(SRC_DIR))
            if f.endswith((".cu", ".cuh"))] + [HEADER]


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, extra_flags=None) -> str:
    if not force and not stale():
        return LIB
    cmd = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", LIB + ".tmp", MAIN]
    if extra_flags:
        cmd[1:1] = list(extra_flags)
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
