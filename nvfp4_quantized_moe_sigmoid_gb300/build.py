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
            if f.endswith((".cu", ".cuh"))] + [os.path.join(ROOT, "include", f) for f in
                                               sorted(os.listdir(os.path.join(ROOT, "include")))]


# The phase-trace variant of the library (-DNVFP4MOE_TRACE): the same kernels
# plus global-timer records at the phase boundaries of the stack kernel, read
# back by nvfp4moe_stack_trace_read. Loaded only when NVFP4MOE_LIB names it.
TRACE_LIB = os.path.join(HERE, "libnvfp4moe_trace.so")


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, extra_flags=None, lib: str = LIB) -> str:
    if not force and not stale(lib):
        return lib
    cmd = [NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-I", os.path.join(ROOT, "include"), "-o", lib + ".tmp", MAIN]
    if extra_flags:
        cmd[1:1] = list(extra_flags)
    subprocess.run(cmd, check=True)
    os.replace(lib + ".tmp", lib)
    return lib


def build_trace(force: bool = False) -> str:
    return build(force, ["-DNVFP4MOE_TRACE"], TRACE_LIB)


if __name__ == "__main__":
    print(build(force=True))
