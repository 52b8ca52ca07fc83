"""Builds ``libtensor_core_tiled.so`` in-tree with nvcc for sm_103a (no CMake, no torch).

Each translation unit compiles in its own nvcc process (in parallel); the objects link into
one shared library whose CUDA runtime is static, so the library loads on a machine without
a GPU driver (symbols can be inspected there; calls need a GPU).
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_NAME = "libtensor_core_tiled.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
# (source, object, extra flags): the GEMM kernel source compiles as two objects in parallel,
# each holding the kernels of a share of the operand layouts (TCT_PART 0 and 1).
SOURCES = [("gemm_sm103a.cu", "gemm_sm103a_part0.o", ["-DTCT_PART=0"]),
           ("gemm_sm103a.cu", "gemm_sm103a_part1.o", ["-DTCT_PART=1"]),
           ("api.cu", "api.o", []), ("softmax_sm103a.cu", "softmax_sm103a.o", []),
           ("probe_sm103a.cu", "probe_sm103a.o", [])]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "tensor_core_tiled.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale():
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(f) > t for f in _deps())


def build(force=False, verbose=False, extra_flags=()):
    """Compile and link the library if any source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    common = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]

    def compile_one(job):
        src, obj_name, flags = job
        obj = os.path.join(BUILD_DIR, obj_name)
        cmd = common + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
