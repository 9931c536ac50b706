"""Build command of the CUDA library librlk_logp.so (sm_103a, in-tree)."""
import glob
import os

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIB_DIR, "librlk_logp.so")
INCLUDE = os.path.join(ROOT, "include")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def commands(nvcc="nvcc"):
    """(argv, output) pairs; empty until the library has sources."""
    src = sources()
    if not src:
        return []
    argv = [nvcc, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
            "-I", INCLUDE, "-I", CSRC, "--threads", "0"] + src + [
            "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64"), "-o", LIB]
    if os.environ.get("RLK_PTXAS_VERBOSE"):
        argv.insert(1, "-Xptxas=-v")
    return [(argv, LIB)]
