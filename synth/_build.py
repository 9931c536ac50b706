"""Build commands for the seeded-input generator (host C and CUDA builds)."""
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_DIR = os.path.join(HERE, "_lib")
HOST_LIB = os.path.join(LIB_DIR, "libsynth_host.so")
DEV_LIB = os.path.join(LIB_DIR, "libsynth_dev.so")


def commands(nvcc="nvcc", cc="gcc"):
    """(argv, output) pairs; the caller runs them (in parallel) after making LIB_DIR."""
    host = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-pthread",
            os.path.join(HERE, "synth_host.c"), "-o", HOST_LIB]
    dev = [nvcc, "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC", "--fmad=false",
           "-gencode", "arch=compute_103a,code=sm_103a",
           os.path.join(HERE, "synth_dev.cu"), "-o", DEV_LIB]
    return [(host, HOST_LIB), (dev, DEV_LIB)]
