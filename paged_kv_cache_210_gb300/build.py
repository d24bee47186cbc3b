"""Build step: compile the CUDA library for sm_103a into ``_build/libpkv.so``.

The CUDA sources (``csrc/*.cu``, compiled for ``compute_103a``/``sm_103a``
only) and the host-only C++ sources (``csrc/*.cpp``: the admission
scheduler) go into one position-independent library with the CUDA runtime
linked statically, so it loads beside any PyTorch build. Rebuilds when a
source or a public header is newer than the library.
"""

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libpkv.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")) +
                  glob.glob(os.path.join(HERE, "csrc", "*.cpp")))


def _stale():
    if not os.path.exists(LIBRARY):
        return True
    newest = max(os.path.getmtime(p) for p in sources() + glob.glob(os.path.join(INCLUDE, "*.h"))
                 + glob.glob(os.path.join(HERE, "csrc", "*.cuh"))
                 + glob.glob(os.path.join(HERE, "csrc", "*.h")))
    return os.path.getmtime(LIBRARY) < newest


def nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libpkv.so if missing or stale; returns its path."""
    if not force and not _stale():
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "-cudart", "static", "-I", INCLUDE, "-o", tmp, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose=True))
