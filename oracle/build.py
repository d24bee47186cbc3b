"""Build step for the CPU oracle (test infrastructure only).

Compiles ``pkv_oracle.cpp`` with the host C++ compiler into
``oracle/_build/libpkv_oracle.so``. Plain ``-O2`` with no architecture flags
and no floating-point contraction, so the same source builds and rounds the
same way on x86_64 and aarch64 hosts.
"""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "pkv_oracle.cpp")
BUILD_DIR = os.path.join(HERE, "_build")
LIBRARY = os.path.join(BUILD_DIR, "libpkv_oracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIBRARY + f".tmp{os.getpid()}"
    # no fused multiply-add contraction: the same results on x86 and Arm hosts
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           "-o", tmp, SOURCE]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True))
