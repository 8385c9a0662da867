"""Build the CPU oracle's shared library (test infrastructure only).

Plain gcc, no vectorising or fast-math flags that could change rounding:
``-ffp-contract=off`` keeps every multiply and add a separately rounded IEEE
binary32/binary64 operation (gcc fuses them by default on aarch64).
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libnvfp4_oracle.so")
SOURCES = [os.path.join(HERE, "nvfp4_oracle.c")]
HEADERS = [os.path.join(HERE, "nvfp4_oracle.h")]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in SOURCES + HEADERS)


def build(force: bool = False) -> str:
    """Compile ``libnvfp4_oracle.so`` if missing or out of date; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-Wextra", "-o", tmp] + SOURCES + ["-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
