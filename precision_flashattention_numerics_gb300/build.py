"""Build libpasa.so in-tree with nvcc for sm_103a (one translation unit, seconds)."""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "pasa_lib.cu")
LIB = os.path.join(HERE, "libpasa.so")
NVCC_FLAGS = [
    "-std=c++17", "-O3", "-lineinfo",
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-shared", "-Xcompiler", "-fPIC",
]


def _sources():
    out = [os.path.join(HERE, "..", "include", "pasa.h")]
    for f in sorted(os.listdir(os.path.join(HERE, "csrc"))):
        out.append(os.path.join(HERE, "csrc", f))
    return out


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile csrc/pasa_lib.cu into libpasa.so next to this file; returns its path."""
    if not force and not needs_build():
        return LIB
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *NVCC_FLAGS, "-o", tmp, SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
