"""Build the tensor-core operand-layout self-test (test support, not part of
libsss) into tests/tc_selftest/_build/libsss_selftest.so for sm_103a."""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libsss_selftest.so")
SRC = os.path.join(HERE, "tc_selftest.cu")


def build(force: bool = False) -> str:
    root = os.path.dirname(os.path.dirname(HERE))
    csrc = os.path.join(root, "selective_ssm_scan_gb300", "csrc")
    deps = [SRC] + [os.path.join(csrc, h) for h in os.listdir(csrc) if h.endswith(".cuh")]
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(d) <= os.path.getmtime(LIB) for d in deps)):
        return LIB
    os.makedirs(OUT, exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
           "-Xcompiler", "-fPIC", "-shared", "-I", os.path.join(root, "include"), SRC, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {SRC}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
