"""Compile the test-only CUDA helpers in this folder (sm_103a) next to their
sources.  Used by __graft_entry__.build() and, when the helper is missing, by
the tests that need it."""

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
PROBES = {"curand_philox_probe": "curand_philox_probe.cu"}


def probe_path(name):
    return os.path.join(HERE, f"lib{name}.so")


def build(name="curand_philox_probe", force=False):
    out = probe_path(name)
    src = os.path.join(HERE, PROBES[name])
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    cmd = [nvcc if os.path.exists(nvcc) else "nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O2",
           "-std=c++17", "-Xcompiler", "-fPIC", "-shared", "-cudart", "static", "-o", out, src]
    subprocess.run(cmd, check=True)
    return out


if __name__ == "__main__":
    for n in PROBES:
        print(build(n, force=True))
