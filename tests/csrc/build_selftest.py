"""Builds the test-only tensor-core self-test library (tests/csrc/umma_selftest.cu)."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
OUT = os.path.join(HERE, "_build", "libumma_selftest.so")
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def build() -> str:
    from gated_deltanet_linear_conv1d_gb300 import build as gdn_build
    src = os.path.join(HERE, "umma_selftest.cu")
    deps = [src, os.path.join(gdn_build.CSRC, "umma.cuh"), os.path.join(gdn_build.CSRC, "device.cuh")]
    if os.path.exists(OUT) and os.path.getmtime(OUT) >= max(os.path.getmtime(d) for d in deps):
        return OUT
    os.makedirs(os.path.dirname(OUT), exist_ok=True)
    tmp = OUT + f".tmp{os.getpid()}"
    cmd = [gdn_build.nvcc(), *gdn_build.ARCH, *gdn_build.NVCC_FLAGS, "-shared", "-o", tmp, src,
           "-cudart", "static"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build())
