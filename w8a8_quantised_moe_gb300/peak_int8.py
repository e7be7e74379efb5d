"""Measure the contraction rates behind the layer's compute roofline (the
cases are listed in peak_int8.cu): tcgen05 kind::f16 on int8-valued fp16
operands (one CTA and CTA pairs, A in shared or tensor memory), tcgen05
kind::f8f6f4 (E4M3) and mma.sync s8.  Builds the program in-tree with nvcc,
runs it on the current GPU and prints its JSON line.

    python -m w8a8_quantised_moe_gb300.peak_int8
"""
import os
import subprocess
import sys

from w8a8_quantised_moe_gb300 import build as lib_build

HERE = os.path.dirname(os.path.abspath(__file__))


def main() -> int:
    exe = os.path.join(lib_build.BUILD, "peak_int8")
    os.makedirs(lib_build.BUILD, exist_ok=True)
    subprocess.run([lib_build.nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-I", os.path.join(lib_build.ROOT, "include"), "-I", HERE,
                    os.path.join(HERE, "peak_int8.cu"), "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    sys.stdout.write(r.stdout)
    sys.stderr.write(r.stderr)
    return r.returncode


if __name__ == "__main__":
    sys.exit(main())
