"""Build and run the GB300 micro-benchmarks in probes.cu (a measurement tool).

    python -m tiled_attention_flashattention_gb300.probes

Compiles probes.cu for sm_103a into the package's _build_probes/ folder with
nvcc and runs it on GPU 0: per-SM instruction rates of the softmax's
instruction mix, the issue rate of back-to-back tcgen05.mma by shape and
operand source, and single-thread synchronisation latencies.
"""
import os
import subprocess
import sys

from .. import _build

HERE = os.path.dirname(os.path.abspath(__file__))


def main() -> int:
    out_dir = os.path.join(os.path.dirname(HERE), "_build_probes")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "probes")
    cmd = [_build._nvcc(), *_build.ARCH, "-O3", "-std=c++17", "-I", _build.INCLUDE, "-I", _build.CSRC,
           os.path.join(HERE, "probes.cu"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        return r.returncode
    return subprocess.run([exe]).returncode


if __name__ == "__main__":
    sys.exit(main())
