"""Build the fp64 CPU oracle (``fmha_oracle.c``) into ``oracle/liboracle.so``.

TEST INFRASTRUCTURE: the oracle is the parity checker for the CUDA library; it
is built here so that tests, the smoke check and the benchmark's CPU-baseline
leg can load it.  Plain C, no architecture-specific flags, so the same source
builds on x86_64 and aarch64 hosts.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fmha_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    base = [cc, "-O2", "-std=c99", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       stdout=subprocess.PIPE, stderr=subprocess.PIPE)
    except subprocess.CalledProcessError:
        # No OpenMP runtime on this host: the serial build computes the same.
        subprocess.run(base, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
