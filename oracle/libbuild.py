"""Compile the CPU oracle (``oracle.c``) into ``liboracle.so`` with the host C compiler.

Test infrastructure: the oracle is built beside the GPU library so the tests, the smoke check
and the benchmark's CPU-baseline leg can load it; compiling it does not run it, and nothing on the
GPU path links or calls it.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

# -ffp-contract=off: no fused multiply-adds, so every fp64 step rounds exactly as written and
# the result is the same on x86-64 and aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_library(source: str = SOURCE, output: str = LIBRARY) -> str:
    """Compile ``source`` to the shared library ``output`` and return its path."""
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no host C compiler (gcc/cc) found to build the oracle")
    tmp = output + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, output)
    return output


def build(force: bool = False) -> str:
    """Build ``liboracle.so`` unless it is already newer than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= os.path.getmtime(SOURCE)):
        return LIBRARY
    return compile_library()


if __name__ == "__main__":
    print(build(force=True))
