"""Build libmla.so (sm_103a) in-tree with nvcc, and its bounds-checked twin libmla_checks.so.

    python -m sparse_latent_attention_norm_b300.build [--force] [-v] [--checks]

libmla_checks.so is the same library compiled with MLA_CHECKS: every gather index, TMA
coordinate and output row is checked before use; a failed check records MLA_ERR_BOUNDS in the
status word and skips the access instead of trapping. It is a diagnostic build (the checks cost
a little time); the product is libmla.so.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libmla.so")
LIB_CHECKS = os.path.join(PKG, "libmla_checks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources() -> list[str]:
    out = [os.path.join(INCLUDE, "mla.h")]
    for f in sorted(os.listdir(CSRC)):
        if f.endswith((".cu", ".cuh", ".h")):
            out.append(os.path.join(CSRC, f))
    return out


def nvcc_command(output: str = LIB, extra: list[str] | None = None) -> list[str]:
    nvcc = os.environ.get("NVCC", "nvcc")
    return [nvcc, *ARCH, "-lineinfo", "-O3", "-std=c++17", "-shared", "-Xcompiler", "-fPIC,-fvisibility=hidden",
            f"-I{INCLUDE}", *(extra or []), "-o", output, os.path.join(CSRC, "mla.cu")]


def build(force: bool = False, verbose: bool = False, checks: bool = False) -> str:
    """Compile libmla.so (or, with checks=True, libmla_checks.so) unless it is newer than every
    source. Returns its path."""
    lib = LIB_CHECKS if checks else LIB
    if not force and os.path.exists(lib):
        t = os.path.getmtime(lib)
        if all(os.path.getmtime(s) <= t for s in sources()):
            return lib
    tmp = lib + ".tmp"
    extra = (["-Xptxas", "-v"] if verbose else []) + (["-DMLA_CHECKS"] if checks else [])
    cmd = nvcc_command(tmp, extra)
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed building libmla.so")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checks="--checks" in sys.argv))
