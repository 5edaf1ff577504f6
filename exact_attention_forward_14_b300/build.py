"""Build the CUDA libraries of this package in-tree with nvcc (sm_103a only).

    python -m exact_attention_forward_14_b300.build [--force] [--verbose]

Produces, next to this file:
  libattn_b300.so           the attention library (C ABI in include/attn_b300.h)
  libattn_selftest.so       single-tile tensor-core layout checks used by the tests, and
                            the MUFU exp2 throughput microbenchmark
  libattn_watchdog_test.so  test-only build of the library whose Q barrier is
                            never armed, so every launch ends through the
                            watchdog (bounded wait -> ATTN_ERR_TIMEOUT)
"""
from __future__ import annotations

import argparse
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2",
    "-shared",
    "-I" + INCLUDE, "-I" + CSRC,
]

# name -> (sources, extra nvcc flags)
TARGETS = {
    "libattn_b300.so": (["attn_api.cu"], []),
    "libattn_selftest.so": (["selftest_umma.cu", "mufu_rate.cu"], []),
    "libattn_watchdog_test.so": (["attn_api.cu"], ["-DATTN_TEST_NEVER_ARM_Q"]),
}


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> list[str]:
    deps = (glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h"))
            + [os.path.abspath(__file__)])
    built = []
    for name, (srcs, extra) in TARGETS.items():
        out = os.path.join(PKG, name)
        if not force and not _stale(out, deps):
            continue
        tmp = out + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *NVCC_FLAGS, *extra, *(["-Xptxas", "-v"] if verbose else []),
               *[os.path.join(CSRC, s) for s in srcs], "-o", tmp]
        if verbose:
            print(" ".join(cmd), flush=True)
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
        built.append(out)
    return built


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args(argv)
    for p in build(force=a.force, verbose=a.verbose):
        print("built", p)
    return 0


if __name__ == "__main__":
    sys.exit(main())
