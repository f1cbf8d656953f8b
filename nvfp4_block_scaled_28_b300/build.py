"""Build the in-tree shared libraries for sm_103a.

``libnvfp4_b300.so``   the C-ABI library of include/nvfp4.h: one nvcc
                       invocation over every ``csrc/*.cu``;
``libnvfp4_probe.so``  the measurement library of include/nvfp4_probe.h
                       (the dense FP4 tensor-core peak probe, ``probe/``);
                       it is not part of the product library;
``libnvfp4_b300_debug.so``  the same C ABI and kernels compiled with
                       NVFP4_DEBUG_CHECKS (and relocatable device code):
                       every index a kernel forms for a global or shared
                       access is checked, a failure recorded in the device
                       error word and the access skipped. Loaded instead of
                       the product library when NVFP4_B300_DEBUG=1.

All link the CUDA runtime statically; the driver API is reached at run time
through cudaGetDriverEntryPointByVersion, so the libraries load on machines
without a GPU driver. No fast-math: the quantizer's bytes depend on IEEE
binary32 division, reciprocal and multiplication.

A library is rebuilt when the SHA-256 of its inputs (every source and header
it is built from, this file, and the nvcc command line) differs from the one
recorded beside it when it was last built; file times play no part, so a
copied tree or a restored checkout cannot skip a rebuild.
"""
from __future__ import annotations

import glob
import hashlib
import json
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
PROBE_SRC = os.path.join(PKG_DIR, "probe")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libnvfp4_b300.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
PROBE_LIB_PATH = os.path.join(PKG_DIR, "libnvfp4_probe.so")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libnvfp4_b300_debug.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-shared",
              "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
              "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build")
    return cand


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def probe_sources():
    return sorted(glob.glob(os.path.join(PROBE_SRC, "*.cu")))


def _headers():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


class Target:
    def __init__(self, path, srcs, extra_flags=()):
        self.path = path
        self.srcs = srcs
        self.extra_flags = list(extra_flags)

    @property
    def stamp(self):
        return self.path + ".sha256"

    def command(self, out):
        return ([nvcc()] + ARCH_FLAGS + NVCC_FLAGS + self.extra_flags +
                ["-I", INCLUDE, "-I", CSRC, "-o", out] + self.srcs)

    def digest(self):
        h = hashlib.sha256()
        for p in self.srcs + _headers() + [os.path.abspath(__file__)]:
            h.update(os.path.relpath(p, ROOT).encode())
            with open(p, "rb") as f:
                h.update(hashlib.sha256(f.read()).digest())
        # the command line without the output path and the nvcc location
        h.update(json.dumps(ARCH_FLAGS + NVCC_FLAGS + self.extra_flags).encode())
        return h.hexdigest()

    def up_to_date(self):
        if not (os.path.exists(self.path) and os.path.exists(self.stamp)):
            return False
        with open(self.stamp) as f:
            return f.read().strip() == self.digest()


def product_target():
    return Target(LIB_PATH, sources())


def probe_target():
    return Target(PROBE_LIB_PATH, probe_sources())


def debug_target():
    return Target(DEBUG_LIB_PATH, sources(), ["-DNVFP4_DEBUG_CHECKS", "-rdc=true"])


def up_to_date() -> bool:
    return product_target().up_to_date()


def _build(t: Target, force: bool, verbose: bool) -> str:
    if not force and t.up_to_date():
        return t.path
    digest = t.digest()
    tmp = t.path + ".tmp.%d" % os.getpid()
    cmd = t.command(tmp)
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.splitext(t.path)[0] + ".build.log"
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError("nvcc failed (see %s)" % log)
    if verbose:
        sys.stdout.write(res.stdout + res.stderr)
    os.replace(tmp, t.path)
    with open(t.stamp, "w") as f:
        f.write(digest + "\n")
    return t.path


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the product library, and beside it the probe and debug ones."""
    path = _build(product_target(), force, verbose)
    _build(probe_target(), force, verbose)
    _build(debug_target(), force, verbose)
    return path


def build_probe(force: bool = False, verbose: bool = False) -> str:
    return _build(probe_target(), force, verbose)


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
