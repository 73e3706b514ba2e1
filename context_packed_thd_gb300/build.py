"""Build libcpthd.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel to an object file
under _build/ and linked into context_packed_thd_gb300/libcpthd.so. A
rebuild happens only when a source, a header or the flags changed.

    python -m context_packed_thd_gb300.build [--force] [--verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import hashlib
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcpthd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


class NvccMissing(RuntimeError):
    pass


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise NvccMissing("nvcc not found: the CUDA 13 toolkit is required to build libcpthd")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _fingerprint(extra=()) -> str:
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")))
    for f in files:
        h.update(f.encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + list(extra)).encode())
    return h.hexdigest()


def build(force: bool = False, verbose: bool = False, extra_flags=(), build_dir: str = BUILD,
          lib: str = LIB) -> str:
    """Compile and link libcpthd.so (or, with another build_dir / lib, a
    variant of it built with extra_flags); returns its path."""
    os.makedirs(build_dir, exist_ok=True)
    stamp = os.path.join(build_dir, "fingerprint")
    fp = _fingerprint(extra_flags)
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == fp:
                return lib
    nvcc = _nvcc()
    flags = NVCC_FLAGS + list(extra_flags)
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp, "w") as f:
        f.write(fp)
    return lib


def build_wait_test() -> str:
    """A test-only variant of the library, built with CPTHD_WAIT_TEST: its
    waits give up after 5 ms instead of 2 s, and the attention forward
    withholds one signal so that a wait must run out (CPTHD_ERR_TIMEOUT):
    by default the data-relay warp's arrivals for key block 1, or, after
    cpthd_wait_test_mode(2), the hand-off flags of the pieces of cut items.
    Kept apart from libcpthd.so under _build/; only the timeout tests load
    it."""
    d = os.path.join(BUILD, "wait_test")
    return build(extra_flags=("-DCPTHD_WAIT_TEST",), build_dir=d, lib=os.path.join(d, "libcpthd_wait_test.so"))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv))
