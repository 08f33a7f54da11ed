"""Build libpagedkv.so in-tree with nvcc for sm_103a (GB300).

Every translation unit under csrc/ is compiled in parallel, then linked into
one shared library next to this file.  A stamp of the sources and flags skips
the build when nothing changed.
"""

import hashlib
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
                     "-I", os.path.join(ROOT, "include")]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-I",
             os.path.join(ROOT, "include")]


# per-file extra flags (none: the prefill softmax calls the hardware exp2
# through inline PTX, so no unit needs fast-math code generation)
EXTRA_FLAGS = {}


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    srcs = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))
    hdrs = sorted(f for f in os.listdir(CSRC) if f.endswith((".cuh", ".h")))
    return srcs, hdrs


def _stamp(srcs, hdrs):
    h = hashlib.sha256()
    for f in srcs + hdrs:
        with open(os.path.join(CSRC, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    with open(os.path.join(ROOT, "include", "pagedkv.h"), "rb") as fh:
        h.update(fh.read())
    h.update(" ".join(NVCC_FLAGS + CXX_FLAGS).encode() + repr(sorted(EXTRA_FLAGS.items())).encode())
    return h.hexdigest()


def build_variant(tag, defines, verbose=False):
    """A separate copy of the library compiled with extra -D definitions, for
    tests that need a behaviour the product build must not have (the
    wait-timeout test: a 1 ms wait limit and one decode tile never copied).
    It lands beside the product library as libpagedkv_<tag>.so, from its own
    object directory, and is rebuilt only when sources or definitions change."""
    import fcntl

    lib = os.path.join(HERE, f"libpagedkv_{tag}.so")
    flags = [f"-D{k}={v}" for k, v in sorted(defines.items())]
    with open(lib + ".lock", "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(False, verbose, lib=lib, build_dir=os.path.join(BUILD, tag),
                                 extra=flags)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def build(force=False, verbose=False):
    """Compile and link the library; return its path.  Raises on compiler errors.

    Processes that build at the same time (one per rank under torchrun) take
    turns through a lock file next to the library; the later ones find the
    fresh stamp and return at once."""
    import fcntl

    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    with open(LIB + ".lock", "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            return _build_locked(force, verbose)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build_locked(force, verbose, lib=LIB, build_dir=BUILD, extra=()):
    srcs, hdrs = _sources()
    stamp = _stamp(srcs, hdrs) + ("" if not extra else " " + " ".join(extra))
    stamp_file = lib + ".stamp"
    if not force and os.path.exists(lib) and os.path.exists(stamp_file):
        with open(stamp_file) as f:
            if f.read().strip() == stamp:
                return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, src + ".o")
        path = os.path.join(CSRC, src)
        if src.endswith(".cu"):
            cmd = ([nvcc] + NVCC_FLAGS + EXTRA_FLAGS.get(src, []) + list(extra)
                   + ["-c", path, "-o", obj])
        else:
            cmd = ["g++"] + CXX_FLAGS + list(extra) + ["-c", path, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    with open(stamp_file, "w") as f:
        f.write(stamp)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
