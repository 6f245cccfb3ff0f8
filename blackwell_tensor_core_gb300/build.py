"""Build step for the CUDA library: compiles csrc/*.cu for sm_103a with nvcc
(one translation unit per process, in parallel) and links libbwgemm.so into
this package directory.  Run as ``python -m blackwell_tensor_core_gb300.build``
or through ``__graft_entry__.build()``.

The library's ``bwg_version()`` ends with the hash of the code it was built
from (every csrc file and the public header, comments removed); a library
whose hash differs from the sources on disk, or that does not load on this
machine, is rebuilt."""
from __future__ import annotations

import hashlib
import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD_DIR = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libbwgemm.so")
HEADER = os.path.join(ROOT, "include", "bwgemm.h")
SOURCES = ["api.cu", "gemm_tc.cu", "gemm_small_m.cu", "probes.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def code_only(text: str) -> str:
    """C/C++/CUDA source with comments and blank space removed, so that a hash
    of it changes with the code, not with its comments."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def library_files() -> list:
    """Every file the library is compiled from: csrc/* and the public header."""
    names = sorted(f for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h")))
    return [os.path.join(CSRC, f) for f in names] + [HEADER]


def source_hash(paths=None) -> str:
    """16 hex digits of SHA-256 over the code-only text of `paths` (default:
    every library source), in order."""
    h = hashlib.sha256()
    for path in (paths if paths is not None else library_files()):
        with open(path, encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def built_version(path: str = LIB):
    """bwg_version() of the library at `path`, read in a child process (so that
    this process does not keep a stale copy loaded); None if it cannot load."""
    if not os.path.exists(path):
        return None
    code = ("import ctypes,sys; L=ctypes.CDLL(sys.argv[1]); L.bwg_version.restype=ctypes.c_char_p; "
            "print(L.bwg_version().decode())")
    try:
        r = subprocess.run([sys.executable, "-c", code, path], capture_output=True, text=True, timeout=60)
    except (OSError, subprocess.SubprocessError):
        return None
    return r.stdout.strip() if r.returncode == 0 else None


def _up_to_date() -> bool:
    """The library exists, loads on this machine and was built from the
    sources as they are now (its version string carries their hash)."""
    v = built_version()
    return v is not None and v.endswith("source " + source_hash())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and _up_to_date():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "-I" + os.path.join(ROOT, "include"), "--expt-relaxed-constexpr",
                    '-DBWG_SOURCE_HASH="%s"' % source_hash()]
    if os.environ.get("BWG_PTXAS_VERBOSE"):
        flags += ["-Xptxas", "-v"]

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + objs + ["-lcudart_static", "-lrt", "-ldl", "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
