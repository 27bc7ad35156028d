"""Builds libkda.so in-tree from csrc/*.cu for sm_103a (nvcc, no cmake).

Each translation unit compiles in parallel; the shared library links against
the shared CUDA runtime so it shares one runtime with the host process.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libkda.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(_nvcc())), "lib64")


def _inputs():
    return (sorted(glob.glob(os.path.join(CSRC, "*.cu")))
            + sorted(glob.glob(os.path.join(CSRC, "*.h")))
            + sorted(glob.glob(os.path.join(INCLUDE, "*.h"))))


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                    "-I" + INCLUDE, "-I" + CSRC, "--expt-relaxed-constexpr"]
    if verbose:
        flags += ["-Xptxas", "-v"]
    flags += list(extra_flags or [])
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
        r = subprocess.run([nvcc] + flags + ["-c", src, "-o", obj], capture_output=True,
                           text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s:\n%s%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 4))) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose:
        for _, err in results:
            print(err)
    tmp = LIB + ".tmp%d" % os.getpid()
    link = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + [o for o, _ in results]
    link += ["-Xlinker", "-rpath," + _cuda_lib_dir()]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
