"""Compile the CUDA library (libfa_gb300.so) in-tree for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into one shared object with a C ABI (include/fa.h).  Re-running is a
no-op unless a source or header is newer than the library.

A second build of the same sources with FA_TEST_HOOKS defined
(libfa_gb300_testhooks.so) adds one test-only switch that makes a kernel's
producer withhold a load, so that the failure-detection tests can make a
bounded wait expire.  Only those tests load it; the product library has
neither the switch nor the code behind it.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libfa_gb300.so")
TEST_HOOKS_DIR = os.path.join(OUT_DIR, "test_hooks")
TEST_HOOKS_LIB = os.path.join(TEST_HOOKS_DIR, "libfa_gb300_testhooks.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]
VARIANTS = {
    "product": (OUT_DIR, LIB, []),
    "test_hooks": (TEST_HOOKS_DIR, TEST_HOOKS_LIB, ["-DFA_TEST_HOOKS"]),
}


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        [os.path.join(ROOT, "include", "fa.h")]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def _compile(src: str, out_dir: str, defines: list, verbose_ptxas: bool) -> str:
    obj = os.path.join(out_dir, os.path.basename(src) + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *defines, "-c", src, "-o", obj]
    if verbose_ptxas:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose_ptxas:
        sys.stderr.write(r.stderr)
    return obj


def _link(objs: list, lib: str) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose_ptxas: bool = False, variants=("product",)) -> str:
    """Build the requested variants (all translation units of all of them in
    parallel); returns the product library's path."""
    todo = [v for v in variants if force or _stale(VARIANTS[v][1])]
    if todo:
        srcs = _sources()
        jobs = []
        for v in todo:
            out_dir, _, defines = VARIANTS[v]
            os.makedirs(out_dir, exist_ok=True)
            jobs += [(v, s, out_dir, defines) for s in srcs]
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            objs = list(ex.map(lambda j: (j[0], _compile(j[1], j[2], j[3], verbose_ptxas)), jobs))
        for v in todo:
            _link([o for vv, o in objs if vv == v], VARIANTS[v][1])
    return LIB


def build_test_hooks(force: bool = False) -> str:
    build(force=force, variants=("test_hooks",))
    return TEST_HOOKS_LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv,
                variants=tuple(VARIANTS) if "--all" in sys.argv else ("product",)))
