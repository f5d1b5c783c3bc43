"""Builds libfa.so in-tree with nvcc for sm_103a (and nothing else).

Each translation unit compiles in parallel into ``_build/`` and links into
``exact_io_aware_05_gb300/libfa.so`` with the static CUDA runtime.  No torch
types or headers are involved: the library is a plain C ABI (include/fa.h).

With ``test_variant=True`` the same pool also compiles the API and the two
tile-loop units with ``FA_TEST_WITHHOLD=1`` into ``_build/waittest/`` and links
them with the other product objects into ``libfa_waittest.so``: a library for
the tests of the bounded-wait timeout path only (one launch may leave out one
mbarrier arrive).  Nothing in the package loads it; libfa.so never contains it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(PKG, "libfa.so")
TEST_SO = os.path.join(PKG, "libfa_waittest.so")
SOURCES = ["fa_api.cu", "fa_fwd_sm103.cu", "fa_fwd_f32.cu", "fa_bwd_sm103.cu", "fa_bwd_noalloc.cu",
           "fa_decode_sm103.cu", "fa_fp8_sm103.cu"]
# the units that read FA_TEST_WITHHOLD; the test library takes the others from the product build
TEST_SOURCES = ["fa_api.cu", "fa_fwd_sm103.cu", "fa_bwd_sm103.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or install the CUDA toolkit)")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fa.h"))
    return files


def up_to_date(so: str = SO) -> bool:
    if not os.path.exists(so):
        return False
    t = os.path.getmtime(so)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False, test_variant: bool = False) -> str:
    """Builds libfa.so (and, with test_variant, libfa_waittest.so) unless up to date."""
    if not force and up_to_date() and (not test_variant or up_to_date(TEST_SO)):
        return SO
    os.makedirs(os.path.join(BUILD, "waittest"), exist_ok=True)
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                    "-I", os.path.join(ROOT, "include"), "-I", CSRC]
    if ptxas_info:
        flags += ["-Xptxas", "-v"]

    def compile_one(job: tuple[str, bool]) -> str:
        src, test = job
        obj = os.path.join(BUILD, "waittest" if test else "", src.replace(".cu", ".o"))
        cmd = [cc, *flags, *(["-DFA_TEST_WITHHOLD=1"] if test else []), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose or ptxas_info:
            sys.stdout.write(r.stdout + r.stderr)
        return obj

    jobs = [(src, False) for src in SOURCES] + ([(src, True) for src in TEST_SOURCES] if test_variant else [])
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(compile_one, jobs))
    prod = objs[:len(SOURCES)]
    _link(cc, prod, SO)
    if test_variant:
        test_objs = dict(zip(TEST_SOURCES, objs[len(SOURCES):]))
        _link(cc, [test_objs.get(src, o) for src, o in zip(SOURCES, prod)], TEST_SO)
    return SO


def _link(cc: str, objs: list[str], so: str) -> None:
    tmp = so + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, so)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv,
          test_variant="--test-variant" in sys.argv)
    print(SO)
