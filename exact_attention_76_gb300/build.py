"""Builds libfa_gb300.so in-tree for sm_103a with nvcc (no cmake, no torch
extension machinery).  Each .cu translation unit compiles in parallel; the
objects link into one shared library with the static CUDA runtime.

    python -m exact_attention_76_gb300.build          # build if stale
    python -m exact_attention_76_gb300.build --force  # rebuild
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfa_gb300.so")
SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu", "fa_fp8q.cu", "fa_decode.cu"]
HEADERS = ["fa_common.cuh", "fa_host.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Kernels whose warpgroups redistribute registers with setmaxnreg: the shares
# add up to the launch allocation only if the compiled kernel uses exactly
# this many registers per thread (source, mangled-name fragment, registers).
REGISTER_PLANS = [("fa_bwd.cu", "fa_bwd_main_kernelILi128E", 128)]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "fa.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def check_registers(ptxas_log: str, fragment: str, regs: int, src: str) -> None:
    """Fails the build unless every kernel whose mangled name contains
    `fragment` was compiled to exactly `regs` registers per thread (ptxas -v:
    an entry function line, then its "Used N registers" line)."""
    found = 0
    current = None
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current is not None and fragment in current:
            found += 1
            if int(m.group(1)) != regs:
                raise RuntimeError(f"{src}: {current} uses {m.group(1)} registers per thread; its setmaxnreg "
                                   f"split needs exactly {regs}")
            current = None
    if found == 0:
        raise RuntimeError(f"{src}: no register report for a kernel matching {fragment}")


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        plans = [pl for pl in REGISTER_PLANS if pl[0] == src]
        flags = extra if (extra or not plans) else ["-Xptxas", "-v"]
        cmd = [cc, *ARCH, *FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{p.stderr}")
        for _, frag, regs in plans:
            check_registers(p.stderr, frag, regs, src)
        return obj, p.stderr if (verbose or ptxas_info) else ""

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", "-cudart", "static", "-o", tmp,
           *[o for o, _ in results], "-ldl", "-lpthread", "-lrt"]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)
