"""Build libzyfa.so (the C-ABI library) in-tree for sm_103a with nvcc.

The three translation units compile in parallel; the shared library lands next to this file, where
``fp8_causal_prefill_gb300.api`` loads it.  Run as ``python -m fp8_causal_prefill_gb300.build``.
"""
from __future__ import annotations

import os
import re
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzyfa.so")
SOURCES = ["zyfa_api.cu", "zyfa_kernels_fp8.cu", "zyfa_kernels_fp8_exact.cu", "zyfa_kernels_bf16.cu",
           "zyfa_hadamard.cu", "zyfa_probe.cu"]
# The attention kernel splits its registers between warpgroups at run time (setmaxnreg); the split is
# sized for exactly this many registers per thread at launch, which every instantiation must get.
KERNEL_REGS = 168
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def check_kernel_registers(src: str, ptxas_log: str) -> None:
    """Refuse a build whose attention kernel would not launch with the register count its run-time
    warpgroup split assumes (a smaller count would make the split wait forever)."""
    current, checked = None, 0
    for line in ptxas_log.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            current = m.group(1)
            continue
        m = re.search(r"Used (\d+) registers", line)
        if m and current and "zyfa_fwd_kernel" in current:
            if int(m.group(1)) != KERNEL_REGS:
                raise RuntimeError(f"{src}: {current} uses {m.group(1)} registers, the register split needs "
                                   f"{KERNEL_REGS}")
            current = None
            checked += 1
    if "kernels" in src and checked == 0:
        raise RuntimeError(f"{src}: no register report found for the attention kernel")


def _inputs_newer(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "zyfa.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if any source is newer than the library) and return the library path."""
    if not force and not _inputs_newer(LIB):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc, *ARCH, *FLAGS, "-Xptxas=-v", "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        check_kernel_registers(src, r.stderr)
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
