"""Build libpkx.so in-tree with nvcc for sm_103a.

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into ``paged_kv_extend_gb300/libpkx.so`` with the CUDA runtime linked
statically (so the library loads on a machine without a GPU).  Rebuilds only
when a source or header is newer than the library.
"""
from __future__ import annotations

import glob
import os
import re
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpkx.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "-I" + os.path.join(ROOT, "include"), *ARCH]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _inputs():
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                  + glob.glob(os.path.join(ROOT, "include", "*.h")))
    return srcs, hdrs


def needs_build() -> bool:
    if not os.path.exists(LIB):
        return True
    srcs, hdrs = _inputs()
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in srcs + hdrs + [__file__])


# Kernels that hand registers between warpgroups with setmaxnreg, and the
# source file that states the launch register count the split assumes.
SPLIT_KERNELS = (("attn_kernel", "attention.cu"), ("mla_pair_kernel", "mla_pair_kernel.cuh"))


def check_attention_registers(ptxas_log: str) -> None:
    """The attention kernels hand registers between warpgroups with
    setmaxnreg; the split adds up only if every instantiation launches with
    exactly the register count the kernel source assumes (REGS_LAUNCH).
    Refuse to build otherwise: a wrong split would stall the kernel."""
    for kernel, fname in SPLIT_KERNELS:
        src = open(os.path.join(CSRC, fname)).read()
        m = re.search(r"REGS_LAUNCH = (\d+)", src)
        if not m:
            raise RuntimeError(f"{fname}: REGS_LAUNCH not found")
        want = int(m.group(1))
        found = 0
        current = None
        for line in ptxas_log.splitlines():
            fm = re.search(r"Compiling entry function '(\S+)'", line) or \
                re.search(r"Function properties for (\S+)", line)
            if fm:
                current = fm.group(1)
            rm = re.search(r"Used (\d+) registers", line)
            if rm and current and kernel in current:
                found += 1
                if int(rm.group(1)) != want:
                    raise RuntimeError(
                        f"{current} uses {rm.group(1)} registers at launch, the register "
                        f"split assumes {want}; not building")
        if found == 0:
            raise RuntimeError(f"no {kernel} register report from ptxas; not building")


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libpkx.so; returns its path."""
    if not force and not needs_build():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs, _ = _inputs()
    nvcc = _nvcc()
    procs = []
    objs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
        if os.path.basename(src) == "attention.cu":
            cmd.insert(1, "-Xptxas=-v")
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        else:
            if os.path.basename(src) == "attention.cu":
                check_attention_registers(out.decode(errors="replace"))
            if verbose and out:
                print(out.decode(errors="replace"), file=sys.stderr)
    if failed:
        msg = "\n".join(f"{s}:\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
