"""Builds libfsp.so (planner + fused step) for sm_103a with nvcc, in-tree.

Usage: ``python -m fsdp_sharded_mixed_pass_gb300.build`` or ``build()``.
Translation units compile in parallel; the result goes to
``fsdp_sharded_mixed_pass_gb300/_build/libfsp.so``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libfsp.so")
SOURCES = ("fsp_plan.cpp", "fsp_step.cu", "fsp_host.cu", "fsp_unshard.cu", "fsp_params.cu")
ARCH = ("-gencode", "arch=compute_103a,code=sm_103a")


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def compile_shared(sources, out, includes, extra=()) -> None:
    """Compile ``sources`` in parallel to objects next to ``out``, then link it."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off",
            "-Xptxas", "-v", *[f"-I{i}" for i in includes], *extra]
    procs, objs = [], []
    for src in sources:
        obj = os.path.join(os.path.dirname(out), os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = base + (["-x", "cu"] if src.endswith(".cu") else []) + ["-c", src, "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    logs = []
    for src, p in procs:
        log, _ = p.communicate()
        logs.append(log)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{log}")
    tmp = out + ".tmp"
    link = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, out)
    with open(out + ".ptxas.txt", "w") as f:
        f.write("\n".join(logs))


def build() -> str:
    compile_shared([os.path.join(CSRC, s) for s in SOURCES], LIB, [os.path.join(ROOT, "include"), CSRC])
    return LIB


if __name__ == "__main__":
    print(build())
    sys.exit(0)
