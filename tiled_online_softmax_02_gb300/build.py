"""Builds libattn.so (the CUDA library behind include/attn.h) in-tree with nvcc
for sm_103a.  Translation units compile in parallel; the link uses the static
CUDA runtime, so the library loads on machines without a GPU driver (its
entry points then report ATTN_ERR_CUDA on the first CUDA call)."""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libattn.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", f"-I{INCLUDE}"]
# Per-file flags.  dsa_select.cu computes scores whose exact fp32 rounding
# decides an index set: no multiply may be fused into an add there, including
# the packed f32x2 pairs (which an explicit .rn does not keep apart).
FILE_FLAGS = {"dsa_select.cu": ["-fmad=false"]}


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libattn.so")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: tuple[str, ...] = (),
          out_path: str | None = None) -> str:
    """Compile every csrc/*.cu for sm_103a and link libattn.so; returns its path.
    ``extra_flags`` / ``out_path`` build a variant next to (not over) the
    default library, e.g. with a different -D setting."""
    lib = out_path or LIB
    if not force and not extra_flags and out_path is None and up_to_date():
        return LIB
    nvcc = _nvcc()
    objdir = BUILD if out_path is None else os.path.join(BUILD, "variant_" + os.path.basename(lib))
    os.makedirs(objdir, exist_ok=True)
    procs = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *FILE_FLAGS.get(os.path.basename(src), []), *extra_flags, "-c", src,
               "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, obj, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                                 text=True)))
    objs, failed = [], []
    for src, obj, pr in procs:
        out, _ = pr.communicate()
        if out and (verbose or pr.returncode):
            sys.stdout.write(out)
        if pr.returncode != 0:
            failed.append(src)
        objs.append(obj)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-shared", *ARCH, "-o", tmp, *objs], check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
