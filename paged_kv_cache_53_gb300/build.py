"""Builds libpagedattn.so (the sm_103a CUDA library) in-tree with nvcc.

Each .cu file is compiled to an object in parallel, then linked into
paged_kv_cache_53_gb300/_build/libpagedattn.so.  Nothing is installed.  Run as
`python -m paged_kv_cache_53_gb300.build [--force] [--ptxas-info]`.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libpagedattn.so")
SOURCES = ["pa_api.cu", "pa_cache_ops.cu", "pa_decode.cu", "pa_prefill.cu",
           "pa_decode_static.cu", "pa_shared_prefix.cu", "pa_block_manager.cpp",
           "pa_sha256.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn")


def _flags(ptxas_info: bool):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", "-DNDEBUG"]
    if ptxas_info:
        f += ["-Xptxas", "-v"]
    return f


def _inputs():
    deps = [os.path.join(CSRC, s) for s in SOURCES]
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def build(force: bool = False, ptxas_info: bool = False, verbose: bool = False) -> str:
    """Compiles the library unless it is up to date; returns its path."""
    if not force and not ptxas_info and up_to_date():
        return LIB
    nvcc = _nvcc()
    objdir = os.path.join(BUILD, "obj")
    os.makedirs(objdir, exist_ok=True)
    flags = _flags(ptxas_info)

    def compile_one(src):
        obj = os.path.join(objdir, os.path.splitext(src)[0] + ".o")
        cmd = [nvcc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, _, r in results:
        log.append(f"== {src}\n{r.stdout}{r.stderr}")
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-6000:]}")
    if ptxas_info or verbose:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
            f.write("\n".join(log))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for _, o, _ in results],
           "-Xcompiler", "-fPIC", "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    return LIB


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true",
                    help="compile with -Xptxas -v and keep the report in _build/ptxas.log")
    args = ap.parse_args(argv)
    path = build(force=args.force, ptxas_info=args.ptxas_info, verbose=True)
    print(path)


if __name__ == "__main__":
    sys.exit(main())
