"""Build libsab.so in-tree with nvcc for sm_103a (GB300).

Usage: ``python -m streaming_attention_block_gb300.build [--verbose-ptxas] [--debug-bounds]``.
Translation units compile in parallel; the shared library is linked with the
static CUDA runtime, so it needs only the driver at run time.  The debug
variant (``libsab_debug.so``, ``-DSAB_DEBUG_BOUNDS``) adds the device-side
index checks; it is the same ABI and is selected with ``SAB_LIBRARY``.
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libsab.so")
DEBUG_LIB = os.path.join(HERE, "libsab_debug.so")
SOURCES = ["sab_api.cu", "chunk_attn.cu", "kv_append.cu", "qk_rope.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsab.so")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    return r.returncode, r.stdout + r.stderr


def build(verbose_ptxas: bool = False, force: bool = False, debug_bounds: bool = False,
          both: bool = False) -> str:
    """Build libsab.so (or, with ``debug_bounds``, libsab_debug.so; with
    ``both``, the two in one parallel batch).  Returns the (first) path."""
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", os.path.join(HERE, "..", "include")]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "sab.h")]
    newest_src = max(os.path.getmtime(p) for p in deps)
    variants = [(LIB, BUILD, [])] if not debug_bounds or both else []
    if debug_bounds or both:
        variants.append((DEBUG_LIB, os.path.join(BUILD, "debug"), ["-DSAB_DEBUG_BOUNDS"]))
    todo = [v for v in variants
            if force or verbose_ptxas or not os.path.exists(v[0]) or os.path.getmtime(v[0]) < newest_src]
    jobs = []
    for lib, bdir, defs in todo:
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            obj = os.path.join(bdir, src.replace(".cu", ".o"))
            jobs.append((lib, obj, [cc] + common + defs + ["-c", os.path.join(CSRC, src), "-o", obj]))
    if jobs:
        with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            results = list(ex.map(lambda j: _run(j[2]), jobs))
        for (lib, obj, cmd), (rc, out) in zip(jobs, results):
            if out.strip() and (verbose_ptxas or rc != 0):
                sys.stderr.write(out)
            if rc != 0:
                raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{out}")
    for lib, _, _ in todo:
        tmp = lib + ".tmp"
        objs = [j[1] for j in jobs if j[0] == lib]
        rc, out = _run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs)
        if rc != 0:
            raise RuntimeError(f"link failed:\n{out}")
        os.replace(tmp, lib)
    return variants[0][0]


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true")
    a = ap.parse_args()
    print(build(verbose_ptxas=a.verbose_ptxas, force=a.force, debug_bounds=a.debug_bounds))
