"""Build libsab.so in-tree with nvcc for sm_103a (GB300).

Usage: ``python -m streaming_attention_block_gb300.build [--verbose-ptxas]``.
Translation units compile in parallel; the shared library is linked with the
static CUDA runtime, so it needs only the driver at run time.
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


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    common = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2",
                     "-I", os.path.join(HERE, "..", "include")]
    if verbose_ptxas:
        common += ["-Xptxas", "-v"]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(HERE, "..", "include", "sab.h")]
    newest_src = max(os.path.getmtime(p) for p in deps)
    if not force and not verbose_ptxas and os.path.exists(LIB) and os.path.getmtime(LIB) >= newest_src:
        return LIB
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        jobs.append((obj, [cc] + common + ["-c", os.path.join(CSRC, src), "-o", obj]))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda j: _run(j[1]), jobs))
    for (obj, cmd), (rc, out) in zip(jobs, results):
        if out.strip() and (verbose_ptxas or rc != 0):
            sys.stderr.write(out)
        if rc != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(obj)}:\n{out}")
    tmp = LIB + ".tmp"
    rc, out = _run([cc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + [j[0] for j in jobs])
    if rc != 0:
        raise RuntimeError(f"link failed:\n{out}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(verbose_ptxas=a.verbose_ptxas, force=a.force))
