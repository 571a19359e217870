"""Build libkivi.so (CUDA, sm_103a) in-tree with nvcc.

The translation units compile in parallel, then link into one shared
library next to this file.  No torch headers or libraries are involved: the
library exposes only the C ABI of include/kivi.h.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libkivi.so")
SOURCES = ["kivi_api.cu", "kivi_pack.cu", "kivi_decode.cu", "kivi_decode_d64.cu",
           "kivi_decode_d128.cu", "kivi_decode_d256.cu", "kivi_decode_probs_d64.cu",
           "kivi_decode_probs_d128.cu", "kivi_decode_probs_d256.cu", "kivi_decode_fused_d64.cu",
           "kivi_decode_fused_d128.cu", "kivi_decode_fused_d256.cu", "kivi_probs.cu", "kivi_noalloc.cu",
           "kivi_prefill_attn.cu"]
HEADERS = ["kivi_internal.cuh", "kivi_decode_impl.cuh", "kivi_pack_impl.cuh", "kivi_append_impl.cuh",
           "kivi_mma.cuh", "kivi_tcgen05.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division and rounding stay exact: no --use_fast_math anywhere.
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libkivi needs the CUDA toolkit to build")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if stale) and return the path of libkivi.so."""
    deps_common = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "kivi.h")]
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    objs = []
    jobs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        op = os.path.join(objdir, src.replace(".cu", ".o"))
        objs.append(op)
        if force or _stale(op, [sp] + deps_common):
            cmd = [nvcc()] + ARCH + FLAGS + list(extra_flags) + ["-c", sp, "-o", op]
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    if jobs:
        with cf.ThreadPoolExecutor(len(jobs)) as ex:
            for out in ex.map(run, jobs):
                if verbose and out.strip():
                    print(out)
    if force or jobs or _stale(LIB, objs):
        run([nvcc()] + ARCH + ["-shared", "-o", LIB + ".tmp"] + objs + ["-lcudart_static", "-lrt",
                                                                           "-lpthread", "-ldl"])
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas" in sys.argv else ()))
