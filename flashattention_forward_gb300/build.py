"""Compile the CUDA library (sm_103a) into an in-tree shared library.

Each translation unit is compiled by nvcc in parallel, then linked with
``nvcc -shared``.  The result lives at ``flashattention_forward_gb300/_build/
libfa_gb300.so`` (git-ignored).  Run ``python -m flashattention_forward_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libfa_gb300.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["fa_api.cu", "fa_noalloc.cu", "fa_prologue.cu", "fa_prefill_kt.cu", "fa_prefill3_kt.cu", "fa_prefill3_kt_i8.cu", "fa_prefill3_vec5.cu", "fa_prefill_t1.cu", "fa_prefill_pv8.cu", "fa_prefill3_vec5_i8.cu", "fa_decode.cu", "fa_prefill_d64.cu", "fa_prefill_d128.cu", "fa_prefill_d192.cu",
           "fa_prefill_d192_fp8.cu",
           "fa_prefill_i8.cu", "fa_prefill_q8.cu", "fa_bwd.cu"]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return path


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(HERE, "..", "include", "fa_gb300.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    cc = nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                    "--expt-relaxed-constexpr",
                    "-I", os.path.join(HERE, "..", "include")]
    if ptxas_v:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    errs = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose or ptxas_v or r.returncode != 0:
            sys.stderr.write(f"--- {s}\n{r.stdout}{r.stderr}")
    if errs:
        raise RuntimeError("nvcc failed for " + ", ".join(s for s, _ in errs))
    tmp = LIB + f".tmp{os.getpid()}"
    link = [cc] + ARCH + ["-shared", "-o", tmp] + [o for _, o, _ in results] + ["-lcuda"] * 0
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_v="-v" in sys.argv))
