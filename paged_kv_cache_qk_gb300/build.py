"""Build libpkvqk.so (the C-ABI library) in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_qk_gb300.build [--verbose-ptxas]

Each .cu under csrc/ is compiled in parallel to an object under _build/,
then linked into paged_kv_cache_qk_gb300/libpkvqk.so (CUDA runtime linked
statically, no libcuda link: the TMA encoder is fetched through the runtime's
driver entry-point query).
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libpkvqk.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "norm_rope_append.cu", "decode.cu", "combine.cu", "decode_static_ws.cu",
           "prefill.cu"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def build(verbose_ptxas: bool = False, force: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    deps.append(os.path.join(ROOT, "include", "pkvqk.h"))
    if not force and os.path.exists(LIB):
        t = os.path.getmtime(LIB)
        if all(os.path.getmtime(d) < t for d in deps) and os.path.getmtime(__file__) < t:
            return LIB
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
                    "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]
    if verbose_ptxas:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for s in srcs:
        o = os.path.join(BUILD, os.path.basename(s).replace(".cu", ".o"))
        objs.append(o)
        procs.append((s, subprocess.Popen([nvcc(), *flags, "-c", s, "-o", o],
                                          stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        txt = out.decode(errors="replace")
        if verbose_ptxas or p.returncode != 0:
            sys.stderr.write(txt)
        if p.returncode != 0:
            failed.append(s)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    tmp = LIB + ".tmp"
    r = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs],
                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        sys.stderr.write(r.stdout.decode(errors="replace"))
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args()
    print(build(verbose_ptxas=args.verbose_ptxas, force=args.force))


if __name__ == "__main__":
    main()
