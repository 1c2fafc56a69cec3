"""Build the native libraries in-tree with nvcc for sm_103a (GB300).

    python -m streaming_kv_cache_duo_gb300.build

Produces ``streaming_kv_cache_duo_gb300/libduo_attn.so`` (the C ABI of
include/duo_attn.h) and ``duo_synth/libduo_synth.so`` (the CUDA half of the
seeded input generator). Translation units compile in parallel; no cmake.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include")]

LIBS = {
    os.path.join(PKG, "libduo_attn.so"): [os.path.join(CSRC, f) for f in
                                          ("duo_api.cu", "append.cu", "decode.cu", "prefill.cu", "selftest.cu")],
    os.path.join(ROOT, "duo_synth", "libduo_synth.so"): [os.path.join(ROOT, "duo_synth", "csrc", "synth.cu")],
}


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def _stale(out, srcs):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    deps = list(srcs) + [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + \
        [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> None:
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    jobs = []
    for lib, srcs in LIBS.items():
        if force or _stale(lib, srcs):
            jobs.append((lib, srcs))
    if not jobs:
        return
    compile_cmds = {}
    for lib, srcs in jobs:
        for src in srcs:
            obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
            compile_cmds[obj] = [cc, *ARCH, *FLAGS, "-c", src, "-o", obj]
    workers = max(1, min(len(compile_cmds), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        outs = list(ex.map(_run, compile_cmds.values()))
    if verbose:
        for o in outs:
            sys.stdout.write(o)
    for lib, srcs in jobs:
        objs = [os.path.join(BUILD, os.path.basename(s).replace(".cu", ".o")) for s in srcs]
        tmp = lib + ".tmp"
        _run([cc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
