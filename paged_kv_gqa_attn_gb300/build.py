"""Compile the CUDA library in-tree: paged_kv_gqa_attn_gb300/_lib/libpaged_attn.so (sm_103a).

Each .cu file is compiled to an object in parallel, then linked into one shared library with
the CUDA runtime linked statically.  Run ``python -m paged_kv_gqa_attn_gb300.build``.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libpaged_attn.so")
# The instrumented variant (-DPA_TIMELINE: per-CTA %globaltimer stamps in the verify kernel, per-role
# clock64 sums in the prefill kernel, read back by paged_attn_timeline_read_verify / _prefill) is a
# separate library that only the timeline tool loads; the product library above never carries the
# instrumentation.
TIMELINE_DIR = os.path.join(LIB_DIR, "timeline")
TIMELINE_LIB_PATH = os.path.join(TIMELINE_DIR, "libpaged_attn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA library cannot be built")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date(timeline: bool = False) -> bool:
    path = TIMELINE_LIB_PATH if timeline else LIB_PATH
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, timeline: bool = False) -> str:
    out_dir, lib_path = (TIMELINE_DIR, TIMELINE_LIB_PATH) if timeline else (LIB_DIR, LIB_PATH)
    if not force and up_to_date(timeline):
        return lib_path
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    procs = []
    objs = []
    for src in _sources():
        obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [cc, *ARCH, *NVCC_FLAGS, *(["-DPA_TIMELINE"] if timeline else []), "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if verbose or pr.returncode != 0:
            sys.stdout.write(out.decode(errors="replace"))
        if pr.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed on {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, timeline="--timeline" in sys.argv))
