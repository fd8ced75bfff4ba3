"""Build libscout.so and libscoutgen.so in-tree with nvcc for sm_103a.

    python -m block_sparse_kv_pred_gb300.build

Each translation unit compiles in its own process; the objects are linked into
shared libraries next to this file.  No CMake, no torch extension machinery.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
          "-Xcompiler", "-pthread", "-I" + os.path.join(ROOT, "include")]

LIBS = {
    "libscout.so": [os.path.join(PKG, "csrc", f) for f in
                    ("api.cu", "digest.cu", "score_topk.cu", "sparse_attn.cu", "merge.cu", "predict_q.cu",
                     "recall.cu", "lists.cu", "cpu_attend.cpp")],
    "libscoutgen.so": [os.path.join(PKG, "workload", "gen.cu")],
}


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [nvcc(), *ARCH, *CFLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def lib_path(name: str) -> str:
    return os.path.join(PKG, name)


def build(verbose: bool = False, extra: list[str] | None = None) -> dict[str, str]:
    os.makedirs(BUILD, exist_ok=True)
    extra = list(extra or [])
    out = {}
    srcs = [s for v in LIBS.values() for s in v]
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        objs = dict(zip(srcs, ex.map(lambda s: _compile(s, extra), srcs)))
    for name, lib_srcs in LIBS.items():
        target = lib_path(name)
        tmp = target + ".tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *[objs[s] for s in lib_srcs], "-lcudart", "-Xcompiler", "-pthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed for {name}:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, target)
        out[name] = target
        if verbose:
            print("built", target)
    return out


if __name__ == "__main__":
    build(verbose=True, extra=sys.argv[1:])
