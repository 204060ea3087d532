"""Build libtq.so in-tree with nvcc for sm_103a (GB300).

    python -m kv_cache_vector_gb300.build [--force] [--verbose]

Each translation unit is compiled in parallel, then linked into
``kv_cache_vector_gb300/libtq.so`` with the CUDA runtime linked statically,
so the library loads without a CUDA toolkit on the library path.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libtq.so")
BUILD_DIR = os.path.join(ROOT, "_build")
# (source, specialisation macros TQ_UNIT_<name>)
CODEC_DIMS = (8, 16, 32, 64, 128, 256)
ATTN_DIMS = (32, 64, 128, 256)
UNITS = ([("tq_api.cpp", {}), ("tq_launch.cu", {}), ("tq_noalloc.cu", {})]
         + [("tq_codec.cu", {"D": d}) for d in CODEC_DIMS]
         + [("tq_attn.cu", {"D": 128, "KB": kb}) for kb in (2, 3, 4)]
         + [("tq_attn_generic.cu", {"D": d, "KB": kb}) for d in ATTN_DIMS for kb in (2, 3, 4)]
         + [("tq_prefill.cu", {"KB": kb}) for kb in (2, 3, 4)]
         + [("tq_qjl.cu", {"D": d}) for d in (32, 64, 128)])
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libtq.so")
    return cand


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "tq.h"))
    return files


def _stale() -> bool:
    if not os.path.exists(OUT):
        return True
    stamp = OUT + ".defines"
    want = os.environ.get("TQ_NVCC_DEFINES", "")
    if (open(stamp).read() if os.path.exists(stamp) else "") != want:
        return True
    t = os.path.getmtime(OUT)
    return any(os.path.getmtime(f) > t for f in _deps())


def _compile(unit, verbose: bool) -> str:
    src, defs = unit
    stem = os.path.splitext(src)[0] + "".join(f"_{k.lower()}{v}" for k, v in defs.items())
    obj = os.path.join(BUILD_DIR, stem + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", os.path.join(ROOT, "include"), "-c", os.path.join(CSRC, src), "-o", obj]
    for k, v in defs.items():
        cmd.insert(1, f"-DTQ_UNIT_{k}={v}")
    # extra preprocessor definitions, space separated (TQ_NVCC_DEFINES="A=1 B")
    for d in os.environ.get("TQ_NVCC_DEFINES", "").split():
        cmd.insert(1, f"-D{d}")
    if src.endswith(".cu"):
        cmd[1:1] = ["-Xptxas", "-v"] if verbose else []
    else:
        cmd[1:1] = ["-x", "cu"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        sys.stderr.write(r.stdout + r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return OUT
    os.makedirs(BUILD_DIR, exist_ok=True)
    workers = max(1, min(len(UNITS), os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        objs = list(ex.map(lambda u: _compile(u, verbose), UNITS))
    tmp = OUT + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, OUT)
    with open(OUT + ".defines", "w") as f:
        f.write(os.environ.get("TQ_NVCC_DEFINES", ""))
    return OUT


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))
