"""Build libqkv.so in-tree: nvcc for sm_103a only, one object per .cu, compiled in parallel.

    python quantized_kv_cache_write_gb300/build.py [--force] [--ptxas-verbose]
    python -c "import __graft_entry__ as g; g.build()"

(Run it as a file, not with -m: importing the package first would load a stale library.)
"""

from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(HERE, "libqkv.so")

SOURCES = [
    "api.cu",
    "write.cu",
    "merge.cu",
    "calib.cu",
    "gather_int8_side.cu",
    "gather_int8_inline.cu",
    "gather_e4m3.cu",
    "gather_bf16.cu",
    "gather_noalloc.cu",
    "gather_umma_int8_side.cu",
    "gather_paged_int8_side.cu",
    "gather_paged_int8_inline.cu",
    "gather_paged_e4m3.cu",
    "gather_paged_bf16.cu",
    "gather_f16q_int8_side.cu",
    "gather_f16q_int8_inline.cu",
    "gather_f16q_e4m3.cu",
    "gather_f16q_f16.cu",
]
HEADERS = ["qkv_internal.cuh", "gather_attn.cuh", "gather_umma.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqkv.so")
    return cand


def _stale(outputs_mtime: float) -> bool:
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "qkv.h")]
    return any(os.path.getmtime(d) > outputs_mtime for d in deps)


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True) -> str:
    """Compile csrc/*.cu and link libqkv.so next to this file. Returns the library path.

    Processes that build at the same time (one per GPU under torchrun) take turns on a lock
    file; a later one finds the library fresh and returns."""
    if not force and os.path.exists(LIB_PATH) and not _stale(os.path.getmtime(LIB_PATH)):
        return LIB_PATH
    import fcntl
    os.makedirs(BUILD_DIR, exist_ok=True)
    with open(os.path.join(BUILD_DIR, ".lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)
        try:
            if not force and os.path.exists(LIB_PATH) and not _stale(os.path.getmtime(LIB_PATH)):
                return LIB_PATH
            return _build(ptxas_verbose, quiet)
        finally:
            fcntl.flock(lock, fcntl.LOCK_UN)


def _build(ptxas_verbose: bool, quiet: bool) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []

    def compile_one(src: str):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, p.returncode, p.stdout + p.stderr

    with ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    log = []
    for src, obj, rc, out in results:
        log.append(f"== {src}\n{out}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{out}")
    if ptxas_verbose:
        with open(os.path.join(BUILD_DIR, "ptxas.txt"), "w") as f:
            f.write("\n".join(log))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[r[1] for r in results]]
    p = subprocess.run(cmd, capture_output=True, text=True)
    if p.returncode != 0:
        raise RuntimeError(f"link failed:\n{p.stdout}{p.stderr}")
    os.replace(tmp, LIB_PATH)
    if not quiet:
        print(f"built {LIB_PATH}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, ptxas_verbose=args.ptxas_verbose, quiet=False))
