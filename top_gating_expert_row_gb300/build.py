"""Build libmoerouter.so for sm_103a with nvcc, in-tree.

Translation units compile in parallel (fwd.cu once per score function x logits
dtype, plus sort.cu, bwd.cu, api.cu) and link into one shared library with the
static CUDA runtime, so loading it needs no CUDA library path.

    python -m top_gating_expert_row_gb300.build [--verbose]
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
LIB = os.path.join(HERE, "libmoerouter.so")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", CSRC, "-I", INCLUDE]

UNITS = [
    ("fwd_s0_d0", "fwd.cu", ["-DMR_SCORE_FN=0", "-DMR_IN_BF16=0"]),
    ("fwd_s0_d1", "fwd.cu", ["-DMR_SCORE_FN=0", "-DMR_IN_BF16=1"]),
    ("fwd_s1_d0", "fwd.cu", ["-DMR_SCORE_FN=1", "-DMR_IN_BF16=0"]),
    ("fwd_s1_d1", "fwd.cu", ["-DMR_SCORE_FN=1", "-DMR_IN_BF16=1"]),
    ("sort", "sort.cu", []),
    ("bwd", "bwd.cu", []),
    ("aux_loss", "aux_loss.cu", []),
    ("api", "api.cu", []),
]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "moe_router.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, jobs: int | None = None) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _sources_mtime():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_unit(unit):
        name, src, defs = unit
        obj = os.path.join(BUILD, name + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *defs, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {name}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    jobs = jobs or min(len(UNITS), os.cpu_count() or 4)
    with ThreadPoolExecutor(max_workers=jobs) as ex:
        results = list(ex.map(compile_unit, UNITS))
    if verbose:
        for _, log in results:
            sys.stderr.write(log)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results],
           "-lpthread", "-ldl", "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--force", action="store_true")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose))
