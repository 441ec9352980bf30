"""Build the in-tree CUDA library libhla_gb300.so for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked into one shared
library under causal_prefix_scan_gb300/_lib/.  No cmake, no setuptools.
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
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libhla_gb300.so"
LIB_PATH = os.path.join(OUT_DIR, LIB_NAME)

SOURCES = ["hla_api.cu", "hla_fwd_tc.cu"] + [f"hla_fwd_tc_f{i}.cu" for i in range(12)] + \
    ["hla_fwd_simt.cu", "hla_combine.cu", "hla_decode.cu", "hla_noalloc.cu", "hla_bwd_simt.cu", "hla_bwd_tc.cu", "hla_bwd_norm.cu", "hla_bwd_norm_tc.cu", "hla_bwd_split.cu"] + \
    [f"hla_bwd_{t}_c{c}.cu" for t in ("f32", "bf16") for c in (16, 32, 64)] + ["hla_fwd3_simt.cu", "hla_fwd3_tc.cu", "hla_scan_tc.cu", "hla_fwd3_maps.cu"] + \
    [f"hla_fwd3_{t}_c{c}.cu" for t in ("f32", "bf16") for c in (16, 32, 64)]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "hla.h"), __file__]
    return max(os.path.getmtime(f) for f in files)


def _compile(src: str, extra: list[str]) -> str:
    obj = os.path.join(OBJ_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc()] + ARCH + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj


def build(force: bool = False, verbose: bool = False, extra: list[str] | None = None) -> str:
    """Compile every CUDA source for sm_103a and link libhla_gb300.so; returns its path."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _deps_mtime():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    extra = list(extra or [])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra), SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}", file=sys.stderr)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
