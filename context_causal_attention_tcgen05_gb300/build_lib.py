"""Builds libcp_attn.so in-tree for sm_103a with nvcc (no cmake).

Each CUDA translation unit under csrc/ is compiled in parallel to an object
file under _build/, then linked into the package directory.  Run as
``python -m context_causal_attention_tcgen05_gb300.build_lib``.

``--debug`` (``build(debug=True)``) builds libcp_attn_debug.so instead, with
-DCP_DEBUG: every kernel checks the indices it computes against its buffers'
extents, skips an access that fails and records the failure, which
cp_check_device_status reports as CP_ERR_DEVICE_INDEX.  Load it by setting
CP_ATTN_LIBRARY to its path before the binding loads the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_NAME = "libcp_attn.so"
LIB_PATH = os.path.join(PKG_DIR, LIB_NAME)
DEBUG_BUILD_DIR = os.path.join(PKG_DIR, "_build_debug")
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libcp_attn_debug.so")

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = [
    "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"), "-I", CSRC,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcp_attn.so")


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(nvcc: str, src: str, extra: list[str], build_dir: str) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    cmd = [nvcc, *ARCH_FLAGS, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(verbose: bool = False, extra_flags: list[str] | None = None, debug: bool = False) -> str:
    """Compile every csrc/*.cu and link libcp_attn.so (libcp_attn_debug.so with the
    index checks when debug); returns the library path."""
    nvcc = _nvcc()
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    extra = list(extra_flags or []) + (["-DCP_DEBUG"] if debug else [])
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        results = list(ex.map(lambda s: _compile(nvcc, s, extra, build_dir), srcs))
    objs = [o for o, _ in results]
    if verbose:
        for (_o, err), s in zip(results, srcs):
            if err.strip():
                print(f"[{os.path.basename(s)}]\n{err}", file=sys.stderr)
    tmp = lib_path + ".tmp"
    cmd = [nvcc, *ARCH_FLAGS, "-shared", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    v = "-v" in sys.argv
    flags = ["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None
    print(build(verbose=v or bool(flags), extra_flags=flags, debug="--debug" in sys.argv))
