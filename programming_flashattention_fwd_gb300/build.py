"""Build libfa_gb300.so in-tree with nvcc for sm_103a (no torch extension machinery).

    python -m programming_flashattention_fwd_gb300.build [--verbose] [--force]

The translation units (kernels, host API, host pipeline) compile in parallel; the result lands next to
this file.  A rebuild is skipped when the library is newer than every source.
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
BUILD_DIR = os.path.join(PKG, "_build")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfa_gb300.so")


def sources():
    return [os.path.join(CSRC, f) for f in ("fa_fwd_sm103.cu", "fa_fwd1_sm103.cu", "gemm_sm103.cu", "softmax_sm103.cu", "fa_api.cpp",
                                                  "host_pipeline.cpp", "host_noalloc.cu")]


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = glob.glob(os.path.join(CSRC, "*")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), out: str = LIB_PATH) -> str:
    """Compile and link the library; returns its path."""
    if not force and not extra_flags and not _stale(out):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", f"-I{INCLUDE}", f"-I{CSRC}",
              *ARCH, *extra_flags]
    if verbose:
        common += ["-Xptxas", "-v"]
    tag = f"{os.getpid()}"

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.basename(src) + f".{tag}.o")
        lang = [] if src.endswith(".cu") else ["-x", "cu"]
        cmd = [cc, *common, *lang, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            sys.stderr.write(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=6) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = out + f".tmp{tag}"
    cmd = [cc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *objs, "-o", tmp, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out)
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--force", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=a.verbose))


if __name__ == "__main__":
    main()
