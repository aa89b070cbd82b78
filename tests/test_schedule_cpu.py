"""Host-side check of the persistent attention kernels' work schedule (csrc/schedule.h, the
same functions the kernels call): tests/schedule_check.cpp is compiled with the host compiler
and walks every CTA's rounds for 24 thousand shape x mask x grid-size combinations -- every
query tile visited exactly once, the right KV head, every needed key tile read and none past
the mask (beyond the padding rows of a ragged last tile), every TMA box starting inside k/v."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "programming_flashattention_fwd_gb300", "csrc")


def cuda_include():
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.exists(os.path.join(base, "include", "cuda_runtime.h")):
            return os.path.join(base, "include")
    nvcc = shutil.which("nvcc")
    if nvcc:
        inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
        if os.path.exists(os.path.join(inc, "cuda_runtime.h")):
            return inc
    return None


def test_schedule_covers_every_tile_once(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = cuda_include()
    if not cxx or not inc:
        pytest.skip("needs a host C++ compiler and the CUDA headers")
    exe = str(tmp_path / "schedule_check")
    src = os.path.join(ROOT, "tests", "schedule_check.cpp")
    r = subprocess.run([cxx, "-std=c++17", "-O2", f"-I{CSRC}", f"-I{os.path.join(ROOT, 'include')}", f"-I{inc}",
                        src, "-o", exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
