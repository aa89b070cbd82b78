"""Float64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package smoke check and the benchmark's CPU-baseline leg may
import this module.  The product (the CUDA library and its Python binding) never does,
and this module imports nothing from the product.

The arithmetic lives in ``fa_oracle.c`` (plain C, float64, one query row at a time); this
file compiles it with gcc and marshals arguments through ctypes.  What it computes, with
the passages it follows, is documented at the top of ``fa_oracle.c``:

    o[b,h,i,:] = sum_j softmax_j(scale * q[b,h,i,:] . k[b,h/g,j,:]) * v[b,h/g,j,:]
    lse[b,h,i] = ln sum_j exp(scale * q . k_j)          (natural log)

over the allowed keys j < Sk -- and j <= i when causal == 1 (top-left), j <= i + Sk - Sq when
causal == 2 (bottom-right) -- with g = Hq / Hkv.  A row with no allowed key gets o = 0 and
lse = -inf.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from typing import Optional, Sequence, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")

_handles = {}


def build(plant: int = 0, out_dir: Optional[str] = None) -> str:
    """Compile the oracle into a shared library and return its path.

    ``plant`` selects a deliberately wrong variant (0 = the real oracle); the test suite
    uses planted variants to show that its pins catch each mistake.
    """
    if out_dir is None:
        out_dir = _BUILD_DIR if plant == 0 else tempfile.mkdtemp(prefix="fa_oracle_plant_")
    os.makedirs(out_dir, exist_ok=True)
    name = "libfa_oracle.so" if plant == 0 else f"libfa_oracle_plant{plant}.so"
    out = os.path.join(out_dir, name)
    if plant == 0 and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
           f"-DFA_ORACLE_PLANT={int(plant)}", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes handle on one compiled copy of the oracle."""

    def __init__(self, path: str):
        self.path = path
        self.lib = ctypes.CDLL(path)
        f = self.lib.fa_oracle_rows
        f.restype = ctypes.c_int
        f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
                      ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                      ctypes.c_int]
        d = self.lib.fa_oracle_decode
        d.restype = ctypes.c_double
        d.argtypes = [ctypes.c_uint16, ctypes.c_int]
        self.lib.fa_oracle_max_threads.restype = ctypes.c_int

    def max_threads(self) -> int:
        return int(self.lib.fa_oracle_max_threads())

    def decode(self, bits: int, is_fp16: bool) -> float:
        return float(self.lib.fa_oracle_decode(int(bits) & 0xFFFF, int(bool(is_fp16))))

    def rows(self, q, k, v, is_fp16: bool, causal: int, scale: float,
             rows: np.ndarray, nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """Evaluate the query rows listed in ``rows`` (an n x 3 array of (b, h, i)).

        causal: 0 none, 1 top-left (j <= i), 2 bottom-right (j <= i + Sk - Sq); True means 1.

        q is [B, Hq, Sq, D], k and v are [B, Hkv, Sk, D]: 16-bit patterns (numpy uint16)
        or torch bf16/fp16 tensors.  Returns (o [n, D] float64, lse [n] float64).
        """
        qb, kb, vb = (_bits(x) for x in (q, k, v))
        B, Hq, Sq, D = qb.shape
        Bk, Hkv, Sk, Dk = kb.shape
        if vb.shape != kb.shape or Bk != B or Dk != D:
            raise ValueError("shape mismatch between q, k and v")
        r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
        n = r.shape[0]
        o = np.empty((n, D), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        st = self.lib.fa_oracle_rows(qb.ctypes.data, kb.ctypes.data, vb.ctypes.data,
                                     int(bool(is_fp16)), B, Hq, Hkv, Sq, Sk, D,
                                     int(causal), float(scale), r.ctypes.data, n,
                                     o.ctypes.data, lse.ctypes.data, int(nthreads))
        if st != 0:
            raise ValueError(f"oracle rejected its arguments (status {st})")
        return o, lse

    def full(self, q, k, v, is_fp16: bool, causal: int, scale: float,
             nthreads: int = 0) -> Tuple[np.ndarray, np.ndarray]:
        """Every query row: returns (o [B, Hq, Sq, D], lse [B, Hq, Sq]) in float64."""
        qb = _bits(q)
        B, Hq, Sq, D = qb.shape
        rows = all_rows(B, Hq, Sq)
        o, lse = self.rows(qb, k, v, is_fp16, causal, scale, rows, nthreads)
        return o.reshape(B, Hq, Sq, D), lse.reshape(B, Hq, Sq)


def all_rows(B: int, H: int, S: int) -> np.ndarray:
    """All (b, h, i) triples in row-major order."""
    b, h, i = np.meshgrid(np.arange(B), np.arange(H), np.arange(S), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int64)


def _bits(x) -> np.ndarray:
    """16-bit patterns of a bf16/fp16 torch tensor, or a uint16 numpy array, as uint16."""
    if isinstance(x, np.ndarray):
        if x.dtype != np.uint16:
            raise TypeError("numpy inputs must hold uint16 bit patterns")
        return np.ascontiguousarray(x)
    import torch  # only for tensors handed in by the caller
    t = x.detach().to("cpu").contiguous()
    if t.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("torch inputs must be bf16 or fp16")
    return t.view(torch.int16).numpy().view(np.uint16)


def load(plant: int = 0) -> Oracle:
    """Build (if needed) and load the oracle; planted variants are built in a temp dir."""
    if plant not in _handles:
        _handles[plant] = Oracle(build(plant))
    return _handles[plant]


def rows(*args, **kwargs):
    return load().rows(*args, **kwargs)


def full(*args, **kwargs):
    return load().full(*args, **kwargs)


__all__: Sequence[str] = ["build", "load", "Oracle", "rows", "full", "all_rows"]
