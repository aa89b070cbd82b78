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
_SRCS = [_SRC, os.path.join(_HERE, "ops_oracle.c")]
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
    if plant == 0 and os.path.exists(out) and all(os.path.getmtime(out) >= os.path.getmtime(x) for x in _SRCS):
        return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-D_DEFAULT_SOURCE", "-fPIC", "-shared", "-fopenmp",
           f"-DFA_ORACLE_PLANT={int(plant)}", *_SRCS, "-o", tmp, "-lm"]
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
        g = self.lib.fa_oracle_gemm_entries
        g.restype = ctypes.c_int
        g.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                      ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                      ctypes.c_void_p]
        sm = self.lib.fa_oracle_softmax_rows
        sm.restype = ctypes.c_int
        sm.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                       ctypes.c_int64, ctypes.c_void_p]
        self.lib.fa_oracle_gelu_tanh.restype = ctypes.c_double
        self.lib.fa_oracle_gelu_tanh.argtypes = [ctypes.c_double]

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


    # ---------------------------------------------------------------- building blocks
    def gemm_entries(self, a, b, is_fp16: bool, entries, bias=None, epilogue: int = 0) -> np.ndarray:
        """epilogue(A @ B) at the listed (m, n) entries; A [M,K], B [K,N] 16-bit (bits or tensors).
        epilogue: 0 none, 1 + bias[n], 2 tanh-GELU(. + bias[n]); bias is float32 [N]."""
        ab, bb = _bits(a), _bits(b)
        M, K = ab.shape
        Kb, N = bb.shape
        if Kb != K:
            raise ValueError("inner dimensions differ")
        e = np.ascontiguousarray(np.asarray(entries, dtype=np.int64).reshape(-1, 2))
        out = np.empty(e.shape[0], dtype=np.float64)
        bptr = None
        if epilogue:
            bias = np.ascontiguousarray(np.asarray(_as_numpy(bias), dtype=np.float32).reshape(-1))
            if bias.shape[0] != N:
                raise ValueError("bias must have N entries")
            bptr = bias.ctypes.data
        st = self.lib.fa_oracle_gemm_entries(ab.ctypes.data, bb.ctypes.data, int(bool(is_fp16)), M, N, K,
                                             bptr, int(epilogue), e.ctypes.data, e.shape[0], out.ctypes.data)
        if st != 0:
            raise ValueError(f"oracle rejected its arguments (status {st})")
        return out

    def gemm_full(self, a, b, is_fp16: bool, bias=None, epilogue: int = 0) -> np.ndarray:
        ab, bb = _bits(a), _bits(b)
        M, N = ab.shape[0], bb.shape[1]
        mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
        ent = np.stack([mm.ravel(), nn.ravel()], axis=1)
        return self.gemm_entries(ab, bb, is_fp16, ent, bias, epilogue).reshape(M, N)

    def softmax_rows(self, x, row_ids=None) -> np.ndarray:
        """Row softmax of the listed rows of x [rows, cols] (fp32 array/tensor or bf16 tensor)."""
        xf, xb = None, None
        try:
            import torch
            if isinstance(x, torch.Tensor) and x.dtype == torch.bfloat16:
                xb = _bits(x)
            elif isinstance(x, torch.Tensor):
                xf = np.ascontiguousarray(x.detach().cpu().float().numpy())
        except ImportError:
            pass
        if xf is None and xb is None:
            xf = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
        arr = xf if xf is not None else xb
        rows, cols = arr.shape
        ids = np.arange(rows, dtype=np.int64) if row_ids is None else np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
        out = np.empty((ids.shape[0], cols), dtype=np.float64)
        st = self.lib.fa_oracle_softmax_rows(xf.ctypes.data if xf is not None else None,
                                             xb.ctypes.data if xb is not None else None,
                                             rows, cols, ids.ctypes.data, ids.shape[0], out.ctypes.data)
        if st != 0:
            raise ValueError(f"oracle rejected its arguments (status {st})")
        return out

    def gelu_tanh(self, h: float) -> float:
        return float(self.lib.fa_oracle_gelu_tanh(float(h)))


def _as_numpy(x):
    if isinstance(x, np.ndarray):
        return x
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().float().numpy()
    except ImportError:
        pass
    return np.asarray(x)


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
