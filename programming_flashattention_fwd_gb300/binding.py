"""ctypes binding of libfa_gb300.so -- argument marshalling only.

Every step of the attention computation runs in the library's CUDA kernel; this module
only turns torch tensors into device pointers, sizes and a stream handle, and raises
FaError on a non-zero status.  The library must exist (built by ``build.build()``); a
missing library raises at the first call -- there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa_gb300.so")

STATUS = {
    0: "FA_OK", 1: "FA_ERR_NULL_PTR", 2: "FA_ERR_BAD_DIM", 3: "FA_ERR_HEADS",
    4: "FA_ERR_UNSUPPORTED_D", 5: "FA_ERR_ALIGN", 6: "FA_ERR_ALIAS", 7: "FA_ERR_SCALE",
    8: "FA_ERR_NO_DEVICE", 9: "FA_ERR_ARCH", 10: "FA_ERR_TENSORMAP", 11: "FA_ERR_LAUNCH",
    12: "FA_ERR_DEVICE_TIMEOUT", 13: "FA_ERR_CAUSAL", 14: "FA_ERR_SHAPE", 15: "FA_ERR_ARG",
    16: "FA_ERR_TOO_LARGE",
}

# FA_HOST_NOALLOC_MAX_BYTES of include/fa.h: the fixed staging area of fa_fwd_host_noalloc.
HOST_NOALLOC_MAX_BYTES = 64 << 20

_lib = None
_lock = threading.Lock()

_FWD_ARGS = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_void_p]


class FaError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    for name in ("fa_fwd", "fa_fwd_fp16"):
        f = getattr(lib, name)
        f.restype = ctypes.c_int
        f.argtypes = _FWD_ARGS
    lib.fa_fwd_select.restype = ctypes.c_int
    lib.fa_fwd_select.argtypes = _FWD_ARGS + [ctypes.c_int, ctypes.c_int]
    lib.fa_fwd_debug.restype = ctypes.c_int
    lib.fa_fwd_debug.argtypes = _FWD_ARGS + [ctypes.c_int, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_int, ctypes.c_float]
    lib.fa_fwd_host.restype = ctypes.c_int
    lib.fa_fwd_host.argtypes = ([ctypes.c_void_p] * 10 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int,
                                                                                ctypes.c_int, ctypes.c_void_p])
    lib.fa_fwd_host_noalloc.restype = ctypes.c_int
    lib.fa_fwd_host_noalloc.argtypes = ([ctypes.c_void_p] * 5 + [ctypes.c_int] * 7 + [ctypes.c_float, ctypes.c_int,
                                                                                     ctypes.c_int, ctypes.c_void_p])
    lib.fa_strerror.restype = ctypes.c_char_p
    lib.fa_strerror.argtypes = [ctypes.c_int]
    lib.fa_device_status.restype = ctypes.c_int
    lib.fa_device_status.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_uint32)]
    lib.fa_gemm.restype = ctypes.c_int
    lib.fa_gemm.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] * 6 + [ctypes.c_void_p]
    lib.fa_softmax_rows.restype = ctypes.c_int
    lib.fa_softmax_rows.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_void_p]
    return lib


def load_library(path: Optional[str] = None) -> ctypes.CDLL:
    """Load (once) and return the CUDA library; raises if it is missing."""
    global _lib
    lib = _lib
    if lib is not None and path is None:
        return lib
    with _lock:
        if _lib is not None and (path is None or path == LIB_PATH):
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise FaError(-1, f"CUDA library not built: {p} is missing "
                              "(run programming_flashattention_fwd_gb300.build.build())")
        lib = _declare(ctypes.CDLL(p))
        if p == LIB_PATH:
            _lib = lib
        return lib


def fa_strerror(status: int) -> str:
    return load_library().fa_strerror(int(status)).decode()


# The current stream's raw handle straight from torch's C layer when it offers that (one call
# instead of building a torch.cuda.Stream object: a few microseconds less per launch).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)
_cur_device = getattr(torch._C, "_cuda_getDevice", None)


def _stream_handle(stream) -> int:
    if stream is None:
        if _raw_stream is not None and _cur_device is not None:
            return int(_raw_stream(_cur_device()))
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _check_stream_device(stream, device: torch.device) -> None:
    """A torch.cuda.Stream passed with tensors must belong to their device: the library
    enqueues on the stream but encodes and launches on the current device."""
    if isinstance(stream, torch.cuda.Stream) and stream.device != device:
        raise ValueError(f"stream is on {stream.device} but the tensors are on {device}")


def _check_same_device(tensors) -> Optional[torch.device]:
    """All non-empty CUDA tensors on one device; returns it (None if every tensor is empty)."""
    dev = None
    for name, t in tensors:
        if t.numel() and t.is_cuda:
            if dev is None:
                dev = t.device
            elif t.device != dev:
                raise ValueError(f"{name} is on {t.device} but another tensor is on {dev}: "
                                 "every tensor of one call must be on the same GPU")
    return dev


def _check_tensors(q, k, v, o, lse):
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous ([B, H, S, D] dense layout)")
        if t.numel() and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    _check_same_device((("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)))
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4 or o.dim() != 4 or lse.dim() != 3:
        raise ValueError("q, k, v, o must be 4-D [B, H, S, D] and lse 3-D [B, Hq, Sq]")
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("k and v must be [B, Hkv, Sk, D] with q's B and D")
    if o.shape != q.shape or tuple(lse.shape) != tuple(q.shape[:3]):
        raise ValueError("o must match q's shape and lse must be [B, Hq, Sq]")
    if not (q.dtype == k.dtype == v.dtype == o.dtype) or lse.dtype != torch.float32:
        raise ValueError("q, k, v, o share one 16-bit dtype; lse is float32")


def _causal_code(causal) -> int:
    """False/0: none; True/1: top-left (j <= i); 2 or "bottom_right": j <= i + Sk - Sq."""
    if causal in ("bottom_right", "bottom-right"):
        return 2
    if causal in ("top_left", "top-left"):
        return 1
    return int(causal)


class _OnDevice:
    """Makes `device` current for the library call when it is not already (the C ABI works on
    the current device); a no-op otherwise, so the common call pays nothing."""
    __slots__ = ("idx", "prev")

    def __init__(self, device: Optional[torch.device]):
        self.idx = device.index if device is not None and device.type == "cuda" else None
        self.prev = None

    def __enter__(self):
        if self.idx is not None:
            cur = _cur_device() if _cur_device is not None else torch.cuda.current_device()
            if cur != self.idx:
                self.prev = cur
                torch.cuda.set_device(self.idx)
        return self

    def __exit__(self, *exc):
        if self.prev is not None:
            torch.cuda.set_device(self.prev)
        return False


def _call(fn_name: str, q, k, v, o, lse, causal: bool, scale: float, stream, extra=()):
    _check_tensors(q, k, v, o, lse)
    dev = q.device if q.is_cuda else None
    if dev is not None:
        _check_stream_device(stream, dev)
    B, Hq, Sq, D = q.shape
    Hkv, Sk = k.shape[1], k.shape[2]
    lib = load_library()
    with _OnDevice(dev):
        st = getattr(lib, fn_name)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                                   B, Hq, Hkv, Sq, Sk, D, _causal_code(causal), float(scale),
                                   _stream_handle(stream), *extra)
    if st != 0:
        raise FaError(st, fa_strerror(st))


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """bf16 attention forward into caller-allocated o [B,Hq,Sq,D] and lse [B,Hq,Sq] fp32."""
    if q.dtype != torch.bfloat16:
        raise ValueError("fa_fwd takes bf16 tensors (use fa_fwd_fp16 for fp16)")
    _call("fa_fwd", q, k, v, o, lse, causal, scale, stream)


def fa_fwd_fp16(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """fp16 attention forward into caller-allocated o and lse."""
    if q.dtype != torch.float16:
        raise ValueError("fa_fwd_fp16 takes fp16 tensors")
    _call("fa_fwd_fp16", q, k, v, o, lse, causal, scale, stream)


def fa_fwd_debug(q, k, v, o, lse, causal: bool, scale: float, timeout_ns: int = 0,
                 inject: int = 0, kernel: int = 0, tau: float = -1.0, stream=None) -> None:
    """Test hook: the forward with an explicit watchdog limit, fault-injection mask, kernel
    variant and lazy-rescale threshold tau (log2 units; negative = the default 12)."""
    _call("fa_fwd_debug", q, k, v, o, lse, causal, scale, stream,
          extra=(int(q.dtype == torch.float16), int(timeout_ns), int(inject), int(kernel), float(tau)))


def fa_fwd_select(q, k, v, o, lse, causal, scale: float, kernel: int = 0, stream=None) -> None:
    """The forward with an explicit kernel variant (0 automatic, 1 two query tiles per CTA
    with 128-key steps, 2 one query tile per CTA with 64-key steps, 3 one query tile per CTA
    with 128-key steps, D 128 only); bf16 or fp16."""
    _call("fa_fwd_select", q, k, v, o, lse, causal, scale, stream,
          extra=(int(q.dtype == torch.float16), int(kernel)))


def fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, causal, scale: float,
                chunks: int = 0, stream=None) -> None:
    """The forward on host (CPU, ideally pinned) tensors q_h, k_h, v_h into host o_h, lse_h,
    staged through the caller's device buffers q_d .. lse_d of the same shapes; copies in,
    kernels and copies back overlap chunk by chunk.  Asynchronous on `stream`."""
    _check_tensors(q_d, k_d, v_d, o_d, lse_d)
    for name, h, d in (("q_h", q_h, q_d), ("k_h", k_h, k_d), ("v_h", v_h, v_d), ("o_h", o_h, o_d),
                       ("lse_h", lse_h, lse_d)):
        if not isinstance(h, torch.Tensor) or h.is_cuda or not h.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
        if h.shape != d.shape or h.dtype != d.dtype:
            raise ValueError(f"{name} must match its device buffer's shape and dtype")
    B, Hq, Sq, D = q_d.shape
    Hkv, Sk = k_d.shape[1], k_d.shape[2]
    dev = q_d.device if q_d.is_cuda else None
    if dev is not None:
        _check_stream_device(stream, dev)
    with _OnDevice(dev):
        st = load_library().fa_fwd_host(
            q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(), lse_h.data_ptr(),
            q_d.data_ptr(), k_d.data_ptr(), v_d.data_ptr(), o_d.data_ptr(), lse_d.data_ptr(),
            B, Hq, Hkv, Sq, Sk, D, _causal_code(causal), float(scale), int(q_d.dtype == torch.float16), int(chunks),
            _stream_handle(stream))
    if st != 0:
        raise FaError(st, fa_strerror(st))


def fa_fwd_host_noalloc(q_h, k_h, v_h, o_h, lse_h, causal, scale: float, chunks: int = 0,
                        stream=None) -> None:
    """fa_fwd_host without caller-owned device buffers, for callers that cannot allocate device
    memory: the staging area is the library's fixed HOST_NOALLOC_MAX_BYTES device array, shared
    by every call on the device (calls on different streams must not overlap in time).
    q_h .. lse_h are contiguous CPU tensors (pinned for overlap); asynchronous on `stream`."""
    for name, h in (("q_h", q_h), ("k_h", k_h), ("v_h", v_h), ("o_h", o_h), ("lse_h", lse_h)):
        if not isinstance(h, torch.Tensor) or h.is_cuda or not h.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CPU tensor")
    if q_h.dim() != 4 or k_h.dim() != 4 or k_h.shape != v_h.shape or o_h.shape != q_h.shape or \
            tuple(lse_h.shape) != tuple(q_h.shape[:3]) or q_h.shape[0] != k_h.shape[0] or q_h.shape[3] != k_h.shape[3]:
        raise ValueError("q_h, o_h [B,Hq,Sq,D], k_h, v_h [B,Hkv,Sk,D] and lse_h [B,Hq,Sq] expected")
    if not (q_h.dtype == k_h.dtype == v_h.dtype == o_h.dtype) or q_h.dtype not in (torch.bfloat16, torch.float16) \
            or lse_h.dtype != torch.float32:
        raise ValueError("q_h, k_h, v_h, o_h share one 16-bit dtype; lse_h is float32")
    B, Hq, Sq, D = q_h.shape
    Hkv, Sk = k_h.shape[1], k_h.shape[2]
    # the staging area is taken on the current device: with a stream given, that is its device
    dev = stream.device if isinstance(stream, torch.cuda.Stream) else None
    with _OnDevice(dev):
        st = load_library().fa_fwd_host_noalloc(
            q_h.data_ptr(), k_h.data_ptr(), v_h.data_ptr(), o_h.data_ptr(), lse_h.data_ptr(),
            B, Hq, Hkv, Sq, Sk, D, _causal_code(causal), float(scale), int(q_h.dtype == torch.float16), int(chunks),
            _stream_handle(stream))
    if st != 0:
        raise FaError(st, fa_strerror(st))


def attention(q, k, v, causal=False, scale: Optional[float] = None, stream=None,
              kernel: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Allocate o and lse on q's device and run the forward; returns (o, lse)."""
    if scale is None:
        scale = 1.0 / math.sqrt(q.shape[-1])
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if kernel:
        fa_fwd_select(q, k, v, o, lse, causal, scale, kernel, stream)
    elif q.dtype == torch.float16:
        fa_fwd_fp16(q, k, v, o, lse, causal, scale, stream)
    else:
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def fa_device_status(stream=None) -> Tuple[int, int]:
    """Synchronise the stream, read and clear the watchdog word: (status, raw word)."""
    w = ctypes.c_uint32(0)
    st = load_library().fa_device_status(_stream_handle(stream), ctypes.byref(w))
    return int(st), int(w.value)


def gemm(a, b, bias=None, epilogue: int = 0, out_fp32: bool = False, c=None, stream=None):
    """C = epilogue(A @ B) on the GPU (fa_gemm): a [M,K], b [K,N] bf16/fp16 CUDA tensors,
    bias [N] float32 for epilogue 1 (+bias) and 2 (tanh-GELU(. + bias)).  Returns c."""
    if a.dim() != 2 or b.dim() != 2 or a.shape[1] != b.shape[0]:
        raise ValueError("a must be [M, K] and b [K, N]")
    if a.dtype != b.dtype or a.dtype not in (torch.bfloat16, torch.float16):
        raise ValueError("a and b share one 16-bit dtype")
    for name, t in (("a", a), ("b", b)):
        if not (t.is_cuda and t.is_contiguous()):
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if a.device != b.device:
        raise ValueError(f"a is on {a.device} but b is on {b.device}")
    _check_stream_device(stream, a.device)
    M, K = a.shape
    N = b.shape[1]
    if c is None:
        c = torch.empty((M, N), dtype=torch.float32 if out_fp32 else a.dtype, device=a.device)
    if epilogue and (bias is None or bias.dtype != torch.float32 or bias.numel() != N or not bias.is_cuda):
        raise ValueError("epilogues 1 and 2 need a float32 CUDA bias of N entries")
    if c.device != a.device or (epilogue and bias.device != a.device):
        raise ValueError("c and bias must be on a's device")
    with _OnDevice(a.device):
        st = load_library().fa_gemm(a.data_ptr(), b.data_ptr(), c.data_ptr(), bias.data_ptr() if epilogue else None,
                                    M, N, K, 0 if a.dtype == torch.bfloat16 else 1, int(bool(out_fp32)),
                                    int(epilogue), _stream_handle(stream))
    if st != 0:
        raise FaError(st, fa_strerror(st))
    return c


def softmax_rows(x, y=None, stream=None):
    """Row softmax on the GPU (fa_softmax_rows): x [rows, cols] float32 or bf16 CUDA tensor;
    y defaults to a new tensor (pass y=x for in place).  Returns y."""
    if x.dim() != 2 or x.dtype not in (torch.float32, torch.bfloat16) or not (x.is_cuda and x.is_contiguous()):
        raise ValueError("x must be a contiguous 2-D float32 or bf16 CUDA tensor")
    if y is None:
        y = torch.empty_like(x)
    if y.shape != x.shape or y.dtype != x.dtype or not y.is_contiguous() or y.device != x.device:
        raise ValueError("y must match x (shape, dtype, device)")
    _check_stream_device(stream, x.device)
    with _OnDevice(x.device):
        st = load_library().fa_softmax_rows(x.data_ptr(), y.data_ptr(), x.shape[0], x.shape[1],
                                            0 if x.dtype == torch.float32 else 1, _stream_handle(stream))
    if st != 0:
        raise FaError(st, fa_strerror(st))
    return y
