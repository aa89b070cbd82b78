"""The C-ABI library builds, loads, exports every function include/fa.h declares, and
rejects bad arguments with the documented status code before making any CUDA call.

Every call in this file is rejected by validation (or is an empty problem), so none of
them reaches the CUDA runtime: they are safe on machines with or without a GPU."""
import math
import os
import re

import pytest

from programming_flashattention_fwd_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    path = fa_build.build()
    from programming_flashattention_fwd_gb300 import binding
    return binding.load_library(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_\w+)\s*\(", text)))


def declared_status_codes():
    text = open(HEADER).read()
    return {m.group(1): int(m.group(2)) for m in re.finditer(r"\b(FA_\w+)\s*=\s*(\d+)", text)}


def test_header_declares_the_entry_points():
    fns = declared_functions()
    for name in ("fa_fwd", "fa_fwd_fp16", "fa_strerror", "fa_device_status", "fa_fwd_debug", "fa_gemm",
                 "fa_softmax_rows", "fa_fwd_select"):
        assert name in fns


def test_library_exports_every_declared_function(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/fa.h but not exported"


def test_strerror_covers_every_code(lib):
    codes = declared_status_codes()
    assert len(codes) == 17 and sorted(codes.values()) == list(range(17))
    msgs = set()
    for name, val in codes.items():
        msg = lib.fa_strerror(val).decode()
        assert msg.startswith(name), (name, msg)
        msgs.add(msg)
    assert len(msgs) == len(codes)
    assert lib.fa_strerror(999).decode() == "unknown fa status code"


# Fake, 16-byte aligned, non-overlapping "device" addresses: validation never dereferences them.
Q, K, V, O, L = 0x10000000, 0x20000000, 0x30000000, 0x40000000, 0x50000000
GOOD = dict(B=1, Hq=4, Hkv=2, Sq=256, Sk=256, D=128, causal=1, scale=0.125)


def call(lib, fn="fa_fwd", q=Q, k=K, v=V, o=O, lse=L, **over):
    a = dict(GOOD, **over)
    return getattr(lib, fn)(q, k, v, o, lse, a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["D"],
                            a["causal"], a["scale"], None)


@pytest.mark.parametrize("fn", ["fa_fwd", "fa_fwd_fp16"])
@pytest.mark.parametrize("over,code", [
    (dict(B=-1), 2), (dict(Sq=-5), 2), (dict(Sk=-1), 2), (dict(Sk=0), 2),
    (dict(Hq=0), 3), (dict(Hkv=0), 3), (dict(Hq=6, Hkv=4), 3), (dict(Hq=2, Hkv=4), 3),
    (dict(D=32), 4), (dict(D=96), 4), (dict(D=192), 4), (dict(D=512), 4),
    (dict(scale=math.nan), 7), (dict(scale=math.inf), 7),
    (dict(B=100000, Hq=100000, Hkv=1), 2),
    (dict(causal=3), 13), (dict(causal=-1), 13),
])
def test_invalid_arguments(lib, fn, over, code):
    assert call(lib, fn, **over) == code


def test_empty_problems_are_noops(lib):
    # B == 0 or Sq == 0 returns FA_OK without touching memory, even with NULL pointers
    assert call(lib, q=None, k=None, v=None, o=None, lse=None, B=0) == 0
    assert call(lib, q=None, k=None, v=None, o=None, lse=None, Sq=0) == 0
    assert call(lib, Sq=0, Sk=0) == 0


@pytest.mark.parametrize("which", ["q", "k", "v", "o", "lse"])
def test_null_pointers(lib, which):
    assert call(lib, **{which: None}) == 1


@pytest.mark.parametrize("which,addr", [("q", Q + 8), ("k", K + 2), ("v", V + 4), ("o", O + 8), ("lse", L + 2)])
def test_misaligned_pointers(lib, which, addr):
    assert call(lib, **{which: addr}) == 5


def test_lse_needs_only_4_byte_alignment(lib):
    # A 4-byte aligned lse passes the alignment check and is then rejected by the overlap
    # check (it sits inside o), so the call never reaches the CUDA runtime.
    assert call(lib, lse=O + 4) == 6


@pytest.mark.parametrize("over", [dict(o=Q), dict(o=K + 64), dict(lse=V), dict(lse=O + 16)])
def test_overlapping_outputs(lib, over):
    assert call(lib, **over) == 6


def test_debug_entry_point_validates_the_same_way(lib):
    f = lib.fa_fwd_debug
    assert f(Q, K, V, O, L, 1, 3, 2, 8, 8, 128, 0, 1.0, None, 0, 0, 0, 0, -1.0) == 3
    assert f(Q, K, V, O, L, 1, 2, 2, 8, 8, 80, 0, 1.0, None, 1, 0, 0, 0, -1.0) == 4
    assert f(Q, K, V, O, L, 1, 2, 2, 8, 8, 256, 0, 1.0, None, 0, 0, 0, 1, -1.0) == 4   # kernel 1 has no D 256
    assert f(Q, K, V, O, L, 1, 2, 2, 8, 8, 128, 0, 1.0, None, 0, 0, 0, 5, -1.0) == 15  # no kernel 5
    assert f(Q, K, V, O, L, 1, 2, 2, 8, 8, 128, 0, 1.0, None, 0, 0, 0, 0, float("nan")) == 15
    assert f(Q, K, V, O, L, 1, 2, 2, 8, 8, 128, 0, 1.0, None, 0, 0, 0, 0, 15.5) == 15
    # valid tau values pass validation (the overlapping lse then stops the call before CUDA)
    for tau in (0.0, 8.0, 15.0, -1.0):
        assert f(Q, K, V, O, O + 16, 1, 2, 2, 8, 8, 128, 0, 1.0, None, 0, 0, 0, 3, tau) == 6


# fa_gemm(a, b, c, bias, M, N, K, dtype, out_fp32, epilogue, stream) -- every call rejected before CUDA
GG = dict(M=256, N=512, K=128, dtype=0, out=0, epi=2)
A_, B_, C_, BIAS = 0x60000000, 0x70000000, 0x80000000, 0x90000000


def gemm_call(lib, a=A_, b=B_, c=C_, bias=BIAS, **over):
    g = dict(GG, **over)
    return lib.fa_gemm(a, b, c, bias, g["M"], g["N"], g["K"], g["dtype"], g["out"], g["epi"], None)


@pytest.mark.parametrize("over,code", [
    (dict(M=-1), 2), (dict(K=-8), 2), (dict(K=0), 2),
    (dict(dtype=2), 15), (dict(out=3), 15), (dict(epi=3), 15), (dict(epi=-1), 15),
    (dict(K=12), 14), (dict(N=100), 14),
    (dict(a=None), 1), (dict(c=None), 1), (dict(bias=None), 1),
    (dict(a=A_ + 8), 5), (dict(c=C_ + 2), 5), (dict(bias=BIAS + 2), 5),
    (dict(c=A_ + 64), 6), (dict(c=BIAS - 64, bias=BIAS), 6),
])
def test_gemm_invalid_arguments(lib, over, code):
    assert gemm_call(lib, **over) == code


def test_gemm_empty_and_bias_optional(lib):
    assert gemm_call(lib, M=0) == 0 and gemm_call(lib, N=0, a=None, b=None, c=None) == 0
    # no bias needed without an epilogue: rejected later only by the overlap check here
    assert gemm_call(lib, epi=0, bias=None, c=A_ + 16) == 6


@pytest.mark.parametrize("args,code", [
    ((Q, O, -1, 8, 0), 2), ((Q, O, 4, 0, 0), 2), ((Q, O, 4, 8, 2), 15), ((None, O, 4, 8, 0), 1),
    ((Q + 2, O, 4, 8, 0), 5), ((Q + 1, O, 4, 8, 1), 5), ((Q, Q + 8, 4, 8, 0), 6), ((Q, O, 0, 8, 0), 0),
])
def test_softmax_invalid_arguments(lib, args, code):
    x, y, rows, cols, dtype = args
    assert lib.fa_softmax_rows(x, y, rows, cols, dtype, None) == code


@pytest.mark.parametrize("D,dtype,kernel,code", [
    (128, 0, 4, 15), (128, 2, 1, 15), (128, 0, -1, 15),
    (256, 0, 1, 4), (192, 0, 0, 4), (256, 0, 3, 4), (64, 0, 3, 4), (192, 1, 2, 4),
])
def test_select_invalid_arguments(lib, D, dtype, kernel, code):
    assert lib.fa_fwd_select(Q, K, V, O, L, 1, 4, 2, 256, 256, D, 1, 0.1, None, dtype, kernel) == code


def test_select_valid_pairs_pass_validation(lib):
    # every supported (kernel, D) pair gets past validation: an overlapping lse makes each
    # call stop at the overlap check instead, before any CUDA call
    for kernel, D in ((0, 64), (0, 128), (0, 256), (1, 64), (1, 128), (2, 64), (2, 128), (2, 256), (3, 128)):
        assert lib.fa_fwd_select(Q, K, V, O, O + 16, 1, 4, 2, 256, 256, D, 1, 0.1, None, 0, kernel) == 6


# fa_fwd_host(q_h, k_h, v_h, o_h, lse_h, q_d, k_d, v_d, o_d, lse_d, sizes..., dtype, chunks, stream)
QH, KH, VH, OH, LH = 0xA0000000, 0xB0000000, 0xC0000000, 0xD0000000, 0xE0000000


def call_host(lib, dtype=0, chunks=0, **over):
    a = dict(GOOD, qh=QH, kh=KH, vh=VH, oh=OH, lh=LH, q=Q, k=K, v=V, o=O, lse=L)
    a.update(over)
    return lib.fa_fwd_host(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["q"], a["k"], a["v"], a["o"], a["lse"],
                           a["B"], a["Hq"], a["Hkv"], a["Sq"], a["Sk"], a["D"], a["causal"], a["scale"], dtype,
                           chunks, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), 15), (dict(dtype=-1), 15), (dict(chunks=-1), 15), (dict(chunks=65), 15),
    (dict(D=96), 4), (dict(Hq=3), 3), (dict(causal=3), 13), (dict(scale=math.inf), 7), (dict(Sk=0), 2),
    (dict(qh=None), 1), (dict(lh=None), 1), (dict(o=None), 1),
    (dict(q=Q + 8), 5), (dict(lse=L + 2), 5),
    # written ranges must be disjoint from every other range
    (dict(oh=QH + 64), 6), (dict(lh=OH + 4), 6), (dict(oh=Q), 6), (dict(qh=K + 16), 6), (dict(lh=KH), 6),
    (dict(o=L), 6), (dict(k=V), 6),
])
def test_host_entry_point_invalid_arguments(lib, kw, code):
    assert call_host(lib, **kw) == code


def test_host_entry_point_empty_and_shared_inputs(lib):
    # empty problems are no-ops before any pointer is looked at
    assert call_host(lib, B=0, qh=None, kh=None, vh=None, oh=None, lh=None) == 0
    assert call_host(lib, Sq=0) == 0
    # host inputs may share memory (they are only read): the call then gets as far as the
    # overlap checks of the written ranges, here a clash of lse_h with o_h
    assert call_host(lib, kh=QH, vh=QH, lh=OH) == 6


# fa_fwd_host_noalloc(q_h, k_h, v_h, o_h, lse_h, sizes..., dtype, chunks, stream): the device
# staging area is the library's own, so only host pointers are passed.
def call_noalloc(lib, dtype=0, chunks=0, **over):
    a = dict(GOOD, qh=QH, kh=KH, vh=VH, oh=OH, lh=LH)
    a.update(over)
    return lib.fa_fwd_host_noalloc(a["qh"], a["kh"], a["vh"], a["oh"], a["lh"], a["B"], a["Hq"], a["Hkv"],
                                   a["Sq"], a["Sk"], a["D"], a["causal"], a["scale"], dtype, chunks, None)


@pytest.mark.parametrize("kw,code", [
    (dict(dtype=2), 15), (dict(chunks=-1), 15), (dict(chunks=65), 15),
    (dict(D=96), 4), (dict(Hq=3), 3), (dict(causal=3), 13), (dict(scale=math.nan), 7), (dict(Sk=0), 2),
    (dict(B=-1), 2), (dict(qh=None), 1), (dict(lh=None), 1),
    (dict(oh=QH + 64), 6), (dict(lh=OH + 4), 6), (dict(lh=KH), 6),
    # staging needs more than the 64 MiB area: q alone is 2 * 32 * 4096 * 128 * 2 B = 64 MiB
    (dict(B=2, Hq=32, Hkv=8, Sq=4096, Sk=4096, D=128), 16),
    # 16-bit q, k, v, o at 4 * 16 * 1024 * 64 * 2 B = 8 MiB each + lse fits; eight times the keys does not
    (dict(B=4, Hq=16, Hkv=16, Sq=1024, Sk=8192, D=64), 16),
    # a key count whose byte product would overflow 64 bits is still only "too large"
    (dict(B=1, Hq=1, Hkv=1, Sq=1, Sk=2**31 - 1, D=256), 16),
])
def test_noalloc_entry_point_rejects_before_any_cuda_call(lib, kw, code):
    assert call_noalloc(lib, **kw) == code


def test_noalloc_entry_point_empty_problems(lib):
    assert call_noalloc(lib, B=0, qh=None, kh=None, vh=None, oh=None, lh=None) == 0
    assert call_noalloc(lib, Sq=0) == 0


def test_noalloc_capacity_matches_the_header():
    from programming_flashattention_fwd_gb300 import binding
    text = open(HEADER).read()
    m = re.search(r"#define FA_HOST_NOALLOC_MAX_BYTES \((\d+)ull << (\d+)\)", text)
    assert m and int(m.group(1)) << int(m.group(2)) == binding.HOST_NOALLOC_MAX_BYTES


def test_noalloc_capacity_boundary(lib):
    """The 64 MiB staging area holds q, k, v, o and lse, each rounded up to 256 bytes.  D = 64,
    one head, Sq = 64: q and o take 8192 bytes each, lse 256, k and v 128 * Sk each.  Sk = 262078
    needs 67108608 bytes (fits), Sk = 262080 needs 67109120 (does not).  Both calls pass o_h
    overlapping q_h, so the one that fits stops at the overlap check, before any CUDA call."""
    over = dict(B=1, Hq=1, Hkv=1, Sq=64, D=64, causal=0, oh=QH + 64)
    assert 2 * 8192 + 256 + 2 * 128 * 262078 <= 64 << 20 < 2 * 8192 + 256 + 2 * 128 * 262080
    assert call_noalloc(lib, Sk=262078, **over) == 6
    assert call_noalloc(lib, Sk=262080, **over) == 16
