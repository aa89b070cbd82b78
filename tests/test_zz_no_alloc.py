"""GPU test of fa_fwd_host_noalloc, the host-memory forward for callers that cannot allocate
device memory (its staging area is a fixed device array inside the library).

Two calls in a row, on different inputs, shapes and types, go through the C ABI of the new
entry point; each result must be bit-identical to fa_fwd_host's -- the entry point with
caller-allocated device staging buffers -- since the same kernels run on the same values (the
parity tolerances, max |dO| <= 2e-2, mean |dO| <= 2e-3, max |dLSE| <= 1e-3, are checked as
well, so that a failure says how far off it is).  The second call reuses the staging area the
first call left filled, so a result that leaned on stale or zeroed staging would show there,
and so would staging slices that overlap.

The file name sorts last so that a run stopping at the first failure has run every other test
first; the test also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

from programming_flashattention_fwd_gb300 import build as fa_build
from programming_flashattention_fwd_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa_build.build()
    from programming_flashattention_fwd_gb300 import binding
    binding.load_library()
    return binding


def host_outputs(q):
    o = torch.full(q.shape, float("nan"), dtype=q.dtype).pin_memory()
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32).pin_memory()
    return o, lse


def with_caller_staging(fa, w, qh, kh, vh):
    """The existing host entry point, staged through device buffers this test allocates."""
    oh, lh = host_outputs(qh)
    qd, kd, vd = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (qh, kh, vh))
    od = torch.empty(qh.shape, dtype=qh.dtype, device="cuda")
    ld = torch.empty(qh.shape[:3], dtype=torch.float32, device="cuda")
    fa.fa_fwd_host(qh, kh, vh, oh, lh, qd, kd, vd, od, ld, w.causal, w.softmax_scale, chunks=3)
    torch.cuda.synchronize()
    return oh, lh


def noalloc_c_abi(fa, w, qh, kh, vh, stream):
    """fa_fwd_host_noalloc called straight through the C ABI (ctypes), no device buffer passed."""
    oh, lh = host_outputs(qh)
    st = fa.load_library().fa_fwd_host_noalloc(
        ctypes.c_void_p(qh.data_ptr()), ctypes.c_void_p(kh.data_ptr()), ctypes.c_void_p(vh.data_ptr()),
        ctypes.c_void_p(oh.data_ptr()), ctypes.c_void_p(lh.data_ptr()),
        w.B, w.Hq, w.Hkv, w.Sq, w.Sk, w.D, w.causal, ctypes.c_float(w.softmax_scale),
        int(w.is_fp16), 3, ctypes.c_void_p(stream.cuda_stream))
    assert st == 0, fa.fa_strerror(st)
    return oh, lh


def assert_close(o, lse, o_ref, l_ref):
    """Within the parity tolerances, then bit for bit (the header promises identical results)."""
    d = (o.double() - o_ref.double()).abs().numpy()
    assert np.isfinite(d).all(), "o has non-finite entries where the reference has none"
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS, (d.max(), d.mean())
    l, lr = lse.double().numpy(), l_ref.double().numpy()
    fin = np.isfinite(lr)
    assert np.array_equal(fin, np.isfinite(l))
    assert np.abs(l[fin] - lr[fin]).max(initial=0.0) <= LSE_ABS
    assert torch.equal(o, o_ref), "o differs from fa_fwd_host's in some bits"
    assert torch.equal(lse, l_ref), "lse differs from fa_fwd_host's in some bits"


def test_noalloc_matches_caller_staged_entry_point_on_two_calls_in_a_row(fa):
    first = Workload("noalloc_a", 2, 8, 2, 700, 700, 128, "bf16", 1, seed=9001)       # GQA, causal, ragged tail
    second = Workload("noalloc_b", 1, 6, 3, 333, 517, 64, "fp16", 2, seed=9002,      # bottom-right, fp16
                      q_std=2.0, k_std=2.0)
    inputs = []
    for w in (first, second):
        q, k, v = make_qkv(w)
        inputs.append((w, q.pin_memory(), k.pin_memory(), v.pin_memory()))
    refs = [with_caller_staging(fa, w, qh, kh, vh) for w, qh, kh, vh in inputs]

    s = torch.cuda.Stream()
    outs = [noalloc_c_abi(fa, w, qh, kh, vh, s) for w, qh, kh, vh in inputs]   # back to back, one stream
    s.synchronize()
    assert fa.fa_device_status() == (0, 0)
    for (o, lse), (o_ref, l_ref) in zip(outs, refs):
        assert_close(o, lse, o_ref, l_ref)


def test_noalloc_problem_filling_most_of_the_staging_area(fa):
    """q, k, v, o and lse of this problem take 62.75 MiB of the 64 MiB area, so the slices run
    up to its end; the result must still agree with the caller-staged entry point."""
    w = Workload("noalloc_big", 1, 32, 32, 2000, 2000, 128, "bf16", 1, seed=9003)
    need = 4 * (w.B * w.Hq * w.Sq * w.D * 2) + w.B * w.Hq * w.Sq * 4
    assert need <= fa.HOST_NOALLOC_MAX_BYTES and need > 0.95 * fa.HOST_NOALLOC_MAX_BYTES
    q, k, v = make_qkv(w)
    qh, kh, vh = q.pin_memory(), k.pin_memory(), v.pin_memory()
    o_ref, l_ref = with_caller_staging(fa, w, qh, kh, vh)
    s = torch.cuda.Stream()
    o, lse = noalloc_c_abi(fa, w, qh, kh, vh, s)
    s.synchronize()
    assert fa.fa_device_status() == (0, 0)
    assert_close(o, lse, o_ref, l_ref)
