"""GPU tests of the host-memory entry point fa_fwd_host: host (pinned or pageable) inputs and
outputs, copies overlapped with the kernels chunk by chunk.

Its results must be bit-identical to fa_fwd on the same inputs (every output row is computed
by the same kernel in the same order), whatever the chunk count, including chunks that cross
a batch boundary and chunk counts above B * Hkv; a few rows are also checked against the
float64 oracle with the parity tolerances.  The call must start after the work already on the
caller's stream and the caller's stream must wait for the last copy back.
"""
import numpy as np
import pytest
import torch

from programming_flashattention_fwd_gb300 import build as fa_build
from programming_flashattention_fwd_gb300.inputs import Workload, make_qkv, sample_rows

pytestmark = pytest.mark.gpu

MAX_ABS, LSE_ABS = 2e-2, 1e-3


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa_build.build()
    from programming_flashattention_fwd_gb300 import binding
    binding.load_library()
    return binding


def host_buffers(q, k, v, pinned):
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t.clone())
    qh, kh, vh = pin(q), pin(k), pin(v)
    oh = pin(torch.full(q.shape, float("nan"), dtype=q.dtype))
    lh = pin(torch.full(q.shape[:3], float("nan"), dtype=torch.float32))
    return qh, kh, vh, oh, lh


def device_buffers(q, k, v):
    qd, kd, vd = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (q, k, v))
    od = torch.empty(q.shape, dtype=q.dtype, device="cuda")
    ld = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    return qd, kd, vd, od, ld


def reference_device_run(fa, w, q, k, v):
    o = torch.empty(q.shape, dtype=q.dtype, device="cuda")
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    fn = fa.fa_fwd_fp16 if w.is_fp16 else fa.fa_fwd
    fn(q.cuda(), k.cuda(), v.cuda(), o, lse, w.causal, w.softmax_scale)
    torch.cuda.synchronize()
    return o.cpu(), lse.cpu()


CASES = [
    # name, B, Hq, Hkv, Sq, Sk, D, dtype, causal, chunks
    ("cross_batch", 3, 8, 2, 300, 300, 128, "bf16", 1, 4),     # runs [1,3) and [4,6) span two batches
    ("fp16_bottom_right", 2, 4, 4, 129, 257, 64, "fp16", 2, 3),
    ("prefill_gqa", 1, 16, 8, 1000, 4096, 128, "bf16", 2, 0),
    ("d256", 2, 8, 1, 513, 513, 256, "bf16", 0, 5),             # capped at B * Hkv = 2
    ("one_chunk", 1, 4, 2, 64, 64, 128, "bf16", 1, 1),
    ("chunks_above_groups", 1, 4, 2, 64, 64, 128, "bf16", 1, 64),
    ("one_head_per_chunk", 2, 6, 3, 200, 333, 64, "fp16", 0, 6),
    ("auto_cross", 3, 8, 4, 160, 200, 64, "bf16", 1, 0),   # automatic: 4 runs of 3 KV heads, one crossing a batch
]


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_host_entry_matches_device_entry(fa, orc, case, pinned):
    name, B, Hq, Hkv, Sq, Sk, D, dtype, causal, chunks = case
    w = Workload(name, B, Hq, Hkv, Sq, Sk, D, dtype, causal, seed=4242 + B * Sq + D)
    q, k, v = make_qkv(w)
    hb = host_buffers(q, k, v, pinned)
    db = device_buffers(q, k, v)
    s = torch.cuda.Stream()
    fa.fa_fwd_host(*hb, *db, w.causal, w.softmax_scale, chunks=chunks, stream=s)
    s.synchronize()
    assert fa.fa_device_status() == (0, 0)
    o_ref, l_ref = reference_device_run(fa, w, q, k, v)
    assert torch.equal(hb[3], o_ref), "o differs from fa_fwd"
    assert torch.equal(hb[4], l_ref), "lse differs from fa_fwd"
    # a handful of rows against the float64 oracle as well
    rows = sample_rows(w, n=24)
    o_o, l_o = orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
    o_g = hb[3][rows[:, 0], rows[:, 1], rows[:, 2]].double().numpy()
    l_g = hb[4][rows[:, 0], rows[:, 1], rows[:, 2]].double().numpy()
    assert np.abs(o_g - o_o).max() <= MAX_ABS
    fin = np.isfinite(l_o)
    assert np.array_equal(fin, np.isfinite(l_g))
    assert np.abs(l_g[fin] - l_o[fin]).max(initial=0.0) <= LSE_ABS


def test_host_entry_orders_after_and_before_the_callers_stream(fa):
    """Work already on the stream (a long sleep, then a NaN fill of the device output buffer)
    runs before the pipeline; syncing only the caller's stream is enough to read the results."""
    w = Workload("order", 2, 16, 4, 2048, 2048, 128, "bf16", 1, seed=77)
    q, k, v = make_qkv(w)
    hb = host_buffers(q, k, v, True)
    db = device_buffers(q, k, v)
    o_ref, l_ref = reference_device_run(fa, w, q, k, v)
    s = torch.cuda.Stream()
    for _ in range(3):
        hb[3].fill_(float("nan"))
        with torch.cuda.stream(s):
            torch.cuda._sleep(20_000_000)
            db[3].fill_(float("nan"))
            db[4].fill_(float("nan"))
        fa.fa_fwd_host(*hb, *db, w.causal, w.softmax_scale, chunks=4, stream=s)
        s.synchronize()
        assert torch.equal(hb[3], o_ref) and torch.equal(hb[4], l_ref)
    assert fa.fa_device_status() == (0, 0)


def test_host_entry_back_to_back_calls_reuse_buffers(fa):
    """Two calls in a row on one stream with the same staging buffers and different inputs:
    the second call's copies must not overwrite the first call's inputs while it still runs."""
    w1 = Workload("a", 1, 8, 2, 1024, 1024, 128, "bf16", 0, seed=5)
    w2 = w1.with_(seed=6)
    (q1, k1, v1), (q2, k2, v2) = make_qkv(w1), make_qkv(w2)
    h1, h2 = host_buffers(q1, k1, v1, True), host_buffers(q2, k2, v2, True)
    db = device_buffers(q1, k1, v1)
    s = torch.cuda.Stream()
    fa.fa_fwd_host(*h1, *db, 0, w1.softmax_scale, chunks=2, stream=s)
    fa.fa_fwd_host(*h2, *db, 0, w2.softmax_scale, chunks=2, stream=s)
    s.synchronize()
    for h, (q, k, v), w in ((h1, (q1, k1, v1), w1), (h2, (q2, k2, v2), w2)):
        o_ref, l_ref = reference_device_run(fa, w, q, k, v)
        assert torch.equal(h[3], o_ref) and torch.equal(h[4], l_ref)


def test_host_entry_binding_rejects_bad_tensors(fa):
    w = Workload("x", 1, 2, 1, 16, 16, 64, "bf16", 0, seed=1)
    q, k, v = make_qkv(w)
    hb = host_buffers(q, k, v, True)
    db = device_buffers(q, k, v)
    with pytest.raises(ValueError):
        fa.fa_fwd_host(db[0], *hb[1:], *db, 0, 0.125)               # a device tensor as host input
    with pytest.raises(ValueError):
        fa.fa_fwd_host(*hb[:3], hb[3][:, :1].contiguous(), hb[4], *db, 0, 0.125)   # wrong shape
    with pytest.raises(fa.FaError):
        fa.fa_fwd_host(*hb, *db, 0, 0.125, chunks=100)


def test_host_entry_two_calls_in_flight(fa):
    """Calls on two caller streams, each with its own staging buffers and host outputs, enqueued
    alternately without synchronising in between (the benchmark's end-to-end pattern): the
    shared internal streams and events must keep every call's copies and kernels ordered."""
    w = Workload("inflight", 2, 8, 2, 700, 900, 128, "bf16", 2, seed=31)
    q, k, v = make_qkv(w)
    o_ref, l_ref = reference_device_run(fa, w, q, k, v)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    hbs = [host_buffers(q, k, v, True) for _ in range(2)]
    dbs = [device_buffers(q, k, v) for _ in range(2)]
    for i in range(6):
        fa.fa_fwd_host(*hbs[i % 2], *dbs[i % 2], w.causal, w.softmax_scale, chunks=3, stream=streams[i % 2])
    torch.cuda.synchronize()
    assert fa.fa_device_status() == (0, 0)
    for hb in hbs:
        assert torch.equal(hb[3], o_ref) and torch.equal(hb[4], l_ref)
