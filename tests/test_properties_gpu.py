"""GPU checks at the benchmark workloads' full sizes through properties of attention that hold
at any size, so they need no oracle and cover every output row (the parity tests compare
sampled rows with the float64 oracle at these sizes).

  - causal: row i depends only on keys <= i.  Perturbing every key and value row from a
    cut-off c on leaves rows < c bit-identical (O and LSE), for a cut-off on a tile boundary
    and one inside a tile, on both attention kernels;
  - identical value rows: if every value row of a KV head is the same vector v, every output
    row of its query heads is v up to the 16-bit rounding of P and of O, and LSE (which does not
    depend on V) is unchanged bit for bit;
  - grouped-query heads with equal query rows produce equal outputs, bit for bit;
  - without a mask, permuting the key/value rows of a head together leaves the output
    unchanged up to rounding order (parity tolerances: 2e-2 max, 2e-3 mean on O, 1e-3 on LSE).
"""
import pytest
import torch

from programming_flashattention_fwd_gb300 import build as fa_build
from programming_flashattention_fwd_gb300.inputs import EXTRA_WORKLOADS, WORKLOADS, make_qkv

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = 2e-2, 2e-3, 1e-3
ALL = {**WORKLOADS, **EXTRA_WORKLOADS}


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa_build.build()
    from programming_flashattention_fwd_gb300 import binding
    binding.load_library()
    return binding


def forward(fa, w, q, k, v):
    o = torch.full(q.shape, float("nan"), dtype=q.dtype, device="cuda")
    lse = torch.full(q.shape[:3], float("nan"), dtype=torch.float32, device="cuda")
    fn = fa.fa_fwd_fp16 if w.is_fp16 else fa.fa_fwd
    fn(q, k, v, o, lse, w.causal, w.softmax_scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == (0, 0)
    assert not torch.isnan(o).any() and not torch.isnan(lse).any(), "an output row was not written"
    return o, lse


def inputs(w):
    return tuple(t.cuda() for t in make_qkv(w))


@pytest.mark.parametrize("name,cuts", [
    ("gqa_causal_b2_h32kv8_s4096", (2048, 1000)),
    ("mha_causal_b4_h16_s1024_d64", (512, 300)),
    ("gqa_causal_b2_h32kv8_s4096_d256", (1024, 2500)),
])
def test_causal_rows_ignore_later_keys(fa, name, cuts):
    w = ALL[name]
    assert w.causal == 1 and w.Sq == w.Sk
    q, k, v = inputs(w)
    o, lse = forward(fa, w, q, k, v)
    g = torch.Generator(device="cuda").manual_seed(4321)
    for c in cuts:
        k2, v2 = k.clone(), v.clone()
        k2[:, :, c:] = (3 * torch.randn(k2[:, :, c:].shape, device="cuda", generator=g)).to(k.dtype)
        v2[:, :, c:] = (3 * torch.randn(v2[:, :, c:].shape, device="cuda", generator=g)).to(v.dtype)
        o2, lse2 = forward(fa, w, q, k2, v2)
        assert torch.equal(o2[:, :, :c], o[:, :, :c]), f"cut {c}: a row before the cut changed"
        assert torch.equal(lse2[:, :, :c], lse[:, :, :c]), f"cut {c}: an lse before the cut changed"
        # and the rows from the cut on do see the new keys
        assert not torch.equal(o2[:, :, c:], o[:, :, c:])


@pytest.mark.parametrize("name", ["gqa_causal_b2_h32kv8_s4096", "mha_fp16_b8_h16_s2000_std2"])
def test_identical_value_rows_give_that_row(fa, name):
    w = ALL[name]
    q, k, v = inputs(w)
    _, lse = forward(fa, w, q, k, v)
    v1 = v[:, :, :1].expand_as(v).contiguous()          # every value row of a KV head = its row 0
    o1, lse1 = forward(fa, w, q, k, v1)
    assert torch.equal(lse1, lse), "lse must not depend on the values"
    group = w.Hq // w.Hkv
    want = v[:, :, 0].repeat_interleave(group, dim=1).unsqueeze(2).float()   # [B, Hq, 1, D]
    err = (o1.float() - want).abs()
    # P is rounded to 16 bits before the product and O on the way out: a relative error
    # of at most 2^-8 on each element, plus a small absolute floor for values near zero
    bound = want.abs() * 2.0 ** -7 + 1e-6
    assert bool((err <= bound).all()), f"max excess {(err - bound).max().item():.3e}"


def test_gqa_heads_with_equal_queries_match(fa):
    w = ALL["gqa_causal_b2_h32kv8_s4096"]
    q, k, v = inputs(w)
    group = w.Hq // w.Hkv
    q1 = q.view(w.B, w.Hkv, group, w.Sq, w.D)[:, :, :1].expand(-1, -1, group, -1, -1).reshape(q.shape).contiguous()
    o, lse = forward(fa, w, q1, k, v)
    ov = o.view(w.B, w.Hkv, group, w.Sq, w.D)
    lv = lse.view(w.B, w.Hkv, group, w.Sq)
    for h in range(1, group):
        assert torch.equal(ov[:, :, h], ov[:, :, 0]) and torch.equal(lv[:, :, h], lv[:, :, 0]), f"head {h} of a group"


@pytest.mark.parametrize("name", ["mha_fp16_b8_h16_s2000_std2", "mha_b4_h16_s2048_d256"])
def test_key_value_permutation_without_mask(fa, name):
    w = ALL[name]
    assert w.causal == 0
    q, k, v = inputs(w)
    o, lse = forward(fa, w, q, k, v)
    g = torch.Generator(device="cuda").manual_seed(99)
    perm = torch.randperm(w.Sk, device="cuda", generator=g)
    o2, lse2 = forward(fa, w, q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous())
    d = (o2.float() - o.float()).abs()
    assert d.max().item() <= MAX_ABS and d.mean().item() <= MEAN_ABS, (d.max().item(), d.mean().item())
    assert (lse2 - lse).abs().max().item() <= LSE_ABS
