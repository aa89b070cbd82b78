"""Pins for the float64 oracle, checked against things other than itself.

Each pin is a function of an oracle handle that raises AssertionError on a mismatch.  They
run against the real oracle, and ``test_planted_mistakes_are_caught`` runs them against
copies of the oracle built with one deliberate mistake each (wrong GQA head, causal bound
off by one, transposed key operand, dropped scale, reversed value rows, wrong normaliser,
stray log-sum-exp term) to show that every such mistake fails at least one pin.

What pins what:
  - torch's scaled_dot_product_attention in float64 on CPU (an independent library
    routine the oracle never calls) for O, including GQA (enable_gqa), top-left causal
    (is_causal) and bottom-right causal (an explicit lower-right boolean mask), on shapes
    with Sq != Sk, odd D and tiny heads; rows left without keys are checked to be 0 / -inf;
  - torch.logsumexp over the masked score matrix for the log-sum-exp;
  - numpy's and torch's own bf16/fp16 decoders for every 16-bit pattern;
  - closed forms: scale = 0 (uniform weights), all keys equal, one key, two keys
    (softmax of two logits is the logistic function, scipy.special.expit);
  - invariants: identical value rows, permutation of key/value rows (non-causal),
    causal rows independent of future keys, saturation under huge logits.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::UserWarning")


def _rand_bits(shape, dtype, rng_seed, std=1.0):
    g = torch.Generator().manual_seed(rng_seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def _rows_all(B, H, S):
    return oracle.all_rows(B, H, S)


SHAPES = [
    # B, Hq, Hkv, Sq, Sk, D
    (1, 1, 1, 1, 1, 1),
    (2, 4, 2, 5, 5, 3),
    (1, 4, 1, 7, 3, 8),
    (1, 6, 3, 3, 9, 16),
    (2, 2, 2, 17, 17, 4),
    (1, 8, 2, 9, 12, 5),
]


def _allowed(Sq, Sk, causal):
    """Boolean [Sq, Sk] mask of allowed keys (built from torch.tril, not from the oracle)."""
    ones = torch.ones(Sq, Sk, dtype=torch.bool)
    if causal == 0:
        return ones
    return ones.tril(0 if causal == 1 else Sk - Sq)


def pin_sdpa(orc):
    """O against torch SDPA (float64, CPU), LSE against torch.logsumexp, for no mask,
    top-left causal (SDPA's own is_causal) and bottom-right causal (explicit mask)."""
    seed = 10
    for (B, Hq, Hkv, Sq, Sk, D) in SHAPES:
        for dtype in (torch.bfloat16, torch.float16):
            for causal in (0, 1, 2):
                seed += 1
                q = _rand_bits((B, Hq, Sq, D), dtype, seed)
                k = _rand_bits((B, Hkv, Sk, D), dtype, seed + 1000)
                v = _rand_bits((B, Hkv, Sk, D), dtype, seed + 2000)
                scale = 0.37 if D > 1 else 1.3
                o, lse = orc.full(q, k, v, dtype == torch.float16, causal, scale)
                qd, kd, vd = q.double(), k.double(), v.double()
                mask = _allowed(Sq, Sk, causal)
                if causal == 2:
                    ref = F.scaled_dot_product_attention(qd, kd, vd, attn_mask=mask,
                                                         scale=scale, enable_gqa=True)
                else:
                    ref = F.scaled_dot_product_attention(qd, kd, vd, is_causal=causal == 1,
                                                         scale=scale, enable_gqa=True)
                live = mask.any(dim=1).numpy()            # rows with at least one key
                np.testing.assert_allclose(o[:, :, live], ref.numpy()[:, :, live], rtol=0, atol=1e-12)
                assert np.all(o[:, :, ~live] == 0.0)      # empty softmax: o = 0
                kx = kd.repeat_interleave(Hq // Hkv, dim=1)
                s = scale * torch.einsum("bhid,bhjd->bhij", qd, kx)
                s = s.masked_fill(~mask, float("-inf"))
                np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(),
                                           rtol=0, atol=1e-12)


def pin_decoders(orc):
    """Every bf16 / fp16 bit pattern decodes to numpy's / torch's value."""
    bits = np.arange(65536, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    bf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    for x in range(0, 65536, 7):   # a stride coprime to the field widths covers all classes
        got = orc.decode(x, True)
        assert (math.isnan(got) and math.isnan(f16[x])) or got == f16[x], (x, got, f16[x])
        got = orc.decode(x, False)
        assert (math.isnan(got) and math.isnan(bf[x])) or got == bf[x], (x, got, bf[x])
    for x in (0x0000, 0x0001, 0x03FF, 0x0400, 0x3C00, 0x7BFF, 0x7C00, 0x8001, 0xFBFF, 0xFC00):
        assert orc.decode(x, True) == f16[x]


def pin_identical_value_rows(orc):
    """All value rows equal -> every output row equals that value row."""
    B, Hq, Hkv, S, D = 1, 4, 2, 11, 6
    q = _rand_bits((B, Hq, S, D), torch.bfloat16, 1)
    k = _rand_bits((B, Hkv, S, D), torch.bfloat16, 2)
    row = _rand_bits((1, Hkv, 1, D), torch.bfloat16, 3)
    v = row.expand(B, Hkv, S, D).contiguous()
    for causal in (False, True):
        o, _ = orc.full(q, k, v, False, causal, 0.5)
        want = row.double().repeat_interleave(Hq // Hkv, dim=1).expand(B, Hq, S, D)
        np.testing.assert_allclose(o, want.numpy(), rtol=0, atol=1e-14)


def pin_single_key(orc):
    """Sk = 1 -> o = v_0 and lse = scale * q . k_0 for every row."""
    B, Hq, Hkv, Sq, D = 2, 3, 1, 4, 5
    q = _rand_bits((B, Hq, Sq, D), torch.float16, 4)
    k = _rand_bits((B, Hkv, 1, D), torch.float16, 5)
    v = _rand_bits((B, Hkv, 1, D), torch.float16, 6)
    o, lse = orc.full(q, k, v, True, False, 0.25)
    qd, kd, vd = q.double().numpy(), k.double().numpy(), v.double().numpy()
    for b in range(B):
        for h in range(Hq):
            for i in range(Sq):
                np.testing.assert_allclose(o[b, h, i], vd[b, 0, 0], rtol=0, atol=1e-14)
                want = 0.25 * float(np.dot(qd[b, h, i], kd[b, 0, 0]))
                assert abs(lse[b, h, i] - want) < 1e-12


def pin_permutation(orc):
    """Non-causal: permuting key and value rows together changes nothing."""
    B, Hq, Hkv, Sq, Sk, D = 1, 2, 2, 6, 13, 7
    q = _rand_bits((B, Hq, Sq, D), torch.bfloat16, 7)
    k = _rand_bits((B, Hkv, Sk, D), torch.bfloat16, 8)
    v = _rand_bits((B, Hkv, Sk, D), torch.bfloat16, 9)
    perm = torch.randperm(Sk, generator=torch.Generator().manual_seed(3))
    o1, l1 = orc.full(q, k, v, False, False, 0.4)
    o2, l2 = orc.full(q, k[:, :, perm].contiguous(), v[:, :, perm].contiguous(), False, False, 0.4)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def pin_causal_future(orc):
    """Causal: row i does not move when keys/values j > i change, and does move when a
    key j <= i changes."""
    B, H, S, D = 1, 2, 9, 4
    q = _rand_bits((B, H, S, D), torch.bfloat16, 10)
    k = _rand_bits((B, H, S, D), torch.bfloat16, 11)
    v = _rand_bits((B, H, S, D), torch.bfloat16, 12)
    o1, l1 = orc.full(q, k, v, False, True, 0.6)
    for i in range(S):
        k2, v2 = k.clone(), v.clone()
        k2[:, :, i + 1:] = _rand_bits(k2[:, :, i + 1:].shape, torch.bfloat16, 100 + i)
        v2[:, :, i + 1:] = _rand_bits(v2[:, :, i + 1:].shape, torch.bfloat16, 200 + i)
        o2, l2 = orc.full(q, k2, v2, False, True, 0.6)
        np.testing.assert_array_equal(o1[:, :, i], o2[:, :, i])
        np.testing.assert_array_equal(l1[:, :, i], l2[:, :, i])
        k3 = k.clone()
        k3[:, :, i] += 1.0
        _, l3 = orc.full(q, k3, v, False, True, 0.6)
        assert np.all(l3[:, :, i] != l1[:, :, i])


def pin_scale_zero(orc):
    """scale = 0 -> uniform weights: o_i = mean of the allowed v_j, lse_i = ln |J_i|, where
    |J_i| = Sk, min(i+1, Sk) (top-left) or clamp(i+1+Sk-Sq, 0, Sk) (bottom-right)."""
    B, Hq, Hkv, D = 1, 4, 2, 3
    for (Sq, Sk) in ((10, 7), (4, 9)):
        q = _rand_bits((B, Hq, Sq, D), torch.float16, 13)
        k = _rand_bits((B, Hkv, Sk, D), torch.float16, 14)
        v = _rand_bits((B, Hkv, Sk, D), torch.float16, 15)
        vd = v.double().numpy()
        for causal in (0, 1, 2):
            o, lse = orc.full(q, k, v, True, causal, 0.0)
            for h in range(Hq):
                for i in range(Sq):
                    n = (Sk, min(i + 1, Sk), max(0, min(i + 1 + Sk - Sq, Sk)))[causal]
                    if n == 0:
                        assert np.all(o[0, h, i] == 0.0) and lse[0, h, i] == -math.inf
                        continue
                    np.testing.assert_allclose(o[0, h, i], vd[0, h // 2, :n].mean(axis=0), rtol=0, atol=1e-14)
                    assert abs(lse[0, h, i] - math.log(n)) < 1e-14


def pin_equal_keys(orc):
    """All key rows equal -> o_i = mean of allowed v_j, lse_i = scale*q_i.k + ln |J_i|."""
    B, H, Sq, Sk, D = 1, 2, 8, 8, 5
    q = _rand_bits((B, H, Sq, D), torch.bfloat16, 16)
    krow = _rand_bits((B, H, 1, D), torch.bfloat16, 17)
    k = krow.expand(B, H, Sk, D).contiguous()
    v = _rand_bits((B, H, Sk, D), torch.bfloat16, 18)
    qd, kd, vd = q.double().numpy(), krow.double().numpy(), v.double().numpy()
    for causal in (False, True):
        o, lse = orc.full(q, k, v, False, causal, 0.8)
        for h in range(H):
            for i in range(Sq):
                n = i + 1 if causal else Sk
                np.testing.assert_allclose(o[0, h, i], vd[0, h, :n].mean(axis=0), rtol=0, atol=1e-13)
                want = 0.8 * float(np.dot(qd[0, h, i], kd[0, h, 0])) + math.log(n)
                assert abs(lse[0, h, i] - want) < 1e-12


def pin_two_keys_logistic(orc):
    """Two keys: the weight of key 1 is the logistic function of s1 - s0."""
    from scipy.special import expit, logsumexp
    B, H, Sq, Sk, D = 1, 1, 5, 2, 4
    q = _rand_bits((B, H, Sq, D), torch.float16, 19)
    k = _rand_bits((B, H, Sk, D), torch.float16, 20)
    v = _rand_bits((B, H, Sk, D), torch.float16, 21)
    o, lse = orc.full(q, k, v, True, False, 0.9)
    qd, kd, vd = q.double().numpy()[0, 0], k.double().numpy()[0, 0], v.double().numpy()[0, 0]
    for i in range(Sq):
        s = 0.9 * (kd @ qd[i])
        w1 = expit(s[1] - s[0])
        np.testing.assert_allclose(o[0, 0, i], vd[0] + w1 * (vd[1] - vd[0]), rtol=0, atol=1e-13)
        assert abs(lse[0, 0, i] - logsumexp(s)) < 1e-13


def pin_bottom_right_future(orc):
    """Bottom-right causal: row i does not move when keys/values j > i + Sk - Sq change."""
    B, H, Sq, Sk, D = 1, 2, 5, 9, 4
    q = _rand_bits((B, H, Sq, D), torch.bfloat16, 30)
    k = _rand_bits((B, H, Sk, D), torch.bfloat16, 31)
    v = _rand_bits((B, H, Sk, D), torch.bfloat16, 32)
    o1, l1 = orc.full(q, k, v, False, 2, 0.6)
    for i in range(Sq):
        last = i + Sk - Sq
        k2, v2 = k.clone(), v.clone()
        k2[:, :, last + 1:] = _rand_bits(k2[:, :, last + 1:].shape, torch.bfloat16, 300 + i)
        v2[:, :, last + 1:] = _rand_bits(v2[:, :, last + 1:].shape, torch.bfloat16, 400 + i)
        o2, l2 = orc.full(q, k2, v2, False, 2, 0.6)
        np.testing.assert_array_equal(o1[:, :, i], o2[:, :, i])
        np.testing.assert_array_equal(l1[:, :, i], l2[:, :, i])


def pin_huge_logits(orc):
    """Logits far beyond exp's range stay finite: the largest one takes all the weight."""
    B, H, S, D = 1, 1, 4, 8
    q = torch.full((B, H, 1, D), 200.0).to(torch.float16)
    kv = torch.tensor([1.0, -1.0, 2.0, 0.5]).view(1, 1, S, 1).expand(B, H, S, D)
    k = (kv * 100.0).to(torch.float16).contiguous()
    v = torch.arange(S * D, dtype=torch.float32).view(1, 1, S, D).to(torch.float16)
    o, lse = orc.full(q, k, v, True, False, 1.0)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(o[0, 0, 0], v.double().numpy()[0, 0, 2], rtol=0, atol=1e-12)
    assert abs(lse[0, 0, 0] - 200.0 * 200.0 * D) < 1e-6


PINS = [pin_sdpa, pin_decoders, pin_identical_value_rows, pin_single_key, pin_permutation,
        pin_causal_future, pin_bottom_right_future, pin_scale_zero, pin_equal_keys,
        pin_two_keys_logistic, pin_huge_logits]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(orc, pin):
    pin(orc)


PLANTS = {1: "wrong GQA head mapping", 2: "causal bound off by one",
          3: "transposed key operand", 4: "scale dropped", 5: "reversed value rows",
          6: "normalised by key count", 7: "stray log-sum-exp term",
          8: "bottom-right offset with the wrong sign"}


@pytest.mark.parametrize("plant", sorted(PLANTS), ids=[PLANTS[p] for p in sorted(PLANTS)])
def test_planted_mistakes_are_caught(plant):
    bad = oracle.load(plant)
    caught = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{PLANTS[plant]}' passed every pin"


def test_oracle_rejects_bad_rows(orc):
    q = _rand_bits((1, 2, 3, 4), torch.bfloat16, 1)
    k = _rand_bits((1, 2, 3, 4), torch.bfloat16, 2)
    with pytest.raises(ValueError):
        orc.rows(q, k, k, False, False, 1.0, np.array([[0, 2, 0]]))
    with pytest.raises(ValueError):
        orc.rows(q, k, k, False, False, 1.0, np.array([[0, 0, 3]]))


def test_rows_match_full(orc):
    """Sampled-row evaluation equals the same rows of the full evaluation (bit for bit)."""
    from programming_flashattention_fwd_gb300.inputs import WORKLOADS, make_qkv, sample_rows
    w = WORKLOADS["mha_b1_h2_s128_d64"]
    q, k, v = make_qkv(w)
    o, lse = orc.full(q, k, v, w.is_fp16, w.causal, w.softmax_scale)
    rows = sample_rows(w, n=40)
    o2, l2 = orc.rows(q, k, v, w.is_fp16, w.causal, w.softmax_scale, rows)
    np.testing.assert_array_equal(o2, o[rows[:, 0], rows[:, 1], rows[:, 2]])
    np.testing.assert_array_equal(l2, lse[rows[:, 0], rows[:, 1], rows[:, 2]])
