"""Pins for the oracle's building blocks (matrix product, bias + tanh-GELU epilogue, row
softmax), checked against things other than the oracle itself:

  - the product against numpy's float64 matmul of the decoded inputs (a library routine),
    and the closed forms A = I (C = B) and B = ones (row sums);
  - the epilogue against torch.nn.functional.gelu(approximate="tanh") in float64 (library),
    gelu(0) = 0, gelu(h) - gelu(-h) = h (tanh is odd), gelu(h) -> h for large h;
  - the row softmax against scipy.special.softmax, rows summing to 1, shift invariance, a
    constant row giving 1/cols, and finite results for inputs far beyond exp's range.

Planted mistakes 9 (B read as [N, K]), 10 (no max subtraction) and 11 (wrong cubic GELU
coefficient) must each fail at least one of these pins.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F
from scipy.special import softmax as sp_softmax

import oracle


def _rand(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def pin_gemm_matmul(orc):
    for (M, N, K) in ((1, 1, 1), (5, 7, 3), (17, 9, 33), (8, 24, 16)):
        for dtype in (torch.bfloat16, torch.float16):
            a, b = _rand((M, K), dtype, M + K), _rand((K, N), dtype, N + 7)
            c = orc.gemm_full(a, b, dtype == torch.float16)
            np.testing.assert_allclose(c, a.double().numpy() @ b.double().numpy(), rtol=0, atol=1e-12)


def pin_gemm_closed_forms(orc):
    K, N = 12, 10
    b = _rand((K, N), torch.bfloat16, 3)
    eye = torch.eye(K).to(torch.bfloat16)
    np.testing.assert_array_equal(orc.gemm_full(eye, b, False), b.double().numpy())
    a = _rand((6, K), torch.float16, 4)
    ones = torch.ones(K, N).to(torch.float16)
    np.testing.assert_allclose(orc.gemm_full(a, ones, True), np.repeat(a.double().numpy().sum(1, keepdims=True), N, 1),
                               rtol=0, atol=1e-12)


def pin_epilogue_library(orc):
    M, N, K = 9, 11, 16
    a, b = _rand((M, K), torch.bfloat16, 5), _rand((K, N), torch.bfloat16, 6)
    bias = _rand((N,), torch.float32, 7)
    h = a.double() @ b.double() + bias.double()
    np.testing.assert_allclose(orc.gemm_full(a, b, False, bias, 1), h.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(orc.gemm_full(a, b, False, bias, 2), F.gelu(h, approximate="tanh").numpy(),
                               rtol=0, atol=1e-12)


def pin_gelu_closed_forms(orc):
    assert orc.gelu_tanh(0.0) == 0.0
    for hv in (0.1, 0.7, 1.3, 2.9, 5.0):
        assert abs(orc.gelu_tanh(hv) - orc.gelu_tanh(-hv) - hv) < 1e-14
    assert abs(orc.gelu_tanh(30.0) - 30.0) < 1e-12 and abs(orc.gelu_tanh(-30.0)) < 1e-12
    # one value known in closed form: at h = 1 the tanh argument is sqrt(2/pi) * 1.044715
    z = math.sqrt(2.0 / math.pi) * 1.044715
    assert abs(orc.gelu_tanh(1.0) - 0.5 * (1.0 + math.tanh(z))) < 1e-15


def pin_softmax_library(orc):
    for (R, C) in ((1, 1), (3, 7), (5, 128), (2, 1000)):
        x = _rand((R, C), torch.float32, R * C, std=3.0)
        np.testing.assert_allclose(orc.softmax_rows(x), sp_softmax(x.double().numpy(), axis=1), rtol=0, atol=1e-15)
        xb = x.to(torch.bfloat16)
        np.testing.assert_allclose(orc.softmax_rows(xb), sp_softmax(xb.double().numpy(), axis=1), rtol=0, atol=1e-15)


def pin_softmax_invariants(orc):
    x = torch.round(_rand((4, 33), torch.float32, 11, std=2.0) * 8) / 8   # x + 5 is exact in fp32
    y = orc.softmax_rows(x)
    np.testing.assert_allclose(y.sum(1), 1.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(orc.softmax_rows(x + 5.0), y, rtol=0, atol=1e-14)
    np.testing.assert_allclose(orc.softmax_rows(np.full((2, 9), 3.25, np.float32)), 1.0 / 9.0, rtol=0, atol=1e-16)
    big = np.array([[1000.0, 999.0, -1000.0], [88.0, 89.0, 90.0]], dtype=np.float32)
    yb = orc.softmax_rows(big)
    assert np.all(np.isfinite(yb))
    np.testing.assert_allclose(yb[0, :2], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))], rtol=0, atol=1e-15)


OPS_PINS = [pin_gemm_matmul, pin_gemm_closed_forms, pin_epilogue_library, pin_gelu_closed_forms,
            pin_softmax_library, pin_softmax_invariants]


@pytest.mark.parametrize("pin", OPS_PINS, ids=[p.__name__ for p in OPS_PINS])
def test_pin(orc, pin):
    pin(orc)


OPS_PLANTS = {9: "B read as [N, K]", 10: "softmax without max subtraction", 11: "wrong GELU cubic coefficient"}


@pytest.mark.parametrize("plant", sorted(OPS_PLANTS), ids=[OPS_PLANTS[p] for p in sorted(OPS_PLANTS)])
def test_planted_mistakes_are_caught(plant):
    bad = oracle.load(plant)
    caught = []
    for pin in OPS_PINS:
        try:
            with np.errstate(all="ignore"):
                pin(bad)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, f"planted mistake '{OPS_PLANTS[plant]}' passed every pin"
