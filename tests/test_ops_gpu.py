"""GPU parity of the standalone building blocks (through the C ABI) against the float64 oracle.

Tolerances, derived from the arithmetic:
  - matrix product (fp32 accumulation of exact 16-bit products): per entry
        |C - C_ref| <= 2^-14 * sum_k |A[m,k] B[k,n]|  +  out_rounding * |C_ref|
    with out_rounding = 2^-8 for a 16-bit output (half an ulp of bf16 is 2^-9; fp16 is finer)
    and 2^-22 for an fp32 output; with tanh-GELU the accumulation term is scaled by the
    largest slope of gelu (1.13) and the hardware tanh (error below 2^-10.9) adds
    0.5 * |h| * 2^-10 for the pre-activation h = A B + bias;
  - row softmax (exp2 approximation, relative error ~2^-22, fp32 sums): |y - y_ref| <=
    1e-5 * y_ref + 1e-7 for fp32 output, 2^-8 * y_ref + 1e-7 for bf16 output.
"""
import numpy as np
import pytest
import torch

import oracle
from programming_flashattention_fwd_gb300 import build as fa_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    fa_build.build()
    from programming_flashattention_fwd_gb300 import binding
    binding.load_library()
    return binding


def _rand(shape, dtype, seed, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * std).to(dtype)


def check_gemm(c_gpu, ref, abs_sum, out_fp32, epilogue, what, h_ref=None):
    c = c_gpu.double().cpu().numpy() if isinstance(c_gpu, torch.Tensor) else c_gpu
    assert np.all(np.isfinite(c)), what
    rel = 2.0 ** -22 if out_fp32 else 2.0 ** -8
    tol = 2.0 ** -14 * abs_sum + rel * np.abs(ref)
    if epilogue == 2:
        tol = 1.13 * 2.0 ** -14 * abs_sum + rel * np.abs(ref) + 0.5 * np.abs(h_ref) * 2.0 ** -10
    err = np.abs(c - ref)
    bad = err > tol + 1e-6
    assert not bad.any(), f"{what}: {bad.sum()} entries out of tolerance, worst excess {(err - tol).max():.3e}"


CASES = [(1, 8, 8), (128, 256, 64), (200, 264, 72), (129, 520, 200), (300, 136, 1024), (77, 1024, 16)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("out_fp32", [False, True])
@pytest.mark.parametrize("epilogue", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", CASES)
def test_gemm_small(fa, orc, dtype, out_fp32, epilogue, M, N, K):
    td = torch.bfloat16 if dtype == "bf16" else torch.float16
    a, b = _rand((M, K), td, M * 7 + K), _rand((K, N), td, N * 3 + K)
    bias = _rand((N,), torch.float32, N + 1)
    c = fa.gemm(a.cuda(), b.cuda(), bias.cuda() if epilogue else None, epilogue, out_fp32)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == (0, 0)
    ref = orc.gemm_full(a, b, dtype == "fp16", bias if epilogue else None, epilogue)
    h_ref = orc.gemm_full(a, b, dtype == "fp16", bias, 1) if epilogue == 2 else None
    abs_sum = np.abs(a.double().numpy()) @ np.abs(b.double().numpy())
    check_gemm(c, ref, abs_sum, out_fp32, epilogue, f"{dtype} out_fp32={out_fp32} epi={epilogue} {M}x{N}x{K}", h_ref)


@pytest.mark.parametrize("epilogue", [0, 2])
def test_gemm_large_sampled(fa, orc, epilogue):
    """4096 x 4096 x 4096 bf16, checked on 600 seeded entries plus tile corners."""
    M = N = K = 4096
    a, b = _rand((M, K), torch.bfloat16, 1), _rand((K, N), torch.bfloat16, 2)
    bias = _rand((N,), torch.float32, 3)
    c = fa.gemm(a.cuda(), b.cuda(), bias.cuda(), epilogue).cpu()
    rng = np.random.default_rng(4)
    ent = [tuple(x) for x in np.stack([rng.integers(0, M, 600), rng.integers(0, N, 600)], 1)]
    ent += [(m, n) for m in (0, 127, 128, M - 1) for n in (0, 255, 256, N - 1)]
    ent = np.asarray(sorted(set(ent)), dtype=np.int64)
    ref = orc.gemm_entries(a, b, False, ent, bias, epilogue)
    h_ref = orc.gemm_entries(a, b, False, ent, bias, 1)
    ad, bd = np.abs(a.double().numpy()), np.abs(b.double().numpy())
    abs_sum = np.einsum("ek,ke->e", ad[ent[:, 0]], bd[:, ent[:, 1]])
    check_gemm(c.double().numpy()[ent[:, 0], ent[:, 1]], ref, abs_sum, False, epilogue, f"4096^3 epi={epilogue}", h_ref)


def check_softmax(y_gpu, ref, bf16, what):
    y = y_gpu.double().cpu().numpy()
    tol = (2.0 ** -8 if bf16 else 1e-5) * ref + 1e-7
    err = np.abs(y - ref)
    assert np.all(np.isfinite(y)), what
    assert (err <= tol).all(), f"{what}: worst excess {(err - tol).max():.3e}"


# every path: register groups of 32 .. 256 threads with 1 .. 8 vectors, the shared-memory path
# with two and one row buffers, the vectorised and scalar two-pass paths, ragged widths
SOFTMAX_SHAPES = [(1, 1), (3, 7), (7, 8), (1000, 33), (33, 256), (5, 129), (64, 1000), (9, 1024), (6, 2048),
                  (10, 4096), (3, 8200), (2, 16384), (2, 20000), (3, 32768), (2, 50000), (2, 60000), (4, 65544),
                  (1, 262144), (2, 70001)]


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("rows,cols", SOFTMAX_SHAPES)
def test_softmax_rows(fa, orc, bf16, rows, cols):
    x = _rand((rows, cols), torch.bfloat16 if bf16 else torch.float32, rows * 131 + cols, std=4.0)
    y = fa.softmax_rows(x.cuda())
    torch.cuda.synchronize()
    check_softmax(y, orc.softmax_rows(x), bf16, f"{rows}x{cols} bf16={bf16}")


def test_softmax_in_place_and_unaligned_width(fa, orc):
    for bf16 in (False, True):
        x = _rand((37, 1001), torch.bfloat16 if bf16 else torch.float32, 5, std=3.0)
        xd = x.cuda()
        fa.softmax_rows(xd, xd)
        torch.cuda.synchronize()
        check_softmax(xd, orc.softmax_rows(x), bf16, f"in place bf16={bf16}")


def test_softmax_large_sampled(fa, orc):
    rows, cols = 65536, 4096
    x = _rand((rows, cols), torch.float32, 9, std=4.0)
    y = fa.softmax_rows(x.cuda()).cpu()
    ids = np.unique(np.concatenate([np.random.default_rng(1).integers(0, rows, 64), [0, rows - 1]]))
    check_softmax(y[torch.from_numpy(ids)], orc.softmax_rows(x, ids), False, "65536x4096 sampled")
