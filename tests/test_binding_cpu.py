"""Host-side argument checks of the Python binding that need no GPU: tensors of one call on
different GPUs are rejected before the library is called (the C ABI works on the current
device only, so a mismatch would otherwise launch on one GPU over another GPU's memory)."""
import pytest
import torch

from programming_flashattention_fwd_gb300 import binding


class FakeCuda(torch.Tensor):
    """A CPU tensor that reports itself as living on a given CUDA device (no GPU needed)."""
    _dev = torch.device("cuda", 0)

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return self._dev


def on(idx, shape, dtype=torch.bfloat16):
    t = torch.Tensor._make_subclass(FakeCuda, torch.zeros(shape, dtype=dtype))
    t._dev = torch.device("cuda", idx)
    return t


def tensors(devs):
    B, Hq, Hkv, S, D = 1, 2, 1, 8, 64
    shapes = [(B, Hq, S, D), (B, Hkv, S, D), (B, Hkv, S, D), (B, Hq, S, D), (B, Hq, S)]
    dts = [torch.bfloat16] * 4 + [torch.float32]
    return [on(d, s, dt) for d, s, dt in zip(devs, shapes, dts)]


def test_same_device_passes_the_checks():
    q, k, v, o, lse = tensors([1, 1, 1, 1, 1])
    binding._check_tensors(q, k, v, o, lse)
    assert binding._check_same_device((("q", q), ("k", k))) == torch.device("cuda", 1)


@pytest.mark.parametrize("odd", range(5))
def test_a_tensor_on_another_gpu_is_rejected(odd, monkeypatch):
    devs = [0] * 5
    devs[odd] = 1
    q, k, v, o, lse = tensors(devs)
    called = []
    monkeypatch.setattr(binding, "load_library", lambda *a: called.append(1))
    with pytest.raises(ValueError, match="same GPU"):
        binding.fa_fwd(q, k, v, o, lse, True, 0.125)
    assert not called, "the library must not be reached"


def test_host_entry_point_checks_its_device_buffers():
    q, k, v, o, lse = tensors([0, 0, 1, 0, 0])
    qh, kh, vh, oh, lh = (torch.zeros(t.shape, dtype=t.dtype) for t in (q, k, v, o, lse))
    with pytest.raises(ValueError, match="same GPU"):
        binding.fa_fwd_host(qh, kh, vh, oh, lh, q, k, v, o, lse, True, 0.125)
