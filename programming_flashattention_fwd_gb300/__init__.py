"""GB300 (sm_103a) FlashAttention forward: a C-ABI CUDA library and its Python binding.

``fa_fwd`` / ``fa_fwd_fp16`` / ``attention`` call into ``libfa_gb300.so`` (built from
``csrc/`` by ``build.build()``).  The library is loaded on first use and a missing or
unloadable library raises immediately: there is no CPU fallback.
"""
from .inputs import WORKLOADS, Workload, make_qkv, sample_rows  # noqa: F401


def __getattr__(name):
    # The CUDA binding is imported lazily so that the input generators can be used on
    # machines without a GPU; any call into the binding loads the library or raises.
    if name in ("fa_fwd", "fa_fwd_fp16", "attention", "fa_strerror", "fa_device_status",
                "FaError", "load_library", "STATUS", "fa_fwd_debug", "fa_fwd_select", "gemm",
                "softmax_rows"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
