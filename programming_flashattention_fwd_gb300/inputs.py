"""Seeded synthetic inputs and named workloads for the attention forward pass.

This module is shared by the CUDA path's tests, the benchmark and the oracle-side checks.
It holds no attention arithmetic: it only draws random tensors, names workload shapes and
picks query rows to sample.

Workloads are the five shapes the pages' problem is exercised on (no dataset is involved;
every input is synthetic):

    mha_b1_h2_s128_d64           B=1  Hq=Hkv=2   S=128    D=64   bf16  non-causal
    mha_causal_b4_h16_s1024_d64  B=4  Hq=Hkv=16  S=1024   D=64   bf16  causal
    gqa_causal_b2_h32kv8_s4096   B=2  Hq=32 Hkv=8 S=4096  D=128  bf16  causal
    gqa_causal_b1_h32kv8_s16384  B=1  Hq=32 Hkv=8 S=16384 D=128  bf16  causal
    mha_fp16_b8_h16_s2000_std2   B=8  Hq=Hkv=16  S=2000   D=128  fp16  non-causal,
                                 q and k drawn with std 2 (large logits), v with std 1

Seed semantics: a CPU ``torch.Generator`` seeded with the workload's seed draws float32
standard normals in the order q [B,Hq,Sq,D], k [B,Hkv,Sk,D], v [B,Hkv,Sk,D]; each is
multiplied by its standard deviation and rounded (round-to-nearest-even) to the 16-bit
type.  Both the GPU path and the oracle consume exactly these rounded values.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Dict, List, Optional, Tuple

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Sk: int
    D: int
    dtype: str          # "bf16" or "fp16"
    causal: int         # 0 none, 1 top-left (j <= i), 2 bottom-right (j <= i + Sk - Sq)
    seed: int
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    scale: Optional[float] = None   # None -> 1/sqrt(D)

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.bfloat16 if self.dtype == "bf16" else torch.float16

    @property
    def is_fp16(self) -> bool:
        return self.dtype == "fp16"

    def flops(self) -> float:
        """Attention forward FLOPs: 4*B*Hq*Sq*Sk*D, halved when causal (the benchmark's
        convention for the square causal workloads)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Sk * self.D
        return f / 2.0 if self.causal else f

    def compulsory_bytes(self) -> int:
        """|Q| + |K| + |V| + |O| (16-bit) + |LSE| (fp32)."""
        q = self.B * self.Hq * self.Sq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.Sk * self.D * 2
        return 2 * q + kv + self.B * self.Hq * self.Sq * 4

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("mha_b1_h2_s128_d64", 1, 2, 2, 128, 128, 64, "bf16", False, 0),
        Workload("mha_causal_b4_h16_s1024_d64", 4, 16, 16, 1024, 1024, 64, "bf16", True, 1),
        Workload("gqa_causal_b2_h32kv8_s4096", 2, 32, 8, 4096, 4096, 128, "bf16", True, 2),
        Workload("gqa_causal_b1_h32kv8_s16384", 1, 32, 8, 16384, 16384, 128, "bf16", True, 3),
        Workload("mha_fp16_b8_h16_s2000_std2", 8, 16, 16, 2000, 2000, 128, "fp16", False, 4,
                 q_std=2.0, k_std=2.0, v_std=1.0),
    ]
}

# Head dimension 256 (the tile-size / head-dimension variants): the same GQA causal shape and a
# non-causal one, served by the one-query-tile kernel.
EXTRA_WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("gqa_causal_b2_h32kv8_s4096_d256", 2, 32, 8, 4096, 4096, 256, "bf16", True, 12),
        Workload("mha_b4_h16_s2048_d256", 4, 16, 16, 2048, 2048, 256, "bf16", False, 13),
    ]
}
ALL_WORKLOADS: Dict[str, Workload] = {**WORKLOADS, **EXTRA_WORKLOADS}

# The workload the benchmark times by default (GQA, causal, D=128, 275 GFLOP per call).
DEFAULT_BENCH_WORKLOAD = "gqa_causal_b2_h32kv8_s4096"


def make_qkv(w: Workload, device: str = "cpu") -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Draw q, k, v for workload ``w`` with the seed semantics in the module docstring."""
    g = torch.Generator(device="cpu").manual_seed(int(w.seed))
    shapes = ((w.B, w.Hq, w.Sq, w.D), (w.B, w.Hkv, w.Sk, w.D), (w.B, w.Hkv, w.Sk, w.D))
    stds = (w.q_std, w.k_std, w.v_std)
    out = []
    for shp, std in zip(shapes, stds):
        x = torch.randn(shp, generator=g, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        out.append(x.to(w.torch_dtype).to(device))
    return out[0], out[1], out[2]


def sample_rows(w: Workload, n: int = 256, seed: Optional[int] = None,
                edge: bool = True) -> np.ndarray:
    """Seeded (b, h, i) triples to check at full size: ``n`` distinct uniform draws plus,
    when ``edge`` is set, deterministic edge rows (first/last row of the first two tiles,
    the first row of the last tile, the last row; first and last head; first and last
    batch).  Returns an int64 array of shape [m, 3] without duplicates."""
    rng = np.random.default_rng(w.seed if seed is None else seed)
    total = w.B * w.Hq * w.Sq
    n = min(n, total)
    flat = rng.choice(total, size=n, replace=False)
    b = flat // (w.Hq * w.Sq)
    h = (flat // w.Sq) % w.Hq
    i = flat % w.Sq
    rows: List[Tuple[int, int, int]] = list(zip(b.tolist(), h.tolist(), i.tolist()))
    if edge:
        last_tile_first = ((w.Sq - 1) // 128) * 128
        idx = sorted({x for x in (0, 127, 128, last_tile_first, w.Sq - 1) if 0 <= x < w.Sq})
        for bb in sorted({0, w.B - 1}):
            for hh in sorted({0, w.Hq - 1}):
                for ii in idx:
                    rows.append((bb, hh, ii))
    uniq = sorted(set(rows))
    return np.asarray(uniq, dtype=np.int64).reshape(-1, 3)


__all__ = ["Workload", "WORKLOADS", "EXTRA_WORKLOADS", "ALL_WORKLOADS", "DEFAULT_BENCH_WORKLOAD", "make_qkv",
           "sample_rows"]
