"""Seeded synthetic inputs and the workload table.

This module only draws random numbers and describes shapes; it holds none of
the attention arithmetic, so both the CUDA path's tests and the float64 oracle
may use it.

Recipe (every workload): ``torch.manual_seed(seed)`` on the CPU generator,
then float32 ``randn`` drawn in the order Q, K, V, dO, each rounded once to
bf16 (round-to-nearest-even, ``Tensor.to(torch.bfloat16)``).  Both sides read
the same bf16 bits.
"""
from __future__ import annotations

from dataclasses import dataclass, asdict

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Tq: int
    Tk: int
    d: int
    causal: bool
    seed: int
    dO_std: float = 1.0
    window: int = 0  # causal sliding window in keys (0 = none)
    dv_: int = 0     # head size of V and O when it differs from d (0 = same as d)

    @property
    def dv(self) -> int:
        return self.dv_ or self.d

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def pairs_per_head(self) -> int:
        """Unmasked (query, key) pairs of one head (bottom-right causal
        alignment; with a window W, row i sees keys (i + off - W, i + off])."""
        if not self.causal:
            return self.Tq * self.Tk
        off = self.Tk - self.Tq
        if self.window <= 0 and self.Tq == self.Tk:
            return self.Tq * (self.Tq + 1) // 2
        total = 0
        for i in range(self.Tq):
            end = max(0, min(self.Tk, i + off + 1))
            beg = max(0, i + off - self.window + 1) if self.window > 0 else 0
            total += max(0, end - beg)
        return total

    def flops(self, part: str) -> float:
        """Algorithmic flops per head, two per multiply-add of each product:
        fwd S = QK^T and O = PV: 2*pairs*(d + dv); bwd S, dP = dO V^T, dV, dK,
        dQ: 2*pairs*(3 d + 2 dv).  With dv = d: 4, 10 and 14 * pairs * d."""
        d, dv = self.d, self.dv
        per_pair = {"fwd": 2 * (d + dv), "bwd": 2 * (3 * d + 2 * dv), "fwdbwd": 2 * (4 * d + 3 * dv)}[part]
        return float(per_pair) * self.pairs_per_head() * self.B * self.Hq

    def as_dict(self) -> dict:
        return asdict(self)


# The workloads the library is measured and checked on.  The last one is the
# local-attention layer of "The Autograd Memory Trap" (section "Assumptions and
# Uncertainties", item 3: sliding-window layers that see at most 2080 keys),
# at the headline GQA shape.
WORKLOADS = {
    "single_head_T256_d64": Workload("single_head_T256_d64", 1, 1, 1, 256, 256, 64, False, 1),
    "mha_B4_H16_T2048_d64_causal": Workload("mha_B4_H16_T2048_d64_causal", 4, 16, 16, 2048, 2048, 64, True, 2),
    "gqa_B2_H32x8_T8192_d128_causal": Workload("gqa_B2_H32x8_T8192_d128_causal", 2, 32, 8, 8192, 8192, 128, True, 3),
    "gqa_B1_H32x8_Tq4096_Tk8032_d128": Workload("gqa_B1_H32x8_Tq4096_Tk8032_d128", 1, 32, 8, 4096, 8032, 128, False,
                                                4, dO_std=0.1),
    "long_B1_H16_T32768_d128_causal": Workload("long_B1_H16_T32768_d128_causal", 1, 16, 16, 32768, 32768, 128, True, 5),
    "swa_B1_H32x8_T8192_W2080_d128": Workload("swa_B1_H32x8_T8192_W2080_d128", 1, 32, 8, 8192, 8192, 128, True, 6,
                                              window=2080),
}
WORKLOAD_ORDER = list(WORKLOADS)
# The workload the headline throughput is quoted on.
HEADLINE = "gqa_B2_H32x8_T8192_d128_causal"


def make_inputs(w: Workload, seed: int | None = None):
    """Return bf16 CPU tensors (Q, K, V, dO) with [B, H, T, d] layout."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed if seed is None else seed)
    Q = torch.randn(w.B, w.Hq, w.Tq, w.d, generator=g, dtype=torch.float32)
    K = torch.randn(w.B, w.Hkv, w.Tk, w.d, generator=g, dtype=torch.float32)
    V = torch.randn(w.B, w.Hkv, w.Tk, w.dv, generator=g, dtype=torch.float32)
    dO = torch.randn(w.B, w.Hq, w.Tq, w.dv, generator=g, dtype=torch.float32)
    if w.dO_std != 1.0:
        dO = dO * w.dO_std
    return tuple(t.to(torch.bfloat16) for t in (Q, K, V, dO))


def make_custom(B, Hq, Hkv, Tq, Tk, d, causal, seed, dO_std=1.0, dv=None):
    """Inputs for an ad-hoc shape (edge-case tests).  The draws do not depend
    on the mask, so a windowed case takes the same inputs as its causal one.
    ``dv`` sets the head size of V and dO (default d)."""
    return make_inputs(Workload("custom", B, Hq, Hkv, Tq, Tk, d, causal, seed, dO_std, dv_=dv or 0))
