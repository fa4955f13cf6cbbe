"""The algorithmic flop count behind every TFLOP/s figure: visible (query,
key) pairs per head, counted by brute force over the mask definition
(bottom-right causal alignment, optional sliding window), and the per-pair
flop factors of the five backward and two forward contractions."""
import pytest
import torch

from tiled_attention_05_gb300.inputs import WORKLOADS, Workload


def brute_pairs(Tq, Tk, causal, window=0):
    i = torch.arange(Tq)[:, None]
    j = torch.arange(Tk)[None, :]
    if not causal:
        return Tq * Tk
    vis = j <= i + (Tk - Tq)
    if window > 0:
        vis &= j > i + (Tk - Tq) - window
    return int(vis.sum())


@pytest.mark.parametrize("Tq, Tk, causal, window", [
    (1, 1, False, 0), (7, 13, False, 0), (256, 256, True, 0), (300, 300, True, 0),
    (32, 8032, True, 0), (600, 257, True, 0),            # Tq < Tk and Tq > Tk (empty first rows)
    (300, 300, True, 1), (300, 300, True, 77), (40, 90, True, 70), (1, 5000, True, 300),
    (600, 257, True, 100), (129, 129, True, 128),
])
def test_pairs_match_brute_force(Tq, Tk, causal, window):
    w = Workload("t", 1, 1, 1, Tq, Tk, 64, causal, 0, window=window)
    assert w.pairs_per_head() == brute_pairs(Tq, Tk, causal, window)


def test_flop_factors():
    w = Workload("t", 2, 4, 2, 100, 90, 64, False, 0)
    pairs = w.pairs_per_head() * w.B * w.Hq
    assert w.flops("fwd") == 4 * pairs * 64      # QK^T and PV
    assert w.flops("bwd") == 10 * pairs * 64     # S, dP, dV, dK, dQ
    assert w.flops("fwdbwd") == 14 * pairs * 64
    v = Workload("t", 1, 2, 1, 50, 60, 128, True, 0, dv_=64)
    pv = v.pairs_per_head() * v.Hq
    assert v.flops("fwd") == 2 * pv * (128 + 64)
    assert v.flops("bwd") == 2 * pv * (3 * 128 + 2 * 64)


def test_headline_workload_totals():
    # B=2, 32 query heads, T=8192 causal, d=128: T(T+1)/2 pairs per head
    w = WORKLOADS["gqa_B2_H32x8_T8192_d128_causal"]
    assert w.pairs_per_head() == 8192 * 8193 // 2
    assert round(w.flops("fwd") / 1e9, 1) == 1099.6
    assert round(w.flops("bwd") / 1e9, 1) == 2749.1
    assert round(w.flops("fwdbwd") / 1e9, 1) == 3848.8
    s = WORKLOADS["swa_B1_H32x8_T8192_W2080_d128"]
    assert s.pairs_per_head() == brute_pairs(8192, 8192, True, 2080)
