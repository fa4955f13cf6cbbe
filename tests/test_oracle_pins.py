"""Pins for the float64 oracle: what the pages and the mathematics fix.

Nothing here compares the oracle with itself.  The pins are:
  * a library implementation of the same definition (torch float64
    scaled_dot_product_attention, differentiated by torch autograd) -- the
    page's own comparison pattern, "What Ordinary Autograd Saves", section "The
    way out is recomputation", run in double;
  * central finite differences of the loss <O, dO> (independent of the
    hand-derived gradient formulas);
  * the tiled online-softmax recurrence of "What Ordinary Autograd Saves",
    section "The implementation under test", restated here in float64 with
    ragged tiles -- it must land on the oracle's definition;
  * closed forms and special cases (one key, constant V, causal row 0, key
    shift, V = identity exposing the softmax rows, a 2x2 case by hand);
  * invariants of the gradients (sum_j dS_ij = 0 so sum_j dK_j = 0;
    D = rowsum(dO * O); dV = P^T dO; GQA = expanded heads summed);
  * the saved-payload numbers printed on the page (tests/golden/);
  * mutation: planted mistakes in a copy of the oracle source must fail a pin.
"""
from __future__ import annotations

import math
import os
import re
import shutil
import subprocess

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden")


def rnd(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g, dtype=torch.float64) * scale).numpy()


def make(B, Hq, Hkv, Tq, Tk, d, dv=None, seed=0):
    dv = d if dv is None else dv
    return (rnd((B, Hq, Tq, d), seed), rnd((B, Hkv, Tk, d), seed + 1), rnd((B, Hkv, Tk, dv), seed + 2),
            rnd((B, Hq, Tq, dv), seed + 3))


def visible_mask(Tq, Tk, causal, window=0):
    i = torch.arange(Tq)[:, None]
    j = torch.arange(Tk)[None, :]
    if not causal:
        return torch.ones(Tq, Tk, dtype=torch.bool)
    m = j <= i + (Tk - Tq)
    if window > 0:
        m = m & (j > i + (Tk - Tq) - window)
    return m


def torch_reference(Q, K, V, dO, causal, scale, window=0):
    """torch float64 SDPA (GQA by repeat_interleave) + autograd; returns O, L, dQ, dK, dV."""
    Qt, Kt, Vt = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    G = Q.shape[1] // K.shape[1]
    Ke, Ve = Kt.repeat_interleave(G, dim=1), Vt.repeat_interleave(G, dim=1)
    mask = visible_mask(Q.shape[2], K.shape[2], causal, window)
    O = F.scaled_dot_product_attention(Qt, Ke, Ve, attn_mask=mask, scale=scale)
    S = (Qt @ Ke.transpose(-1, -2)) * scale
    L = torch.logsumexp(S.masked_fill(~mask, -math.inf), dim=-1)
    (O * torch.tensor(dO)).sum().backward()
    return O.detach().numpy(), L.detach().numpy(), Qt.grad.numpy(), Kt.grad.numpy(), Vt.grad.numpy()


SHAPES = [
    # B, Hq, Hkv, Tq, Tk, d, causal
    (1, 1, 1, 13, 13, 8, False),
    (2, 4, 2, 17, 23, 8, False),
    (1, 4, 1, 19, 19, 16, True),
    (2, 2, 2, 9, 30, 4, True),   # Tq < Tk: bottom-right causal
    (1, 2, 1, 1, 1, 4, False),
    (1, 8, 2, 33, 40, 8, False),
]


def rel(a, b):
    """Max abs error relative to the largest reference magnitude (floored at 1e-3 for all-zero references)."""
    return float(np.max(np.abs(a - b)) / max(1e-3, np.max(np.abs(b))))


def fd_grads(lib, Q, K, V, dO, causal, scale, h=1e-6, window=0):
    def loss(Q_, K_, V_):
        O, _ = lib.forward(Q_, K_, V_, causal, scale, window=window)
        return float(np.sum(O * dO))

    grads = []
    for idx, X in enumerate((Q, K, V)):
        g = np.zeros_like(X)
        it = np.nditer(X, flags=["multi_index"])
        for _ in it:
            mi = it.multi_index
            args = [Q.copy(), K.copy(), V.copy()]
            args[idx][mi] += h
            lp = loss(*args)
            args[idx][mi] -= 2 * h
            lm = loss(*args)
            g[mi] = (lp - lm) / (2 * h)
        grads.append(g)
    return grads


def tiled_recurrence(Q, K, V, causal, scale, bq=32, bk=32):
    """Online-softmax tiled forward in float64: outer loop over query blocks,
    inner over key blocks, running max / sum / unnormalised output per row, one
    rescale when the max moves, normalise once at the end."""
    B, Hq, Tq, d = Q.shape
    Hkv, Tk, dv = K.shape[1], K.shape[2], V.shape[3]
    G = Hq // Hkv
    O = np.zeros((B, Hq, Tq, dv))
    L = np.zeros((B, Hq, Tq))
    vis = visible_mask(Tq, Tk, causal).numpy()
    for b in range(B):
        for h in range(Hq):
            q, k, v = Q[b, h], K[b, h // G], V[b, h // G]
            for i in range(0, Tq, bq):
                nq = min(bq, Tq - i)
                m = np.full(nq, -np.inf)
                l = np.zeros(nq)
                acc = np.zeros((nq, dv))
                for j in range(0, Tk, bk):
                    nk = min(bk, Tk - j)
                    S = (q[i:i + nq] @ k[j:j + nk].T) * scale
                    S = np.where(vis[i:i + nq, j:j + nk], S, -np.inf)
                    m_new = np.maximum(m, S.max(axis=1))
                    base = np.where(np.isneginf(m_new), 0.0, m_new)
                    alpha = np.where(np.isneginf(m), 0.0, np.exp(m - base))
                    P = np.exp(S - base[:, None])
                    l = l * alpha + P.sum(axis=1)
                    acc = acc * alpha[:, None] + P @ v[j:j + nk]
                    m = m_new
                O[b, h, i:i + nq] = acc / l[:, None]
                L[b, h, i:i + nq] = m + np.log(l)
    return O, L


# ----------------------------------------------------------------- pin suite
def pin_suite(lib, quick=False):
    """Run the pins on ``lib``; return the names of those that fail."""
    failed = []
    shapes = SHAPES[:4] if quick else SHAPES
    for n, (B, Hq, Hkv, Tq, Tk, d, causal) in enumerate(shapes):
        Q, K, V, dO = make(B, Hq, Hkv, Tq, Tk, d, seed=10 * n)
        scale = 1.0 / math.sqrt(d) * (1.3 if n % 2 else 1.0)
        O, L = lib.forward(Q, K, V, causal, scale)
        dQ, dK, dV, D = lib.backward(Q, K, V, dO, causal, scale)
        Or, Lr, dQr, dKr, dVr = torch_reference(Q, K, V, dO, causal, scale)
        for name, a, b, tol in (("O", O, Or, 1e-12), ("L", L, Lr, 1e-12), ("dQ", dQ, dQr, 1e-11),
                                ("dK", dK, dKr, 1e-11), ("dV", dV, dVr, 1e-11)):
            if not np.all(np.isfinite(a)) or rel(a, b) > tol:
                failed.append(f"torch:{name}:{n}")
        if not np.allclose(D, np.sum(dO * O, axis=-1), rtol=0, atol=1e-12):
            failed.append(f"D-identity:{n}")
        if not np.allclose(dK.sum(axis=2), 0.0, atol=1e-12):
            failed.append(f"sum-dK:{n}")
    # sliding window against the band-masked library reference
    for n, (Tq, Tk, W) in enumerate(((23, 23, 5), (9, 30, 7))):
        Q, K, V, dO = make(1, 4, 2, Tq, Tk, 8, seed=200 + n)
        O, L = lib.forward(Q, K, V, True, 0.4, window=W)
        dQ, dK, dV, _ = lib.backward(Q, K, V, dO, True, 0.4, window=W)
        ref = torch_reference(Q, K, V, dO, True, 0.4, window=W)
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), (O, L, dQ, dK, dV), ref):
            if not np.all(np.isfinite(a)) or rel(a, b) > 1e-11:
                failed.append(f"window:{name}:{n}")
    # V and O narrower or wider than Q and K (d != dv), against torch float64
    for n, (d, dv, causal) in enumerate(((8, 12, True), (12, 8, False))):
        Q, K, V, dO = make(2, 4, 2, 19, 23, d, dv=dv, seed=300 + n)
        O, L = lib.forward(Q, K, V, causal, 0.35)
        dQ, dK, dV, _ = lib.backward(Q, K, V, dO, causal, 0.35)
        ref = torch_reference(Q, K, V, dO, causal, 0.35)
        for name, a, b in zip(("O", "L", "dQ", "dK", "dV"), (O, L, dQ, dK, dV), ref):
            if a.shape != b.shape or not np.all(np.isfinite(a)) or rel(a, b) > 1e-11:
                failed.append(f"dv:{name}:{n}")
    # finite differences on a tiny causal GQA problem
    Q, K, V, dO = make(1, 2, 1, 7, 7, 4, seed=99)
    for causal in (True, False):
        dQ, dK, dV, _ = lib.backward(Q, K, V, dO, causal, 0.7)
        for name, a, b in zip(("dQ", "dK", "dV"), (dQ, dK, dV), fd_grads(lib, Q, K, V, dO, causal, 0.7)):
            if rel(a, b) > 1e-7:
                failed.append(f"fd:{name}:{causal}")
    return failed


def test_pin_suite_passes(oracle_lib):
    assert pin_suite(oracle_lib) == []


# ----------------------------------------------------------------- individual pins
@pytest.mark.parametrize("shape", SHAPES)
def test_forward_and_grads_match_torch_float64(oracle_lib, shape):
    B, Hq, Hkv, Tq, Tk, d, causal = shape
    Q, K, V, dO = make(B, Hq, Hkv, Tq, Tk, d, seed=5)
    scale = 0.9 / math.sqrt(d)
    O, L = oracle_lib.forward(Q, K, V, causal, scale)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, causal, scale)
    Or, Lr, dQr, dKr, dVr = torch_reference(Q, K, V, dO, causal, scale)
    assert rel(O, Or) < 1e-12 and rel(L, Lr) < 1e-12
    assert rel(dQ, dQr) < 1e-11 and rel(dK, dKr) < 1e-11 and rel(dV, dVr) < 1e-11


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(oracle_lib, causal):
    Q, K, V, dO = make(1, 2, 1, 9, 9, 4, seed=3)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, causal, 0.5)
    fQ, fK, fV = fd_grads(oracle_lib, Q, K, V, dO, causal, 0.5)
    assert rel(dQ, fQ) < 1e-7 and rel(dK, fK) < 1e-7 and rel(dV, fV) < 1e-7


@pytest.mark.parametrize("Tq,Tk,causal", [(100, 77, False), (77, 77, True), (40, 100, True), (64, 64, False)])
def test_tiled_online_softmax_recurrence_equals_definition(oracle_lib, Tq, Tk, causal):
    Q, K, V, _ = make(1, 4, 2, Tq, Tk, 8, seed=Tq + Tk)
    O, L = oracle_lib.forward(Q, K, V, causal, 0.35)
    Ot, Lt = tiled_recurrence(Q, K, V, causal, 0.35)
    assert np.max(np.abs(O - Ot)) < 1e-13
    assert np.max(np.abs(L - Lt)) < 1e-13


def test_single_key(oracle_lib):
    Q, K, V, dO = make(2, 4, 2, 5, 1, 8, seed=7)
    O, L = oracle_lib.forward(Q, K, V, False, 0.3)
    G = 2
    for h in range(4):
        assert np.allclose(O[:, h], np.broadcast_to(V[:, h // G], O[:, h].shape), atol=1e-15)
        assert np.allclose(L[:, h], 0.3 * np.einsum("btd,bd->bt", Q[:, h], K[:, h // G, 0]), atol=1e-14)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, False, 0.3)
    assert np.max(np.abs(dQ)) < 1e-15 and np.max(np.abs(dK)) < 1e-15
    want = dO.reshape(2, 2, 2, 5, 8).sum(axis=(2, 3))[:, :, None, :]
    assert np.allclose(dV, want, atol=1e-13)


def test_constant_values_give_constant_output(oracle_lib):
    Q, K, V, _ = make(1, 2, 2, 11, 17, 8, seed=8)
    V[:] = np.arange(8)[None, None, None, :] * 0.25 - 1.0
    for causal in (False, True):
        O, _ = oracle_lib.forward(Q, K, V, causal, 0.4)
        assert np.allclose(O, V[:, :, :1, :], atol=1e-14)


def test_causal_first_row(oracle_lib):
    Q, K, V, dO = make(1, 2, 2, 12, 12, 8, seed=9)
    O, L = oracle_lib.forward(Q, K, V, True, 0.6)
    assert np.allclose(O[:, :, 0], V[:, :, 0], atol=1e-15)
    assert np.allclose(L[:, :, 0], 0.6 * np.sum(Q[:, :, 0] * K[:, :, 0], axis=-1), atol=1e-14)
    dQ, _, _, _ = oracle_lib.backward(Q, K, V, dO, True, 0.6)
    assert np.max(np.abs(dQ[:, :, 0])) < 1e-15


def test_key_shift_moves_L_not_O(oracle_lib):
    Q, K, V, _ = make(1, 4, 2, 10, 14, 8, seed=10)
    c = rnd((8,), 77)
    O1, L1 = oracle_lib.forward(Q, K, V, False, 0.5)
    O2, L2 = oracle_lib.forward(Q, K + c, V, False, 0.5)
    assert np.allclose(O1, O2, atol=1e-13)
    assert np.allclose(L2 - L1, 0.5 * Q @ c, atol=1e-12)


def test_identity_values_expose_softmax_rows(oracle_lib):
    # With V = I (dv = Tk) each output row is the probability row itself.
    Tq, Tk = 9, 6
    Q, K, _, _ = make(1, 1, 1, Tq, Tk, 4, seed=11)
    V = np.eye(Tk)[None, None]
    for causal in (False, True):
        P, L = oracle_lib.forward(Q, K, V, causal, 0.8)
        vis = visible_mask(Tq, Tk, causal).numpy()
        has_key = vis.any(axis=1)
        # rows with a visible key sum to one; rows without one (causal, Tq > Tk) are zero
        assert np.allclose(P[0, 0].sum(-1), has_key.astype(float), atol=1e-14)
        assert np.all(P >= 0)
        assert np.all(P[0, 0][~vis] == 0)
        # the ratio of two visible probabilities is the exp of their score difference
        S = 0.8 * Q[0, 0] @ K[0, 0].T
        i = Tq - 1
        assert np.allclose(P[0, 0, i, 1] / P[0, 0, i, 0], math.exp(S[i, 1] - S[i, 0]), rtol=1e-13)


def test_dV_is_Pt_dO(oracle_lib):
    Tq, Tk, d = 8, 5, 4
    Q, K, V, dO = make(1, 1, 1, Tq, Tk, d, seed=12)
    for causal in (False, True):
        P, _ = oracle_lib.forward(Q, K, np.eye(Tk)[None, None], causal, 0.5)
        _, _, dV, _ = oracle_lib.backward(Q, K, V, dO, causal, 0.5)
        assert np.allclose(dV[0, 0], P[0, 0].T @ dO[0, 0], atol=1e-14)


def test_two_by_two_by_hand(oracle_lib):
    # q0 = k0 = (1, 0), q1 = k1 = (0, 1), scale 1: row 0 scores (1, 0), row 1 scores (0, 1).
    Q = np.array([[[[1.0, 0.0], [0.0, 1.0]]]])
    K = Q.copy()
    V = np.array([[[[1.0, 2.0], [3.0, 4.0]]]])
    O, L = oracle_lib.forward(Q, K, V, False, 1.0)
    e = math.e
    assert np.allclose(O[0, 0, 0], [(e * 1 + 3) / (e + 1), (e * 2 + 4) / (e + 1)], atol=1e-15)
    assert np.allclose(O[0, 0, 1], [(1 + e * 3) / (e + 1), (2 + e * 4) / (e + 1)], atol=1e-15)
    assert np.allclose(L[0, 0], [math.log(e + 1), math.log(e + 1)], atol=1e-15)
    # causal: row 0 sees key 0 only
    O, L = oracle_lib.forward(Q, K, V, True, 1.0)
    assert np.allclose(O[0, 0, 0], [1.0, 2.0]) and abs(L[0, 0, 0] - 1.0) < 1e-15


def test_gqa_equals_expanded_heads_summed(oracle_lib):
    Q, K, V, dO = make(2, 6, 2, 11, 13, 8, seed=13)
    G = 3
    Ke, Ve = np.repeat(K, G, axis=1), np.repeat(V, G, axis=1)
    for causal in (False, True):
        O, L = oracle_lib.forward(Q, K, V, causal, 0.4)
        Oe, Le = oracle_lib.forward(Q, Ke, Ve, causal, 0.4)
        assert np.array_equal(O, Oe) and np.array_equal(L, Le)
        dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, causal, 0.4)
        dQe, dKe, dVe, _ = oracle_lib.backward(Q, Ke, Ve, dO, causal, 0.4)
        assert np.allclose(dQ, dQe, atol=1e-14)
        assert np.allclose(dK, dKe.reshape(2, 2, G, 13, 8).sum(2), atol=1e-13)
        assert np.allclose(dV, dVe.reshape(2, 2, G, 13, 8).sum(2), atol=1e-13)


def test_empty_key_rows_policy(oracle_lib):
    # causal with Tq > Tk: rows i < Tq - Tk see no key.
    Tq, Tk = 12, 5
    Q, K, V, dO = make(1, 2, 1, Tq, Tk, 4, seed=14)
    O, L = oracle_lib.forward(Q, K, V, True, 0.5)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, True, 0.5)
    empty = Tq - Tk
    assert np.all(O[:, :, :empty] == 0) and np.all(np.isneginf(L[:, :, :empty]))
    assert np.all(dQ[:, :, :empty] == 0)
    # the remaining rows are exactly the Tq = Tk causal problem on the last Tk rows
    O2, L2 = oracle_lib.forward(Q[:, :, empty:], K, V, True, 0.5)
    _, dK2, dV2, _ = oracle_lib.backward(Q[:, :, empty:], K, V, dO[:, :, empty:], True, 0.5)
    assert np.array_equal(O[:, :, empty:], O2) and np.array_equal(L[:, :, empty:], L2)
    assert np.allclose(dK, dK2, atol=1e-15) and np.allclose(dV, dV2, atol=1e-15)


def test_row_subset_equals_full(oracle_lib):
    Q, K, V, _ = make(1, 4, 1, 50, 60, 8, seed=15)
    O, L = oracle_lib.forward(Q, K, V, True, 0.3)
    Os, Ls = oracle_lib.forward(Q, K, V, True, 0.3, rows=(17, 29))
    assert np.array_equal(Os[:, :, 17:29], O[:, :, 17:29]) and np.array_equal(Ls[:, :, 17:29], L[:, :, 17:29])
    assert np.all(np.isnan(Os[:, :, :17]))


def test_thread_count_does_not_change_results(oracle_lib):
    Q, K, V, dO = make(1, 4, 2, 40, 40, 8, seed=16)
    a = oracle_lib.backward(Q, K, V, dO, True, 0.3, nthreads=1)
    b = oracle_lib.backward(Q, K, V, dO, True, 0.3, nthreads=4)
    for x, y in zip(a, b):
        assert np.allclose(x, y, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("d,dv,causal", [(8, 16, True), (16, 8, True), (4, 12, False), (64, 128, True)])
def test_value_head_size_differs(oracle_lib, d, dv, causal):
    """V and O may have a head size dv other than d ("What Ordinary Autograd
    Saves", section "The implementation under test": the value width is read
    from V's shape): torch float64 and finite differences agree."""
    Q, K, V, dO = make(1, 4, 2, 21, 26, d, dv=dv, seed=d * 100 + dv)
    O, L = oracle_lib.forward(Q, K, V, causal, 0.3)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, causal, 0.3)
    assert O.shape == (1, 4, 21, dv) and dQ.shape == Q.shape and dK.shape == K.shape and dV.shape == V.shape
    Or, Lr, dQr, dKr, dVr = torch_reference(Q, K, V, dO, causal, 0.3)
    assert rel(O, Or) < 1e-12 and rel(L, Lr) < 1e-12
    assert rel(dQ, dQr) < 1e-11 and rel(dK, dKr) < 1e-11 and rel(dV, dVr) < 1e-11
    if d <= 16:
        Qs, Ks, Vs, dOs = (t[:, :2, :6] if t.shape[1] == 4 else t[:, :1, :6] for t in (Q, K, V, dO))
        got = oracle_lib.backward(Qs, Ks, Vs, dOs, causal, 0.3)[:3]
        for a, b in zip(got, fd_grads(oracle_lib, Qs, Ks, Vs, dOs, causal, 0.3)):
            assert rel(a, b) < 1e-7


@pytest.mark.parametrize("Tq,Tk,W", [(40, 40, 1), (40, 40, 7), (33, 70, 16), (70, 33, 5), (64, 64, 200)])
def test_sliding_window_matches_torch_float64(oracle_lib, Tq, Tk, W):
    Q, K, V, dO = make(2, 4, 2, Tq, Tk, 8, seed=Tq + W)
    O, L = oracle_lib.forward(Q, K, V, True, 0.45, window=W)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, True, 0.45, window=W)
    vis = visible_mask(Tq, Tk, True, W)
    if bool(vis.any(dim=1).all()):
        Or, Lr, dQr, dKr, dVr = torch_reference(Q, K, V, dO, True, 0.45, window=W)
        assert rel(O, Or) < 1e-12 and rel(L, Lr) < 1e-12
        assert rel(dQ, dQr) < 1e-11 and rel(dK, dKr) < 1e-11 and rel(dV, dVr) < 1e-11
    # rows without a visible key follow the empty-row policy
    empty = ~vis.any(dim=1).numpy()
    assert np.all(O[:, :, empty] == 0) and np.all(np.isneginf(L[:, :, empty]))


def test_window_wider_than_keys_is_plain_causal(oracle_lib):
    Q, K, V, dO = make(1, 2, 1, 30, 45, 8, seed=21)
    a = oracle_lib.forward(Q, K, V, True, 0.3)
    b = oracle_lib.forward(Q, K, V, True, 0.3, window=45)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    ga = oracle_lib.backward(Q, K, V, dO, True, 0.3)
    gb = oracle_lib.backward(Q, K, V, dO, True, 0.3, window=1000)
    # (the backward's per-thread partial sums are added in a run-dependent order)
    assert all(np.allclose(x, y, rtol=0, atol=1e-14) for x, y in zip(ga, gb))


def test_window_of_one_sees_only_the_diagonal(oracle_lib):
    Tq, Tk = 12, 20
    off = Tk - Tq
    Q, K, V, dO = make(1, 1, 1, Tq, Tk, 4, seed=22)
    O, L = oracle_lib.forward(Q, K, V, True, 0.5, window=1)
    assert np.allclose(O[0, 0], V[0, 0, off:], atol=1e-15)
    assert np.allclose(L[0, 0], 0.5 * np.sum(Q[0, 0] * K[0, 0, off:], axis=-1), atol=1e-14)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, True, 0.5, window=1)
    assert np.max(np.abs(dQ)) < 1e-15 and np.max(np.abs(dK)) < 1e-15
    assert np.allclose(dV[0, 0, off:], dO[0, 0], atol=1e-15) and np.all(dV[0, 0, :off] == 0)


def test_window_backward_matches_finite_differences(oracle_lib):
    Q, K, V, dO = make(1, 2, 1, 9, 9, 4, seed=23)
    dQ, dK, dV, _ = oracle_lib.backward(Q, K, V, dO, True, 0.6, window=3)
    fQ, fK, fV = fd_grads(oracle_lib, Q, K, V, dO, True, 0.6, window=3)
    assert rel(dQ, fQ) < 1e-7 and rel(dK, fK) < 1e-7 and rel(dV, fV) < 1e-7


# ----------------------------------------------------------------- saved payload (golden)
def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            rows.append(line.split())
    return rows[0], rows[1:]


def test_saved_payload_matches_page_table(oracle_lib):
    header, rows = read_golden("p1_saved_payload.txt")
    d = 32
    for r in rows:
        T, tiled_kib, dense_kib = int(r[0]), int(r[1]), int(r[2])
        dense = oracle_lib.saved_bytes("dense", 1, 1, 1, T, T, d, d, elem_bytes=4, prob_bytes=4)
        assert dense == dense_kib * 1024
        ckpt = oracle_lib.saved_bytes("checkpoint", 1, 1, 1, T, T, d, d, elem_bytes=4)
        assert ckpt == 3 * T * d * 4
        keep = oracle_lib.saved_bytes("keep_o_l", 1, 1, 1, T, T, d, d, elem_bytes=4, stat_bytes=4)
        assert keep == ckpt + T * d * 4 + T * 4
    # "about 4x at T = 128 and 25x at T = 1024" (tiled / checkpointed)
    t128 = int(rows[0][1]) * 1024 / oracle_lib.saved_bytes("checkpoint", 1, 1, 1, 128, 128, d, d, elem_bytes=4)
    t1024 = int(rows[3][1]) * 1024 / oracle_lib.saved_bytes("checkpoint", 1, 1, 1, 1024, 1024, d, d, elem_bytes=4)
    assert round(t128) == 4 and round(t1024) == 25


def test_dense_payload_reproduced_with_saved_tensor_hooks(oracle_lib):
    """The page's instrument (count stashed bytes once per storage view) on the dense definition."""

    class Payload:
        def __init__(self):
            self.seen, self.bytes = set(), 0

        def pack(self, t):
            key = (t.untyped_storage().data_ptr(), t.storage_offset(), tuple(t.shape), tuple(t.stride()), t.dtype)
            if key not in self.seen:
                self.seen.add(key)
                self.bytes += t.numel() * t.element_size()
            return t.detach()

    def dense(Q, K, V):
        return torch.softmax((Q @ K.T) / math.sqrt(Q.shape[-1]), -1) @ V

    for T in (128, 256, 512, 1024):
        torch.manual_seed(0)
        Q, K, V = (torch.randn(T, 32, requires_grad=True) for _ in range(3))
        p = Payload()
        with torch.autograd.graph.saved_tensors_hooks(p.pack, lambda t: t):
            dense(Q, K, V).sum().backward()
        assert p.bytes == oracle_lib.saved_bytes("dense", 1, 1, 1, T, T, 32, 32, elem_bytes=4, prob_bytes=4)


# ----------------------------------------------------------------- mutation
MUTANTS = {
    "dS-sign": ("p[j] * (dP[j] - Di)", "p[j] * (dP[j] + Di)"),
    "gqa-index-forward": ("kvh = h / G;", "kvh = h % Hkv;"),
    "dK-scale-dropped": ("dk[c] += scale * dS * q[c];", "dk[c] += dS * q[c];"),
    "causal-off-by-one": ("(int64_t)(z.Tk - z.Tq) + 1;", "(int64_t)(z.Tk - z.Tq);"),
    "lse-max-dropped": ("*lse = m + std::log(l);", "*lse = std::log(l);"),
    "dP-wrong-operand": ("s += g[c] * v[c];", "s += g[c] * Kh[j * z.d + c];"),
    "dQ-uses-q": ("dq[c] += scale * dS * k[c];", "dq[c] += scale * dS * q[c];"),
    "window-off-by-one": ("- z.window + 1;", "- z.window;"),
    "dP-over-d-not-dv": ("for (int c = 0; c < dv; ++c) s += g[c] * v[c];", "for (int c = 0; c < d; ++c) s += g[c] * v[c];"),
    "softmax-not-normalised": ("for (int64_t j = *j0; j < n; ++j) p[j] /= l;", ""),
    "max-not-subtracted": ("p[j] = std::exp(p[j] - m);", "p[j] = std::exp(p[j]);"),
    "scale-dropped-forward": ("s *= z.scale;", ""),
    "D-without-p": ("Di += p[j] * s;", "Di += s;"),
    "dV-without-p": ("dvv[c] += p[j] * g[c];", "dvv[c] += g[c];"),
    "gqa-index-backward": ("const int64_t h = kvh * G + t / Tq,", "const int64_t h = kvh + (t / Tq) * Hkv,"),
    "causal-top-left": ("int64_t e = i + (int64_t)(z.Tk - z.Tq) + 1;", "int64_t e = i + 1;"),
    "window-ignores-offset": ("int64_t b = i + (int64_t)(z.Tk - z.Tq) - z.window + 1;", "int64_t b = i - z.window + 1;"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    if shutil.which("g++") is None:
        pytest.skip("no g++")
    src = open(oracle._SRC).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation anchor missing: {old}"
    mutant_src = tmp_path / "mutant.cpp"
    mutant_src.write_text(src.replace(old, new))
    out = str(tmp_path / "libmutant.so")
    oracle.build(force=True, src=str(mutant_src), out=out)
    lib = oracle.OracleLib(out)
    assert pin_suite(lib, quick=True) != [], f"planted mistake {name} went unnoticed"
