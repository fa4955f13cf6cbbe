"""The forward and backward calls inside a captured CUDA graph.

Both calls only enqueue work on the caller's stream (no host synchronisation,
no allocation by the library), so a training step can capture them once and
replay the graph.  The test captures forward + backward on static buffers,
then replays the graph on fresh inputs copied into those buffers and checks
every output of every replay against the float64 oracle.  It covers both
backward variants (d = 64 with the deeper rings, d = 128) and a non-causal
shape whose short last round runs split work items.
"""
import pytest
import torch

import oracle
from tests.parity import assert_close, assert_L_close
from tiled_attention_05_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tiled_attention_05_gb300 as lib

    lib.load()
    return lib


@pytest.mark.parametrize("shape", [(1, 4, 2, 300, 300, 64, True), (1, 4, 2, 300, 300, 128, True),
                                   (1, 3, 1, 200, 385, 64, False)],
                         ids=lambda s: "x".join(map(str, s)))
def test_forward_and_backward_replay_in_a_cuda_graph(fa, shape):
    B, Hq, Hkv, Tq, Tk, d, causal = shape
    dev = torch.device("cuda")
    static = [t.to(dev) for t in make_custom(B, Hq, Hkv, Tq, Tk, d, causal, seed=1)]
    sQ, sK, sV, sdO = static

    # warm-up on a side stream (first-call set-up happens outside the capture)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        O, L = fa.fa_forward(sQ, sK, sV, causal)
        fa.fa_backward(sQ, sK, sV, O, sdO, L, causal)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gO, gL = fa.fa_forward(sQ, sK, sV, causal)
        gdQ, gdK, gdV = fa.fa_backward(sQ, sK, sV, gO, sdO, gL, causal)

    for seed in (2, 3):
        host = make_custom(B, Hq, Hkv, Tq, Tk, d, causal, seed=seed)
        for dst, src in zip(static, host):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        Q, K, V, dO = host
        Or, Lr = oracle.forward(Q, K, V, causal)
        dQr, dKr, dVr, _ = oracle.backward(Q, K, V, dO, causal)
        assert_close(f"O seed {seed}", gO.cpu(), Or)
        assert_L_close(f"L seed {seed}", gL.cpu(), Lr)
        for name, got, ref in (("dQ", gdQ, dQr), ("dK", gdK, dKr), ("dV", gdV, dVr)):
            assert_close(f"{name} seed {seed}", got.cpu(), ref)
