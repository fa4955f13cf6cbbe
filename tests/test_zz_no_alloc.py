"""fa_backward_noalloc: the backward pass for callers that cannot allocate
device memory (code running inside a host framework that hands it only its
inputs and outputs, or a loop that must not call cudaMalloc).  It takes no
workspace and uses the library's fixed scratch array instead.

Checked through the C ABI against fa_backward (which gets a workspace from the
caller) on two calls in a row with different problems, so the second call
runs on scratch the first one left behind.  This file is named to be
collected last.
"""
import ctypes

import pytest
import torch

from tests.parity import assert_close
from tiled_attention_05_gb300.inputs import make_custom

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tiled_attention_05_gb300 as lib

    lib.load()
    return lib


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc_via_abi(fa, dims, Q, K, V, O, dO, L):
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    code = fa.load().fa_backward_noalloc(ctypes.byref(dims), _ptr(Q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(L),
                                         _ptr(dQ), _ptr(dK), _ptr(dV),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == fa.FA_OK, fa.status_string(code)
    return dQ, dK, dV


@pytest.mark.parametrize("first,second", [
    ((1, 8, 2, 1000, 1000, 128, True), (2, 4, 4, 333, 517, 64, False)),
])
def test_noalloc_matches_backward_twice(fa, first, second):
    dev = torch.device("cuda")
    for shape in (first, second):
        B, Hq, Hkv, Tq, Tk, d, causal = shape
        Q, K, V, dO = (t.to(dev) for t in make_custom(B, Hq, Hkv, Tq, Tk, d, causal, seed=Tq + Tk))
        dims = fa.make_dims(B, Hq, Hkv, Tq, Tk, d, d, causal, None)
        assert fa.fa_backward_workspace_min_bytes(dims) <= fa.FA_NOALLOC_SCRATCH_BYTES
        O, L = fa.fa_forward(Q, K, V, causal)
        ref = fa.fa_backward(Q, K, V, O, dO, L, causal)
        got = _noalloc_via_abi(fa, dims, Q, K, V, O, dO, L)
        torch.cuda.synchronize()
        assert fa.fa_last_device_status() == fa.FA_OK
        for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
            assert_close(f"{name} {shape}", g.cpu(), r.double().cpu().numpy())


def test_noalloc_rejects_problems_beyond_its_scratch(fa):
    # 2 x 32 heads x 8192 rows needs ~272 MB of workspace: refused before anything is enqueued.
    dims = fa.make_dims(2, 32, 8, 8192, 8192, 128, 128, True, None)
    assert fa.fa_backward_workspace_min_bytes(dims) > fa.FA_NOALLOC_SCRATCH_BYTES
    p = [ctypes.c_void_p(0x1000 * (i + 1)) for i in range(9)]
    code = fa.load().fa_backward_noalloc(ctypes.byref(dims), *p, None)
    assert code == fa.FA_ERR_SCRATCH_TOO_SMALL
    assert "fa_backward" in fa.status_string(code)
