"""Failure detection without a GPU fault: every on-chip wait in the kernels is
bounded.  The library's failure-path test build (libfa_gb300_testhooks.so,
compiled with FA_TEST_HOOKS; the product library has no such switch) can make
a producer withhold one load -- a barrier that nothing completes:

* forward: the Q tile is never loaded, so no MMA can start;
* backward: no dO tile is loaded, so dP^T and dV never start while S^T, the
  P phase and the other roles run up to their waits.

Both head sizes run it: at d = 64 the backward also takes the path where
other roles vouch for the MMA thread's checks.

Every wait then expires (about 2 s) or sees the CTA's abort flag, the CTA
skips its remaining work, lets copies and MMAs already in flight land, frees
its tensor memory and records FA_ERR_TIMEOUT in the device status word.  The
same process then runs a correct forward and backward pass, checked against
the float64 oracle, so the context stays usable."""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import ctypes, sys, time, torch
    sys.path.insert(0, {root!r})
    import tiled_attention_05_gb300 as fa
    from tiled_attention_05_gb300 import build as fa_build
    import oracle
    from tiled_attention_05_gb300.inputs import make_custom
    from tests.parity import assert_close, assert_L_close
    lib = fa.load(fa_build.build_test_hooks())
    lib.fa_test_set_withhold.argtypes = [ctypes.c_int]
    lib.fa_test_set_withhold.restype = None
    Q, K, V, dO = make_custom(1, 4, 2, 300, 333, {d}, True, seed=5)
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = Q.to(dev), K.to(dev), V.to(dev), dO.to(dev)

    def timed_status():
        t0 = time.perf_counter()
        s = fa.fa_last_device_status()
        return s, time.perf_counter() - t0

    lib.fa_test_set_withhold(1)            # forward: withhold Q
    fa.fa_forward(Qd, Kd, Vd, True)
    s_fwd, t_fwd = timed_status()
    lib.fa_test_set_withhold(0)
    O, L = fa.fa_forward(Qd, Kd, Vd, True)
    s_fwd_ok, _ = timed_status()
    lib.fa_test_set_withhold(2)            # backward: withhold dO
    fa.fa_backward(Qd, Kd, Vd, O, dOd, L, True)
    s_bwd, t_bwd = timed_status()
    lib.fa_test_set_withhold(0)
    dQ, dK, dV = fa.fa_backward(Qd, Kd, Vd, O, dOd, L, True)
    s_bwd_ok, _ = timed_status()
    Or, Lr = oracle.forward(Q, K, V, True)
    dQr, dKr, dVr, _ = oracle.backward(Q, K, V, dO, True)
    assert_close("O", O.cpu(), Or)
    assert_L_close("L", L.cpu(), Lr)
    for n, g, r in (("dQ", dQ, dQr), ("dK", dK, dKr), ("dV", dV, dVr)):
        assert_close(n, g.cpu(), r)
    print("STATUS", s_fwd, s_fwd_ok, s_bwd, s_bwd_ok, f"{{t_fwd:.2f}}", f"{{t_bwd:.2f}}")
""")


@pytest.mark.gpu
@pytest.mark.parametrize("d", [64, 128])
def test_withheld_loads_time_out_and_context_survives(d):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, d=d)], cwd=ROOT, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    _, s_fwd, s_fwd_ok, s_bwd, s_bwd_ok, t_fwd, t_bwd = line.split()
    import tiled_attention_05_gb300 as fa

    assert int(s_fwd) == fa.FA_ERR_TIMEOUT
    assert int(s_fwd_ok) == fa.FA_OK
    assert int(s_bwd) == fa.FA_ERR_TIMEOUT
    assert int(s_bwd_ok) == fa.FA_OK
    # the waits give up after about 2 s (plus the exit path's bounded drains)
    assert float(t_fwd) < 10.0 and float(t_bwd) < 10.0, line


def test_only_the_test_build_has_the_withhold_switch():
    """The switch is compiled into the failure-path test build alone."""
    from tiled_attention_05_gb300 import build as fa_build

    prod = ctypes.CDLL(fa_build.build())
    hooks = ctypes.CDLL(fa_build.build_test_hooks())
    assert not hasattr(prod, "fa_test_set_withhold")
    assert hasattr(hooks, "fa_test_set_withhold")
