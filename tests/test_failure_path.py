"""Failure detection without a GPU fault: every on-chip wait in the kernels is
bounded.  A test-only switch (FA_TEST_WITHHOLD_Q=1) makes the forward's
producer withhold the Q tile -- a barrier that nothing completes.  The waits
expire (about 2 s), the kernel stops, the device status word reports
FA_ERR_TIMEOUT, and the same process then runs a correct forward pass."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys, torch
    sys.path.insert(0, {root!r})
    import tiled_attention_05_gb300 as fa
    import oracle
    from tiled_attention_05_gb300.inputs import make_custom
    from tests.parity import assert_close
    Q, K, V, dO = make_custom(1, 2, 1, 200, 300, 128, True, seed=5)
    dev = torch.device("cuda")
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    os.environ["FA_TEST_WITHHOLD_Q"] = "1"
    fa.fa_forward(Qd, Kd, Vd, True)
    s1 = fa.fa_last_device_status()
    os.environ["FA_TEST_WITHHOLD_Q"] = "0"
    O, L = fa.fa_forward(Qd, Kd, Vd, True)
    s2 = fa.fa_last_device_status()
    Or, Lr = oracle.forward(Q, K, V, True)
    assert_close("O", O.cpu(), Or)
    print("STATUS", s1, s2)
""")


@pytest.mark.gpu
def test_withheld_tile_times_out_and_context_survives():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ)
    env.pop("FA_TEST_WITHHOLD_Q", None)
    r = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT)], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("STATUS")][-1]
    _, s1, s2 = line.split()
    import tiled_attention_05_gb300 as fa

    assert int(s1) == fa.FA_ERR_TIMEOUT
    assert int(s2) == fa.FA_OK
