"""Host-side checks of the Python binding: the C library receives only
pointers, so the binding must refuse every tensor whose shape, dtype, layout
or device differs from what the kernels will index.  These run on the CPU and
stop before anything reaches the library."""
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import tiled_attention_05_gb300 as fa

bf = torch.bfloat16


def operands(B=1, Hq=4, Hkv=2, Tq=100, Tk=90, d=64, dv=64):
    Q = torch.zeros(B, Hq, Tq, d, dtype=bf)
    K = torch.zeros(B, Hkv, Tk, d, dtype=bf)
    V = torch.zeros(B, Hkv, Tk, dv, dtype=bf)
    O = torch.zeros(B, Hq, Tq, dv, dtype=bf)
    L = torch.zeros(B, Hq, Tq, dtype=torch.float32)
    return Q, K, V, O, O.clone(), L


@pytest.mark.parametrize("which, shape", [
    ("O", (1, 4, 100, 128)),     # dv of O differs from V's
    ("O", (1, 4, 99, 64)),
    ("dO", (1, 2, 100, 64)),
    ("L", (1, 4, 101)),
    ("L", (1, 4, 100, 1)),
])
def test_backward_rejects_misshapen_saved_state(which, shape):
    Q, K, V, O, dO, L = operands()
    args = dict(O=O, dO=dO, L=L)
    args[which] = torch.zeros(shape, dtype=torch.float32 if which == "L" else bf)
    with pytest.raises(ValueError, match=f"{which} has shape"):
        fa.fa_backward(Q, K, V, args["O"], args["dO"], args["L"], causal=False)


@pytest.mark.parametrize("which", ["dQ", "dK", "dV"])
def test_backward_rejects_misshapen_gradient_buffers(which):
    Q, K, V, O, dO, L = operands()
    bufs = dict(dQ=None, dK=None, dV=None)
    bufs[which] = torch.zeros(1, 4, 100, 32, dtype=bf)
    with pytest.raises(ValueError, match=f"{which} has shape"):
        fa.fa_backward(Q, K, V, O, dO, L, False, **bufs)
    with pytest.raises(ValueError, match=f"{which} has shape"):
        fa.fa_backward_noalloc(Q, K, V, O, dO, L, False, **bufs)


def test_forward_rejects_misshapen_outputs():
    Q, K, V, O, _, L = operands()
    with pytest.raises(ValueError, match="O has shape"):
        fa.fa_forward(Q, K, V, False, O=torch.zeros(1, 4, 100, 128, dtype=bf))
    with pytest.raises(ValueError, match="L has shape"):
        fa.fa_forward(Q, K, V, False, L=torch.zeros(1, 4, 128, dtype=torch.float32))


def test_inconsistent_inputs_rejected():
    Q, K, V, *_ = operands()
    with pytest.raises(ValueError, match="inconsistent"):
        fa.fa_forward(Q, K[:, :, :50], V, False)
    with pytest.raises(ValueError, match="inconsistent"):
        fa.fa_forward(Q, K[..., :32].contiguous(), V, False)
    with pytest.raises(ValueError, match=r"\[B, H, T, d\]"):
        fa.fa_forward(Q[0], K, V, False)


def test_host_tensors_wrong_dtype_and_views_rejected():
    Q, K, V, O, dO, L = operands()
    with pytest.raises(ValueError, match="contiguous CUDA"):
        fa.fa_forward(Q, K, V, False)                       # host memory: no CPU path
    with pytest.raises(ValueError, match="contiguous CUDA"):
        fa.fa_forward(Q.float(), K, V, False)
    with pytest.raises(ValueError, match="contiguous CUDA"):
        fa.fa_backward(Q, K, V, O, dO, L, False)
    Qt = torch.zeros(1, 4, 64, 100, dtype=bf).transpose(2, 3)  # right shape, not contiguous
    with pytest.raises(ValueError, match="contiguous CUDA"):
        fa.fa_forward(Qt, K, V, False)


def test_missing_library_fails_loudly(tmp_path):
    """With no built library and no compiler, loading raises instead of
    falling back to anything else."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    child = textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {root!r})
        import tiled_attention_05_gb300.build as b
        b.OUT_DIR = {str(tmp_path)!r}
        b.LIB = {str(tmp_path / "libfa_gb300.so")!r}
        import tiled_attention_05_gb300 as fa
        try:
            fa.load()
        except Exception as e:
            print("RAISED", type(e).__name__)
        else:
            print("LOADED")
    """)
    env = dict(os.environ, NVCC=str(tmp_path / "no-such-nvcc"))
    r = subprocess.run([sys.executable, "-c", child], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "RAISED" in r.stdout and "LOADED" not in r.stdout
