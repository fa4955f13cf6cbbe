"""Host-side checks of the C ABI that need no GPU: the library builds, loads and
exports every symbol include/fa.h declares; argument validation rejects bad
calls before anything reaches the device; the workspace query matches its
documented size."""
import ctypes
import os
import re

import pytest

import tiled_attention_05_gb300 as fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    return sorted(set(re.findall(r"FA_API\s+[\w\s\*]+?\b(fa_\w+)\s*\(", text)))


def test_header_declares_the_binding_names():
    assert declared_symbols() == sorted(fa.EXPORTED_SYMBOLS)


def test_library_loads_and_exports_every_declared_symbol():
    lib = fa.load()
    raw = ctypes.CDLL(fa.lib_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name
    assert lib is not None


def test_status_strings():
    for code in range(5):
        s = fa.status_string(code)
        assert isinstance(s, str) and s
    assert fa.status_string(0) == "ok"
    assert "unknown" in fa.status_string(99)


def dims(**kw):
    base = dict(B=1, Hq=4, Hkv=2, Tq=100, Tk=90, d=128, dv=128, causal=0, scale=0.0, window=0)
    base.update(kw)
    return fa.FaDims(base["B"], base["Hq"], base["Hkv"], base["Tq"], base["Tk"], base["d"], base["dv"],
                     base["causal"], base["scale"], base["window"])


def call_fwd(d, ptrs=(0x1000, 0x2000, 0x3000, 0x4000, 0x5000)):
    q, k, v, o, l = ptrs
    return fa.load().fa_forward(ctypes.byref(d), q, k, v, o, l, None)


@pytest.mark.parametrize("bad", [
    dict(Hq=3, Hkv=2),       # Hq not a multiple of Hkv
    dict(Hkv=0),             # no kv heads for non-empty Hq
    dict(B=-1),
    dict(Tq=-5),
    dict(causal=2),
    dict(window=64),         # a window needs the causal mask
    dict(causal=1, window=-1),
    dict(scale=float("nan")),
    dict(scale=float("inf")),
])
def test_invalid_dims_rejected(bad):
    assert call_fwd(dims(**bad)) == fa.FA_ERR_INVALID_ARG


@pytest.mark.parametrize("bad", [dict(d=96, dv=96), dict(d=64, dv=96), dict(d=256, dv=256), dict(d=128, dv=32),
                                 dict(Tq=65535 * 256 + 1),                       # Tq size limit
                                 dict(B=1 << 12, Hq=1 << 12, Hkv=1 << 12, Tk=1 << 20)])  # backward grid limit
def test_unsupported_dims(bad):
    assert call_fwd(dims(**bad)) == fa.FA_ERR_UNSUPPORTED


def test_null_and_misaligned_pointers_rejected():
    assert call_fwd(dims(), (0, 0x2000, 0x3000, 0x4000, 0x5000)) == fa.FA_ERR_INVALID_ARG
    assert call_fwd(dims(), (0x1002, 0x2000, 0x3000, 0x4000, 0x5000)) == fa.FA_ERR_INVALID_ARG
    assert call_fwd(dims(), (0x1000, 0x2000, 0x3000, 0x4000, 0x5008)) == fa.FA_ERR_INVALID_ARG


def test_zero_sized_problems_are_noops():
    # nothing to compute: returns before touching the device (null pointers allowed for empty tensors)
    assert call_fwd(dims(B=0), (0, 0, 0, 0, 0)) == fa.FA_OK
    assert call_fwd(dims(Tq=0), (0, 0x2000, 0x3000, 0, 0)) == fa.FA_OK
    assert call_fwd(dims(Hq=0, Hkv=0), (0, 0, 0, 0, 0)) == fa.FA_OK


def test_backward_workspace_validation():
    lib = fa.load()
    d = dims()
    need = fa.fa_backward_workspace_min_bytes(d)
    assert 0 < need < fa.fa_backward_workspace_bytes(d)  # non-causal: the split area is optional
    p = [0x1000 * (i + 1) for i in range(9)]
    # too small, misaligned, null workspace
    for ws, nbytes in ((0x100000, need - 1), (0x100010, need), (0, need)):
        assert lib.fa_backward(ctypes.byref(d), *p, ws, nbytes, None) == fa.FA_ERR_INVALID_ARG


def test_workspace_size_formula():
    up = lambda x: (x + 255) // 256 * 256
    for B, Hq, Tq, Tk, dd, causal, window in ((1, 1, 256, 50, 64, 0, 0), (2, 32, 8192, 8192, 128, 1, 0),
                                              (1, 32, 4096, 8032, 128, 0, 0), (3, 5, 1, 50, 64, 0, 0),
                                              (1, 32, 8192, 8192, 128, 1, 2080), (40, 8, 128, 9000, 64, 0, 0)):
        d = dims(B=B, Hq=Hq, Hkv=1, Tq=Tq, Tk=Tk, d=dd, dv=dd, causal=causal, window=window)
        rows = B * Hq * ((Tq + 127) // 128) * 128
        base = up(up(up(rows * dd * 4) + rows * 4) + rows * 4)
        # key tiles that may be split in two: equal-work items only (no causal mask)
        cap = min(B * 1 * ((Tk + 127) // 128), 128) if not causal else 0
        want = up(base + cap * 2 * 128 * (2 * dd) * 4) + cap * 4
        assert fa.fa_backward_workspace_bytes(d) == up(want)
        assert fa.fa_backward_workspace_min_bytes(d) == base
    assert fa.fa_backward_workspace_bytes(dims(Hq=3, Hkv=2)) == 0
    assert fa.fa_backward_workspace_min_bytes(dims(Hq=3, Hkv=2)) == 0


def test_binding_constants_match_the_header():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    enum = dict((k, int(v)) for k, v in re.findall(r"\b(FA_[A-Z_]+)\s*=\s*(\d+)", text))
    for name in ("FA_OK", "FA_ERR_INVALID_ARG", "FA_ERR_UNSUPPORTED", "FA_ERR_CUDA", "FA_ERR_TIMEOUT",
                 "FA_ERR_SCRATCH_TOO_SMALL", "FA_BWD_PRE", "FA_BWD_MAIN", "FA_BWD_CAST", "FA_BWD_ALL"):
        assert getattr(fa, name) == enum[name], name
    m = re.search(r"#define\s+FA_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m and fa.FA_NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))
    # field order and types of fa_dims as the binding lays them out
    body = re.search(r"typedef struct \{(.*?)\} fa_dims;", text, re.S).group(1)
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    fields = []
    for decl in body.split(";"):
        decl = decl.strip()
        if decl:
            typ, names = decl.split(None, 1)
            fields += [(n.strip(), typ) for n in names.split(",")]
    ctypes_of = {"int": ctypes.c_int, "float": ctypes.c_float}
    assert [(n, ctypes_of[t]) for n, t in fields] == [(n, t) for n, t in fa.FaDims._fields_]
