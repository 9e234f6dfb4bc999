"""The C-ABI library loads, exports every call include/pa.h declares, and
rejects bad arguments on the host before anything reaches a GPU."""
import ctypes
import os
import re

import pytest
import torch

import paged_kv_attention_04_gb300 as P
from paged_kv_attention_04_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_attention_04_gb300 import build
    build.build()
    return P.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pa_cache_write", "pa_forward", "pa_forward_workspace_size", "pa_last_error"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_version(lib):
    assert lib.pa_version() >= 100


def L(**kw):
    base = dict(num_q_heads=32, num_kv_heads=8, head_size=128, num_blocks=100, dtype=torch.bfloat16)
    base.update(kw)
    return P.make_layout(**base)


def test_workspace_size_grows_with_bounds(lib):
    lay = L()
    a = P.pa_forward_workspace_size(lay, 4, 4, 64)
    b = P.pa_forward_workspace_size(lay, 4, 4, 8192)
    c = P.pa_forward_workspace_size(lay, 4, 600, 8192)
    assert 0 < a < b < c
    assert a % 256 == 0


@pytest.mark.parametrize("bad,code", [
    (dict(head_size=96), P.PA_ERR_UNSUPPORTED),
    (dict(num_q_heads=48, num_kv_heads=3), P.PA_ERR_UNSUPPORTED),   # group 16
    (dict(num_q_heads=30, num_kv_heads=8), P.PA_ERR_INVALID),       # not a multiple
    (dict(num_blocks=0), P.PA_ERR_INVALID),
])
def test_bad_layouts_rejected(lib, bad, code):
    lay = L(**bad)
    assert lib.pa_forward_workspace_size(ctypes.byref(lay), 4, 4, 64) == 0
    rc = lib.pa_cache_write(16, 16, 16, 1, 16, 16, ctypes.byref(lay), None, None)
    assert rc == code
    assert P.last_error()


def test_bad_block_size_rejected(lib):
    lay = L()
    lay.block_size = 32
    assert lib.pa_cache_write(16, 16, 16, 1, 16, 16, ctypes.byref(lay), None, None) == \
        P.PA_ERR_UNSUPPORTED


def test_cache_write_argument_checks(lib):
    lay = L()
    assert lib.pa_cache_write(None, None, None, 0, None, None, ctypes.byref(lay), None, None) == P.PA_OK
    assert lib.pa_cache_write(None, 16, 16, 3, 16, 16, ctypes.byref(lay), None, None) == P.PA_ERR_INVALID
    assert lib.pa_cache_write(24, 16, 16, 3, 16, 16, ctypes.byref(lay), None, None) == P.PA_ERR_INVALID
    assert "aligned" in P.last_error()
    assert lib.pa_cache_write(16, 16, 16, -1, 16, 16, ctypes.byref(lay), None, None) == P.PA_ERR_INVALID
    assert lib.pa_cache_write(16, 16, 16, 1, 16, 16, None, None, None) == P.PA_ERR_INVALID


def _fwd(lib, lay, **over):
    a = dict(q=256, kc=256, vc=256, bt=256, maxb=4, sl=256, qsl=256, B=2, T=2, maxq=1, maxs=64,
             scale=0.125, out=256, ws=256, wsb=1 << 30, status=None)
    a.update(over)
    return lib.pa_forward(a["q"], a["kc"], a["vc"], a["bt"], a["maxb"], a["sl"], a["qsl"], a["B"],
                          a["T"], a["maxq"], a["maxs"], ctypes.c_float(a["scale"]), a["out"],
                          a["ws"], a["wsb"], ctypes.byref(lay), a["status"], None)


def test_forward_argument_checks(lib):
    lay = L()
    assert _fwd(lib, lay, B=0, T=0) == P.PA_OK                      # empty step
    assert _fwd(lib, lay, q=None) == P.PA_ERR_INVALID
    assert _fwd(lib, lay, ws=None) == P.PA_ERR_INVALID
    assert _fwd(lib, lay, q=264) == P.PA_ERR_INVALID                # misaligned q
    assert _fwd(lib, lay, ws=272) == P.PA_ERR_INVALID               # misaligned workspace
    assert _fwd(lib, lay, wsb=1024) == P.PA_ERR_INVALID             # workspace too small
    assert "workspace" in P.last_error()
    assert _fwd(lib, lay, maxb=3) == P.PA_ERR_INVALID               # table narrower than 64/16
    assert _fwd(lib, lay, scale=float("nan")) == P.PA_ERR_INVALID
    assert _fwd(lib, lay, T=1) == P.PA_ERR_INVALID                  # fewer tokens than requests
    assert _fwd(lib, lay, maxq=0) == P.PA_ERR_INVALID
    assert _fwd(lib, lay, B=-1) == P.PA_ERR_INVALID


def test_binding_raises_with_message(lib):
    lay = L(head_size=96)
    with pytest.raises(P.PaError) as ei:
        P.pa_forward_workspace_size(lay, 1, 1, 16)
    assert "head_size" in str(ei.value)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "LIB_PATH", str(tmp_path / "libpa.so"))
    monkeypatch.setattr(binding, "_lib", None)
    with pytest.raises(RuntimeError, match="missing"):
        binding.lib()


def test_binding_rejects_host_tensors():
    """A host tensor is refused before any call into the library."""
    import torch
    lay = P.make_layout(8, 2, 64, 4, torch.bfloat16)
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16)
    e = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(P.PaError, match="not a CUDA tensor"):
        P.pa_cache_write(e, e, torch.zeros(1, dtype=torch.int64), kc, kc, lay)
    with pytest.raises(P.PaError, match="not a CUDA tensor"):
        P.pa_forward(e, kc, kc, torch.zeros(1, 1, dtype=torch.int32),
                     torch.ones(1, dtype=torch.int32), torch.tensor([0, 1], dtype=torch.int32),
                     1, 1, 0.125, e, torch.zeros(16, dtype=torch.uint8), lay)
