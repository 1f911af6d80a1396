"""The C-ABI library builds for sm_103a, loads, and exports every symbol that
include/moe.h declares.  Host-only calls (sizes, argument validation) run here;
nothing touches a GPU.  CPU only."""
import ctypes
import os
import re
import shutil

import pytest

import moe_expert_layer_softmax_gb300 as m
from moe_expert_layer_softmax_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    _build.build()
    return m.load()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "moe.h")) as fh:
        text = fh.read()
    return sorted(set(re.findall(r"MOE_API\s+int\s+(moe_\w+)\s*\(", text)))


def test_header_and_binding_agree():
    assert declared_symbols() == sorted(m.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_rows_max_and_workspace(lib):
    s = m.shape(8192, 2048, 32, 4, 1024)
    assert m.rows_max(s) == ((8192 * 4 + 32 * 127 + 127) // 128) * 128
    assert m.rows_max(s) % 128 == 0
    ws = m.workspace_size(s)
    assert ws >= 256 + (8192 // 64) * 32 * 4 + 8192 * 4 * 4
    s1 = m.shape(1, 128, 1, 1, 128)
    assert m.rows_max(s1) == 128


@pytest.mark.parametrize("bad,code", [
    ((0, 128, 8, 2, 128), -1),        # T < 1
    ((16, 128, 8, 9, 128), -1),       # k > E
    ((16, 100, 8, 2, 128), -2),       # d not a multiple of 128
    ((16, 128, 8, 2, 200), -2),       # f not a multiple of 128
    ((16, 128, 300, 2, 128), -2),     # E > 256
    ((16, 128, 64, 33, 128), -2),     # k > 32
])
def test_shape_validation(lib, bad, code):
    with pytest.raises(m.MoEError) as ei:
        m.rows_max(m.shape(*bad))
    assert ei.value.code == code


def test_bad_precision_is_rejected(lib):
    with pytest.raises(m.MoEError) as ei:
        m.workspace_size(m.shape(16, 128, 8, 2, 128, prec=7))
    assert ei.value.code == -1


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="no CPU or eager fallback"):
        m._lib_saved = m._lib
        try:
            m._lib = None
            m.load(str(tmp_path / "nope.so"))
        finally:
            m._lib = m._lib_saved
