"""The C-ABI library loads and exports every symbol include/gdn_spec.h declares.

Runs without a GPU: it loads the shared library and inspects symbols and
constants only; no compute call is made.
"""
import ctypes
import os
import re

import pytest

from gated_delta_rule_spec_gb300 import binding
from gated_delta_rule_spec_gb300 import build as lib_build

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gdn_spec.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_spec_\w+)\s*\(", text)))


def _header_defines():
    out = {}
    for m in re.finditer(r"#define\s+(GDN_SPEC_\w+)\s+(-?\d+)u?", open(HEADER).read()):
        out[m.group(1)] = int(m.group(2))
    return out


@pytest.fixture(scope="module")
def lib():
    lib_build.build()
    return binding.load()


def test_every_declared_function_is_exported(lib):
    names = _declared_functions()
    assert set(names) == set(binding.EXPORTS), names
    for n in names:
        assert hasattr(lib, n), n


def test_host_only_calls(lib):
    assert lib.gdn_spec_abi_version() == _header_defines()["GDN_SPEC_ABI_VERSION"]
    assert lib.gdn_spec_strerror(0) == b"ok"
    assert b"invalid" in lib.gdn_spec_strerror(-1)
    # invalid descriptors are rejected on the host, before any CUDA call
    assert lib.gdn_spec_verify_path(None) is None
    bad = binding.LayerDesc(2, 3, 32, 32, 4, 8, 2, 0, 0, 1.0, 1e-6, 16, 16, 16, 16, 16)
    assert lib.gdn_spec_verify_path(ctypes.byref(bad)) is None
    assert lib.gdn_spec_verify(None, None, None, 0, *([None] * 8), None) == -1
    assert lib.gdn_spec_commit(None, 4, 8, None, 0, None, None) == -1


def test_python_constants_match_header():
    d = _header_defines()
    assert d["GDN_SPEC_GATE_SCALAR"] == binding.GATE_SCALAR
    assert d["GDN_SPEC_GATE_PER_KEY"] == binding.GATE_PER_KEY
    assert d["GDN_SPEC_DTYPE_BF16"] == binding.DTYPE_BF16
    assert d["GDN_SPEC_DTYPE_FP32"] == binding.DTYPE_FP32
    assert d["GDN_SPEC_ST_ACCEPT_RANGE"] == binding.ST_ACCEPT_RANGE
    assert d["GDN_SPEC_ST_SLOT_OOR"] == binding.ST_SLOT_OOR
    assert d["GDN_SPEC_ST_RING_OVERFLOW"] == binding.ST_RING_OVERFLOW
    assert d["GDN_SPEC_ST_CURSOR_CORRUPT"] == binding.ST_CURSOR_CORRUPT
    assert d["GDN_SPEC_ST_TIMEOUT"] == binding.ST_TIMEOUT
    assert d["GDN_SPEC_ST_UNFOLDED"] == binding.ST_UNFOLDED


def test_descriptor_layout_matches_header():
    # field order and sizes of the ctypes mirrors (9 int32 + 2 float + 5 pointers)
    assert ctypes.sizeof(binding.LayerDesc) == 9 * 4 + 2 * 4 + 4 + 5 * 8  # 4 bytes padding
    assert binding.LayerDesc.checkpoint.offset == 48
    assert ctypes.sizeof(binding.CursorDesc) == 8 + 4 * 8


def test_wait_limit_setter_is_host_only_and_restores_the_default(lib):
    """gdn_spec_set_wait_limit only records a number on the host (no CUDA call):
    it returns the previous limit, and 0xFFFFFFFF restores the default 2^20."""
    assert binding.set_wait_limit(7) == 1 << 20
    assert binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT) == 7
    assert binding.set_wait_limit(binding.WAIT_LIMIT_DEFAULT) == 1 << 20
