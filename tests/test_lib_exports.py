"""The C-ABI library builds, loads, and exports every function the header
declares; host-only entry points answer without a GPU."""

import ctypes
import os
import re

import pytest

from speculative_decoding_verification_07_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(binding.LIB_PATH):
        from speculative_decoding_verification_07_gb300 import build
        build.build()
    return binding.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:sv_status|size_t)\s+(\w+)\s*\(", text, flags=re.M)
    assert names, "no declarations found"
    return names


def test_every_declared_function_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
    assert set(_declared_functions()) == set(binding.EXPORTS)


def test_struct_layout_matches(lib):
    assert lib.sv_verify_args_size() == ctypes.sizeof(binding.SvVerifyArgs)


def test_workspace_size_is_host_only(lib):
    a = binding.SvVerifyArgs()
    a.B, a.kmax = 64, 4
    n = ctypes.c_size_t()
    assert lib.sv_workspace_size(ctypes.byref(a), ctypes.byref(n)) == 0
    assert n.value >= 64 * 5 * 4 and n.value % 256 == 0
    a.B = -1
    assert lib.sv_workspace_size(ctypes.byref(a), ctypes.byref(n)) == binding.SV_ERR_INVALID


def test_null_handle_is_rejected_before_any_launch(lib):
    a = binding.SvVerifyArgs()
    assert lib.spec_verify(None, ctypes.byref(a), None, 0, None) == binding.SV_ERR_INVALID
    st = binding.BflState()
    assert lib.bfl_init(None, ctypes.byref(st), None) == binding.SV_ERR_INVALID
    assert lib.kv_rollback_contig(None, 1, None, None, None) == binding.SV_ERR_INVALID


def test_flag_and_status_constants_match_header():
    """The binding's flag and status constants are the header's values (the
    kernel selection flags included)."""
    text = open(HEADER).read()
    defs = dict(re.findall(r"#define\s+(SV_(?:FLAG|ST)_\w+)\s+(\d+)u", text))
    assert "SV_FLAG_STREAM_PATH" in defs and "SV_FLAG_CLUSTER_PATH" in defs
    for name, value in defs.items():
        py = name[3:]  # SV_FLAG_X -> FLAG_X, SV_ST_X -> ST_X
        assert getattr(binding, py) == int(value), name
