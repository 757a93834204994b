"""The C-ABI library builds, loads and exports every function the header
declares; host-only entry points validate their arguments without a GPU."""
import ctypes
import os
import re

import pytest

from sparse_moe_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sparse_moe.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    return _abi.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("moe_ctx_create", "moe_load_weights", "moe_route", "moe_forward_prefill",
                     "moe_forward_decode"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_binding_covers_every_declared_symbol():
    assert set(declared_functions()) == set(_abi.SIGNATURES)


def _cfg(**kw):
    base = dict(hidden=2048, n_experts=256, top_k=8, inter=512, shared_inter=512, n_layers=1,
                max_chunk_rows=4096, wfmt=0)
    base.update(kw)
    return _abi.MoeConfig(*[base[n] for n, _ in _abi.MoeConfig._fields_])


def test_workspace_size_host_only(lib):
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(_cfg()), ctypes.byref(n)) == _abi.MOE_OK
    # at least h (bf16) and o (bf16) for T*k + T grouped rows of a 4096-row chunk
    R = 4096 * 8 + 4096
    assert n.value >= R * 512 * 2 + R * 2048 * 2
    small = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(_cfg(max_chunk_rows=16)), ctypes.byref(small)) == 0
    assert small.value < n.value


@pytest.mark.parametrize("bad", [dict(hidden=100), dict(hidden=0), dict(n_experts=0),
                                 dict(n_experts=2048), dict(top_k=0), dict(top_k=300),
                                 dict(n_experts=4, top_k=5), dict(inter=96), dict(shared_inter=0),
                                 dict(n_layers=0), dict(max_chunk_rows=0),
                                 dict(max_chunk_rows=1 << 20), dict(wfmt=7)])
def test_invalid_configs_rejected(lib, bad):
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(ctypes.byref(_cfg(**bad)), ctypes.byref(n)) == \
        _abi.MOE_ERR_INVALID_ARG


def test_null_arguments_rejected(lib):
    n = ctypes.c_size_t()
    assert lib.moe_workspace_size(None, ctypes.byref(n)) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_workspace_size(ctypes.byref(_cfg()), None) == _abi.MOE_ERR_INVALID_ARG
    h = ctypes.c_void_p()
    # no workspace: rejected before any device call
    assert lib.moe_ctx_create(ctypes.byref(_cfg()), 0, None, 0, ctypes.byref(h)) == \
        _abi.MOE_ERR_WORKSPACE
    assert lib.moe_ctx_create(ctypes.byref(_cfg()), 0, ctypes.c_void_p(0x1001), 1 << 40,
                              ctypes.byref(h)) == _abi.MOE_ERR_WORKSPACE   # misaligned
    assert lib.moe_ctx_destroy(None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_prefill(None, 0, None, 1, None, None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_forward_decode(None, 0, None, None, None) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_route(None, 0, None, 1, None, None, None, None, None, None, None, None) == \
        _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_load_weights(None, 0, None) == _abi.MOE_ERR_INVALID_ARG
    w, m = ctypes.c_double(0.0), ctypes.c_double(0.0)
    assert lib.moe_decode_phase_read(None, ctypes.byref(w), ctypes.byref(m)) == \
        _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_profile_enable(None, 1) == _abi.MOE_ERR_INVALID_ARG
    assert lib.moe_launch_count(None) == 0
    assert lib.moe_last_error(None) == b""
    assert lib.moe_status_string(_abi.MOE_ERR_DEVICE_TIMEOUT) == b"device-side wait timed out"
