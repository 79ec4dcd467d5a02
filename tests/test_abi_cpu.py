"""C-ABI checks that need no GPU: the library builds, loads, exports every
function include/pe.h declares, and rejects bad arguments on the host."""

import ctypes
import os
import re

import pytest

from speculative_drafting_pe_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared():
    text = open(HEADER).read()
    return re.findall(r"^(?:int|void|const char\s*\*)\s+(pe_\w+)\s*\(", text, re.M)


def test_header_declares_the_expected_entry_points():
    names = set(_declared())
    assert {"pe_init_drafter", "pe_draft", "pe_verify_rebuild", "pe_destroy", "pe_last_error"} <= names
    assert names == set(binding.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_abi_version(lib):
    assert lib.pe_abi_version() == 1


def _cfg(**over):
    c = dict(hidden=256, n_layers=4, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=512, vocab=4096,
             rms_eps=1e-6, rope_theta=1e4, page_size=16, k_max=3, dtype=binding.PE_DTYPE_FP32)
    c.update(over)
    return binding.PeConfig(**c)


@pytest.mark.parametrize("over,code", [
    (dict(n_layers=3), -2), (dict(page_size=8), -2), (dict(head_dim=96), -2), (dict(n_kv_heads=3), -2),
    (dict(k_max=0), -2), (dict(k_max=17), -2), (dict(hidden=100), -2), (dict(dtype=7), -1),
    (dict(n_q_heads=2, n_kv_heads=1), -2),   # 2*64 q rows is fine, 1*64 kv rows is not a multiple of 128
])
def test_init_rejects_bad_config_before_touching_a_device(lib, over, code):
    w = binding.PeWeights()
    h = ctypes.c_void_p()
    rc = lib.pe_init_drafter(ctypes.byref(_cfg(**over)), ctypes.byref(w), 1, 0, ctypes.byref(h))
    assert rc == code, lib.pe_last_error()
    assert h.value is None
    assert len(lib.pe_last_error()) > 0


def test_init_rejects_null_weights(lib):
    w = binding.PeWeights()
    h = ctypes.c_void_p()
    assert lib.pe_init_drafter(ctypes.byref(_cfg()), ctypes.byref(w), 1, 0, ctypes.byref(h)) == -1
    assert b"null" in lib.pe_last_error()
    assert lib.pe_init_drafter(None, ctypes.byref(w), 1, 0, ctypes.byref(h)) == -1


def test_draft_and_verify_reject_bad_arguments(lib):
    p = ctypes.c_void_p(16)
    assert lib.pe_draft(None, 1, 1, p, p, p, p, p, 1, 1, p, p, p, None, p, None) == -1
    # K outside 1..31 and B < 1 fail before any launch
    args = [p, p, p, 1, 1, p, p, p, p, p, p, None, p, p, p, None]
    assert lib.pe_verify_rebuild(None, 4, 0, *args) == -1
    assert lib.pe_verify_rebuild(None, 4, 32, *args) == -1
    assert lib.pe_verify_rebuild(None, 0, 4, *args) == -1
    nul = [None, None, None, 1, 1] + [None] * 11
    assert lib.pe_verify_rebuild(None, 4, 4, *nul) == -1
    assert lib.pe_last_launch_count(None) == 0
    lib.pe_destroy(None)
