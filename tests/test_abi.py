"""The C ABI library builds, loads without a GPU and exports every symbol the header declares."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cacheblend.h")


def _declared():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:cb_status|const char\*|int32_t)\s+(cb_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib_path():
    from rag_kv_cache_gb300.build import build

    return build()


def test_header_declares_the_blend_calls():
    names = _declared()
    for n in ("cb_rope_rerotate", "cb_kv_deviation", "cb_hkvd_topk", "cb_fuse_scatter", "cb_hkvd_attention",
              "cb_blend_layer", "cb_plan_create", "cb_plan_destroy", "cb_check"):
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(cb_\w+)$", out, flags=re.M))
    assert set(_declared()) <= exported, set(_declared()) - exported
    lib = ctypes.CDLL(lib_path)
    for n in _declared():
        assert hasattr(lib, n)


def test_binding_lists_match_header(lib_path):
    from rag_kv_cache_gb300 import _lib

    assert sorted(_lib.EXPORTS) == _declared()
    lib = _lib.load(lib_path)
    assert lib.cb_version() == 100


def test_host_validation_without_gpu(lib_path):
    # argument checks run on the host before any CUDA call, so they work with no device
    from rag_kv_cache_gb300 import _lib

    lib = _lib.load(lib_path)
    h = ctypes.c_void_p()
    bad = _lib.CbConfig(2, 256, 32, 4, 3, 64, 1e4, 0, 15, 15)  # hq not a multiple of hkv
    assert lib.cb_plan_create(ctypes.byref(bad), ctypes.byref(h)) == 1
    assert b"multiple" in lib.cb_last_error_string()
    bad = _lib.CbConfig(2, 256, 32, 4, 2, 96, 1e4, 0, 15, 15)  # head_dim 96
    assert lib.cb_plan_create(ctypes.byref(bad), ctypes.byref(h)) == 2
    bad = _lib.CbConfig(2, 256, 32, 4, 2, 64, 1e4, 0, 10, 20)  # r2 > r1
    assert lib.cb_plan_create(ctypes.byref(bad), ctypes.byref(h)) == 1
    assert lib.cb_rope_rerotate(None, None, None, None, None, None, None, 1, 1, 1, 1, None) == 1
    assert lib.cb_blend_layer(None, 1, None, None) == 1
    assert lib.cb_check(None) == 1
    # a projection call without a plan is refused before any argument is read
    assert lib.cb_qkv_projection_indexed(None, None, 0, 64, None, None, 1, None, 0, None, None, None, None, None) == 1
    assert b"plan" in lib.cb_last_error_string()
