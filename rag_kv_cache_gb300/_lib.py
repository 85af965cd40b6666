"""ctypes binding of libcacheblend.so (include/cacheblend.h).

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t. Every step of the blend runs in the
library's CUDA kernels. If the library is missing or cannot be loaded, every
call raises: there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcacheblend.so")

CB_OK = 0
STATUS = {0: "CB_OK", 1: "CB_ERR_INVALID_ARG", 2: "CB_ERR_UNSUPPORTED", 3: "CB_ERR_CUDA",
          4: "CB_ERR_TIMEOUT", 5: "CB_ERR_DEVICE_CHECK"}
ROPE_STYLES = {"half": 0, "interleaved": 1}
DEVIATIONS = {"v": 0, "kv": 1}  # cb_deviation
FILTERS = {"keep": 0, "reselect": 1}  # cb_filter
STAGES = {"deviation": 0, "topk": 1, "fuse": 2, "attention": 3}  # cb_stage

# every symbol include/cacheblend.h declares
EXPORTS = ("cb_plan_create", "cb_plan_destroy", "cb_layer_sizes", "cb_rope_rerotate", "cb_kv_deviation",
           "cb_kv_deviation_kv", "cb_hkvd_topk", "cb_fuse_scatter", "cb_hkvd_attention", "cb_decode_attention",
           "cb_attention_sparsity", "cb_output_deviation", "cb_qkv_projection", "cb_qkv_projection_indexed",
           "cb_blend_layer", "cb_blend_stage", "cb_blend_request", "cb_hkvd_select_noalloc",
           "cb_attention_uses_paired_tiles", "cb_test_attention_wait_timeout", "cb_test_decode_wait_timeout",
           "cb_test_projection_wait_timeout", "cb_check",
           "cb_last_error_string", "cb_version")


class CbConfig(ctypes.Structure):
    _fields_ = [("n_chunks", ctypes.c_int32), ("chunk_len", ctypes.c_int32), ("n_suffix", ctypes.c_int32),
                ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("rope_theta", ctypes.c_double), ("rope_style", ctypes.c_int32),
                ("r1_pct", ctypes.c_int32), ("r2_pct", ctypes.c_int32),
                ("deviation", ctypes.c_int32), ("filter", ctypes.c_int32)]


class CbLayerIO(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "k_old", "v_old", "k_new", "v_new", "q", "cand", "dev", "sel_tok", "sel_row",
        "k_fused", "v_fused", "q_rot", "out")]


class CacheBlendError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library {path} is missing: build it with "
                           "`python -m rag_kv_cache_gb300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(path)
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float
    sig = {
        "cb_plan_create": (i32, [ctypes.POINTER(CbConfig), ctypes.POINTER(vp)]),
        "cb_plan_destroy": (i32, [vp]),
        "cb_layer_sizes": (i32, [vp, i32] + [ctypes.POINTER(i32)] * 4),
        "cb_rope_rerotate": (i32, [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, vp]),
        "cb_kv_deviation": (i32, [vp, vp, vp, vp, i32, vp, vp]),
        "cb_kv_deviation_kv": (i32, [vp, vp, vp, vp, vp, vp, i32, vp, vp]),
        "cb_hkvd_topk": (i32, [vp, vp, vp, i32, i32, vp, vp, vp]),
        "cb_fuse_scatter": (i32, [vp, vp, vp, vp, vp, vp, i32, vp]),
        "cb_hkvd_attention": (i32, [vp, vp, vp, i32, vp, vp, i32, f32, vp, vp]),
        "cb_decode_attention": (i32, [vp, vp, vp, vp, i32, f32, vp, vp]),
        "cb_attention_sparsity": (i32, [vp, vp, vp, i32, vp, vp, i32, f32, f32, vp, vp, vp, vp, vp]),
        "cb_output_deviation": (i32, [vp, vp, vp, i32, vp, vp]),
        "cb_qkv_projection": (i32, [vp, vp, i32, i32, vp, i32, vp, i32, vp, vp, vp, vp, vp]),
        "cb_qkv_projection_indexed": (i32, [vp, vp, i32, i32, vp, vp, i32, vp, i32, vp, vp, vp, vp, vp]),
        "cb_blend_layer": (i32, [vp, i32, ctypes.POINTER(CbLayerIO), vp]),
        "cb_blend_stage": (i32, [vp, i32, ctypes.POINTER(CbLayerIO), i32, vp]),
        "cb_blend_request": (i32, [vp, i32, ctypes.POINTER(CbLayerIO), vp]),
        "cb_hkvd_select_noalloc": (i32, [vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp]),
        "cb_attention_uses_paired_tiles": (i32, [vp, i32]),
        "cb_test_attention_wait_timeout": (i32, [vp, vp, vp, i32, vp, vp, i32, vp, vp]),
        "cb_test_decode_wait_timeout": (i32, [vp, vp, vp, vp, i32, vp, vp]),
        "cb_test_projection_wait_timeout": (i32, [vp, vp, i32, i32, vp, vp, vp, vp, vp]),
        "cb_check": (i32, [vp]),
        "cb_last_error_string": (ctypes.c_char_p, []),
        "cb_version": (i32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != CB_OK:
        raise CacheBlendError(status, load().cb_last_error_string().decode())
