"""ctypes view of include/mqa_decode.h: the struct, the status codes and the
entry points of libmqa_decode.so. Loading fails loudly when the library has
not been built; there is no fallback."""

from __future__ import annotations

import ctypes
import os
import re

from .build import INCLUDE, lib_path

MQA_OK = 0
MQA_ERR_INVALID_ARG = 1
MQA_ERR_UNSUPPORTED = 2
MQA_ERR_CUDA = 3
MQA_ERR_WORKSPACE = 4

MQA_BF16 = 0
MQA_F32 = 1
MQA_U8 = 2
MQA_FP8_E5M2 = 3

MQA_VARIANT_AUTO = 0
MQA_VARIANT_CUDA_CORE = 1
MQA_VARIANT_TENSOR_CORE = 2

MQA_DEVERR_POS_RANGE = 0x1
MQA_DEVERR_PAGE_RANGE = 0x2
MQA_DEVERR_SEQ_LEN = 0x4
MQA_DEVERR_TIMEOUT = 0x8
MQA_DEVERR_U8_SCALE = 0x10

c_i32 = ctypes.c_int32
c_vp = ctypes.c_void_p


class KVLayout(ctypes.Structure):
    """mqa_kv_layout"""

    _fields_ = [
        ("cache_dtype", c_i32),
        ("batch", c_i32),
        ("h_q", c_i32),
        ("h_kv", c_i32),
        ("head_dim", c_i32),
        ("paged", c_i32),
        ("k_cache", c_vp),
        ("v_cache", c_vp),
        ("capacity", ctypes.c_int64),
        ("page_size", c_i32),
        ("num_pages", c_i32),
        ("max_pages_per_seq", c_i32),
        ("window", c_i32),
        ("block_table", c_vp),
        ("k_scale_zero", c_vp),
        ("v_scale_zero", c_vp),
        ("wait_limit_ns", ctypes.c_uint64),
    ]


_PROTOTYPES = {
    "kv_append_rope": (c_i32, [ctypes.POINTER(KVLayout), c_vp, c_vp, c_vp, c_vp, ctypes.c_double, c_vp, c_vp, c_vp]),
    "gqa_decode_attention": (
        c_i32,
        [ctypes.POINTER(KVLayout), c_vp, c_vp, c_i32, ctypes.c_float, c_i32, c_vp, c_i32, c_vp, c_vp,
         ctypes.c_size_t, c_i32, c_vp, c_vp],
    ),
    "splitkv_combine": (c_i32, [c_vp, c_vp, c_i32, c_i32, c_i32, c_i32, c_vp, c_i32, c_vp, c_vp]),
    "mqa_decode_step": (
        c_i32,
        [ctypes.POINTER(KVLayout), c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, ctypes.c_double, ctypes.c_float, c_i32, c_vp,
         c_vp, c_i32, c_vp, c_vp, ctypes.c_size_t, c_i32, c_vp, c_vp],
    ),
    "kv_append_rope_multi": (
        c_i32, [ctypes.POINTER(KVLayout), c_i32, c_vp, c_vp, c_vp, c_vp, ctypes.c_double, c_vp, c_vp, c_vp]),
    "gqa_decode_attention_multi": (
        c_i32,
        [ctypes.POINTER(KVLayout), c_i32, c_vp, c_vp, c_i32, ctypes.c_float, c_i32, c_vp, c_i32, c_vp, c_vp,
         ctypes.c_size_t, c_i32, c_vp, c_vp],
    ),
    "mqa_decode_step_multi": (
        c_i32,
        [ctypes.POINTER(KVLayout), c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, ctypes.c_double, ctypes.c_float, c_i32,
         c_vp, c_vp, c_i32, c_vp, c_vp, ctypes.c_size_t, c_i32, c_vp, c_vp],
    ),
    "gqa_prefill_attention": (
        c_i32, [ctypes.POINTER(KVLayout), c_i32, c_vp, c_vp, c_i32, ctypes.c_float, c_vp, c_i32, c_vp, c_vp, c_vp]),
    "mqa_prefill_step": (
        c_i32,
        [ctypes.POINTER(KVLayout), c_i32, c_vp, c_vp, c_vp, c_vp, c_vp, c_i32, ctypes.c_double, ctypes.c_float, c_vp,
         c_vp, c_i32, c_vp, c_vp, c_vp],
    ),
    "mqa_choose_splits_multi": (c_i32, [ctypes.POINTER(KVLayout), c_i32, c_i32, c_i32]),
    "mqa_workspace_size_multi": (ctypes.c_size_t, [ctypes.POINTER(KVLayout), c_i32, c_i32, c_i32, c_i32]),
    "mqa_step_launches": (c_i32, [ctypes.POINTER(KVLayout), c_i32, c_i32, c_i32, c_i32, ctypes.POINTER(c_i32)]),
    "mqa_choose_splits": (c_i32, [ctypes.POINTER(KVLayout), c_i32, c_i32]),
    "mqa_workspace_size": (ctypes.c_size_t, [ctypes.POINTER(KVLayout), c_i32, c_i32, c_i32]),
    "mqa_status_string": (ctypes.c_char_p, [c_i32]),
    "mqa_last_cuda_error": (ctypes.c_char_p, []),
}

_LIB = None


def header_functions() -> list[str]:
    """Names of the functions include/mqa_decode.h declares."""
    text = open(os.path.join(INCLUDE, "mqa_decode.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*MQA_API\s+(?:const\s+)?[A-Za-z_]\w*\s*\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return [n for n in names if n not in ("if", "while", "for", "switch", "return", "sizeof")]


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmqa_decode.so (once) and attach the prototypes."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise ImportError(
            f"libmqa_decode.so is not built ({p} missing); run `python -c \"import __graft_entry__ as g; g.build()\"`"
        )
    lib = ctypes.CDLL(p)
    for name, (res, args) in _PROTOTYPES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib
