"""ctypes loader of libpagedkv.so (the C ABI in include/pagedkv.h).

The library is built in-tree (paged_kv_decode_26_gb300/libpagedkv.so) by
``paged_kv_decode_26_gb300.build``.  There is no fallback: if the library is
missing or fails to load, every entry point raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

PKV_OK, PKV_ERR_INVALID, PKV_ERR_UNSUPPORTED, PKV_ERR_CUDA, PKV_ERR_WORKSPACE, PKV_ERR_NO_BLOCKS = range(6)
PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2

DEVERR_BLOCK_ID = 0x1
DEVERR_CONTEXT = 0x2
DEVERR_SLOT = 0x4
DEVERR_PAIR = 0x8
DEVERR_TIMEOUT = 0x10

# Launch-shape override knobs (pkv_tune_knob), by lower-case name.
TUNE_AUTO = -2147483648
TUNE_KNOBS = {name: i for i, name in enumerate(
    ["decode_mma", "decode_hpc", "decode_stages", "decode_wpt", "decode_qpw", "decode_split",
     "decode_order", "decode_pdl", "mq_tc", "mq_tc_stages", "mq_lpt", "mq_stages", "swap_bulk",
     "swap_chunk", "swap_stages", "swap_ctas", "swap_hint", "decode_stream"])}

# Every symbol include/pagedkv.h declares, with (restype, argtypes).
_p, _i, _i32, _i64, _sz, _f = C.c_void_p, C.c_int, C.c_int32, C.c_int64, C.c_size_t, C.c_float
SIGNATURES = {
    "pkv_status_string": (C.c_char_p, [_i]),
    "pkv_last_error_detail": (C.c_char_p, []),
    "pkv_version": (_i, []),
    "pkv_set_tuning": (_i, [_i, _i]),
    "pkv_get_tuning": (_i, [_i]),
    "pkv_device_errors": (_i, [C.POINTER(C.c_uint32), _i]),
    "pkv_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i, _i]),
    "pkv_decode_split_tokens": (_i, [_i, _i, _i, _i, _i, _i]),
    "pkv_decode_launch_shape": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _i, _i, _p]),
    "paged_attn_decode": (_i, [_p, _i, _p, _p, _p, _i, _p, _i, _p, _i, _i, _i, _i, _i, _i, _f,
                               _i, _i, _p, _sz, _p]),
    "paged_attn_decode_append": (_i, [_p, _i, _p, _p, _p, _i, _p, _i, _p, _i, _i, _i, _i, _i,
                                      _i, _f, _i, _i, _p, _sz, _p, _p, _p, _p]),
    "paged_attn_decode_append_host": (_i, [_p, _i, _p, _sz, _i, _p, _i, _p, _p, _p, _i, _p, _i,
                                           _p, _i, _i, _i, _i, _i, _i, _f, _i, _i, _p, _sz, _p,
                                           _p, _p, _p]),
    "pkv_decode_batched_workspace_bytes": (_sz, [_p, _i, _i, _i, _i, _i, _i, _i]),
    "pkv_decode_batched_plan": (_i, [_p, _p, _i, _i, _i, _i, _i, _i, _i, _f, _i, _i, _p, _sz,
                                     _p]),
    "paged_attn_decode_batched": (_i, [_p, _p]),
    "paged_attn_decode_noalloc": (_i, [_p, _i, _p, _p, _p, _i, _p, _i, _p, _i, _i, _i, _i, _i,
                                       _i, _f, _i, _i, _p]),
    "paged_attn_multi_query": (_i, [_p, _i, _p, _p, _i, _i, _p, _p, _i, _p, _i, _p, _i, _i, _i,
                                    _i, _i, _i, _f, _i, _p]),
    "kv_append": (_i, [_p, _p, _p, _p, _i, _p, _i, _i, _i, _i, _i, _p]),
    "swap_blocks": (_i, [_p, _p, _sz, _p, _i, _i64, _i64, _p]),
    "swap_blocks_kv": (_i, [_p, _p, _p, _p, _sz, _p, _i, _i64, _i64, _p]),
    "pkv_block_manager_create": (_p, [_i, _i]),
    "pkv_block_manager_create_with_free": (_p, [_i, _i, _p, _i]),
    "pkv_block_manager_destroy": (None, [_p]),
    "pkv_block_allocate": (_i, [_p, C.POINTER(_i32)]),
    "pkv_block_free": (_i, [_p, _i32]),
    "pkv_block_add_reference": (_i, [_p, _i32]),
    "pkv_block_free_count": (_i, [_p]),
    "pkv_block_ref_count": (_i, [_p, _i32]),
    "pkv_block_free_ids": (_i, [_p, _p, _i]),
    "pkv_append_slots": (_i, [_p, _p, _i, _p, _i, _p]),
    "pkv_append_slots_cow": (_i, [_p, _p, _i, _p, _i, _p, _p, C.POINTER(_i)]),
    "pkv_defrag": (_i, [_p, _p, _i, _i, _p, _i, C.POINTER(_i)]),
    "pkv_device_rebuild_free_list": (_i, [_p, _p, _p, _i, _p]),
    "pkv_device_append_slots": (_i, [_p, _p, _p, _p, _i, _p, _i, _i, _i, _p, _p]),
    "pkv_device_free_blocks": (_i, [_p, _p, _p, _p, _i, _i, _p]),
}

_lib = None
_lock = threading.Lock()


class PagedKVError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = status
        name = lib().pkv_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{where}: {name}" + (f" ({detail})" if detail else ""))


def lib():
    """The loaded library (loads on first use; raises if it is not built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -c 'import paged_kv_decode_26_gb300.build as b; b.build()'` "
                        "(there is no CPU fallback)")
                L = C.CDLL(LIB_PATH)
                for name, (res, args) in SIGNATURES.items():
                    fn = getattr(L, name)
                    fn.restype = res
                    fn.argtypes = args
                _lib = L
    return _lib


def check(status: int, where: str) -> None:
    if status != PKV_OK:
        detail = lib().pkv_last_error_detail()
        raise PagedKVError(status, where, detail.decode() if detail else "")
