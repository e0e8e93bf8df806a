"""ctypes loader for libpkv.so and the declarations of its C ABI (include/pkv.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any operation.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpkv.so")

PKV_OK = 0
STATUS_NAMES = {
    0: "PKV_OK", -1: "PKV_ERR_INVALID_ARG", -2: "PKV_ERR_SHAPE", -3: "PKV_ERR_ALIGNMENT",
    -4: "PKV_ERR_WORKSPACE_TOO_SMALL", -5: "PKV_ERR_CUDA", -6: "PKV_ERR_DEVICE",
    -7: "PKV_ERR_NO_SPACE", -8: "PKV_ERR_NOT_FOUND",
}
DEV_BLOCK_ID = 0x1
DEV_SLOT = 0x2
DEV_SEQ_LEN = 0x4
DEV_COPY_CONFLICT = 0x8
DEV_TIMEOUT = 0x10
DEV_TABLE_RANGE = 0x20
DEV_PREFIX = 0x40
DECODE_GENERIC = 0x1
DECODE_NO_TCGEN05 = 0x2
DECODE_TEST_WITHHOLD = 0x100      # test control of the failure path (see pkv.h)


class CacheDesc(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim_k", ctypes.c_int32),
                ("head_dim_v", ctypes.c_int32)]


# name -> (restype, argtypes); mirrors include/pkv.h
_P = ctypes.c_void_p
_i32, _i64, _u64 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
_f32, _sz = ctypes.c_float, ctypes.c_size_t
_DESC = ctypes.POINTER(CacheDesc)
SIGNATURES = {
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int, _P]),
    "pkv_slot_mapping": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _i64, _P, _P]),
    "pkv_kv_append": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _P, _i64, _P]),
    "pkv_copy_blocks": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _i32, _P]),
    "pkv_kv_append_e4m3": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _P, _P, _P, _i64, _P]),
    "pkv_copy_blocks_e4m3": (ctypes.c_int, [_DESC, _P, _P, _P, _P, _i32, _P]),
    "pkv_decode_auto_splits_e4m3": (_i32, [_DESC, _i32, _i32, _i32]),
    "pkv_paged_decode_attn_e4m3": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P, _P, _P,
                                                  _i32, _P, _f32, _i32, _P, _sz, _P, _P, _i32,
                                                  _P]),
    "pkv_interleave_slot_mapping": (ctypes.c_int, [_DESC, _i64, _i64, _i32, _i32, _P, _i32,
                                                   _P, _P, _P]),
    "pkv_interleave_partition_len": (_i64, [_i64, _i32, _i32, _i32]),
    "pkv_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32]),
    "pkv_decode_auto_splits": (_i32, [_DESC, _i32, _i32, _i32]),
    "pkv_paged_decode_attn": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P, _i32, _P, _f32,
                                             _i32, _P, _sz, _P, _P, _i32, _P]),
    "pkv_paged_decode_attn_partial": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P, _i32,
                                                     _P, _f32, _i32, _P, _P, _i32, _P]),
    "pkv_paged_decode_attn_noalloc": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P, _i32,
                                                     _P, _f32, _i32, _P, _P, _i32, _P]),
    "pkv_paged_decode_attn_partial_e4m3": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P,
                                                          _P, _P, _i32, _P, _f32, _i32, _P,
                                                          _P, _i32, _P]),
    "pkv_paged_decode_attn_noalloc_e4m3": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P,
                                                          _P, _P, _i32, _P, _f32, _i32, _P,
                                                          _P, _i32, _P]),
    "pkv_decode_multi_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, _i32]),
    "pkv_decode_multi_auto_splits": (_i32, [_DESC, _i32, _i32, _i32, _i32, _i32]),
    "pkv_paged_decode_attn_multi": (ctypes.c_int, [_DESC, _P, _i32, _i32, _i32, _P, _P, _P,
                                                   _i32, _P, _f32, _i32, _P, _sz, _P, _P, _i32,
                                                   _P]),
    "pkv_decode_multi_auto_splits_e4m3": (_i32, [_DESC, _i32, _i32, _i32, _i32]),
    "pkv_paged_decode_attn_multi_e4m3": (ctypes.c_int, [_DESC, _P, _i32, _i32, _i32, _P, _P,
                                                        _P, _P, _P, _i32, _P, _f32, _i32, _P,
                                                        _sz, _P, _P, _i32, _P]),
    "pkv_lse_merge": (ctypes.c_int, [_i32, _P, _P, _i64, _i32, _P, _P, _P]),
    "pkv_decode_cascade_splits": (ctypes.c_int, [_DESC, _i32, _i32, _i32, _i32,
                                                 ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "pkv_decode_cascade_workspace_size": (_sz, [_DESC, _i32, _i32, _i32, _i32, _i32, _i32]),
    "pkv_paged_decode_attn_cascade": (ctypes.c_int, [_DESC, _P, _i32, _i32, _P, _P, _P, _i32, _P,
                                                     _i32, _P, _f32, _i32, _i32, _P, _sz, _P, _P,
                                                     _i32, _P]),
    "pkv_test_enable_withhold": (ctypes.c_int, [ctypes.c_int]),
    "pkv_bm_create": (_P, [_i32, _i32, _P]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_add_sequence": (ctypes.c_int, [_P, ctypes.POINTER(_i64)]),
    "pkv_bm_fork": (ctypes.c_int, [_P, _i64, ctypes.POINTER(_i64)]),
    "pkv_bm_append": (ctypes.c_int, [_P, _i64, _i32, _P, _P, _P, _i32, ctypes.POINTER(_i32)]),
    "pkv_bm_free": (ctypes.c_int, [_P, _i64]),
    "pkv_bm_block_table": (ctypes.c_int, [_P, _i64, _P, _i32, ctypes.POINTER(_i32),
                                          ctypes.POINTER(_i64)]),
    "pkv_bm_num_free": (_i32, [_P]),
    "pkv_bm_ref_count": (_i32, [_P, _i32]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python paged_kv_cache_93_gb300/_build.py, or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


class PkvError(RuntimeError):
    def __init__(self, where: str, status: int, message: str):
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)} ({message})")
        self.status = status
