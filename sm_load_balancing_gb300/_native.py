"""ctypes view of libskdecode.so (argument marshalling only).

The library must have been built (``sm_load_balancing_gb300.build.build()``);
there is no fallback of any kind: a missing library raises at import time of
the first call.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libskdecode.so")

SKD_OK, SKD_EINVAL, SKD_EUNSUPPORTED, SKD_ECUDA, SKD_EPLAN, SKD_ESIZE = range(6)
SKD_KIND_GQA, SKD_KIND_MLA = 0, 1
SKD_PLAN_STREAMK, SKD_PLAN_ROUND_ROBIN, SKD_PLAN_FIXED_SPLIT = 0, 1, 2
SKD_DEVERR_PLAN, SKD_DEVERR_SEQLEN, SKD_DEVERR_PAGE, SKD_DEVERR_TIMEOUT, SKD_DEVERR_INDEX = 1, 2, 4, 8, 16
SKD_GRANULE = 16

# every symbol include/skdecode.h declares, with (restype, argtypes)
_c_int, _c_size, _vp, _f = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_float


class Shape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("q_tokens", ctypes.c_int32),
                ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim_qk", ctypes.c_int32), ("head_dim_v", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_pages_per_req", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("v_row_stride", ctypes.c_int32),
                ("scale", ctypes.c_float), ("causal", ctypes.c_int32), ("kind", ctypes.c_int32)]


SIGNATURES = {
    "skd_abi_version": (_c_int, []),
    "skd_status_string": (ctypes.c_char_p, [_c_int]),
    "skd_device_sm_count": (_c_int, [_c_int, ctypes.POINTER(ctypes.c_int)]),
    "skd_default_workers": (_c_int, [ctypes.POINTER(Shape), _c_int, ctypes.POINTER(ctypes.c_int)]),
    "skd_plan_bytes": (_c_size, [_c_int, _c_int, _c_int]),
    "skd_decode_plan": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size]),
    "skd_decode_plan_device": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    "skd_decode_plan_weighted": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size]),
    "skd_decode_plan_weighted_device": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size, _vp]),
    "skd_decode_plan_aligned": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size]),
    "skd_decode_plan_aligned_device": (_c_int, [_vp, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _vp, _c_size,
                                                 _vp]),
    "skd_workspace_bytes": (_c_size, [ctypes.POINTER(Shape), _c_int]),
    "skd_workspace_reset": (_c_int, [_vp, _c_size, _vp]),
    "skd_decode_attention": (_c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _c_int,
                                      _vp, _c_size, _vp, _vp, _vp]),
    "skd_read_error": (_c_int, [_vp, ctypes.POINTER(ctypes.c_int32), _vp]),
    "skd_trace_enable": (_c_int, [_vp, _c_size]),
    "skd_set_pdl": (_c_int, [_c_int]),
    "skd_decode_attention_split_combine": (_c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp, _c_int,
                                      _vp, _c_size, _vp, _vp, _vp]),
    "skd_decode_attention_noalloc": (_c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _vp,
                                              _c_int, _vp, _vp, _vp]),
    "skd_decode_attention_sparse": (_c_int, [ctypes.POINTER(Shape), _vp, _vp, _vp, _vp, _vp, _c_int, _vp, _vp,
                                             _c_int, _vp, _c_size, _vp, _vp, _vp]),
    "skd_gather_rows": (_c_int, [_vp, _vp, _vp, ctypes.c_int64, ctypes.c_int64, _vp]),
    "skd_merge_states": (_c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _c_int, _vp]),
}

_lib = None


class SkdError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = _lib.skd_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {msg} (status {status})")


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libskdecode.so is not built ({LIB_PATH}); run "
                              "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def check(fn_name, status):
    if status != SKD_OK:
        raise SkdError(fn_name, status)
