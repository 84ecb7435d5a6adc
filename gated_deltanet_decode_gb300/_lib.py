"""ctypes declarations of the C ABI in ``include/gdn_decode.h``.

Loading fails loudly: there is no fallback when the CUDA library cannot be
found or built.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

GDN_OK = 0
GDN_EINVAL = 1
GDN_ENOMEM = 2
GDN_ECUDA = 3
GDN_EUNSUPPORTED = 4
GDN_ESLOTS = 5

GDN_DEVERR_NONE = 0
GDN_DEVERR_BAD_SLOT = 1
GDN_DEVERR_TIMEOUT = 2

GDN_F32 = 0
GDN_BF16 = 1

GDN_PROBE_TWIN = 0
GDN_PROBE_INPLACE = 1
GDN_PROBE_READ = 2
GDN_PROBE_WRITE = 3

GDN_MAX_POOLS = 4096
GDN_NOALLOC_SCRATCH_SLOTS = 64

# Every symbol the header declares (the export test checks this list against
# include/gdn_decode.h).
EXPORTS = [
    "gdn_last_error", "gdn_abi_version",
    "gdn_state_pool_create", "gdn_state_pool_wrap", "gdn_state_pool_destroy", "gdn_pool_data",
    "gdn_pool_inplace_counter_bytes", "gdn_pool_attach_inplace_counters",
    "gdn_pool_num_slots", "gdn_pool_dims", "gdn_pool_zero_slots", "gdn_pool_copy_slots",
    "conv_state_pool_create", "conv_state_pool_wrap", "conv_state_pool_destroy", "conv_pool_data",
    "conv_pool_num_slots", "conv_pool_zero_slots", "conv_pool_copy_slots",
    "causal_conv1d_decode", "gdn_decode_step", "gdn_layer_decode", "gdn_layer_decode_commit",
    "gdn_layer_decode_noalloc", "gdn_layer_decode_bucket", "gdn_prefill", "gdn_prefill_chunked", "gdn_prefill_chunked_workspace_bytes", "gdn_verify", "causal_conv1d_prefill",
    "gdn_commit", "gdn_validate_slots", "gdn_get_device_error", "gdn_selftest_wait_timeout",
    "gdn_probe_traffic",
]


class gdn_dims(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_int), ("hv", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int)]


_P = ctypes.c_void_p
_I = ctypes.c_int
_PP = ctypes.POINTER(ctypes.c_void_p)

_SIGS = {
    "gdn_last_error": (ctypes.c_char_p, []),
    "gdn_abi_version": (_I, []),
    "gdn_state_pool_create": (_I, [_I, gdn_dims, _P, _PP]),
    "gdn_state_pool_wrap": (_I, [_P, _I, gdn_dims, _PP]),
    "gdn_state_pool_destroy": (_I, [_P]),
    "gdn_pool_data": (_P, [_P]),
    "gdn_pool_inplace_counter_bytes": (ctypes.c_size_t, [_I, gdn_dims]),
    "gdn_pool_attach_inplace_counters": (_I, [_P, _P, ctypes.c_size_t]),
    "gdn_pool_num_slots": (_I, [_P]),
    "gdn_pool_dims": (gdn_dims, [_P]),
    "gdn_pool_zero_slots": (_I, [_P, _P, _I, _P]),
    "gdn_pool_copy_slots": (_I, [_P, _P, _P, _I, _P]),
    "conv_pool_copy_slots": (_I, [_P, _P, _P, _I, _P]),
    "conv_state_pool_create": (_I, [_I, _I, _I, _I, _P, _PP]),
    "conv_state_pool_wrap": (_I, [_P, _I, _I, _I, _I, _PP]),
    "conv_state_pool_destroy": (_I, [_P]),
    "conv_pool_data": (_P, [_P]),
    "conv_pool_num_slots": (_I, [_P]),
    "conv_pool_zero_slots": (_I, [_P, _P, _I, _P]),
    "causal_conv1d_decode": (_I, [_P, _I, _P, _P, _P, _P, _P, _I, _P, _I, _I, _P]),
    "gdn_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gdn_layer_decode": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "gdn_layer_decode_commit": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _P]),
    "gdn_layer_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                      _P]),
    "gdn_layer_decode_bucket": (_I, [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I,
                                     _P]),
    "gdn_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "gdn_prefill_chunked": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P, ctypes.c_size_t,
                                 _I, _P]),
    "gdn_prefill_chunked_workspace_bytes": (ctypes.c_size_t, [_I, _I, _I]),
    "gdn_verify": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]),
    "causal_conv1d_prefill": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _P]),
    "gdn_commit": (_I, [_P, _P, _I, _P]),
    "gdn_validate_slots": (_I, [_P, _P, _I, _I, _I, _P]),
    "gdn_get_device_error": (_I, [ctypes.POINTER(ctypes.c_int), _P]),
    "gdn_probe_traffic": (_I, [_P, _P, _P, _I, _I, _P, _P]),
    "gdn_selftest_wait_timeout": (_I, [_I, _P]),
}

_lock = threading.Lock()
_lib = None


def lib_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libgdn_decode.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build() if build_if_missing else _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"GDN decode library not found at {path}")
            L = ctypes.CDLL(path)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib
