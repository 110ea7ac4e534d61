"""ctypes view of libpagedkv.so (the C ABI declared in include/pa.h).

Loading never falls back to anything: if the library is missing, every call
raises. Build it with ``python -m paged_kv_cache_114_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpagedkv.so")

PA_F16, PA_BF16, PA_F32, PA_FP8_E4M3 = 0, 1, 2, 3
ABI_VERSION = 4  # PA_ABI_VERSION this binding is written for
PA_OK = 0
PA_PARTITION_BALANCED = -1
STATUS = {
    0: "ok", -1: "null pointer", -2: "unsupported or mismatched dtype", -3: "unsupported shape",
    -4: "misaligned pointer", -5: "workspace missing or too small", -6: "invalid argument",
    -7: "CUDA runtime error", -8: "copy pairs violate the distinct-destination rule",
}
DEVERR_BLOCK_ID, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_POSITION, DEVERR_TIMEOUT = 1, 2, 4, 8, 16

# Every symbol include/pa.h declares.
EXPORTED = (
    "pa_slot_mapping", "pa_write_kv", "pa_copy_blocks", "pa_check_copy_pairs", "pa_decode",
    "pa_decode_workspace_bytes", "pa_decode_default_partition", "pa_get_device_error",
    "pa_status_string", "pa_abi_version", "pa_decode_static_workspace", "pa_decode_kernel_name",
    "pa_prefill", "pa_prefill_workspace_bytes", "pa_prefill_kernel_name", "pa_swap_blocks",
    "pa_prefix_hash", "pa_prefix_key_offsets", "pa_test_set_stall",
)
STATIC_WORKSPACE_BYTES = 16 * 1024 * 1024


class PaCache(ctypes.Structure):
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int),
        ("act_dtype", ctypes.c_int),
        ("k_scale", ctypes.c_float),
        ("v_scale", ctypes.c_float),
    ]


class PagedKVError(RuntimeError):
    """A libpagedkv call returned a negative status."""

    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {STATUS.get(status, 'unknown status')} ({status})")
        self.status = status


_lock = threading.Lock()
_lib = None


def _declare(lib):
    i32, i64, vp, sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    cache_p = ctypes.POINTER(PaCache)
    sig = {
        "pa_slot_mapping": (ctypes.c_int, [vp, i32, i32, vp, vp, i64, i32, i64, vp, vp]),
        "pa_write_kv": (ctypes.c_int, [vp, vp, vp, i64, cache_p, vp]),
        "pa_copy_blocks": (ctypes.c_int, [cache_p, i32, vp, i64, vp]),
        "pa_swap_blocks": (ctypes.c_int, [cache_p, cache_p, i32, vp, i64, vp]),
        "pa_prefix_hash": (ctypes.c_int, [vp, vp, vp, i32, i32, ctypes.c_char_p, vp, vp]),
        "pa_prefix_key_offsets": (ctypes.c_int, [vp, i32, i32, vp, vp]),
        "pa_check_copy_pairs": (ctypes.c_int, [vp, i64, i64]),
        "pa_decode": (ctypes.c_int, [vp, i32, i32, cache_p, vp, i32, vp, i32, ctypes.c_float, vp,
                                     ctypes.c_int, i32, vp, sz, vp]),
        "pa_prefill": (ctypes.c_int, [vp, i32, vp, i32, i32, cache_p, vp, i32, vp, ctypes.c_float,
                                      vp, ctypes.c_int, vp, sz, vp]),
        "pa_prefill_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "pa_prefill_kernel_name": (ctypes.c_char_p, [i32, i32, i32, i32, i32, i32, i32, i32]),
        "pa_decode_static_workspace": (ctypes.c_int, [vp, i32, i32, cache_p, vp, i32, vp, i32,
                                                      ctypes.c_float, vp, ctypes.c_int, i32, vp]),
        "pa_decode_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "pa_decode_default_partition": (i32, [i32, i32, i32, i32]),
        "pa_decode_kernel_name": (ctypes.c_char_p, [i32, i32, i32, i32, i32, i32]),
        "pa_get_device_error": (ctypes.c_int, [ctypes.POINTER(i32), vp]),
        "pa_test_set_stall": (ctypes.c_int, [i32, ctypes.c_uint32]),
        "pa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "pa_abi_version": (ctypes.c_int, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m paged_kv_cache_114_gb300.build` (there is no fallback)")
                loaded = _declare(ctypes.CDLL(LIB_PATH))
                if loaded.pa_abi_version() != ABI_VERSION:
                    raise RuntimeError(
                        f"{LIB_PATH} has ABI version {loaded.pa_abi_version()}, this binding needs "
                        f"{ABI_VERSION}: rebuild it with `python -m paged_kv_cache_114_gb300.build`")
                _lib = loaded
    return _lib


def check(fn: str, status: int) -> None:
    if status != PA_OK:
        raise PagedKVError(fn, status)
