"""The C ABI library on a host without a GPU: it builds, loads, exports every
symbol include/pa.h declares, and its host-only entry points behave.

No call here touches a device.
"""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_114_gb300 import build
    build.build()
    import paged_kv_cache_114_gb300 as pa
    return pa.lib()


def _header_functions():
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pa_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    import paged_kv_cache_114_gb300 as pa
    assert _header_functions() == sorted(pa.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _header_functions():
        assert hasattr(lib, name), name
    nm = os.popen(f"nm -D --defined-only {lib._name}").read()
    for name in _header_functions():
        assert re.search(rf"\bT {name}\b", nm), f"{name} not exported as a text symbol"


def test_static_workspace_size_matches_header():
    """The binding's copy of PA_STATIC_WORKSPACE_BYTES is the header's value."""
    import paged_kv_cache_114_gb300 as pa
    text = open(os.path.join(ROOT, "include", "pa.h")).read()
    m = re.search(r"#define PA_STATIC_WORKSPACE_BYTES \(([0-9u*\s]+)\)", text)
    assert m is not None
    value = 1
    for f in m.group(1).split("*"):
        value *= int(f.strip().rstrip("u"))
    assert value == pa.STATIC_WORKSPACE_BYTES


def test_version_and_status_strings(lib):
    import paged_kv_cache_114_gb300._lib as L
    assert lib.pa_abi_version() == L.ABI_VERSION == 4
    assert lib.pa_status_string(0) == b"ok"
    assert lib.pa_status_string(-5).startswith(b"workspace")
    assert lib.pa_status_string(12345) == b"unknown status"


def test_workspace_bytes(lib):
    # N * Hq * ceil(L / P) * (D + 2) floats; no workspace when one partition covers L
    assert lib.pa_decode_workspace_bytes(8, 32, 8, 128, 32768, 512) == 8 * 32 * 64 * 130 * 4
    assert lib.pa_decode_workspace_bytes(8, 32, 8, 128, 512, 512) == 0
    assert lib.pa_decode_workspace_bytes(8, 32, 8, 128, 4096, 0) == 0
    assert lib.pa_decode_workspace_bytes(4, 4, 4, 64, 33, 16) == 4 * 4 * 3 * 66 * 4
    # the balanced mode's size depends on the device's SM count: 0 without a device
    import torch
    if not torch.cuda.is_available():
        assert lib.pa_decode_workspace_bytes(8, 32, 8, 128, 4096, -1) == 0
        assert lib.pa_prefill_workspace_bytes(128, 64, 8, 128, 16, 4) == 0


def test_decode_kernel_name(lib):
    def name(*a):
        r = lib.pa_decode_kernel_name(*a)
        return None if r is None else r.decode()
    # balanced: grouped boxes need b >= 8 and 4 | H_kv; otherwise per-warp boxes
    assert name(32, 32, 128, 16, 2048, -1) == "decode_grouped_kernel+decode_piece_merge_kernel"
    assert name(64, 8, 128, 16, 8192, -1) == "decode_grouped_kernel+decode_piece_merge_kernel"
    assert name(32, 8, 128, 8, 32768, -1) == "decode_grouped_kernel+decode_piece_merge_kernel"
    assert name(4, 4, 64, 4, 33, -1) == "decode_balanced_kernel"
    assert name(6, 6, 128, 16, 100, -1) == "decode_balanced_kernel"
    # fixed split: a reduce only when there is more than one partition
    assert name(32, 8, 128, 32, 32768, 512) == "decode_kernel+decode_reduce_kernel"
    assert name(32, 8, 128, 32, 512, 512) == "decode_kernel"
    assert name(32, 32, 128, 16, 2048, 0) == "decode_kernel"
    # shapes pa_decode rejects
    assert name(32, 32, 96, 16, 2048, 0) is None
    assert name(30, 8, 128, 16, 2048, 0) is None
    assert name(32, 8, 128, 12, 2048, 0) is None
    assert name(32, 8, 128, 16, 2048, 24) is None
    assert name(32, 8, 128, 16, 2048, -2) is None


def test_prefill_kernel_name(lib):
    def name(*a, sms=152):
        r = lib.pa_prefill_kernel_name(*a, sms)
        return None if r is None else r.decode()
    # a few drafts (<= 32 (query, head) rows per KV head, head_dim 128, b >= 16)
    # run on the balanced grouped kernel when a workspace is given; over 16 rows
    # only while the batch has fewer than 4 (sequence, KV head) pairs per SM
    assert name(128, 64, 8, 128, 16, 4, 1) == "prefill_kernel"          # 32 rows, 1024 pairs
    assert name(75, 64, 8, 128, 16, 4, 1) == "multi_grouped_kernel"     # 600 pairs < 608
    assert name(76, 64, 8, 128, 16, 4, 1) == "prefill_kernel"
    assert name(128, 64, 8, 128, 16, 4, 1, sms=300) == "multi_grouped_kernel"
    assert name(16, 64, 8, 128, 16, 4, 1) == "multi_grouped_kernel"
    assert name(16, 64, 8, 128, 16, 4, 0) == "prefill_kernel"
    assert name(128, 64, 8, 128, 16, 2, 1) == "multi_grouped_kernel"    # 16 rows
    assert name(8, 32, 32, 128, 16, 32, 1) == "multi_grouped_kernel"    # MHA, 32 drafts
    assert name(8, 32, 8, 128, 16, 1, 1) == "multi_grouped_kernel"      # 4 rows
    assert name(8, 32, 8, 128, 16, 3, 1) == "multi_grouped_kernel"      # 12 rows
    assert name(8, 32, 4, 128, 16, 2, 1) == "prefill_kernel"            # 16 rows want 8 | H_kv
    assert name(8, 64, 8, 128, 16, 5, 1) == "prefill_kernel"            # 40 rows
    assert name(8, 64, 8, 128, 8, 4, 1) == "prefill_kernel"             # blocks of 8
    assert name(8, 64, 8, 64, 16, 4, 1) == "prefill_kernel"             # head_dim 64
    assert name(3000, 64, 8, 128, 16, 2, 1) == "prefill_kernel"         # over 2048 sequences
    assert name(8, 32, 8, 128, 16, 512, 1) == "prefill_tc_kernel"
    assert name(8, 32, 8, 128, 16, 512, 0) == "prefill_tc_kernel"
    assert name(8, 30, 8, 128, 16, 4, 1) is None
    assert name(8, 64, 8, 128, 16, 4, 1, sms=-1) is None


def test_check_copy_pairs(lib):
    def chk(pairs, nb=16):
        a = np.ascontiguousarray(np.array(pairs, dtype=np.int64).reshape(-1, 2))
        return lib.pa_check_copy_pairs(a.ctypes.data_as(ctypes.c_void_p), a.shape[0], nb)
    assert chk([(1, 2), (1, 3), (4, 5)]) == 0
    assert chk([(1, 2), (3, 2)]) == -8          # duplicate destination
    assert chk([(1, 2), (2, 3)]) == -8          # a destination is also a source
    assert chk([(1, 16)]) == -8                 # out of range
    assert chk([(-1, 3)]) == -8
    assert lib.pa_check_copy_pairs(None, 0, 16) == 0
    assert lib.pa_check_copy_pairs(None, 2, 16) == -1


def test_host_argument_errors_launch_nothing(lib):
    import paged_kv_cache_114_gb300._lib as L
    vp = ctypes.c_void_p
    # a NULL cache is rejected before any CUDA call
    assert lib.pa_decode(vp(0), 1, 1, None, vp(0), 1, vp(0), 1, 1.0, vp(0), 0, 0, vp(0), 0, vp(0)) == -1
    assert lib.pa_write_kv(vp(0), vp(0), vp(0), 1, None, vp(0)) == -1
    assert lib.pa_copy_blocks(None, 1, vp(0), 1, vp(0)) == -1
    assert lib.pa_copy_blocks(None, 0, vp(0), 1, vp(0)) == -6
    assert lib.pa_swap_blocks(None, None, 1, vp(0), 1, vp(0)) == -1
    assert lib.pa_swap_blocks(None, None, 0, vp(0), 1, vp(0)) == -6
    sw_a = L.PaCache(4096, 8192, 64, 16, 8, 128, L.PA_F16, L.PA_F16, 1.0, 1.0)
    sw_b = L.PaCache(4096, 8192, 64, 16, 8, 128, L.PA_BF16, L.PA_BF16, 1.0, 1.0)
    sw_c = L.PaCache(4096, 8192, 64, 16, 4, 128, L.PA_F16, L.PA_F16, 1.0, 1.0)
    assert lib.pa_swap_blocks(ctypes.byref(sw_a), ctypes.byref(sw_b), 1, vp(4096), 1, vp(0)) == -2
    assert lib.pa_swap_blocks(ctypes.byref(sw_a), ctypes.byref(sw_c), 1, vp(4096), 1, vp(0)) == -3
    assert lib.pa_swap_blocks(ctypes.byref(sw_a), ctypes.byref(sw_a), 1, vp(0), 0, vp(0)) == 0
    assert lib.pa_slot_mapping(vp(0), 1, 1, vp(0), vp(0), -1, 4, 8, vp(0), vp(0)) == -6
    assert lib.pa_slot_mapping(vp(0), 1, 1, vp(0), vp(0), 0, 4, 8, vp(0), vp(0)) == 0
    # cache checks: dtype, shape and alignment, all on the host
    good = L.PaCache(4096, 8192, 64, 16, 8, 128, L.PA_F16)
    bad_dtype = L.PaCache(4096, 8192, 64, 16, 8, 128, L.PA_F32)
    bad_dim = L.PaCache(4096, 8192, 64, 16, 8, 100, L.PA_F16)
    misaligned = L.PaCache(4100, 8192, 64, 16, 8, 128, L.PA_F16)
    args = (vp(4096), 1, 8)
    assert lib.pa_decode(*args[:1], 1, 8, ctypes.byref(bad_dtype), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -2
    assert lib.pa_decode(vp(4096), 1, 8, ctypes.byref(bad_dim), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -3
    assert lib.pa_decode(vp(4096), 1, 8, ctypes.byref(misaligned), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -4
    # head grouping: 12 query heads over 8 KV heads is not a whole group
    assert lib.pa_decode(vp(4096), 1, 12, ctypes.byref(good), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -3
    # more than 16 query heads per KV head
    assert lib.pa_decode(vp(4096), 1, 8 * 17, ctypes.byref(good), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -3
    # partition size must be a multiple of 16
    assert lib.pa_decode(vp(4096), 1, 8, ctypes.byref(good), vp(4096), 1, vp(4096), 100, 1.0,
                         vp(4096), 0, 24, vp(0), 0, vp(0)) == -6
    # split-K without a workspace
    assert lib.pa_decode(vp(4096), 1, 8, ctypes.byref(good), vp(4096), 64, vp(4096), 1000, 1.0,
                         vp(4096), 0, 512, vp(0), 0, vp(0)) == -5
    # bad block size (neither a divisor nor a multiple of 16)
    b24 = L.PaCache(4096, 8192, 64, 24, 8, 128, L.PA_F16)
    assert lib.pa_decode(vp(4096), 1, 8, ctypes.byref(b24), vp(4096), 1, vp(4096), 1, 1.0,
                         vp(4096), 0, 0, vp(0), 0, vp(0)) == -3
    # E4M3 caches: act_dtype must be fp16/bf16, scales finite and positive,
    # head_dim 128 or 256 for decode, and prefill does not take them
    def fp8(d=128, act=L.PA_BF16, ks=0.01, vs=0.02):
        return L.PaCache(4096, 8192, 64, 16, 8, d, L.PA_FP8_E4M3, act, ks, vs)
    dec = lambda c: lib.pa_decode(vp(4096), 1, 8, ctypes.byref(c), vp(4096), 1, vp(4096), 1, 1.0,
                                  vp(4096), 0, 0, vp(0), 0, vp(0))
    assert dec(fp8(act=L.PA_F32)) == -2
    assert dec(fp8(act=L.PA_FP8_E4M3)) == -2
    assert dec(fp8(ks=0.0)) == -6
    assert dec(fp8(vs=float("nan"))) == -6
    assert dec(fp8(ks=float("inf"))) == -6
    assert dec(fp8(d=64)) == -3
    assert dec(fp8(d=120)) == -3
    assert lib.pa_write_kv(vp(4096), vp(4096), vp(4096), 1, ctypes.byref(fp8(vs=-1.0)), vp(0)) == -6
    assert lib.pa_prefill(vp(4096), 1, vp(4096), 1, 8, ctypes.byref(fp8(d=64)), vp(4096), 1,
                          vp(4096), 1.0, vp(4096), 0, vp(0), 0, vp(0)) == -3
    # zero sequences is a no-op
    assert lib.pa_decode(vp(0), 0, 8, ctypes.byref(good), vp(0), 1, vp(0), 1, 1.0,
                         vp(0), 0, 0, vp(0), 0, vp(0)) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    import paged_kv_cache_114_gb300._lib as L
    monkeypatch.setattr(L, "_lib", None)
    monkeypatch.setattr(L, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        L.lib()
