"""GPU parity for pa_swap_blocks (preemption by swapping): byte-exact against
the oracle's swap, device <-> pinned host in both directions, FP8 pools, and
the preemption round trip through decode.

Swapping copies a preempted sequence's blocks to host memory and back
("PagedAttention: paging the KV cache", When memory runs out); on GB300 the
host pool is Grace memory reached over NVLink-C2C.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import bits_of, gpu_scenario, to_dev
from workloads import make_random_case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from paged_kv_cache_114_gb300 import build
    build.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def _np_pools(rng, nb, layers, shape, dtype):
    if dtype == np.uint8:
        mk = lambda: rng.integers(0, 256, size=(nb,) + shape, dtype=np.uint8)
    else:
        mk = lambda: rng.integers(0, 2**16, size=(nb,) + shape).astype(np.uint16)
    return [mk() for _ in range(layers)], [mk() for _ in range(layers)]


def _torch(a, where, dev, dtype):
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
    if a.dtype == np.uint16:
        t = t.view(torch.float16 if dtype == "f16" else torch.bfloat16)
    return t.to(dev) if where == "gpu" else t.pin_memory()


@pytest.mark.parametrize("direction", ["gpu->host", "host->gpu", "gpu->gpu"])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "e4m3"])
def test_swap_matches_oracle(dev, direction, dtype):
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(hash((direction, dtype)) % 2**32)
    npdt = np.uint8 if dtype == "e4m3" else np.uint16
    shape = (16, 8, 128)
    sk, sv = _np_pools(rng, 40, 3, shape, npdt)
    dk, dv = _np_pools(rng, 25, 3, shape, npdt)
    pairs = [(int(s), int(d)) for s, d in zip(rng.choice(40, 17, replace=False),
                                              rng.choice(25, 17, replace=False))]
    want_k, want_v = oracle.swap_blocks(sk, sv, dk, dv, pairs)
    s_where, d_where = direction.split("->")
    tk = [_torch(a, s_where, dev, dtype) for a in sk]
    tv = [_torch(a, s_where, dev, dtype) for a in sv]
    uk = [_torch(a, d_where, dev, dtype) for a in dk]
    uv = [_torch(a, d_where, dev, dtype) for a in dv]
    pa.swap_blocks(tk, tv, uk, uv, to_dev(np.array(pairs, dtype=np.int64), dev))
    assert pa.get_device_error(dev) == 0
    for i in range(3):
        assert np.array_equal(bits_of(uk[i]), want_k[i]) and np.array_equal(bits_of(uv[i]), want_v[i])
        assert np.array_equal(bits_of(tk[i]), sk[i])  # the source is untouched


def test_pairs_in_pinned_host_memory(dev):
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(5)
    sk, sv = _np_pools(rng, 8, 1, (16, 2, 64), np.uint16)
    dk, dv = _np_pools(rng, 8, 1, (16, 2, 64), np.uint16)
    pairs = [(1, 2), (7, 0)]
    want_k, want_v = oracle.swap_blocks(sk, sv, dk, dv, pairs)
    uk, uv = [_torch(dk[0], "gpu", dev, "f16")], [_torch(dv[0], "gpu", dev, "f16")]
    p = torch.tensor(pairs, dtype=torch.int64).pin_memory()
    pa.swap_blocks([_torch(sk[0], "gpu", dev, "f16")], [_torch(sv[0], "gpu", dev, "f16")], uk, uv, p)
    assert pa.get_device_error(dev) == 0
    assert np.array_equal(bits_of(uk[0]), want_k[0]) and np.array_equal(bits_of(uv[0]), want_v[0])


def test_pageable_host_memory_is_refused(dev):
    import paged_kv_cache_114_gb300 as pa
    from paged_kv_cache_114_gb300._lib import PaCache, PA_F16, lib
    import ctypes
    k = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device=dev)
    host = np.zeros((4, 16, 2, 64), dtype=np.uint16)  # ordinary (pageable) memory
    src = PaCache(k.data_ptr(), k.data_ptr(), 4, 16, 2, 64, PA_F16, PA_F16, 1.0, 1.0)
    hp = host.ctypes.data
    dst = PaCache(hp, hp, 4, 16, 2, 64, PA_F16, PA_F16, 1.0, 1.0)
    pairs = torch.tensor([[0, 1]], dtype=torch.int64, device=dev)
    st = lib().pa_swap_blocks(ctypes.byref(src), ctypes.byref(dst), 1, ctypes.c_void_p(pairs.data_ptr()),
                              1, ctypes.c_void_p(0))
    assert st == -6
    torch.cuda.synchronize()
    assert pa.get_device_error(dev) == 0


def test_out_of_range_ids_flag_and_skip(dev):
    import paged_kv_cache_114_gb300 as pa
    k = torch.zeros(4, 16, 2, 64, dtype=torch.float16, device=dev)
    h = torch.full((3, 16, 2, 64), 7.0, dtype=torch.float16).pin_memory()
    pa.swap_blocks([k], [k], [h], [h], torch.tensor([[0, 3], [4, 0], [-1, 1], [1, 2]],
                                                    dtype=torch.int64, device=dev))
    assert pa.get_device_error(dev) & pa.DEVERR_BLOCK_ID
    assert torch.all(h[:2] == 7.0) and torch.all(h[2] == 0.0)


@pytest.mark.parametrize("kv", [None, "e4m3"])
def test_preemption_round_trip(dev, kv):
    """Swap a sequence out to a pinned host pool, overwrite its device blocks,
    swap it back in to other block ids and remap its table: pa_decode gives a
    bit-identical output."""
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(61, num_seqs=4, num_q_heads=16, num_kv_heads=4, head_dim=128,
                         block_size=16, seq_lens=[300, 1000, 17, 650], dtype="bf16",
                         pool_factor=2.0, kv_dtype=kv)
    res = gpu_scenario(w, dev, partition_tokens=-1)
    k, v, before = res["k"], res["v"], res["out"].clone()
    s = 1
    nblk = -(-int(w.seq_lens[s]) // w.block_size)
    own = w.block_tables[s, :nblk].astype(np.int64)
    host_k = torch.empty((nblk,) + tuple(k.shape[1:]), dtype=k.dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    pa.swap_blocks([k], [v], [host_k], [host_v],
                   to_dev(np.stack([own, np.arange(nblk)], 1).astype(np.int64), dev))
    k[torch.from_numpy(own).to(dev)] = 0  # the freed blocks are reused by others
    v[torch.from_numpy(own).to(dev)] = 0
    used = set(int(b) for r, L in zip(w.block_tables, w.seq_lens) for b in r[: -(-int(L) // 16)])
    free = np.array([b for b in range(w.num_blocks) if b not in used][:nblk], dtype=np.int64)
    pa.swap_blocks([host_k], [host_v], [k], [v],
                   to_dev(np.stack([np.arange(nblk), free], 1).astype(np.int64), dev))
    tables = w.block_tables.copy()
    tables[s, :nblk] = free
    kw = {"k_scale": w.k_scale, "v_scale": w.v_scale} if kv else {}
    after = pa.decode(to_dev(w.q, dev, w.dtype), k, v, to_dev(tables, dev), to_dev(w.seq_lens, dev),
                      w.scale, max_seq_len=w.max_seq_len, out_dtype=torch.float32,
                      partition_tokens=-1, **kw)
    assert pa.get_device_error(dev) == 0
    assert torch.equal(before, after)


@pytest.mark.parametrize("op", ["swap gpu->host", "copy"])
def test_more_layers_than_one_launch(dev, op):
    """70 layers: the library moves at most 64 per launch, so this takes two
    launches; every layer must match the oracle byte for byte."""
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(70 + len(op))
    layers, shape = 70, (16, 1, 64)
    sk, sv = _np_pools(rng, 12, layers, shape, np.uint16)
    if op == "copy":
        pairs = [(0, 5), (3, 6), (7, 1), (11, 10)]
        want_k, want_v = oracle.copy_blocks(sk, sv, pairs)
        tk = [_torch(a, "gpu", dev, "f16") for a in sk]
        tv = [_torch(a, "gpu", dev, "f16") for a in sv]
        pa.copy_blocks(tk, tv, to_dev(np.array(pairs, dtype=np.int64), dev))
        got_k, got_v = tk, tv
    else:
        dk, dv = _np_pools(rng, 9, layers, shape, np.uint16)
        pairs = [(2, 8), (9, 0), (4, 4)]
        want_k, want_v = oracle.swap_blocks(sk, sv, dk, dv, pairs)
        tk = [_torch(a, "gpu", dev, "f16") for a in sk]
        tv = [_torch(a, "gpu", dev, "f16") for a in sv]
        got_k = [_torch(a, "host", dev, "f16") for a in dk]
        got_v = [_torch(a, "host", dev, "f16") for a in dv]
        pa.swap_blocks(tk, tv, got_k, got_v, to_dev(np.array(pairs, dtype=np.int64), dev))
    torch.cuda.synchronize()
    assert pa.get_device_error(dev) == 0
    for i in range(layers):
        assert np.array_equal(bits_of(got_k[i]), want_k[i]), f"K of layer {i}"
        assert np.array_equal(bits_of(got_v[i]), want_v[i]), f"V of layer {i}"
