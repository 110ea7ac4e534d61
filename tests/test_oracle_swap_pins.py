"""Pins for the oracle's swap (preemption to host memory and back).

Swapping copies a preempted sequence's blocks, all of them, every layer, K and V,
to host memory and later back ("PagedAttention: paging the KV cache", When
memory runs out; "PagedAttention" on learn.pranaymahendrakar.com,
Preemption). The block table is the only indirection, so a swapped-in
sequence may land on other block ids. These tests check the oracle against
that: byte equality per pair, untouched blocks, reduction to the block copy
(pinned on its own) when both pools are one, and the whole preemption round
trip through decode.
"""
import numpy as np

import oracle
from workloads import make_random_case


def _pools(rng, nb, layers=2, shape=(4, 2, 8), dtype=np.uint16):
    ks = [rng.integers(0, 2**16, size=(nb,) + shape).astype(dtype) for _ in range(layers)]
    vs = [rng.integers(0, 2**16, size=(nb,) + shape).astype(dtype) for _ in range(layers)]
    return ks, vs


def test_pairs_copy_blocks_between_pools():
    rng = np.random.default_rng(1)
    sk, sv = _pools(rng, 10)
    dk, dv = _pools(rng, 6)
    pairs = [(9, 0), (2, 5), (2, 3)]
    nk, nv = oracle.swap_blocks(sk, sv, dk, dv, pairs)
    for layer in range(2):
        for s, d in pairs:
            assert np.array_equal(nk[layer][d], sk[layer][s])
            assert np.array_equal(nv[layer][d], sv[layer][s])
        for d in (1, 2, 4):  # not a destination: unchanged
            assert np.array_equal(nk[layer][d], dk[layer][d])
            assert np.array_equal(nv[layer][d], dv[layer][d])
    assert all(a is not b for a, b in zip(nk, dk))  # destination arrays are new


def test_same_pool_reduces_to_copy_blocks():
    rng = np.random.default_rng(2)
    ks, vs = _pools(rng, 12, layers=3)
    pairs = [(1, 7), (1, 8), (4, 0)]
    a = oracle.swap_blocks(ks, vs, ks, vs, pairs)
    b = oracle.copy_blocks(ks, vs, pairs)
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert np.array_equal(x, y)


def test_preemption_round_trip_through_decode():
    """Swap a sequence out, let other sequences overwrite its device blocks,
    swap it back in to different block ids, remap its table: decode gives the
    same output as before preemption, bit for bit (placement independence)."""
    w = make_random_case(7, num_seqs=3, num_q_heads=8, num_kv_heads=2, head_dim=16,
                         block_size=4, seq_lens=[9, 14, 5], dtype="f16", pool_factor=2.0)
    before = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    s = 1
    nblk = -(-int(w.seq_lens[s]) // w.block_size)
    own = [int(b) for b in w.block_tables[s, :nblk]]
    host_k = np.zeros((nblk,) + w.k_cache.shape[1:], dtype=w.k_cache.dtype)
    host_v = np.zeros_like(host_k)
    (hk,), (hv,) = oracle.swap_blocks([w.k_cache], [w.v_cache], [host_k], [host_v],
                                      [(b, i) for i, b in enumerate(own)])
    # other work reuses (overwrites) the freed device blocks
    k_dev, v_dev = w.k_cache.copy(), w.v_cache.copy()
    k_dev[own] = 0x7E00
    v_dev[own] = 0x7E00
    # swap in to blocks nobody owns
    used = set(int(b) for r, L in zip(w.block_tables, w.seq_lens)
               for b in r[: -(-int(L) // w.block_size)])
    free = [b for b in range(w.num_blocks) if b not in used][:nblk]
    (k2,), (v2,) = oracle.swap_blocks([hk], [hv], [k_dev], [v_dev], list(enumerate(free)))
    tables = w.block_tables.copy()
    tables[s, :nblk] = free
    after = oracle.decode(w.q, k2, v2, tables, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(before, after)
