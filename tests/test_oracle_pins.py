"""Pins for the fp64 oracle: what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a worked
value printed on the pages (fixtures under tests/golden/), a closed form, a
library routine (torch's scaled_dot_product_attention in fp64 on the CPU), or
an invariant the pages state (placement independence, shared == private).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from workloads import BlockPool, SeqTable, make_config, make_random_case
from workloads.configs import to_bits


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# slot mapping


def test_ten_token_example(golden_dir):
    """Ten tokens, b=4, table [7, 2, 11]: positions 0-3 -> 7, 4-7 -> 2, 8-9 -> 11;
    token 6 sits in physical block 2 at offset 2."""
    g = _load(golden_dir, "mapping_10tok_b4.json")
    b, n = g["block_size"], g["num_tokens"]
    table = np.array([g["block_table"]], dtype=np.int32)
    slots = oracle.slot_mapping(table, [0] * n, list(range(n)), b)
    assert [int(s) // b for s in slots] == g["physical_block_of_position"]
    t6 = g["token6"]
    assert int(slots[t6["position"]]) // b == t6["physical_block"]
    assert int(slots[t6["position"]]) % b == t6["offset"]
    touched = {int(s) // b for s in slots}
    assert len(touched) * b == g["allocated_slots"]
    assert len(touched) * b - n == g["unused_slots"]


def test_identity_table_slot_is_position():
    """With table[j] = j the pool rows are the sequence itself: slot(t) = t."""
    for b in (1, 2, 4, 8, 16, 32):
        n = 5 * b + 3
        table = np.arange(-(-n // b), dtype=np.int32)[None]
        slots = oracle.slot_mapping(table, [0] * n, range(n), b)
        assert slots.tolist() == list(range(n))
        shifted = (table + 9).astype(np.int32)
        slots = oracle.slot_mapping(shifted, [0] * n, range(n), b)
        assert slots.tolist() == [9 * b + t for t in range(n)]


@pytest.mark.parametrize("b", [1, 4, 8, 16, 32])
def test_slot_waste_formula(b):
    """A sequence of n tokens fills b*ceil(n/b) slots; b*ceil(n/b) - n in [0, b-1]
    of them stay unused, all in its last block."""
    rng = np.random.default_rng(b)
    for n in range(1, 1001):
        if n > 64 and n % 37:
            continue
        nblk = -(-n // b)
        pool = BlockPool(nblk + 7, b, free_order=rng.permutation(nblk + 7))
        s = SeqTable(pool)
        s.admit(n)
        slots = oracle.slot_mapping(np.array([s.table], dtype=np.int32), [0] * n, range(n), b)
        assert len(set(slots.tolist())) == n
        owned = {blk * b + off for blk in s.table for off in range(b)}
        assert set(slots.tolist()) <= owned
        waste = len(owned) - n
        assert waste == b * math.ceil(n / b) - n
        assert 0 <= waste <= b - 1
        last = s.table[-1]
        assert all(x // b == last for x in owned - set(slots.tolist()))


def test_config1_waste_per_sequence():
    """Config 1 lengths {10, 1, 16, 33} at b=4 waste {2, 3, 0, 3} slots."""
    w = make_config(1)
    b = w.block_size
    waste = []
    for s, L in enumerate(w.seq_lens.tolist()):
        slots = oracle.slot_mapping(w.block_tables, [s] * L, range(L), b)
        owned = {int(x) // b for x in slots}
        waste.append(len(owned) * b - L)
    assert waste == [2, 3, 0, 3]
    assert w.block_tables[0, :3].tolist() == [7, 2, 11]


# ----------------------------------------------------------------------------
# KV write and block copy


def test_write_then_gather_round_trip(golden_dir):
    """Writing the ten-token example and gathering it back returns the rows in
    logical order; token 6's row lands in block 2, row 2; every other slot keeps
    its old bytes."""
    g = _load(golden_dir, "mapping_10tok_b4.json")
    b, n = g["block_size"], g["num_tokens"]
    rng = np.random.default_rng(7)
    hkv, d = 3, 8
    k0 = rng.integers(0, 2**16, size=(16, b, hkv, d), dtype=np.uint16)
    v0 = rng.integers(0, 2**16, size=(16, b, hkv, d), dtype=np.uint16)
    key = rng.integers(0, 2**16, size=(n, hkv, d), dtype=np.uint16)
    val = rng.integers(0, 2**16, size=(n, hkv, d), dtype=np.uint16)
    table = np.array([g["block_table"]], dtype=np.int32)
    slots = oracle.slot_mapping(table, [0] * n, range(n), b)
    k1, v1 = oracle.write_kv(k0, v0, key, val, slots)
    t6 = g["token6"]
    assert np.array_equal(k1[t6["physical_block"], t6["offset"]], key[6])
    for h in range(hkv):
        assert np.array_equal(oracle.gather_kv(k1, table[0], n, h), key[:, h])
        assert np.array_equal(oracle.gather_kv(v1, table[0], n, h), val[:, h])
    mask = np.ones(16 * b, dtype=bool)
    mask[slots] = False
    assert np.array_equal(k1.reshape(16 * b, hkv, d)[mask], k0.reshape(16 * b, hkv, d)[mask])
    assert np.array_equal(v1.reshape(16 * b, hkv, d)[mask], v0.reshape(16 * b, hkv, d)[mask])
    # padding slots write nothing
    k2, v2 = oracle.write_kv(k0, v0, key[:2], val[:2], [-1, -1])
    assert np.array_equal(k2, k0) and np.array_equal(v2, v0)


def test_copy_blocks_copies_whole_blocks_every_layer():
    rng = np.random.default_rng(3)
    layers = [rng.integers(0, 2**16, size=(10, 4, 2, 8), dtype=np.uint16) for _ in range(3)]
    vlayers = [rng.integers(0, 2**16, size=(10, 4, 2, 8), dtype=np.uint16) for _ in range(3)]
    pairs = [(1, 7), (1, 8), (4, 2)]
    ks, vs = oracle.copy_blocks(layers, vlayers, pairs)
    for k0, v0, k1, v1 in zip(layers, vlayers, ks, vs):
        for src, dst in pairs:
            assert np.array_equal(k1[dst], k0[src]) and np.array_equal(v1[dst], v0[src])
        untouched = [i for i in range(10) if i not in {7, 8, 2}]
        assert np.array_equal(k1[untouched], k0[untouched])
        assert np.array_equal(v1[untouched], v0[untouched])


# ----------------------------------------------------------------------------
# decode attention


def _sdpa_contiguous(q_bits, K_bits, V_bits, lens, scale, dtype):
    """torch SDPA in fp64 on contiguous per-sequence K/V (the textbook routine)."""
    g = q_bits.shape[1] // K_bits.shape[2]
    outs = []
    for s, L in enumerate(lens):
        q = torch.from_numpy(oracle.bits_to_f64(q_bits[s], dtype))[:, None, :]       # [Hq,1,D]
        K = torch.from_numpy(oracle.bits_to_f64(K_bits[s, :L], dtype)).transpose(0, 1)  # [Hkv,L,D]
        V = torch.from_numpy(oracle.bits_to_f64(V_bits[s, :L], dtype)).transpose(0, 1)
        K = K.repeat_interleave(g, dim=0)
        V = V.repeat_interleave(g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(q, K, V, scale=scale)
        outs.append(o[:, 0, :].numpy())
    return np.stack(outs)


@pytest.mark.parametrize("dtype,hq,hkv,b", [("f16", 4, 4, 4), ("bf16", 8, 2, 8),
                                            ("f16", 6, 3, 16), ("bf16", 4, 1, 1)])
def test_identity_tables_match_contiguous_attention(dtype, hq, hkv, b):
    """Blocks laid out in order reproduce contiguous attention (the math is
    unchanged; only the addresses are indirect)."""
    rng = np.random.default_rng(11)
    d, n = 16, 4
    lens = [1, b + 1, 3 * b, 5 * b - 1]
    m = -(-max(lens) // b)
    Kc = to_bits(rng.standard_normal((n, m * b, hkv, d), dtype=np.float32), dtype)
    Vc = to_bits(rng.standard_normal((n, m * b, hkv, d), dtype=np.float32), dtype)
    q = to_bits(rng.standard_normal((n, hq, d), dtype=np.float32), dtype)
    pool_k = Kc.reshape(n * m, b, hkv, d)   # sequence s owns blocks s*m .. s*m+m-1
    pool_v = Vc.reshape(n * m, b, hkv, d)
    tables = (np.arange(n)[:, None] * m + np.arange(m)[None]).astype(np.int32)
    scale = 0.3
    got = oracle.decode(q, pool_k, pool_v, tables, lens, scale, dtype)
    want = _sdpa_contiguous(q, Kc, Vc, lens, scale, dtype)
    assert np.max(np.abs(got - want)) < 1e-12


def test_placement_permutation_is_invisible():
    """Moving blocks to other physical ids (and remapping the tables) leaves every
    output bit-identical."""
    w = make_random_case(5, num_seqs=6, num_q_heads=8, num_kv_heads=2, head_dim=32,
                         block_size=8, seq_lens=[1, 7, 8, 9, 40, 63], dtype="bf16")
    base = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    t2 = perm[w.block_tables].astype(np.int32)
    moved = oracle.decode(w.q, k2, v2, t2, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(base, moved)


def test_length_one_returns_the_value_row():
    """One token: softmax weight 1, output = V[0] exactly."""
    w = make_random_case(9, num_seqs=3, num_q_heads=4, num_kv_heads=2, head_dim=16,
                         block_size=4, seq_lens=[1, 1, 1], dtype="f16")
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    for s in range(3):
        blk = w.block_tables[s, 0]
        for h in range(4):
            assert np.array_equal(out[s, h], oracle.bits_to_f64(w.v_cache[blk, 0, h // 2], "f16"))


def test_equal_keys_average_the_values():
    """All keys equal: uniform weights, output = mean of the value rows."""
    rng = np.random.default_rng(2)
    b, L, d = 4, 11, 8
    k = np.zeros((3, b, 1, d), dtype=np.uint16)
    k[:] = to_bits(rng.standard_normal(d, dtype=np.float32), "f16")
    v = to_bits(rng.standard_normal((3, b, 1, d), dtype=np.float32), "f16")
    q = to_bits(rng.standard_normal((1, 1, d), dtype=np.float32), "f16")
    table = np.array([[2, 0, 1]], dtype=np.int32)
    out = oracle.decode(q, k, v, table, [L], 0.7, "f16")
    rows = oracle.bits_to_f64(np.concatenate([v[2], v[0], v[1]])[:L, 0], "f16")
    assert np.allclose(out[0, 0], rows.mean(axis=0), rtol=0, atol=1e-14)


def test_two_tokens_closed_form():
    """Two keys: weights are the logistic function of the logit difference."""
    rng = np.random.default_rng(4)
    d = 8
    kf = rng.standard_normal((2, d)).astype(np.float32)
    vf = rng.standard_normal((2, d)).astype(np.float32)
    qf = rng.standard_normal(d).astype(np.float32)
    k = np.zeros((1, 2, 1, d), dtype=np.uint16)
    v = np.zeros((1, 2, 1, d), dtype=np.uint16)
    k[0, :, 0] = to_bits(kf, "f16")
    v[0, :, 0] = to_bits(vf, "f16")
    q = to_bits(qf, "f16")[None, None]
    K = k[0, :, 0].view(np.float16).astype(np.float64)
    V = v[0, :, 0].view(np.float16).astype(np.float64)
    Q = q[0, 0].view(np.float16).astype(np.float64)
    scale = 0.25
    delta = scale * float(Q @ (K[0] - K[1]))
    w0 = 1.0 / (1.0 + math.exp(-delta))
    want = w0 * V[0] + (1.0 - w0) * V[1]
    got = oracle.decode(q, k, v, np.array([[0]], dtype=np.int32), [2], scale, "f16")
    assert np.max(np.abs(got[0, 0] - want)) < 1e-14


def test_zero_length_gives_zeros():
    w = make_random_case(3, num_seqs=2, num_q_heads=2, num_kv_heads=1, head_dim=8,
                         block_size=4, seq_lens=[0, 5], dtype="f16")
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(out[0], np.zeros((2, 8)))
    assert np.all(np.isfinite(out[1]))


def test_tail_slots_never_read():
    """Slots past the length hold NaN in every generated pool; outputs stay finite
    and equal to attention over the valid rows only."""
    w = make_random_case(8, num_seqs=4, num_q_heads=2, num_kv_heads=2, head_dim=8,
                         block_size=8, seq_lens=[3, 9, 15, 17], dtype="bf16")
    out = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.all(np.isfinite(out))


def test_shared_prefix_equals_private_copies():
    """Tables pointing at shared (copy-on-write) prefix blocks give the same output
    as tables whose prefix blocks are private copies."""
    rng = np.random.default_rng(21)
    b, hkv, hq, d = 4, 2, 4, 8
    pool = BlockPool(64, b, free_order=rng.permutation(64))
    root = SeqTable(pool)
    root.admit(10)                        # 2 full blocks + 2 rows of a third
    kids = [root.fork() for _ in range(3)]
    root.free()
    k = to_bits(rng.standard_normal((64, b, hkv, d), dtype=np.float32), "f16")
    v = to_bits(rng.standard_normal((64, b, hkv, d), dtype=np.float32), "f16")
    pairs = []
    for c in kids:
        for _ in range(5):
            p = c.append()
            if p:
                pairs.append(p)
    assert len(pairs) == 2                # the last writer keeps the original block
    ks, vs = oracle.copy_blocks([k], [v], pairs)
    k, v = ks[0], vs[0]
    lens = [c.length for c in kids]
    shared_tables = np.array([c.table for c in kids], dtype=np.int32)
    q = to_bits(rng.standard_normal((3, hq, d), dtype=np.float32), "f16")
    shared = oracle.decode(q, k, v, shared_tables, lens, 0.5, "f16")
    # private: copy every block of every sequence to fresh ids
    k2 = np.concatenate([k, np.zeros((3 * 4, b, hkv, d), np.uint16)])
    v2 = np.concatenate([v, np.zeros((3 * 4, b, hkv, d), np.uint16)])
    priv = np.zeros_like(shared_tables)
    nxt = 64
    for s in range(3):
        for j, blk in enumerate(shared_tables[s]):
            k2[nxt], v2[nxt] = k[blk], v[blk]
            priv[s, j] = nxt
            nxt += 1
    private = oracle.decode(q, k2, v2, priv, lens, 0.5, "f16")
    assert np.array_equal(shared, private)


@pytest.mark.parametrize("b", [1, 3, 4, 16])
def test_online_recurrence_and_partition_combine(b):
    """The blockwise running-max recurrence, and the (m, l, o) partition combine,
    reach textbook softmax attention."""
    rng = np.random.default_rng(b)
    L, d = 50, 16
    K = rng.standard_normal((L, d)) * 2
    V = rng.standard_normal((L, d))
    q = rng.standard_normal(d)
    want = oracle.attention(q[None], K, V, 0.4)[0]
    assert np.max(np.abs(oracle.online_softmax_blocks(q, K, V, 0.4, b) - want)) < 1e-12
    cuts = [0, 7, 8, 30, 50]
    states = [oracle.partition_state(q, K[a:c], V[a:c], 0.4) for a, c in zip(cuts, cuts[1:])]
    assert np.max(np.abs(oracle.combine_partitions(states) - want)) < 1e-12
    assert np.max(np.abs(oracle.combine_partitions([oracle.partition_state(q, K, V, 0.4)]) - want)) < 1e-12


def test_attention_matches_scipy_softmax():
    """Cross-check against scipy's softmax with large logits (shift invariance)."""
    from scipy.special import softmax
    rng = np.random.default_rng(6)
    K = rng.standard_normal((30, 8)) * 40
    V = rng.standard_normal((30, 8))
    q = rng.standard_normal((3, 8))
    want = softmax(0.9 * q @ K.T, axis=1) @ V
    assert np.max(np.abs(oracle.attention(q, K, V, 0.9) - want)) < 1e-12


def test_gqa_mapping_uses_contiguous_groups():
    """Query head h reads KV head h // g: putting distinct constant values in each
    KV head's V identifies which head every query head read."""
    hq, hkv, d, b = 8, 2, 4, 4
    k = np.zeros((2, b, hkv, d), dtype=np.uint16)
    v = np.zeros((2, b, hkv, d), dtype=np.uint16)
    for h in range(hkv):
        v[:, :, h, :] = to_bits(np.full((2, b, d), float(h + 1), np.float32), "f16")
    q = np.zeros((1, hq, d), dtype=np.uint16)
    out = oracle.decode(q, k, v, np.array([[1, 0]], dtype=np.int32), [6], 1.0, "f16")
    assert np.allclose(out[0, :, 0], [1, 1, 1, 1, 2, 2, 2, 2], rtol=0, atol=1e-14)


@pytest.mark.parametrize("dtype,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_widening_matches_torch_conversion(dtype, tdt):
    """Bit patterns widen to the same fp64 values torch's own dtype conversion gives."""
    bits = np.arange(0, 2**16, dtype=np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(tdt).to(torch.float64).numpy()
    with np.errstate(invalid="ignore"):
        got = oracle.bits_to_f64(bits, dtype)
    finite = np.isfinite(want)
    assert np.array_equal(got[finite], want[finite])
    assert np.array_equal(np.isnan(got), np.isnan(want))
