"""The host block manager against the pages' printed allocator numbers.

The block manager only lays out synthetic workloads, but its numbers are the
pages' own: the allocator toy's printed output and the worked memory example.
"""
import json
import math
import os

import numpy as np
import pytest

from workloads import BlockPool, PoolExhausted, SeqTable, kv_bytes_per_token, make_config


def _load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def test_allocator_toy_output(golden_dir):
    g = _load(golden_dir, "allocator_toy.json")
    b, nblk, max_len = g["block_size"], g["pool_blocks"], g["max_len"]
    # contiguous reservation
    used, real = 0, 0
    for name, (p, gen) in g["requests"].items():
        assert used + max_len <= nblk * b
        used += max_len
        real += p + gen
        assert max_len - (p + gen) == g["contiguous"]["wasted"][name]
    assert used == g["contiguous"]["reserved"] and real == g["contiguous"]["really_needed"]
    assert round(100 * (used - real) / used) == g["contiguous"]["waste_pct"]
    # paged, on demand
    pool = BlockPool(nblk, b)
    seqs = {}
    for name, (p, gen) in g["requests"].items():
        s = SeqTable(pool)
        s.admit(p)
        for _ in range(gen):
            s.append()
        seqs[name] = s
        assert len(s.table) == g["paged"]["blocks"][name]
        assert s.length == g["paged"]["tokens"][name]
        assert len(s.table) * b - s.length == g["paged"]["wasted"][name]
    held = sum(len(s.table) for s in seqs.values()) * b
    assert held == g["paged"]["held"]
    assert round(100 * (held - g["paged"]["really_needed"]) / held) == g["paged"]["waste_pct"]
    assert pool.num_free == g["paged"]["blocks_free"]
    # sharing a system prompt
    sh = g["sharing"]
    pool = BlockPool(nblk, b)
    root = SeqTable(pool)
    root.admit(sh["system_tokens"])
    users = [root.fork() for _ in range(sh["users"])]
    root.free()
    assert len(root.table) == 0 and len(users[0].table) == sh["shared_blocks"]
    assert all(pool.ref[i] == sh["refcount"] for i in users[0].table)
    assert sh["users"] * len(users[0].table) == sh["copied_blocks"]
    assert nblk - pool.num_free == sh["shared_blocks"]
    assert (sh["users"] - 1) * sh["shared_blocks"] * b == sh["saved_slots"]


def test_worked_memory_example(golden_dir):
    g = _load(golden_dir, "memory_accounting.json")
    ex = g["worked_example"]
    b = ex["block_size"]
    pool = BlockPool(4096, b)
    seqs = []
    for L in ex["lengths"]:
        s = SeqTable(pool)
        s.admit(L)
        seqs.append(s)
    assert [len(s.table) for s in seqs] == ex["blocks"]
    total = sum(len(s.table) for s in seqs)
    assert total == ex["total_blocks"] and total * b == ex["slots"]
    assert [len(s.table) * b - s.length for s in seqs] == ex["waste"]
    assert sum(ex["waste"]) == ex["total_waste"]
    assert round(100 * sum(ex["lengths"]) / (total * b), 1) == ex["utilisation_pct"]
    reserved = len(ex["lengths"]) * ex["max_len"]
    assert reserved == ex["reserved_slots"]
    assert round(100 * sum(ex["lengths"]) / reserved, 1) == ex["reserved_utilisation_pct"]
    llama = g["llama3_8b_shape"]
    bpt = kv_bytes_per_token(llama["layers"], llama["kv_heads"], llama["head_dim"], llama["dtype_bytes"])
    assert bpt == llama["bytes_per_token"] == ex["bytes_per_token"]
    assert round(reserved * bpt / 1e9, 2) == ex["reserved_gb"]
    assert round(total * b * bpt / 1e6) == ex["paged_mb"]
    assert int(60e9 // (ex["max_len"] * bpt)) == ex["reserve_fit_60gb"]


def test_utilisation_bounds(golden_dir):
    g = _load(golden_dir, "memory_accounting.json")
    u = g["utilisation_bound"]
    S, b = u["mean_len"], u["block_size"]
    # the worst case wastes b-1 slots: S / (S + b - 1)
    assert round(100 * S / (S + b - 1), 1) == u["paged_at_least_pct"]
    assert round(100 * S / u["max_len"], 1) == u["reserve_pct"]
    e = g["eta_bound"]
    s, B = e["seq_len"], e["block_size"]
    bound = 1 - B / (s + B)
    assert round(100 * bound, 2) == e["bound_pct"]
    for L in range(1, 5000, 7):
        eta = L / (math.ceil(L / B) * B)
        assert eta >= L / (L + B) - 1e-15
    m = g["m_kv_70b"]
    bpt = kv_bytes_per_token(m["layers"], m["kv_heads"], m["head_dim"], m["dtype_bytes"])
    assert bpt == m["bytes_per_token"]
    assert round(bpt / 1024) == m["approx_kb_per_token"]


def test_copy_on_write_once_per_sharer():
    """Forking k sequences off a partially filled block: every sharer but the last
    writer copies that one block, exactly once."""
    pool = BlockPool(100, 16, free_order=np.random.default_rng(0).permutation(100))
    root = SeqTable(pool)
    root.admit(40)
    kids = [root.fork() for _ in range(5)]
    root.free()
    pairs = []
    for c in kids:
        for _ in range(30):
            p = c.append()
            if p:
                pairs.append(p)
    assert len(pairs) == 4
    assert len({src for src, _ in pairs}) == 1
    assert len({dst for _, dst in pairs}) == 4
    shared = kids[0].table[:2]
    assert all(k.table[:2] == shared for k in kids)
    assert all(pool.ref[i] == 5 for i in shared)
    for c in kids:
        c.free()
    assert pool.num_free == 100


def test_exhaustion_raises():
    pool = BlockPool(2, 4)
    s = SeqTable(pool)
    s.admit(8)
    with pytest.raises(PoolExhausted):
        s.append()


def test_config_shapes():
    w1 = make_config(1)
    assert w1.seq_lens.tolist() == [10, 1, 16, 33] and w1.num_blocks == 64
    assert w1.key.shape == (60, 4, 64)
    w5 = make_config(5)
    assert w5.copy_pairs.shape == (255, 2)
    assert len(set(w5.copy_pairs[:, 1].tolist())) == 255
    assert not set(w5.copy_pairs[:, 1].tolist()) & set(w5.copy_pairs[:, 0].tolist())
    assert (w5.block_tables[:, :62] == w5.block_tables[0, :62]).all()
    assert w5.seq_lens.min() >= 1016 and w5.seq_lens.max() <= 1512
