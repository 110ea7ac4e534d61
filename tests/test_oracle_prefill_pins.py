"""Pins for the oracle's multi-token (chunked prefill / speculative verify)
attention: what the pages and the mathematics fix.

The i-th of a sequence's n new queries sits at position L - n + i and may
attend to positions 0 .. L - n + i ("PagedAttention: Manage the Cache Without
Moving the Sequence", §The kernel must understand the mapping: masks give the
allowed attention edges, the block table only where rows are stored). Each
test checks the oracle against something other than itself: torch's
scaled_dot_product_attention with its causal mask, the decode oracle (pinned
on its own), closed forms, and invariants of the mask.
"""
import numpy as np
import pytest
import torch

import oracle
from workloads import make_prefill_case


def _contiguous(w):
    """Per sequence, the K/V rows of positions 0 .. L-1 in logical order, fp64."""
    ks, vs = [], []
    for s, L in enumerate(w.seq_lens.tolist()):
        k = np.stack([oracle.gather_kv(w.k_cache, w.block_tables[s], L, h) for h in range(w.num_kv_heads)])
        v = np.stack([oracle.gather_kv(w.v_cache, w.block_tables[s], L, h) for h in range(w.num_kv_heads)])
        ks.append(oracle.bits_to_f64(k, w.dtype))
        vs.append(oracle.bits_to_f64(v, w.dtype))
    return ks, vs


@pytest.mark.parametrize("dtype,hq,hkv,b", [("f16", 4, 4, 4), ("bf16", 8, 2, 16), ("f16", 6, 3, 8)])
def test_whole_prompt_matches_torch_causal_attention(dtype, hq, hkv, b):
    """n = L (the whole prompt at once): every query position equals its row
    index, so the mask is torch's lower-triangular causal mask."""
    lens = [1, 5, 2 * b, 3 * b + 1]
    w = make_prefill_case(21, num_seqs=4, num_q_heads=hq, num_kv_heads=hkv, head_dim=16,
                          block_size=b, seq_lens=lens, q_lens=lens, dtype=dtype)
    got = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                         w.scale, w.dtype)
    ks, vs = _contiguous(w)
    g = hq // hkv
    for s, L in enumerate(lens):
        lo = int(w.q_start[s])
        q = torch.from_numpy(oracle.bits_to_f64(w.q[lo:lo + L], dtype)).permute(1, 0, 2)  # [Hq, L, D]
        k = torch.from_numpy(ks[s]).repeat_interleave(g, dim=0)
        v = torch.from_numpy(vs[s]).repeat_interleave(g, dim=0)
        want = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True,
                                                                scale=w.scale)
        assert np.max(np.abs(got[lo:lo + L] - want.permute(1, 0, 2).numpy())) < 1e-12


def test_one_query_per_sequence_is_decode():
    """n = 1: the single query sits at position L - 1 and sees every token,
    which is decode attention."""
    lens = [1, 7, 33, 64]
    w = make_prefill_case(22, num_seqs=4, num_q_heads=8, num_kv_heads=2, head_dim=32,
                          block_size=8, seq_lens=lens, q_lens=[1, 1, 1, 1], dtype="bf16")
    got = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                         w.scale, w.dtype)
    want = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(got, want)


def test_first_query_of_a_prompt_returns_its_value_row():
    """The query at position 0 may only see token 0: weight 1, output V[0]
    exactly. A chunk that starts later sees more than one token."""
    w = make_prefill_case(23, num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim=16,
                          block_size=4, seq_lens=[9, 9], q_lens=[9, 3], dtype="f16")
    got = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                         w.scale, w.dtype)
    ks, vs = _contiguous(w)
    assert np.array_equal(got[0], vs[0][:, 0, :])
    # sequence 1's first query sits at position 6: not the value row of token 0
    assert not np.allclose(got[int(w.q_start[1])], vs[1][:, 0, :])


def test_future_rows_are_invisible_and_the_own_row_is_seen():
    """Changing K/V at positions after p leaves query p unchanged; changing
    the row at p itself changes it (the mask is inclusive)."""
    L, n = 23, 6
    w = make_prefill_case(24, num_seqs=1, num_q_heads=4, num_kv_heads=2, head_dim=16,
                          block_size=4, seq_lens=[L], q_lens=[n], dtype="bf16")
    base = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                          w.scale, w.dtype)
    b = w.block_size
    for i in range(n):
        p = L - n + i
        k2, v2 = w.k_cache.copy(), w.v_cache.copy()
        for t in range(p + 1, L):
            blk, off = int(w.block_tables[0][t // b]), t % b
            k2[blk, off] ^= np.uint16(0x1234)
            v2[blk, off] ^= np.uint16(0x0421)
        after = oracle.prefill(w.q, w.q_start, k2, v2, w.block_tables, w.seq_lens, w.scale, w.dtype)
        assert np.array_equal(after[i], base[i])
        if p + 1 < L:
            assert not np.array_equal(after[i + 1], base[i + 1])
        k3 = w.k_cache.copy()
        blk, off = int(w.block_tables[0][p // b]), p % b
        k3[blk, off] ^= np.uint16(0x0300)
        own = oracle.prefill(w.q, w.q_start, k3, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
        assert not np.allclose(own[i], base[i])


def test_a_chunk_equals_the_tail_of_the_whole_prompt():
    """Running the last c tokens as a chunk gives the same rows as running the
    whole prompt (chunked prefill changes nothing about the result)."""
    L = 40
    full = make_prefill_case(25, num_seqs=1, num_q_heads=6, num_kv_heads=2, head_dim=32,
                             block_size=8, seq_lens=[L], q_lens=[L], dtype="f16")
    whole = oracle.prefill(full.q, full.q_start, full.k_cache, full.v_cache, full.block_tables,
                           full.seq_lens, full.scale, full.dtype)
    for c in (1, 7, 16, 39):
        part = oracle.prefill(full.q[L - c:], np.array([0, c]), full.k_cache, full.v_cache,
                              full.block_tables, full.seq_lens, full.scale, full.dtype)
        assert np.array_equal(part, whole[L - c:])


def test_placement_permutation_is_invisible_for_chunks():
    w = make_prefill_case(26, num_seqs=3, num_q_heads=8, num_kv_heads=4, head_dim=16,
                          block_size=8, seq_lens=[17, 40, 8], q_lens=[5, 16, 8], dtype="bf16")
    base = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                          w.scale, w.dtype)
    perm = np.random.default_rng(2).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    moved = oracle.prefill(w.q, w.q_start, k2, v2, perm[w.block_tables].astype(np.int32),
                           w.seq_lens, w.scale, w.dtype)
    assert np.array_equal(base, moved)


def test_selected_rows_match_the_full_result():
    w = make_prefill_case(27, num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=16,
                          block_size=4, seq_lens=[13, 6], q_lens=[4, 6], dtype="f16")
    full = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                          w.scale, w.dtype)
    rows = [(0, 0), (3, 7), (5, 2), (9, 5)]
    some = oracle.prefill(w.q, w.q_start, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                          w.scale, w.dtype, rows=rows)
    for t, h in rows:  # fewer heads per product: the last bits may round differently
        assert np.max(np.abs(some[t, h] - full[t, h])) < 1e-12
    assert np.isnan(some[1, 1]).all()
