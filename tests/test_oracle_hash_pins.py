"""Pins for the oracle's prefix-cache keys (device-side prefix hashing).

The pages key cached blocks by their token ids. A hit needs an unbroken chain of
matching block keys from position zero, and the first differing token ends the
chain ("Paged Attention", firehose-demo; "PagedAttention",
learn.pranaymahendrakar.com, Prefix caching: hash each block-aligned prefix of
token ids). Only full blocks are keyed. The oracle reads this as key_j =
SHA-256(key_{j-1} || the block's int32 token ids), starting from a 32-byte
root. These tests check the chain against the pages' worked example and the
properties the pages state. They also check it against the SHA-256 standard's
own test vector and the byte layout written out independently.
"""
import hashlib
import json
import os

import numpy as np
import pytest

import oracle


def test_sha256_standard_vector():
    """FIPS 180-4's one-block example: SHA-256("abc")."""
    assert hashlib.sha256(b"abc").hexdigest() == (
        "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad")


def test_pages_shared_system_prefix(golden_dir):
    """The pages' simulation admits two prompts that share a 16-token system
    prefix: with the keys driving the allocator's prefix cache, the prefix block
    is shared (refcount 2) and the partial tails get private blocks, giving the
    tables the page's allocator produces from a fresh free list."""
    with open(os.path.join(golden_dir, "prefix_sharing_example.json")) as f:
        g = json.load(f)
    b = g["block_size"]
    prompts = [g["system_prefix"] + g["req1_prompt_suffix"], g["system_prefix"] + g["req2_prompt_suffix"]]
    free = list(range(128))
    cache, ref, tables = {}, {}, []
    for p in prompts:
        keys = oracle.prefix_block_keys(p, b)
        assert len(keys) == len(p) // b == 1
        table = []
        for j in range(-(-len(p) // b)):
            key = keys[j] if j < len(keys) else None
            if key is not None and key in cache:
                blk = cache[key]
                ref[blk] += 1
            else:
                blk = free.pop(0)
                ref[blk] = 1
                if key is not None:
                    cache[key] = blk
            table.append(blk)
        tables.append(table)
    assert tables == g["expected_tables"]
    assert ref[tables[0][0]] == g["expected_shared_block_refcount"]


def test_first_differing_token_ends_the_chain():
    rng = np.random.default_rng(1)
    b = 16
    a = rng.integers(0, 128000, size=10 * b).tolist()
    for k in (0, 3, 9):
        for pos in (0, 7, b - 1):
            bb = list(a)
            bb[k * b + pos] += 1
            ka, kb = oracle.prefix_block_keys(a, b), oracle.prefix_block_keys(bb, b)
            assert ka[:k] == kb[:k]
            assert all(x != y for x, y in zip(ka[k:], kb[k:]))


def test_same_block_at_another_position_gets_another_key():
    """A key covers the whole prefix, not the block alone: a repeated block
    does not collide with its first occurrence."""
    block = list(range(16))
    keys = oracle.prefix_block_keys(block * 3, 16)
    assert len(set(keys)) == 3


def test_only_full_blocks_are_keyed():
    for n, b in ((0, 16), (15, 16), (16, 16), (33, 16), (64, 8), (63, 8), (5, 1)):
        assert len(oracle.prefix_block_keys(list(range(n)), b)) == n // b


def test_root_separates_caches():
    t = list(range(64))
    a = oracle.prefix_block_keys(t, 16)
    r = oracle.prefix_block_keys(t, 16, root=bytes([7]) * 32)
    assert all(x != y for x, y in zip(a, r))


def test_message_layout():
    """key_0 for tokens 0x01020304 and -1 at b = 2 hashes 32 zero bytes, then
    each id as four little-endian bytes; key_1 chains on key_0. The bytes are
    written out here by hand."""
    t = [0x01020304, -1, 5, 6]
    k0 = hashlib.sha256(bytes(32) + bytes([4, 3, 2, 1, 255, 255, 255, 255])).digest()
    k1 = hashlib.sha256(k0 + bytes([5, 0, 0, 0, 6, 0, 0, 0])).digest()
    assert oracle.prefix_block_keys(t, 2) == [k0, k1]


@pytest.mark.parametrize("b", [1, 8, 16, 32])
def test_extending_a_sequence_keeps_its_keys(b):
    """Appending tokens never changes the keys of blocks already full."""
    t = list(range(5 * b + 3))
    short = oracle.prefix_block_keys(t, b)
    longer = oracle.prefix_block_keys(t + [99] * (2 * b), b)
    assert longer[:len(short)] == short
