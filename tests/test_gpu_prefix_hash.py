"""GPU parity for pa_prefix_hash: every key byte-equal to the oracle's SHA-256
chain (hashlib), for many block sizes, lengths (empty, partial, exact, long),
roots, and the pages' shared-system-prefix example; bad key ranges flagged."""
import json
import os

import numpy as np
import pytest
import torch

import oracle

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


def _batch(seqs, dev):
    toks = np.concatenate([np.asarray(s, dtype=np.int32) for s in seqs] + [np.zeros(0, np.int32)])
    off = np.concatenate([[0], np.cumsum([len(s) for s in seqs])]).astype(np.int64)
    return torch.from_numpy(toks).to(dev), torch.from_numpy(off).to(dev)


def _want(seqs, b, root=None):
    keys = [k for s in seqs for k in oracle.prefix_block_keys(list(s), b, root)]
    return np.frombuffer(b"".join(keys), dtype=np.uint8).reshape(-1, 32)


@pytest.mark.parametrize("b", [1, 3, 8, 16, 32, 64, 128])
def test_keys_match_oracle(dev, b):
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(b)
    lens = [0, 1, b - 1, b, b + 1, 3 * b, 7 * b + 5] + rng.integers(0, 12 * b, 20).tolist()
    seqs = [rng.integers(-2**31, 2**31, size=n, dtype=np.int64).astype(np.int32) for n in lens]
    toks, off = _batch(seqs, dev)
    for root in (None, bytes(range(32))):
        keys = pa.prefix_hash(toks, off, b, root=root)
        assert pa.get_device_error(dev) == 0
        assert np.array_equal(keys.cpu().numpy(), _want(seqs, b, root))


def test_pages_shared_prefix_example(dev, golden_dir):
    import paged_kv_cache_114_gb300 as pa
    with open(os.path.join(golden_dir, "prefix_sharing_example.json")) as f:
        g = json.load(f)
    seqs = [g["system_prefix"] + g["req1_prompt_suffix"], g["system_prefix"] + g["req2_prompt_suffix"]]
    toks, off = _batch(seqs, dev)
    keys = pa.prefix_hash(toks, off, g["block_size"]).cpu().numpy()
    assert keys.shape == (2, 32) and np.array_equal(keys[0], keys[1])
    assert np.array_equal(keys, _want(seqs, g["block_size"]))


def test_long_batch(dev):
    """512 prompts of up to 4,096 tokens at b = 16, against the oracle."""
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(77)
    seqs = [rng.integers(0, 128000, size=int(n)).astype(np.int32) for n in rng.integers(0, 4097, 512)]
    toks, off = _batch(seqs, dev)
    keys = pa.prefix_hash(toks, off, 16)
    assert pa.get_device_error(dev) == 0
    assert np.array_equal(keys.cpu().numpy(), _want(seqs, 16))


def test_wrong_key_range_is_flagged(dev):
    import paged_kv_cache_114_gb300 as pa
    seqs = [list(range(40)), list(range(33))]
    toks, off = _batch(seqs, dev)
    bad = torch.tensor([0, 2, 4], dtype=torch.int64, device=dev)  # sequence 1 needs 2 keys: ok; 0 needs 2: ok
    out = torch.zeros((4, 32), dtype=torch.uint8, device=dev)
    pa.prefix_hash(toks, off, 16, key_offsets=bad, out=out)
    assert pa.get_device_error(dev) == 0
    bad = torch.tensor([0, 3, 4], dtype=torch.int64, device=dev)  # sequence 0 given 3 slots
    out.zero_()
    pa.prefix_hash(toks, off, 16, key_offsets=bad, out=out)
    assert pa.get_device_error(dev) & pa.DEVERR_SEQ_LEN
    assert torch.count_nonzero(out[:3]) == 0  # sequence 0 wrote nothing


@pytest.mark.parametrize("n_seqs", [0, 1, 5, 8192, 8193, 20000])
def test_key_offsets_on_device(dev, n_seqs):
    """pa_prefix_key_offsets packs floor(len / b) keys per sequence back to
    back, exactly the oracle's key counts summed in order; chunk edges of the
    device scan (8,192 sequences) included."""
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(n_seqs)
    lens = rng.integers(0, 200, n_seqs)
    lens[::7] = 0
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)).to(dev)
    for b in (1, 16, 33):
        got = pa.prefix_key_offsets(off, b).cpu().numpy()
        counts = [len(oracle.prefix_block_keys([0] * int(n), b)) for n in lens] if n_seqs <= 5 \
            else (lens // b).tolist()
        want = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        assert pa.get_device_error(dev) == 0
        assert np.array_equal(got, want)


def test_negative_length_is_flagged_in_offsets(dev):
    import paged_kv_cache_114_gb300 as pa
    off = torch.tensor([0, 40, 30, 64], dtype=torch.int64, device=dev)  # sequence 1 has length -10
    got = pa.prefix_key_offsets(off, 16).cpu().numpy()
    assert pa.get_device_error(dev) & pa.DEVERR_SEQ_LEN
    assert got.tolist() == [0, 2, 2, 4]
