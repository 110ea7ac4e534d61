"""GPU parity for FP8 (E4M3) caches: the CUDA path through the C ABI against the
fp64 oracle.

An FP8 cache halves the bytes per block and changes nothing else about paging
("PagedAttention: paging the KV cache", Fine-tuned models and adapters): the
slot mapping and block tables are the same, the write stores E4M3 codes of
x / scale, the block copy moves codes, and decode reads code * scale. Writes
and copies are compared byte for byte; decode within 2e-3 max abs (plus half
an ulp of a 16-bit output dtype), every partition mode.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import (assert_close, bits_of, gpu_scenario, oracle_scenario,
                           to_dev)
from workloads import make_config, make_random_case
from workloads.configs import to_bits

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


def _check_bytes(res, ref):
    assert np.array_equal(res["slots"].cpu().numpy(), ref["slots"]), "slot mapping differs"
    assert np.array_equal(bits_of(res["k"]), ref["k"]), "K codes differ"
    assert np.array_equal(bits_of(res["v"]), ref["v"]), "V codes differ"


CASES = [
    # act dtype, D, Hq, Hkv, b, lens, partitions
    ("f16", 128, 8, 8, 16, [1, 15, 16, 17, 100, 333], (0, 64, -1)),
    ("bf16", 128, 32, 8, 16, [5, 512, 513, 1000], (0, 128, 512, -1)),
    ("f16", 128, 16, 1, 32, [1, 31, 32, 33, 700], (0, 96, -1)),
    ("bf16", 256, 8, 4, 8, [3, 64, 257], (0, 64, -1)),
    ("f16", 128, 12, 4, 4, [1, 4, 5, 99], (0, 32, -1)),
    ("bf16", 128, 64, 8, 16, [1, 2, 3, 16, 17, 4097], (0, 512, -1)),
    ("f16", 256, 16, 16, 16, [300, 1], (0, 128, -1)),
    ("bf16", 128, 8, 8, 16, [0, 0, 0], (0, -1)),
    ("f16", 128, 32, 2, 64, [1, 63, 64, 65, 1000], (0, 256, -1)),
    ("bf16", 128, 4, 4, 2, [0, 7, 0, 40], (0, 16, -1)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-d{c[1]}-{c[2]}x{c[3]}-b{c[4]}" for c in CASES])
def test_shapes(dev, case):
    dtype, d, hq, hkv, b, lens, parts = case
    w = make_random_case(sum(lens) + d + hq + 7, num_seqs=len(lens), num_q_heads=hq,
                         num_kv_heads=hkv, head_dim=d, block_size=b, seq_lens=lens, dtype=dtype,
                         kv_dtype="e4m3")
    ref = oracle_scenario(w)
    for p in parts:
        for odt in (torch.float32, torch.float16 if dtype == "f16" else torch.bfloat16):
            res = gpu_scenario(w, dev, partition_tokens=p, out_dtype=odt)
            assert res["err"] == 0
            _check_bytes(res, ref)
            assert_close(res["out"], ref["out"], what=f"partition {p} out {odt}")
            for i, L in enumerate(lens):
                if L == 0:
                    assert torch.count_nonzero(res["out"][i]) == 0


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_write_quantisation_edges(dev, dtype):
    """Rows built to hit every rounding case of the write: exact midpoints
    between codes (ties to even), one float32 step either side, values that
    round to +-0, subnormal codes and saturation, with a scale whose quotient
    is exact (7 * 2^-10) and one whose quotient is rounded (the workload's)."""
    import paged_kv_cache_114_gb300 as pa
    hkv, d = 2, 128
    grid = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    mids = (grid[:-1] + grid[1:]) / 2
    for scale in (7.0 / 1024.0, float(np.float32(3.0 / 448.0))):
        vals = np.concatenate([mids, -mids, grid, -grid, [1e-12, -1e-12, 0.0, -0.0, 500.0, -500.0,
                                                          448.0, 460.0, 470.0, -470.0]])
        x = (vals * scale).astype(np.float32)
        # round the inputs to the input dtype; midpoints stay exact at scale 7 * 2^-10
        bits = to_bits(x, dtype)
        n = hkv * d
        rows = -(-bits.size // n)
        key = np.resize(bits, rows * n).reshape(rows, hkv, d)
        value = key[::-1].copy()
        nb, b = rows, 1
        k = np.full((nb, b, hkv, d), 0x7F, dtype=np.uint8)
        v = np.full((nb, b, hkv, d), 0x7F, dtype=np.uint8)
        slots = np.arange(rows, dtype=np.int64)[::-1].copy()
        want_k, want_v = oracle.write_kv_e4m3(k, v, key, value, slots, dtype, scale, scale * 0.5)
        kd, vd = to_dev(k, dev), to_dev(v, dev)
        pa.write_kv(to_dev(key, dev, dtype), to_dev(value, dev, dtype), to_dev(slots, dev), kd, vd,
                    k_scale=scale, v_scale=scale * 0.5)
        assert pa.get_device_error(dev) == 0
        assert np.array_equal(bits_of(kd), want_k), f"K codes differ at scale {scale}"
        assert np.array_equal(bits_of(vd), want_v), f"V codes differ at scale {scale}"


def test_copy_blocks_moves_codes(dev):
    import paged_kv_cache_114_gb300 as pa
    rng = np.random.default_rng(9)
    layers = 3
    ks = [rng.integers(0, 256, size=(40, 16, 8, 128), dtype=np.uint8) for _ in range(layers)]
    vs = [rng.integers(0, 256, size=(40, 16, 8, 128), dtype=np.uint8) for _ in range(layers)]
    pairs = [(3, 30), (3, 31), (7, 0), (39, 12)]
    want_k, want_v = oracle.copy_blocks(ks, vs, pairs)
    kd = [to_dev(k, dev) for k in ks]
    vd = [to_dev(v, dev) for v in vs]
    pa.copy_blocks(kd, vd, to_dev(np.array(pairs, dtype=np.int64), dev))
    assert pa.get_device_error(dev) == 0
    for i in range(layers):
        assert np.array_equal(bits_of(kd[i]), want_k[i]) and np.array_equal(bits_of(vd[i]), want_v[i])


def test_float8_storage_dtype_is_accepted(dev):
    """A cache held as torch.float8_e4m3fn gives the same bytes and output as uint8."""
    w = make_random_case(41, num_seqs=3, num_q_heads=16, num_kv_heads=4, head_dim=128,
                         block_size=16, seq_lens=[40, 1, 300], dtype="bf16", kv_dtype="e4m3")
    import paged_kv_cache_114_gb300 as pa
    outs = []
    for view in (None, torch.float8_e4m3fn):
        k, v = to_dev(w.k_cache, dev), to_dev(w.v_cache, dev)
        if view is not None:
            k, v = k.view(view), v.view(view)
        tables, lens = to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev)
        slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                                w.block_size, w.num_blocks)
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v,
                    k_scale=w.k_scale, v_scale=w.v_scale)
        outs.append(pa.decode(to_dev(w.q, dev, w.dtype), k, v, tables, lens, w.scale,
                              max_seq_len=w.max_seq_len, out_dtype=torch.float32,
                              k_scale=w.k_scale, v_scale=w.v_scale))
    assert torch.equal(outs[0], outs[1])


def test_placement_permutation_bit_identical(dev):
    w = make_random_case(43, num_seqs=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                         block_size=16, seq_lens=[1, 17, 200, 513, 999], dtype="f16",
                         kv_dtype="e4m3")
    base = gpu_scenario(w, dev, partition_tokens=-1)["out"]
    perm = np.random.default_rng(4).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    w.k_cache, w.v_cache = k2, v2
    w.block_tables = perm[w.block_tables].astype(np.int32)
    assert torch.equal(base, gpu_scenario(w, dev, partition_tokens=-1)["out"])


def test_split_matches_single_pass(dev):
    w = make_random_case(44, num_seqs=3, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=32, seq_lens=[4096, 3000, 17], dtype="bf16", kv_dtype="e4m3")
    one = gpu_scenario(w, dev, partition_tokens=0)["out"]
    for p in (512, 16, -1):
        assert torch.max(torch.abs(gpu_scenario(w, dev, partition_tokens=p)["out"] - one)).item() <= 1e-5


@pytest.mark.parametrize("cid,block_size", [(2, None), (3, None), (4, 32), (4, 8), (5, None)])
def test_full_size_configs(dev, cid, block_size):
    """The pages' workload shapes with an FP8 pool: every byte of the writes
    (and config 5's copy-on-write copies) and every (sequence, head) output."""
    w = make_config(cid, block_size=block_size, kv_dtype="e4m3")
    res = gpu_scenario(w, dev)
    ref = oracle_scenario(w)
    assert res["err"] == 0
    _check_bytes(res, ref)
    assert_close(res["out"], ref["out"], what=w.name)


def test_static_workspace_matches(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(45, num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=16, seq_lens=[2000, 7, 900, 1], dtype="bf16", kv_dtype="e4m3")
    k, v = to_dev(w.k_cache, dev), to_dev(w.v_cache, dev)
    args = (to_dev(w.q, dev, w.dtype), k, v, to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev),
            w.scale)
    kw = dict(max_seq_len=w.max_seq_len, out_dtype=torch.float32, k_scale=w.k_scale,
              v_scale=w.v_scale)
    for p in (-1, 256):
        a = pa.decode(*args, partition_tokens=p, **kw)
        b = pa.decode_static_workspace(*args, partition_tokens=p, **kw)
        assert torch.equal(a, b)


def test_decode_step_from_host(dev):
    """DecodeStep on an E4M3 pool: the staged host path gives the oracle's output."""
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(46, num_seqs=6, num_q_heads=16, num_kv_heads=8, head_dim=128,
                         block_size=16, seq_lens=[100, 1, 2000, 37, 512, 64], dtype="f16",
                         kv_dtype="e4m3")
    k, v = to_dev(w.k_cache, dev), to_dev(w.v_cache, dev)
    step = pa.DecodeStep(k, v, num_seqs=w.num_seqs, num_q_heads=w.num_q_heads,
                         num_tokens=len(w.positions), max_blocks_per_seq=w.max_blocks_per_seq,
                         max_seq_len=w.max_seq_len, scale=w.scale, act_dtype=torch.float16,
                         k_scale=w.k_scale, v_scale=w.v_scale)
    views, _ = step.host_buffers()
    tdt = torch.float16
    views["q"].copy_(torch.from_numpy(w.q.view(np.int16)).view(tdt))
    views["key"].copy_(torch.from_numpy(w.key.view(np.int16)).view(tdt))
    views["value"].copy_(torch.from_numpy(w.value.view(np.int16)).view(tdt))
    views["seq_idx"].copy_(torch.from_numpy(w.seq_idx))
    views["positions"].copy_(torch.from_numpy(w.positions))
    views["block_tables"].copy_(torch.from_numpy(w.block_tables))
    views["seq_lens"].copy_(torch.from_numpy(w.seq_lens))
    out = step.run_from_host().clone()
    ref = oracle_scenario(w)
    assert pa.get_device_error(dev) == 0
    assert np.array_equal(bits_of(k), ref["k"])
    assert_close(out, ref["out"], what="DecodeStep e4m3")
