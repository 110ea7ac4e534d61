"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bit-exact for slot mapping, KV writes and block copies; within 2e-3 max abs
for decode outputs (plus half an ulp of the output dtype when it is 16-bit).
"""
import numpy as np
import pytest
import torch

from tests.helpers import assert_close, bits_of, gpu_scenario, oracle_scenario, to_dev
from workloads import make_config, make_config5_steps, make_random_case

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
    assert np.array_equal(bits_of(res["k"]), ref["k"]), "K cache bytes differ"
    assert np.array_equal(bits_of(res["v"]), ref["v"]), "V cache bytes differ"


# ---------------------------------------------------------------- config 1


@pytest.mark.parametrize("partition", [0, 16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.float16])
def test_config1_tiny(dev, partition, out_dtype):
    w = make_config(1)
    res = gpu_scenario(w, dev, partition_tokens=partition, out_dtype=out_dtype)
    ref = oracle_scenario(w)
    assert res["err"] == 0
    _check_bytes(res, ref)
    assert int(ref["slots"][6]) == 10  # token 6 of table [7, 2, 11]: block 2, offset 2
    assert_close(res["out"], ref["out"], what="config 1")


# ---------------------------------------------------------------- shapes and edges

CASES = [
    # dtype, D, Hq, Hkv, b, lens, partitions
    ("f16", 64, 8, 8, 16, [1, 15, 16, 17, 100, 333], (0, 64, -1)),
    ("bf16", 128, 32, 8, 16, [5, 512, 513, 1000], (0, 128, 512, -1)),
    ("f16", 128, 16, 1, 32, [1, 31, 32, 33, 700], (0, 96, -1)),
    ("bf16", 256, 8, 4, 8, [3, 64, 257], (0, 64, -1)),
    ("f16", 128, 12, 4, 4, [1, 4, 5, 99], (0, 32, -1)),
    ("bf16", 64, 6, 6, 1, [1, 2, 17], (0, 16, -1)),
    ("f16", 128, 20, 2, 64, [1, 63, 64, 65, 1000], (0, 256, -1)),
    ("f16", 128, 4, 4, 2, [0, 7, 0, 40], (0, 16, -1)),
    ("bf16", 128, 64, 8, 16, [1, 2, 3, 16, 17, 4097], (0, 512, -1)),
    ("f16", 256, 16, 16, 16, [300, 1], (0, 128, -1)),
    ("bf16", 128, 8, 8, 16, [0, 0, 0], (0, -1)),
    ("f16", 128, 32, 32, 16, [1] * 300 + [2048], (0, -1)),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-d{c[1]}-{c[2]}x{c[3]}-b{c[4]}" for c in CASES])
def test_shapes(dev, case):
    dtype, d, hq, hkv, b, lens, parts = case
    w = make_random_case(sum(lens) + d + hq, num_seqs=len(lens), num_q_heads=hq, num_kv_heads=hkv,
                         head_dim=d, block_size=b, seq_lens=lens, dtype=dtype)
    ref = oracle_scenario(w)
    for p in parts:
        for odt in (torch.float32, torch.float16 if dtype == "f16" else torch.bfloat16):
            res = gpu_scenario(w, dev, partition_tokens=p, out_dtype=odt)
            assert res["err"] == 0
            _check_bytes(res, ref)
            assert_close(res["out"], ref["out"], what=f"partition {p} out {odt}")
            zero_rows = [i for i, L in enumerate(lens) if L == 0]
            for i in zero_rows:
                assert torch.count_nonzero(res["out"][i]) == 0


def test_split_matches_single_pass(dev):
    """Split-K partials merged by the reduce agree with one pass to fp32 rounding."""
    w = make_random_case(77, num_seqs=3, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=32, seq_lens=[4096, 3000, 17], dtype="bf16")
    one = gpu_scenario(w, dev, partition_tokens=0)["out"]
    for p in (512, 256, 1024, 16, -1):
        split = gpu_scenario(w, dev, partition_tokens=p)["out"]
        assert torch.max(torch.abs(split - one)).item() <= 1e-5


def test_placement_permutation_bit_identical(dev):
    """Moving blocks to other physical ids leaves the kernel's output bit-identical."""
    w = make_random_case(31, num_seqs=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                         block_size=16, seq_lens=[1, 17, 200, 513, 999], dtype="f16")
    base = gpu_scenario(w, dev, partition_tokens=-1)["out"]
    perm = np.random.default_rng(3).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    w.k_cache, w.v_cache = k2, v2
    w.block_tables = perm[w.block_tables].astype(np.int32)
    moved = gpu_scenario(w, dev, partition_tokens=-1)["out"]
    assert torch.equal(base, moved)


def test_repeat_is_deterministic(dev):
    w = make_random_case(32, num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=16, seq_lens=[2000, 1500, 900, 3], dtype="bf16")
    for p in (256, -1):
        a = gpu_scenario(w, dev, partition_tokens=p)["out"]
        b = gpu_scenario(w, dev, partition_tokens=p)["out"]
        assert torch.equal(a, b)


# ---------------------------------------------------------------- full-size configs


def _full_config(dev, w, partition=None):
    """The whole scenario on the device and in the oracle; every (sequence,
    head) output row is compared, the pieces the balanced split cuts across
    CTAs (merged by the last arriver) included."""
    res = gpu_scenario(w, dev, partition_tokens=partition)
    ref = oracle_scenario(w)
    assert res["err"] == 0
    _check_bytes(res, ref)
    return res, ref, None


def test_config2_mha_full(dev):
    w = make_config(2)
    res, ref, heads = _full_config(dev, w)
    assert_close(res["out"], ref["out"], heads, what="config 2")


def test_config3_gqa_full(dev):
    w = make_config(3)
    res, ref, heads = _full_config(dev, w)
    assert_close(res["out"], ref["out"], heads, what="config 3")


@pytest.mark.parametrize("partition", [512, -1])
@pytest.mark.parametrize("b", [8, 16, 32])
def test_config4_long_split_full(dev, b, partition):
    w = make_config(4, block_size=b)
    res, ref, heads = _full_config(dev, w, partition=partition)
    assert_close(res["out"], ref["out"], heads, what=f"config 4 b={b} partition {partition}")


def test_config5_prefix_cow_full(dev):
    w = make_config(5)
    res, ref, heads = _full_config(dev, w)
    assert_close(res["out"], ref["out"], heads, what="config 5")
    # shared (copy-on-write) tables equal private copies, bit for bit
    k = res["k"]
    v = res["v"]
    tables = w.block_tables.copy()
    prefix = w.shared_blocks
    nb = w.num_blocks
    extra = w.num_seqs * len(prefix)
    k2 = torch.cat([k, torch.empty((extra,) + tuple(k.shape[1:]), dtype=k.dtype, device=dev)])
    v2 = torch.cat([v, torch.empty((extra,) + tuple(v.shape[1:]), dtype=v.dtype, device=dev)])
    import paged_kv_cache_114_gb300 as pa
    pairs = []
    nxt = nb
    for s in range(w.num_seqs):
        for j, blk in enumerate(prefix):
            pairs.append((blk, nxt))
            tables[s, j] = nxt
            nxt += 1
    pa.copy_blocks([k2], [v2], to_dev(np.array(pairs, dtype=np.int64), dev))
    out2 = pa.decode(to_dev(w.q, dev, w.dtype), k2, v2, to_dev(tables, dev),
                     to_dev(w.seq_lens, dev), w.scale, max_seq_len=w.max_seq_len,
                     out_dtype=torch.float32)
    assert pa.get_device_error(dev) == 0
    assert torch.equal(out2, res["out"])


@pytest.mark.parametrize("kv", [None, "e4m3"])
def test_config5_decode_steps(dev, kv):
    """Config 5 as a decode loop: 32 steps of slot mapping, KV write of one new
    token per sequence and decode, on 256 sequences sharing a 1000-token prefix.
    Step 0 copies the shared partial block for 255 sequences (copy-on-write)
    before the write lands in the copies; steps 8 and 24 open fresh blocks.
    Every step's slots and every output row are compared with the oracle
    running the same loop, and the pools byte for byte at the end."""
    import oracle
    import paged_kv_cache_114_gb300 as pa
    w = make_config5_steps(32, kv_dtype=kv)
    fp8 = kv == "e4m3"
    sc = dict(k_scale=w["k_scale"], v_scale=w["v_scale"]) if fp8 else {}
    if fp8:
        k, v = to_dev(w["k_cache"], dev), to_dev(w["v_cache"], dev)
    else:
        k, v = to_dev(w["k_cache"], dev, w["dtype"]), to_dev(w["v_cache"], dev, w["dtype"])
    ko, vo = w["k_cache"], w["v_cache"]
    part = pa.default_partition(w["num_seqs"], w["num_kv_heads"], 1032, w["block_size"])
    for i, st in enumerate(w["steps"]):
        if len(st["pairs"]):
            pa.copy_blocks([k], [v], to_dev(st["pairs"], dev))
            ks, vs = oracle.copy_blocks([ko], [vo], [tuple(p) for p in st["pairs"].tolist()])
            ko, vo = ks[0], vs[0]
        tables = to_dev(st["block_tables"], dev)
        slots = pa.slot_mapping(tables, to_dev(st["seq_idx"], dev), to_dev(st["positions"], dev),
                                w["block_size"], w["num_blocks"])
        pa.write_kv(to_dev(st["key"], dev, w["dtype"]), to_dev(st["value"], dev, w["dtype"]), slots,
                    k, v, **sc)
        out = torch.full((w["num_seqs"], w["num_q_heads"], w["head_dim"]), float("nan"),
                         dtype=torch.float32, device=dev)
        pa.decode(to_dev(st["q"], dev, w["dtype"]), k, v, tables, to_dev(st["seq_lens"], dev),
                  w["scale"], max_seq_len=int(st["seq_lens"].max()), out=out,
                  partition_tokens=part, **sc)
        assert pa.get_device_error(dev) == 0, f"step {i}"
        so = oracle.slot_mapping(st["block_tables"], st["seq_idx"], st["positions"], w["block_size"])
        assert np.array_equal(slots.cpu().numpy(), so), f"step {i}: slots differ"
        if fp8:
            ko, vo = oracle.write_kv_e4m3(ko, vo, st["key"], st["value"], so, w["dtype"],
                                          w["k_scale"], w["v_scale"])
            want = oracle.decode(st["q"], ko, vo, st["block_tables"], st["seq_lens"], w["scale"],
                                 w["dtype"], kv_dtype="e4m3", k_scale=w["k_scale"],
                                 v_scale=w["v_scale"])
        else:
            ko, vo = oracle.write_kv(ko, vo, st["key"], st["value"], so)
            want = oracle.decode(st["q"], ko, vo, st["block_tables"], st["seq_lens"], w["scale"],
                                 w["dtype"])
        assert_close(out, want, what=f"config 5 step {i}{' e4m3' if fp8 else ''}")
    assert np.array_equal(bits_of(k), ko), "K pool bytes differ after 32 steps"
    assert np.array_equal(bits_of(v), vo), "V pool bytes differ after 32 steps"


# ---------------------------------------------------------------- device-side errors


def test_bad_block_id_is_flagged_not_faulted(dev):
    import oracle
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(41, num_seqs=3, num_q_heads=8, num_kv_heads=8, head_dim=64,
                         block_size=16, seq_lens=[40, 40, 40], dtype="f16")
    want = oracle.decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens, w.scale, w.dtype)
    tables = w.block_tables.copy()
    tables[1, 1] = w.num_blocks + 5  # sequence 1's second block id is out of range
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    for partition in (0, 16, -1):
        out = torch.full((3, 8, 64), float("nan"), dtype=torch.float32, device=dev)
        pa.decode(to_dev(w.q, dev, w.dtype), k, v, to_dev(tables, dev), to_dev(w.seq_lens, dev),
                  w.scale, max_seq_len=40, out=out, partition_tokens=partition)
        assert pa.get_device_error(dev) & pa.DEVERR_BLOCK_ID
        assert torch.all(torch.isfinite(out))
        assert_close(out[0:1], want[0:1])
        assert_close(out[2:3], want[2:3])


def test_bad_lengths_and_slots_are_flagged(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(42, num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim=64,
                         block_size=8, seq_lens=[20, 9], dtype="f16")
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    lens = to_dev(np.array([20, 10_000], dtype=np.int32), dev)
    out = pa.decode(to_dev(w.q, dev, w.dtype), k, v, to_dev(w.block_tables, dev), lens, w.scale,
                    max_seq_len=20, out_dtype=torch.float32, partition_tokens=0)
    assert pa.get_device_error(dev) & pa.DEVERR_SEQ_LEN
    assert torch.all(torch.isfinite(out))
    # write_kv: one slot out of range, one padding slot (-1), one good slot
    key = to_dev(w.key[:1].repeat(3, axis=0), dev, w.dtype)
    slots = torch.tensor([w.num_blocks * 8 + 3, -1, 5], dtype=torch.int64, device=dev)
    before = bits_of(k)
    pa.write_kv(key, key, slots, k, v)
    assert pa.get_device_error(dev) == pa.DEVERR_SLOT
    after = bits_of(k)
    changed = np.argwhere((after != before).reshape(-1, 4 * 64).any(axis=1)).ravel().tolist()
    assert changed in ([5], [])  # only slot 5 may change (same bytes possible)
    assert np.array_equal(after.reshape(-1, 4, 64)[5], w.key[0])
    pa.write_kv(key[1:2], key[1:2], slots[1:2], k, v)
    assert pa.get_device_error(dev) == 0
    # slot mapping: a position beyond the table gives -1 and a flag
    tables = to_dev(w.block_tables, dev)
    sm = pa.slot_mapping(tables, torch.tensor([0, 1, 5], dtype=torch.int32, device=dev),
                         torch.tensor([3, 10**6, 0], dtype=torch.int32, device=dev), 8, w.num_blocks)
    assert pa.get_device_error(dev) & pa.DEVERR_POSITION
    got = sm.cpu().numpy()
    assert got[1] == -1 and got[2] == -1 and got[0] == w.block_tables[0, 0] * 8 + 3
    # copy pairs out of range
    pa.copy_blocks([k], [v], torch.tensor([[0, w.num_blocks + 1]], dtype=torch.int64, device=dev))
    assert pa.get_device_error(dev) & pa.DEVERR_BLOCK_ID


def test_host_errors_raise(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(43, num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim=64,
                         block_size=8, seq_lens=[20, 9], dtype="f16")
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    q = to_dev(w.q, dev, w.dtype)
    with pytest.raises(ValueError):
        pa.decode(q.to(torch.bfloat16), k, v, to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev),
                  w.scale, max_seq_len=20)
    with pytest.raises(pa.PagedKVError):
        pa.decode(q, k, v, to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev), w.scale,
                  max_seq_len=20, partition_tokens=24)
    flat = torch.empty(k.numel() + 8, dtype=k.dtype, device=dev)
    k_off = flat[4:4 + k.numel()].view(k.shape)  # 8-byte offset: not 16-byte aligned
    with pytest.raises(pa.PagedKVError):
        pa.decode(q, k_off, v, to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev), w.scale,
                  max_seq_len=20)
