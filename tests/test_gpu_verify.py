"""GPU parity for pa_prefill's balanced multi-token kernel (a few new tokens per
sequence: at most 32 (query, head) rows per KV head, head_dim 128, blocks of
16 or more tokens) against the fp64 oracle, for 16-bit and E4M3 caches.

Every shape below runs once with a workspace (the balanced kernel, whose
ranges cut sequences into pieces merged by the last arriver) and once
without (the per-sequence kernel); both must match the oracle. Tolerance as
for decode: 2e-3 max abs on fp32 outputs (plus half an ulp of a 16-bit
output dtype).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, bits_of, to_dev
from workloads import make_prefill_case

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


def run(w, dev, *, workspace="auto", out_dtype=torch.float32, max_q_len=None, lens=None,
        tables=None):
    """slot_mapping + write_kv of the new tokens, then prefill."""
    import paged_kv_cache_114_gb300 as pa
    fp8 = w.kv_dtype == "e4m3"
    sc = dict(k_scale=w.k_scale, v_scale=w.v_scale) if fp8 else {}
    k = to_dev(w.k_cache, dev, None if fp8 else w.dtype)
    v = to_dev(w.v_cache, dev, None if fp8 else w.dtype)
    tab = to_dev(w.block_tables if tables is None else tables, dev)
    if len(w.positions):
        slots = pa.slot_mapping(to_dev(w.block_tables, dev), to_dev(w.seq_idx, dev),
                                to_dev(w.positions, dev), w.block_size, w.num_blocks)
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v, **sc)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=out_dtype, device=dev)
    mq = int(np.diff(w.q_start).max()) if max_q_len is None else max_q_len
    pa.prefill(q, k, v, tab, to_dev(w.seq_lens if lens is None else lens, dev),
               to_dev(w.q_start, dev), w.scale, max_q_len=mq, out=out, workspace=workspace, **sc)
    return out, pa.get_device_error(dev), k, v


def reference(w):
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    if w.kv_dtype == "e4m3":
        k, v = oracle.write_kv_e4m3(w.k_cache, w.v_cache, w.key, w.value, slots, w.dtype,
                                    w.k_scale, w.v_scale)
        return oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                              kv_dtype="e4m3", k_scale=w.k_scale, v_scale=w.v_scale), k, v
    k, v = oracle.write_kv(w.k_cache, w.v_cache, w.key, w.value, slots)
    return oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale,
                          w.dtype), k, v


CASES = [
    # dtype, Hq, Hkv, b, seq_lens, q_lens: (tiles of 8 NT rows, R tiles, HG heads)
    # 4 drafts at g = 8: 32 rows, (2, 2, 4); lengths from below one stage to several ranges
    ("bf16", 64, 8, 16, [700, 129, 1000, 50, 4, 17, 2049, 333], [4, 4, 3, 1, 4, 2, 4, 0]),
    # g = 4, 2 drafts: 8 rows, (1, 1, 8)
    ("f16", 32, 8, 32, [300, 2000, 77, 16, 2], [2, 1, 2, 2, 2]),
    # g = 8, 2 drafts: 16 rows, (2, 1, 8)
    ("bf16", 64, 8, 64, [1500, 31, 900], [2, 2, 1]),
    # MHA, 32 drafts: 32 rows of one head each, runs of one column
    ("f16", 32, 32, 16, [600, 40, 33], [32, 17, 32]),
    # g = 6, 5 drafts: 30 rows, a query's heads straddle the two tiles
    ("bf16", 24, 4, 128, [513, 300, 64], [5, 3, 5]),
]


def _ids(c):
    return f"{c[0]}-{c[1]}x{c[2]}-b{c[3]}-n{max(c[5])}"


@pytest.mark.parametrize("kv", [None, "e4m3"])
@pytest.mark.parametrize("case", CASES, ids=[_ids(c) for c in CASES])
def test_multi_kernel_matches_oracle(dev, case, kv):
    import paged_kv_cache_114_gb300 as pa
    dtype, hq, hkv, b, lens, qn = case
    w = make_prefill_case(sum(lens) + 13 * hq + b, num_seqs=len(lens), num_q_heads=hq,
                          num_kv_heads=hkv, head_dim=128, block_size=b, seq_lens=lens, q_lens=qn,
                          dtype=dtype, kv_dtype=kv)
    assert pa.prefill_kernel_name(len(lens), hq, hkv, 128, b, max(qn)) == "multi_grouped_kernel"
    want, kw, vw = reference(w)
    odt16 = torch.float16 if dtype == "f16" else torch.bfloat16
    for workspace in ("auto", None):
        for odt in (torch.float32, odt16):
            out, err, k, v = run(w, dev, workspace=workspace, out_dtype=odt)
            assert err == 0
            if kv == "e4m3":
                assert np.array_equal(bits_of(k), kw) and np.array_equal(bits_of(v), vw)
            assert_close(out, want, what=f"prefill {kv or dtype} workspace={workspace} out {odt}")


def test_multi_kernel_long_verify_full(dev):
    """The long-context verification workload (8 sequences of 32768 tokens,
    32 / 8 heads, 4 drafts each) on the balanced kernel, the launch bench.py
    times; the oracle checks every (query, head) row."""
    import paged_kv_cache_114_gb300 as pa
    from workloads import make_prefill_config
    w = make_prefill_config("verify4_long_bf16_b16")
    assert pa.prefill_kernel_name(w.num_seqs, w.num_q_heads, w.num_kv_heads, 128, 16, 4) == \
        "multi_grouped_kernel"
    out, err, _, _ = run(w, dev)
    assert err == 0
    pick = range(w.num_seqs)
    rows = np.concatenate([np.arange(w.q_start[s], w.q_start[s + 1]) for s in pick])
    want, _, _ = reference_rows(w, [(int(t), h) for t in rows for h in range(w.num_q_heads)])
    assert_close(out[torch.as_tensor(rows, device=dev)], want[rows], what="long verify rows")
    again, _, _, _ = run(w, dev)
    assert torch.equal(out, again)


def test_verify_workload_routes_to_the_per_sequence_kernel(dev):
    """Batches of 32 rows per KV head with 4 or more (sequence, KV head) pairs per
    SM run on the per-sequence kernel even with a workspace, and need none."""
    import paged_kv_cache_114_gb300 as pa
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    n = -(-4 * sms // 8)  # the fewest sequences giving 4 (sequence, KV head) pairs per SM
    assert pa.prefill_kernel_name(n, 64, 8, 128, 16, 4) == "prefill_kernel"
    assert pa.prefill_workspace_bytes(n, 64, 8, 128, 16, 4) == 0
    assert pa.prefill_kernel_name(n - 1, 64, 8, 128, 16, 4) == "multi_grouped_kernel"


def reference_rows(w, rows):
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    k, v = oracle.write_kv(w.k_cache, w.v_cache, w.key, w.value, slots)
    return oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                          rows=rows), k, v


def test_multi_kernel_repeat_is_deterministic(dev):
    w = make_prefill_case(71, num_seqs=6, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[3000, 17, 900, 4096, 5, 640],
                          q_lens=[4, 3, 4, 4, 2, 1], dtype="bf16")
    a, _, _, _ = run(w, dev)
    b, _, _, _ = run(w, dev)
    assert torch.equal(a, b)


def test_multi_kernel_flags_bad_lengths(dev):
    """n_s > L_s: the sequence is skipped and flagged; the others are right."""
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(72, num_seqs=3, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[400, 20, 77], q_lens=[4, 4, 2], dtype="bf16")
    lens = w.seq_lens.copy()
    lens[1] = 3  # 4 queries, 3 tokens
    out, err, _, _ = run(w, dev, lens=lens)
    assert err & pa.DEVERR_SEQ_LEN
    assert torch.isnan(out[4:8]).all()
    want, _, _ = reference(w)
    assert_close(out[:4], want[:4], what="sequence 0")
    assert_close(out[8:], want[8:], what="sequence 2")


def test_multi_kernel_max_q_len_too_small(dev):
    """n_s > max_q_len: flagged, rows past max_q_len untouched, the rest right."""
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(73, num_seqs=2, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[500, 260], q_lens=[4, 2], dtype="bf16")
    out, err, _, _ = run(w, dev, max_q_len=2)
    assert pa.prefill_kernel_name(2, 64, 8, 128, 16, 2) == "multi_grouped_kernel"
    assert err & pa.DEVERR_SEQ_LEN
    want, _, _ = reference(w)
    assert_close(out[:2], want[:2], what="covered rows of sequence 0")
    assert torch.isnan(out[2:4]).all()
    assert_close(out[4:], want[4:], what="sequence 1")


def test_multi_kernel_bad_block_id_is_flagged(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(74, num_seqs=2, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[200, 90], q_lens=[4, 3], dtype="f16")
    tables = w.block_tables.copy()
    tables[0, 3] = w.num_blocks + 5   # tokens 48 .. 63 of sequence 0
    out, err, _, _ = run(w, dev, tables=tables)
    assert err & pa.DEVERR_BLOCK_ID
    assert torch.isfinite(out).all()


def test_workspace_too_small_is_refused(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(75, num_seqs=2, num_q_heads=64, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[100, 90], q_lens=[4, 3], dtype="f16")
    need = pa.prefill_workspace_bytes(2, 64, 8, 128, 16, 4)
    assert need > 0
    small = torch.empty(need - 256, dtype=torch.uint8, device=dev)
    with pytest.raises(pa.PagedKVError, match="workspace"):
        run(w, dev, workspace=small)
