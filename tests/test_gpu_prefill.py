"""GPU parity for multi-token causal attention (pa_prefill) against the fp64
oracle: chunked prefill, whole prompts, speculative verification, and the
degenerate cases (a single query, sequences with no new tokens, bad input).

Tolerance as for decode: 2e-3 max abs on fp32 outputs (plus half an ulp of
a 16-bit output dtype).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, gpu_scenario, to_dev
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


def gpu_prefill(w, dev, out_dtype=torch.float32, max_q_len=None, workspace="auto"):
    """slot_mapping + write_kv of the new tokens, then prefill, on the device."""
    import paged_kv_cache_114_gb300 as pa
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    tables = to_dev(w.block_tables, dev)
    if len(w.positions):
        slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                                w.block_size, w.num_blocks)
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=out_dtype, device=dev)
    qn = np.diff(w.q_start)
    pa.prefill(q, k, v, tables, to_dev(w.seq_lens, dev), to_dev(w.q_start, dev), w.scale,
               max_q_len=int(qn.max()) if max_q_len is None else max_q_len, out=out,
               workspace=workspace)
    err = pa.get_device_error(dev)
    return out, err, (k, v, tables)


def oracle_prefill(w, rows=None):
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    k, v = oracle.write_kv(w.k_cache, w.v_cache, w.key, w.value, slots)
    return oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                          rows=rows)


CASES = [
    # dtype, Hq, Hkv, D, b, seq_lens, q_lens
    ("f16", 4, 4, 64, 8, [10, 1, 16, 33], [10, 1, 5, 33]),            # whole prompts + a chunk
    ("bf16", 64, 8, 128, 16, [700, 129, 64, 1000], [4, 4, 64, 130]),  # verify 4 drafts; 17 row tiles
    ("f16", 32, 8, 128, 32, [300, 2000, 77], [200, 1, 0]),           # chunk, single query, none
    ("bf16", 8, 8, 256, 64, [200, 65], [70, 65]),                    # head_dim 256, b = 64
    ("f16", 16, 2, 128, 128, [513, 300], [129, 300]),                # b = 128: two boxes per block
    ("bf16", 12, 2, 64, 16, [95, 160, 33], [31, 160, 9]),            # g = 6: heads of a query split across warps
    ("f16", 8, 1, 128, 8, [1, 2, 3, 4, 5], [1, 2, 1, 4, 3]),         # tiny sequences, MQA
    # drafts only: 32, 32, 48 and 8 rows per KV head, so the 64-row kernel's
    # warps split each stage's tokens two ways, not at all, and four ways
    ("bf16", 64, 8, 128, 16, [700, 129, 1000, 50], [4, 4, 6, 1]),
    # at most 32 rows per KV head: the balanced kernel with a workspace, the thin
    # launch (two-stage ring, 3 CTAs per SM) without
    ("bf16", 64, 8, 128, 16, [700, 129, 1000, 50], [4, 4, 3, 1]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}x{c[2]}-d{c[3]}-b{c[4]}" for c in CASES])
def test_prefill_matches_oracle(dev, case):
    dtype, hq, hkv, d, b, lens, qn = case
    w = make_prefill_case(sum(lens) + 7 * d + hq, num_seqs=len(lens), num_q_heads=hq,
                          num_kv_heads=hkv, head_dim=d, block_size=b, seq_lens=lens, q_lens=qn,
                          dtype=dtype)
    want = oracle_prefill(w)
    # without a workspace every shape runs on the per-sequence kernels
    for ws in ("auto", None):
        out, err, _ = gpu_prefill(w, dev, workspace=ws)
        assert err == 0
        assert_close(out, want, what=f"prefill fp32, workspace {ws}")
        out16, err, _ = gpu_prefill(w, dev, out_dtype=torch.float16 if dtype == "f16" else torch.bfloat16,
                                    workspace=ws)
        assert err == 0
        assert_close(out16, want, what=f"prefill 16-bit out, workspace {ws}")


def test_single_query_agrees_with_decode(dev):
    """n = 1 for every sequence is decode: the two kernels agree to fp32 rounding."""
    import paged_kv_cache_114_gb300 as pa
    lens = [1, 17, 300, 4096, 1000]
    w = make_prefill_case(51, num_seqs=5, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=lens, q_lens=[1] * 5, dtype="bf16")
    out, err, (k, v, tables) = gpu_prefill(w, dev)
    assert err == 0
    dec = pa.decode(to_dev(w.q, dev, w.dtype), k, v, tables, to_dev(w.seq_lens, dev), w.scale,
                    max_seq_len=max(lens), out_dtype=torch.float32, partition_tokens=0)
    assert torch.max(torch.abs(out - dec)).item() <= 1e-5


def test_repeat_is_deterministic(dev):
    w = make_prefill_case(52, num_seqs=3, num_q_heads=16, num_kv_heads=4, head_dim=128,
                          block_size=16, seq_lens=[900, 64, 333], q_lens=[100, 64, 7], dtype="f16")
    a, _, _ = gpu_prefill(w, dev)
    b, _, _ = gpu_prefill(w, dev)
    assert torch.equal(a, b)


def test_more_queries_than_tokens_is_flagged(dev):
    """n_s > L_s cannot be placed: the sequence is skipped and flagged, nothing faults."""
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(53, num_seqs=2, num_q_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=16, seq_lens=[40, 20], q_lens=[8, 20], dtype="f16")
    lens = w.seq_lens.copy()
    lens[1] = 10  # 20 queries, 10 tokens
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device=dev)
    pa.prefill(q, k, v, to_dev(w.block_tables, dev), to_dev(lens, dev), to_dev(w.q_start, dev),
               w.scale, max_q_len=20, out=out)
    assert pa.get_device_error(dev) & pa.DEVERR_SEQ_LEN
    assert torch.isnan(out[8:]).all()          # sequence 1 left alone
    assert torch.isfinite(out[:8]).all()       # sequence 0 computed


def test_max_q_len_too_small_is_flagged(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(54, num_seqs=1, num_q_heads=8, num_kv_heads=1, head_dim=64,
                          block_size=16, seq_lens=[100], q_lens=[20], dtype="bf16")
    out, err, _ = gpu_prefill(w, dev, max_q_len=8)  # 8 * g = 64 rows covered, 160 needed
    assert err & pa.DEVERR_SEQ_LEN
    want = oracle_prefill(w)
    # the rows the launch did cover are still right
    assert_close(out[:8], want[:8], what="covered rows")


def test_bad_block_id_is_flagged_not_faulted(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(55, num_seqs=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                          block_size=16, seq_lens=[200, 90], q_lens=[30, 5], dtype="f16")
    w.block_tables = w.block_tables.copy()
    w.block_tables[0, 3] = w.num_blocks + 5   # tokens 48 .. 63 of sequence 0
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device=dev)
    pa.prefill(q, k, v, to_dev(w.block_tables, dev), to_dev(w.seq_lens, dev),
               to_dev(w.q_start, dev), w.scale, max_q_len=30, out=out)
    assert pa.get_device_error(dev) & pa.DEVERR_BLOCK_ID
    assert torch.isfinite(out).all()


def test_host_errors_raise(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(56, num_seqs=1, num_q_heads=4, num_kv_heads=4, head_dim=64,
                          block_size=4, seq_lens=[10], q_lens=[2], dtype="f16")
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    with pytest.raises(pa.PagedKVError, match="shape"):  # blocks of 4 tokens are not supported
        pa.prefill(to_dev(w.q, dev, w.dtype), k, v, to_dev(w.block_tables, dev),
                   to_dev(w.seq_lens, dev), to_dev(w.q_start, dev), w.scale, max_q_len=2)
