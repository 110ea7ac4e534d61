"""GPU parity for multi-token causal attention (pa_prefill) over FP8 (E4M3)
caches: the new tokens' rows are quantised by pa_write_kv, then every query
row is compared with the fp64 oracle reading the same codes times the layer
scales. Tolerance as for decode: 2e-3 max abs (plus half an ulp of a 16-bit
output dtype)."""
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


def run(w, dev, out_dtype=torch.float32, workspace="auto"):
    import paged_kv_cache_114_gb300 as pa
    k, v = to_dev(w.k_cache, dev), to_dev(w.v_cache, dev)
    tables = to_dev(w.block_tables, dev)
    sc = dict(k_scale=w.k_scale, v_scale=w.v_scale)
    if len(w.positions):
        slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                                w.block_size, w.num_blocks)
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v, **sc)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=out_dtype, device=dev)
    qn = np.diff(w.q_start)
    pa.prefill(q, k, v, tables, to_dev(w.seq_lens, dev), to_dev(w.q_start, dev), w.scale,
               max_q_len=int(qn.max()), out=out, workspace=workspace, **sc)
    return out, pa.get_device_error(dev), k, v


def reference(w):
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    k, v = oracle.write_kv_e4m3(w.k_cache, w.v_cache, w.key, w.value, slots, w.dtype,
                                w.k_scale, w.v_scale)
    out = oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                         kv_dtype="e4m3", k_scale=w.k_scale, v_scale=w.v_scale)
    return out, k, v


CASES = [
    # act dtype, Hq, Hkv, D, b, seq_lens, q_lens
    ("bf16", 64, 8, 128, 16, [700, 129, 64, 1000], [4, 4, 64, 130]),   # verify + chunks, g = 8
    ("f16", 32, 8, 128, 32, [300, 2000, 77], [200, 1, 0]),            # chunk, single query, none
    ("bf16", 8, 8, 256, 64, [200, 65], [70, 65]),                     # head_dim 256, b = 64
    ("f16", 16, 2, 128, 128, [513, 300], [129, 300]),                 # b = 128
    ("bf16", 12, 2, 128, 16, [95, 160, 33], [31, 160, 9]),            # g = 6
    ("f16", 8, 1, 128, 8, [1, 2, 3, 4, 5], [1, 2, 1, 4, 3]),          # tiny sequences, MQA
    ("bf16", 64, 8, 128, 16, [700, 129, 1000, 50], [4, 4, 6, 1]),      # drafts only: 32/32/48/8 rows
    ("bf16", 64, 8, 128, 16, [700, 129, 1000, 50], [4, 4, 3, 1]),      # at most 32 rows: thin launch
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}-{c[1]}x{c[2]}-d{c[3]}-b{c[4]}" for c in CASES])
def test_prefill_e4m3_matches_oracle(dev, case):
    dtype, hq, hkv, d, b, lens, qn = case
    w = make_prefill_case(sum(lens) + 11 * d + hq, num_seqs=len(lens), num_q_heads=hq,
                          num_kv_heads=hkv, head_dim=d, block_size=b, seq_lens=lens, q_lens=qn,
                          dtype=dtype, kv_dtype="e4m3")
    want, kw, vw = reference(w)
    # without a workspace every shape runs on the per-sequence kernels
    for ws in ("auto", None):
        for odt in (torch.float32, torch.float16 if dtype == "f16" else torch.bfloat16):
            out, err, k, v = run(w, dev, odt, workspace=ws)
            assert err == 0
            assert np.array_equal(bits_of(k), kw) and np.array_equal(bits_of(v), vw)
            assert_close(out, want, what=f"prefill e4m3 out {odt}, workspace {ws}")


def test_single_query_equals_decode(dev):
    """n = 1 per sequence is decode: pa_prefill and pa_decode agree on an FP8 pool."""
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(91, num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                          block_size=16, seq_lens=[17, 1000, 2, 513], q_lens=[1, 1, 1, 1],
                          dtype="bf16", kv_dtype="e4m3")
    out, err, k, v = run(w, dev)
    dec = pa.decode(to_dev(w.q, dev, w.dtype), k, v, to_dev(w.block_tables, dev),
                    to_dev(w.seq_lens, dev), w.scale, max_seq_len=w.max_seq_len,
                    out_dtype=torch.float32, k_scale=w.k_scale, v_scale=w.v_scale)
    assert err == 0
    assert torch.max(torch.abs(out - dec)).item() <= 2e-3
