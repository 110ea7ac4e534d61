"""GPU parity of pa_prefill on the bench's multi-token workloads at full size,
in the launch bench.py times (workspace when the shape can use one), against
the fp64 oracle on every (query row, head) output. Tolerance as for decode:
2e-3 max abs on fp32 outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, to_dev
from workloads import make_prefill_config

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


@pytest.mark.parametrize("name,kv", [("verify4_70b_bf16_b16", None),
                                     ("chunk512_gqa_bf16_b16", None),
                                     ("chunk512_gqa_bf16_b16", "e4m3"),
                                     ("prompt2k_mha_fp16_b16", None)])
def test_prefill_workload_full(dev, name, kv):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_config(name, kv_dtype=kv)
    fp8 = w.kv_dtype == "e4m3"
    sc = dict(k_scale=w.k_scale, v_scale=w.v_scale) if fp8 else {}
    k = to_dev(w.k_cache, dev, None if fp8 else w.dtype)
    v = to_dev(w.v_cache, dev, None if fp8 else w.dtype)
    tables = to_dev(w.block_tables, dev)
    slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                            w.block_size, w.num_blocks)
    pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v, **sc)
    q = to_dev(w.q, dev, w.dtype)
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device=dev)
    max_q = int(np.diff(w.q_start).max())
    pa.prefill(q, k, v, tables, to_dev(w.seq_lens, dev), to_dev(w.q_start, dev), w.scale,
               max_q_len=max_q, out=out, **sc)
    assert pa.get_device_error(dev) == 0
    s_ = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    if fp8:
        ko, vo = oracle.write_kv_e4m3(w.k_cache, w.v_cache, w.key, w.value, s_, w.dtype,
                                      w.k_scale, w.v_scale)
        want = oracle.prefill(w.q, w.q_start, ko, vo, w.block_tables, w.seq_lens, w.scale,
                              w.dtype, kv_dtype="e4m3", k_scale=w.k_scale,
                              v_scale=w.v_scale)
    else:
        ko, vo = oracle.write_kv(w.k_cache, w.v_cache, w.key, w.value, s_)
        want = oracle.prefill(w.q, w.q_start, ko, vo, w.block_tables, w.seq_lens, w.scale,
                              w.dtype)
    assert_close(out, want, what=f"{name}{'_e4m3' if fp8 else ''} every row")
