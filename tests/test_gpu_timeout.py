"""The bounded-wait path, run on purpose without a fault.

Every wait of a kernel for a TMA stage is bounded; when the bound runs out the
kernel sets PA_DEVERR_TIMEOUT, waits for the copies it did issue, and finishes,
so the context stays usable. pa_test_set_stall makes that happen: each TMA
ring issues only its first k stages and the waits for the rest get a bound of
a few milliseconds. Nothing is left in flight, no trap or bad address is
involved, and the next call without the hook must match the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, gpu_scenario, oracle_scenario, to_dev
from workloads import make_prefill_case, make_random_case

pytestmark = pytest.mark.gpu

WAIT_US = 3000  # bound of a stalled wait: 3 ms


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from paged_kv_cache_114_gb300 import build
    build.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


class stall:
    """pa_test_set_stall for the duration of a with-block."""

    def __init__(self, stop_stage):
        self.stop = stop_stage

    def __enter__(self):
        import paged_kv_cache_114_gb300 as pa
        assert pa.lib().pa_test_set_stall(self.stop, WAIT_US) == 0

    def __exit__(self, *exc):
        import paged_kv_cache_114_gb300 as pa
        assert pa.lib().pa_test_set_stall(-1, 0) == 0
        return False


def test_hook_rejects_bad_bounds(dev):
    import paged_kv_cache_114_gb300 as pa
    assert pa.lib().pa_test_set_stall(2, 0) == -6
    assert pa.lib().pa_test_set_stall(2, 2_000_000) == -6
    assert pa.lib().pa_test_set_stall(-1, 0) == 0


# (partition, shape) covering every decode kernel: the single pass, split-K
# with its reduce, the balanced head-grouped kernel and the balanced per-warp one
DECODE = [
    (0, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16")),
    (256, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16")),
    (-1, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype="f16")),
    (-1, dict(num_q_heads=12, num_kv_heads=4, head_dim=128, block_size=4, dtype="f16")),
    # E4M3 pool: the grouped kernel with two consumer warps per KV head
    (-1, dict(num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16, dtype="bf16",
              kv_dtype="e4m3")),
]


@pytest.mark.parametrize("stop", [0, 2])
@pytest.mark.parametrize("partition,shape", DECODE,
                         ids=["single", "split256", "grouped", "per_warp", "grouped_e4m3"])
def test_decode_timeout_then_exact(dev, partition, shape, stop):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(900 + stop, num_seqs=6, seq_lens=[6000, 3000, 300, 77, 16, 8000], **shape)
    expected = pa.decode_kernel_name(w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                                     w.max_seq_len, partition)
    with stall(stop):
        res = gpu_scenario(w, dev, partition_tokens=partition)
    assert res["err"] & pa.DEVERR_TIMEOUT, f"{expected}: the stalled call did not time out"
    # the context is usable: the same scenario again, without the hook, is oracle-exact
    res = gpu_scenario(w, dev, partition_tokens=partition)
    assert res["err"] == 0
    assert_close(res["out"], oracle_scenario(w)["out"], what=f"{expected} after a timeout")


@pytest.mark.parametrize("stop", [0, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_prefill_tc_timeout_then_exact(dev, dtype, stop):
    import paged_kv_cache_114_gb300 as pa
    w = make_prefill_case(950 + stop, num_seqs=3, num_q_heads=16, num_kv_heads=4, head_dim=128,
                          block_size=16, seq_lens=[900, 300, 700], q_lens=[200, 64, 700],
                          dtype=dtype)
    qn = np.diff(w.q_start)
    assert pa.prefill_kernel_name(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                  w.block_size, int(qn.max()), False) == "prefill_tc_kernel"

    def run():
        k = to_dev(w.k_cache, dev, w.dtype)
        v = to_dev(w.v_cache, dev, w.dtype)
        tables = to_dev(w.block_tables, dev)
        slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                                w.block_size, w.num_blocks)
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v)
        out = torch.full(tuple(w.q.shape), float("nan"), dtype=torch.float32, device=dev)
        pa.prefill(to_dev(w.q, dev, w.dtype), k, v, tables, to_dev(w.seq_lens, dev),
                   to_dev(w.q_start, dev), w.scale, max_q_len=int(qn.max()), out=out,
                   workspace=None)
        return out, pa.get_device_error(dev)

    with stall(stop):
        _, err = run()
    assert err & pa.DEVERR_TIMEOUT
    out, err = run()
    assert err == 0
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    k, v = oracle.write_kv(w.k_cache, w.v_cache, w.key, w.value, slots)
    rows = [(int(t), h) for t in np.random.default_rng(stop).integers(0, len(w.q), 40)
            for h in (0, w.num_q_heads - 1)]
    want = oracle.prefill(w.q, w.q_start, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype,
                          rows=rows)
    assert_close(out, want, rows, what="prefill after a timeout")
