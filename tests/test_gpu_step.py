"""pa.DecodeStep: the three calls bound to fixed buffers, driven from pinned
host memory, against the fp64 oracle."""
import numpy as np
import pytest
import torch

from tests.helpers import assert_close, bits_of, oracle_scenario, to_dev
from workloads import make_config, make_random_case



@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from paged_kv_cache_114_gb300 import build
    build.build()
    d = torch.device("cuda", 0)
    torch.cuda.set_device(d)
    return d


def _fill(step, w):
    host, _ = step.host_buffers()
    src = {"q": w.q, "key": w.key, "value": w.value, "seq_idx": w.seq_idx,
           "positions": w.positions, "block_tables": w.block_tables, "seq_lens": w.seq_lens}
    for name, arr in src.items():
        a = np.ascontiguousarray(arr)
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        host[name].view(t.dtype).copy_(t.view(host[name].shape))


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["config1", "gqa_ragged"])
@pytest.mark.parametrize("partition", [None, 0, -1])
def test_decode_step_from_host(dev, case, partition):
    import paged_kv_cache_114_gb300 as pa
    if case == "config1":
        w = make_config(1)
    else:
        w = make_random_case(5150, num_seqs=5, num_q_heads=16, num_kv_heads=4, head_dim=128,
                             block_size=16, seq_lens=[1, 17, 300, 2047, 40], dtype="bf16")
    ref = oracle_scenario(w)
    k = to_dev(w.k_cache, dev, w.dtype)
    v = to_dev(w.v_cache, dev, w.dtype)
    step = pa.DecodeStep(k, v, num_seqs=w.num_seqs, num_q_heads=w.num_q_heads,
                         num_tokens=len(w.positions), max_blocks_per_seq=w.max_blocks_per_seq,
                         max_seq_len=w.max_seq_len, scale=w.scale, partition_tokens=partition)
    _fill(step, w)
    for _ in range(2):  # the step is idempotent: same writes, same output
        out = step.run_from_host().clone()
        assert pa.get_device_error(dev) == 0
        assert_close(out, ref["out"], what=f"{case} partition {partition}")
    assert np.array_equal(bits_of(k), ref["k"]) and np.array_equal(bits_of(v), ref["v"])
    dev_out = step.run()
    step.stream.synchronize()
    assert torch.equal(dev_out.cpu(), out)
    # the same step replayed from a captured graph, on fresh inputs each time:
    # the host output is cleared and q changes, so a replay that did not run (or
    # ran behind the synchronisation) fails
    step.capture_graph()
    host, host_out = step.host_buffers()
    for sign in (-1.0, -1.0):
        host["q"].mul_(sign)
        host_out.fill_(float("nan"))
        got = step.run_from_host().clone()
        inputs = {n: t.to(dev) for n, t in host.items()}
        want = pa.decode(inputs["q"], k, v, inputs["block_tables"], inputs["seq_lens"], w.scale,
                         max_seq_len=w.max_seq_len, out_dtype=torch.float32,
                         partition_tokens=step.partition_tokens)
        assert torch.equal(got, want.cpu())
    assert torch.equal(got, out)  # q negated twice: back to the original step
    assert pa.get_device_error(dev) == 0


def test_layout_is_aligned():
    import paged_kv_cache_114_gb300 as pa
    offsets, total = pa.DecodeStep.layout(torch.float16, N=3, Hq=5, Hkv=1, D=64, T=7, maxB=9)
    assert all(off % 256 == 0 for off, _ in offsets.values())
    ends = sorted((off, off + n) for off, n in offsets.values())
    assert all(a[1] <= b[0] for a, b in zip(ends, ends[1:])) and ends[-1][1] <= total
