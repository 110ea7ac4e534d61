"""pa_decode_static_workspace: split-K decode without a caller workspace.

The entry point serves callers that cannot allocate device memory (a host
application whose own pool owns all device memory, latency-critical paths
where cudaMalloc may synchronise the device, runtimes with no device
allocator). Its partials live in a fixed array inside the library. These tests
check it, through the C ABI, against pa_decode with a caller-allocated
workspace, on two calls in a row (bit for bit: the same kernels run on the
same inputs), and check that a too-large request is refused, including the
balanced mode's fixed-size partials for a large query group. The file is
named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from tests.helpers import to_dev
from workloads import make_random_case

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


def _upload(w, dev):
    return dict(q=to_dev(w.q, dev, w.dtype), k=to_dev(w.k_cache, dev, w.dtype),
                v=to_dev(w.v_cache, dev, w.dtype), tables=to_dev(w.block_tables, dev),
                lens=to_dev(w.seq_lens, dev))


@pytest.mark.parametrize("part", [512, -1])
def test_static_workspace_matches_caller_workspace(dev, part):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(2024, num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         block_size=32, seq_lens=[8192, 5000, 300, 1], dtype="bf16")
    t = _upload(w, dev)
    need = pa.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     w.max_seq_len, part)
    assert 0 < need <= pa.STATIC_WORKSPACE_BYTES
    rng = np.random.default_rng(5)
    for call in range(2):
        # a different query on each call: the array keeps the previous call's partials
        q = t["q"] if call == 0 else torch.from_numpy(
            rng.standard_normal(tuple(t["q"].shape)).astype(np.float32)).to(dev).to(t["q"].dtype)
        want = pa.decode(q, t["k"], t["v"], t["tables"], t["lens"], w.scale,
                         max_seq_len=w.max_seq_len, out_dtype=torch.float32, partition_tokens=part)
        # NaN-filled so a row left unwritten cannot pass on stale memory
        got = torch.full(tuple(q.shape), float("nan"), dtype=torch.float32, device=dev)
        pa.decode_static_workspace(q, t["k"], t["v"], t["tables"], t["lens"], w.scale,
                                   max_seq_len=w.max_seq_len, partition_tokens=part, out=got)
        assert pa.get_device_error(dev) == 0
        assert torch.all(torch.isfinite(got))
        # the same kernels on the same inputs: only where the partials live differs
        assert torch.equal(got, want)


def test_static_workspace_refuses_oversize(dev):
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(2025, num_seqs=2, num_q_heads=8, num_kv_heads=8, head_dim=128,
                         block_size=16, seq_lens=[40, 17], dtype="f16")
    t = _upload(w, dev)
    # claimed lengths this long would need more partials than the array holds
    max_len = 1 << 20
    need = pa.decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim,
                                     max_len, 16)
    assert need > pa.STATIC_WORKSPACE_BYTES
    with pytest.raises(pa.PagedKVError, match="workspace"):
        pa.decode_static_workspace(t["q"], t["k"], t["v"], t["tables"], t["lens"], w.scale,
                                   max_seq_len=max_len, partition_tokens=16)
    assert pa.get_device_error(dev) == 0


def test_static_workspace_refuses_large_group_balanced(dev):
    """The balanced mode's partials scale with the SM count and the query group,
    not the batch: at g = 16, head_dim 128 they exceed the array on a GB300
    even for one sequence, while a fixed partition size still fits."""
    import paged_kv_cache_114_gb300 as pa
    w = make_random_case(2026, num_seqs=1, num_q_heads=32, num_kv_heads=2, head_dim=128,
                         block_size=16, seq_lens=[700], dtype="f16")
    t = _upload(w, dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    need = pa.decode_workspace_bytes(1, 32, 2, 128, w.max_seq_len, -1)
    assert need >= 16 * sms * 16 * 130 * 4
    if need <= pa.STATIC_WORKSPACE_BYTES:
        pytest.skip(f"{sms} SMs: the balanced partials fit the array")
    with pytest.raises(pa.PagedKVError, match="workspace"):
        pa.decode_static_workspace(t["q"], t["k"], t["v"], t["tables"], t["lens"], w.scale,
                                   max_seq_len=w.max_seq_len, partition_tokens=-1)
    want = pa.decode(t["q"], t["k"], t["v"], t["tables"], t["lens"], w.scale,
                     max_seq_len=w.max_seq_len, out_dtype=torch.float32, partition_tokens=256)
    got = pa.decode_static_workspace(t["q"], t["k"], t["v"], t["tables"], t["lens"], w.scale,
                                     max_seq_len=w.max_seq_len, partition_tokens=256,
                                     out_dtype=torch.float32)
    assert pa.get_device_error(dev) == 0
    assert torch.equal(got, want)
