"""Shared helpers for the GPU parity tests: move a workload to the device, run
the scenario through the library, run it through the oracle, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle

ATOL = 2e-3  # max abs error allowed on decode outputs (fp16/bf16 K/V, fp32 accumulate)
TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


def to_dev(a: np.ndarray, dev, dtype: str = None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if dtype is not None:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(TDT[dtype])
    return torch.from_numpy(a).to(dev)


def bits_of(t: torch.Tensor) -> np.ndarray:
    """Stored bits: uint16 patterns of a 16-bit tensor, bytes of an 8-bit one."""
    t = t.detach().cpu().contiguous()
    if t.element_size() == 1:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


def fp8_kw(w) -> dict:
    """Scale keywords of the binding's calls for an E4M3 workload (else none)."""
    return {"k_scale": w.k_scale, "v_scale": w.v_scale} if w.kv_dtype == "e4m3" else {}


def cache_to_dev(w, dev):
    """The workload's K and V pools on the device (uint8 codes for E4M3)."""
    if w.kv_dtype == "e4m3":
        return to_dev(w.k_cache, dev), to_dev(w.v_cache, dev)
    return to_dev(w.k_cache, dev, w.dtype), to_dev(w.v_cache, dev, w.dtype)


def gpu_scenario(w, dev, *, partition_tokens=None, out_dtype=torch.float32, pairs=None):
    """copy_blocks -> slot_mapping -> write_kv -> decode on the device."""
    import paged_kv_cache_114_gb300 as pa
    k, v = cache_to_dev(w, dev)
    pairs = w.copy_pairs if pairs is None else pairs
    if len(pairs):
        pa.copy_blocks([k], [v], to_dev(np.asarray(pairs, dtype=np.int64), dev))
    tables = to_dev(w.block_tables, dev)
    slots = pa.slot_mapping(tables, to_dev(w.seq_idx, dev), to_dev(w.positions, dev),
                            w.block_size, w.num_blocks)
    if len(w.positions):
        pa.write_kv(to_dev(w.key, dev, w.dtype), to_dev(w.value, dev, w.dtype), slots, k, v,
                    **fp8_kw(w))
    # NaN-filled so a row the kernel fails to write cannot pass on stale memory
    out = torch.full((w.num_seqs, w.num_q_heads, w.head_dim), float("nan"), dtype=out_dtype,
                     device=dev)
    pa.decode(to_dev(w.q, dev, w.dtype), k, v, tables, to_dev(w.seq_lens, dev), w.scale,
              max_seq_len=max(w.max_seq_len, 1), out=out, partition_tokens=partition_tokens,
              **fp8_kw(w))
    err = pa.get_device_error(dev)
    return {"k": k, "v": v, "slots": slots, "out": out, "err": err}


def oracle_scenario(w, pairs=None, heads=None):
    """The same scenario through the fp64 oracle."""
    pairs = w.copy_pairs if pairs is None else pairs
    k, v = w.k_cache, w.v_cache
    if len(pairs):
        ks, vs = oracle.copy_blocks([k], [v], [tuple(p) for p in np.asarray(pairs).tolist()])
        k, v = ks[0], vs[0]
    slots = oracle.slot_mapping(w.block_tables, w.seq_idx, w.positions, w.block_size)
    if w.kv_dtype == "e4m3":
        k, v = oracle.write_kv_e4m3(k, v, w.key, w.value, slots, w.dtype, w.k_scale, w.v_scale)
        out = oracle.decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype, pairs=heads,
                            kv_dtype="e4m3", k_scale=w.k_scale, v_scale=w.v_scale)
    else:
        k, v = oracle.write_kv(k, v, w.key, w.value, slots)
        out = oracle.decode(w.q, k, v, w.block_tables, w.seq_lens, w.scale, w.dtype, pairs=heads)
    return {"k": k, "v": v, "slots": slots, "out": out}


def half_ulp(x: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    mant = {torch.float16: 10, torch.bfloat16: 7, torch.float32: 23}[dtype]
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return 0.5 * 2.0 ** (np.floor(np.log2(ax)) - mant)


def assert_close(got: torch.Tensor, want: np.ndarray, heads=None, what=""):
    g = got.detach().float().cpu().double().numpy()
    if heads is not None:
        idx = tuple(np.array(heads).T)
        g, want = g[idx], want[idx]
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    tol = ATOL + (half_ulp(want, got.dtype) if got.dtype != torch.float32 else 0.0)
    err = np.abs(g - want)
    worst = float(np.max(err - tol)) if err.size else -1.0
    assert worst <= 0, f"{what}: max abs error {float(err.max()):.3e} exceeds tolerance"
    return float(err.max()) if err.size else 0.0
