"""Torch-facing binding of the C ABI: argument marshalling only.

Each function checks that its tensors are on one CUDA device with the expected
dtype and layout, turns them into pointers, and calls the matching ``pa_*``
entry point on the current stream. All arithmetic runs in the library's CUDA
kernels; there is no other code path.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Sequence

import torch

from . import _lib

_DTYPES = {torch.float16: _lib.PA_F16, torch.bfloat16: _lib.PA_BF16, torch.float32: _lib.PA_F32}
# Storage types of an E4M3 cache: raw bytes, or torch's own float8 type.
FP8_CACHE_DTYPES = (torch.uint8, torch.float8_e4m3fn)


def is_fp8_cache(t: torch.Tensor) -> bool:
    return t.dtype in FP8_CACHE_DTYPES


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _on(device: torch.device):
    """Make ``device`` current for one library call: the library looks up its
    per-device state (error word, SM count, static workspace) and launches on
    the current device, which must be the one the tensors live on."""
    return torch.cuda.device(device)


def _need(cond: bool, msg: str) -> None:
    if not cond:
        raise ValueError(msg)


def _cuda(*ts: torch.Tensor) -> torch.device:
    dev = ts[0].device
    for t in ts:
        _need(t.is_cuda, "tensors must live on a CUDA device")
        _need(t.device == dev, "tensors must live on one device")
        _need(t.is_contiguous(), "tensors must be contiguous")
    return dev


def make_cache(k_cache: torch.Tensor, v_cache: torch.Tensor, *,
               act_dtype: Optional[torch.dtype] = None, k_scale: Optional[float] = None,
               v_scale: Optional[float] = None) -> _lib.PaCache:
    """pa_cache for one layer's pool, k/v shaped [num_blocks, block_size, H_kv, D].

    16-bit caches (float16 / bfloat16) take no other argument. E4M3 caches
    (uint8 or float8_e4m3fn codes) take ``act_dtype`` (the dtype of q, key and
    value) and the layer's ``k_scale`` / ``v_scale``: a code c stands for
    value(c) * scale.
    """
    _cuda(k_cache, v_cache)
    _need(k_cache.dim() == 4 and k_cache.shape == v_cache.shape, "k/v caches: [NB, b, H_kv, D], same shape")
    nb, b, hkv, d = k_cache.shape
    if is_fp8_cache(k_cache):
        _need(is_fp8_cache(v_cache), "caches must both be E4M3 codes")
        _need(act_dtype in (torch.float16, torch.bfloat16), "E4M3 caches: act_dtype float16 or bfloat16")
        _need(k_scale is not None and v_scale is not None, "E4M3 caches need k_scale and v_scale")
        return _lib.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, b, hkv, d,
                            _lib.PA_FP8_E4M3, _DTYPES[act_dtype], float(k_scale), float(v_scale))
    _need(k_cache.dtype == v_cache.dtype and k_cache.dtype in (torch.float16, torch.bfloat16),
          "caches must both be float16, both bfloat16 or both E4M3 codes")
    code = _DTYPES[k_cache.dtype]
    return _lib.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, b, hkv, d, code, code, 1.0, 1.0)


def _check_act(t: torch.Tensor, k_cache: torch.Tensor, what: str) -> None:
    if is_fp8_cache(k_cache):
        _need(t.dtype in (torch.float16, torch.bfloat16),
              f"{what} must be float16 or bfloat16 with an E4M3 cache")
    else:
        _need(t.dtype == k_cache.dtype, f"{what} dtype must match the cache")


def slot_mapping(block_tables: torch.Tensor, seq_idx: torch.Tensor, positions: torch.Tensor,
                 block_size: int, num_blocks: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int64 pool slot of each (sequence, position) token."""
    dev = _cuda(block_tables, seq_idx, positions)
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2, "block_tables: int32 [N, maxB]")
    _need(seq_idx.dtype == torch.int32 and positions.dtype == torch.int32, "seq_idx/positions: int32")
    _need(seq_idx.shape == positions.shape and seq_idx.dim() == 1, "seq_idx/positions: [T]")
    if out is None:
        out = torch.empty(positions.shape[0], dtype=torch.int64, device=dev)
    _need(out.dtype == torch.int64 and out.shape == positions.shape, "out: int64 [T]")
    _cuda(out, block_tables)
    with _on(dev):
        st = _lib.lib().pa_slot_mapping(_ptr(block_tables), block_tables.shape[0], block_tables.shape[1],
                                    _ptr(seq_idx), _ptr(positions), positions.shape[0], block_size,
                                    num_blocks, _ptr(out), _stream(dev))
    _lib.check("pa_slot_mapping", st)
    return out


def write_kv(key: torch.Tensor, value: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor, *, k_scale: Optional[float] = None,
             v_scale: Optional[float] = None) -> None:
    """k_cache/v_cache row at each slot <- the token's key/value rows (in place).

    E4M3 caches store e4m3(x / k_scale) and e4m3(x / v_scale) of the float16 /
    bfloat16 rows."""
    dev = _cuda(key, value, slot_mapping, k_cache, v_cache)
    _need(key.shape == value.shape and key.dim() == 3, "key/value: [T, H_kv, D]")
    _need(key.shape[1:] == k_cache.shape[2:], "key/value rows must match the cache's [H_kv, D]")
    _need(key.dtype == value.dtype, "key and value must share a dtype")
    _check_act(key, k_cache, "key/value")
    _need(slot_mapping.dtype == torch.int64 and slot_mapping.shape == key.shape[:1], "slot_mapping: int64 [T]")
    cache = make_cache(k_cache, v_cache, act_dtype=key.dtype, k_scale=k_scale, v_scale=v_scale)
    with _on(dev):
        st = _lib.lib().pa_write_kv(_ptr(key), _ptr(value), _ptr(slot_mapping), key.shape[0],
                                ctypes.byref(cache), _stream(dev))
    _lib.check("pa_write_kv", st)


def check_copy_pairs(pairs_host: torch.Tensor, num_blocks: int) -> None:
    """Host-side check of copy pairs (ids in range, distinct destinations, none a source)."""
    _need(pairs_host.device.type == "cpu" and pairs_host.dtype == torch.int64, "pairs: host int64 [P, 2]")
    p = pairs_host.contiguous()
    st = _lib.lib().pa_check_copy_pairs(_ptr(p), p.shape[0], num_blocks)
    _lib.check("pa_check_copy_pairs", st)


def copy_blocks(k_caches: Sequence[torch.Tensor], v_caches: Sequence[torch.Tensor],
                pairs: torch.Tensor) -> None:
    """For every (src, dst) pair and every layer, block dst <- block src (in place)."""
    _need(len(k_caches) == len(v_caches) and len(k_caches) > 0, "one k and one v cache per layer")
    dev = _cuda(pairs, *k_caches, *v_caches)
    _need(pairs.dtype == torch.int64 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs: int64 [P, 2]")
    fp8 = dict(act_dtype=torch.float16, k_scale=1.0, v_scale=1.0)  # codes are copied as bytes
    arr = (_lib.PaCache * len(k_caches))(
        *[make_cache(k, v, **(fp8 if is_fp8_cache(k) else {})) for k, v in zip(k_caches, v_caches)])
    with _on(dev):
        st = _lib.lib().pa_copy_blocks(arr, len(k_caches), _ptr(pairs), pairs.shape[0], _stream(dev))
    _lib.check("pa_copy_blocks", st)


def _pool(k_cache: torch.Tensor, v_cache: torch.Tensor) -> _lib.PaCache:
    """pa_cache for a pool on the GPU or in pinned host memory (for swaps)."""
    for t in (k_cache, v_cache):
        _need(t.is_cuda or t.is_pinned(), "swap pools: CUDA tensors or pinned host tensors")
        _need(t.is_contiguous(), "tensors must be contiguous")
    _need(k_cache.dim() == 4 and k_cache.shape == v_cache.shape, "k/v caches: [NB, b, H_kv, D], same shape")
    _need(k_cache.dtype == v_cache.dtype, "k and v share a dtype")
    nb, b, hkv, d = k_cache.shape
    if is_fp8_cache(k_cache):
        return _lib.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, b, hkv, d,
                            _lib.PA_FP8_E4M3, _lib.PA_F16, 1.0, 1.0)  # codes move as bytes
    _need(k_cache.dtype in (torch.float16, torch.bfloat16), "caches: float16, bfloat16 or E4M3")
    code = _DTYPES[k_cache.dtype]
    return _lib.PaCache(k_cache.data_ptr(), v_cache.data_ptr(), nb, b, hkv, d, code, code, 1.0, 1.0)


def swap_blocks(src_k: Sequence[torch.Tensor], src_v: Sequence[torch.Tensor],
                dst_k: Sequence[torch.Tensor], dst_v: Sequence[torch.Tensor],
                pairs: torch.Tensor, device: Optional[torch.device] = None) -> None:
    """For every (src, dst) pair and layer: block dst of the destination pools
    <- block src of the source pools (K and V). Pools live on the GPU or in
    pinned host memory (swap out: GPU -> host; swap in: host -> GPU). Runs on
    the current stream of ``device`` (default: the pairs' device, else the
    current one)."""
    n = len(src_k)
    _need(n > 0 and len(src_v) == n and len(dst_k) == n and len(dst_v) == n,
          "one k and one v pool per layer on both sides")
    _need(pairs.dtype == torch.int64 and pairs.dim() == 2 and pairs.shape[1] == 2, "pairs: int64 [P, 2]")
    _need(pairs.is_contiguous() and (pairs.is_cuda or pairs.is_pinned()),
          "pairs: contiguous, on the GPU or in pinned host memory")
    if device is None:
        device = pairs.device if pairs.is_cuda else torch.device("cuda", torch.cuda.current_device())
    srcs = (_lib.PaCache * n)(*[_pool(k, v) for k, v in zip(src_k, src_v)])
    dsts = (_lib.PaCache * n)(*[_pool(k, v) for k, v in zip(dst_k, dst_v)])
    with torch.cuda.device(device):
        st = _lib.lib().pa_swap_blocks(srcs, dsts, n, _ptr(pairs), pairs.shape[0], _stream(device))
    _lib.check("pa_swap_blocks", st)


def prefix_key_offsets(token_offsets: torch.Tensor, block_size: int,
                       out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """int64 [N + 1] first key of each sequence when full-block keys are packed
    back to back (``out[s + 1] - out[s]`` = floor(len_s / block_size)),
    computed on the device by pa_prefix_key_offsets."""
    dev = _cuda(token_offsets)
    _need(token_offsets.dtype == torch.int64 and token_offsets.dim() == 1, "token_offsets: int64 [N + 1]")
    if out is None:
        out = torch.empty_like(token_offsets)
    _cuda(out, token_offsets)
    _need(out.dtype == torch.int64 and out.shape == token_offsets.shape, "out: int64 [N + 1]")
    with _on(dev):
        st = _lib.lib().pa_prefix_key_offsets(_ptr(token_offsets), token_offsets.shape[0] - 1,
                                              int(block_size), _ptr(out), _stream(dev))
    _lib.check("pa_prefix_key_offsets", st)
    return out


def prefix_hash(token_ids: torch.Tensor, token_offsets: torch.Tensor, block_size: int, *,
                key_offsets: Optional[torch.Tensor] = None, root: Optional[bytes] = None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefix-cache keys of every full block: key_j = SHA-256(key_{j-1} ||
    int32 ids of block j), key_{-1} = ``root`` (32 bytes, zeros by default).
    ``token_offsets`` (int64 [N + 1]) splits ``token_ids`` (int32) into
    sequences; returns uint8 [sum_s floor(len_s / block_size), 32]. Without
    ``key_offsets`` the library computes the packed layout
    (:func:`prefix_key_offsets`); only its last entry, the key count, is read
    back to size ``out`` when ``out`` is not given."""
    dev = _cuda(token_ids, token_offsets)
    _need(token_ids.dtype == torch.int32 and token_ids.dim() == 1, "token_ids: int32 [T]")
    _need(token_offsets.dtype == torch.int64 and token_offsets.dim() == 1, "token_offsets: int64 [N + 1]")
    n = token_offsets.shape[0] - 1
    if key_offsets is None:
        key_offsets = prefix_key_offsets(token_offsets, block_size)
    _cuda(key_offsets, token_ids)
    _need(key_offsets.dtype == torch.int64 and key_offsets.shape == token_offsets.shape,
          "key_offsets: int64 [N + 1]")
    if out is None:
        total = int(key_offsets[-1].item()) if n > 0 else 0
        out = torch.empty((total, 32), dtype=torch.uint8, device=dev)
    _cuda(out, token_ids)
    _need(out.dtype == torch.uint8 and out.dim() == 2 and out.shape[1] == 32, "out: uint8 [K, 32]")
    _need(root is None or len(root) == 32, "root: 32 bytes")
    with _on(dev):
        st = _lib.lib().pa_prefix_hash(_ptr(token_ids), _ptr(token_offsets), _ptr(key_offsets), n,
                                       int(block_size), None if root is None else bytes(root),
                                       _ptr(out), _stream(dev))
    _lib.check("pa_prefix_hash", st)
    return out


def decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_seq_len: int, partition_tokens: int) -> int:
    return int(_lib.lib().pa_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                    max_seq_len, partition_tokens))


def new_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  max_seq_len: int, partition_tokens: int, device) -> Optional[torch.Tensor]:
    """A workspace for pa_decode (None when the call needs none); reusable for
    any later call of the same mode and shape."""
    n = decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                               partition_tokens)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def default_partition(num_seqs: int, num_kv_heads: int, max_seq_len: int, block_size: int) -> int:
    v = int(_lib.lib().pa_decode_default_partition(num_seqs, num_kv_heads, max_seq_len, block_size))
    if v < 0 and v != _lib.PA_PARTITION_BALANCED:
        _lib.check("pa_decode_default_partition", v)
    return v


def decode_kernel_name(num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                       max_seq_len: int, partition_tokens: int) -> str:
    """Which kernel(s) :func:`decode` launches for this shape and partition choice."""
    name = _lib.lib().pa_decode_kernel_name(num_q_heads, num_kv_heads, head_dim, block_size,
                                            max_seq_len, partition_tokens)
    if name is None:
        raise _lib.PagedKVError("pa_decode_kernel_name", -3)  # PA_ERR_SHAPE
    return name.decode()


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           seq_lens: torch.Tensor, scale: float, *, max_seq_len: int,
           out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
           partition_tokens: Optional[int] = None,
           workspace: Optional[torch.Tensor] = None, k_scale: Optional[float] = None,
           v_scale: Optional[float] = None) -> torch.Tensor:
    """Paged decode attention: out[s, h] over the first seq_lens[s] tokens of sequence s.

    ``max_seq_len`` bounds ``seq_lens`` (it sizes the launch, so the call never
    reads the lengths back). ``partition_tokens`` = 0 runs one pass per
    (sequence, KV head); a multiple of 16 runs split-K with a reduce;
    ``PA_PARTITION_BALANCED`` (-1) gives every warp an equal share of the
    work; None picks the library's default for this shape. The workspace,
    when a split needs one, comes from the caller (see :func:`new_workspace`)
    or is allocated here. E4M3 caches take the layer's ``k_scale`` and
    ``v_scale``; q is then float16 or bfloat16.
    """
    dev = _cuda(q, k_cache, v_cache, block_tables, seq_lens)
    _need(q.dim() == 3 and q.shape[2] == k_cache.shape[3], "q: [N, Hq, D] with the cache's D")
    _check_act(q, k_cache, "q")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == q.shape[0], "block_tables: int32 [N, maxB]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.shape == (q.shape[0],), "seq_lens: int32 [N]")
    n, hq, d = q.shape
    if out is None:
        out = torch.empty((n, hq, d), dtype=out_dtype or q.dtype, device=dev)
    _cuda(out, q)
    _need(out.shape == q.shape and out.dtype in _DTYPES, "out: [N, Hq, D] of float16/bfloat16/float32")
    nb, b, hkv, _ = k_cache.shape
    if partition_tokens is None:
        partition_tokens = default_partition(n, hkv, max_seq_len, b)
    if workspace is None:
        workspace = new_workspace(n, hq, hkv, d, max_seq_len, partition_tokens, dev)
    if workspace is not None:
        _cuda(workspace, q)
    cache = make_cache(k_cache, v_cache, act_dtype=q.dtype, k_scale=k_scale, v_scale=v_scale)
    with _on(dev):
        st = _lib.lib().pa_decode(_ptr(q), n, hq, ctypes.byref(cache), _ptr(block_tables),
                              block_tables.shape[1], _ptr(seq_lens), int(max_seq_len), float(scale),
                              _ptr(out), _DTYPES[out.dtype], int(partition_tokens), _ptr(workspace),
                              0 if workspace is None else workspace.numel() * workspace.element_size(),
                              _stream(dev))
    _lib.check("pa_decode", st)
    return out


def prefill_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                            block_size: int, max_q_len: int) -> int:
    return int(_lib.lib().pa_prefill_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                     block_size, max_q_len))


def new_prefill_workspace(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                          block_size: int, max_q_len: int, device) -> Optional[torch.Tensor]:
    """A workspace for pa_prefill (None when the shape needs none); reusable
    for any later call of the same shape, one call at a time."""
    n = prefill_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_q_len)
    return torch.empty(n, dtype=torch.uint8, device=device) if n else None


def prefill_kernel_name(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                        block_size: int, max_q_len: int, with_workspace: bool = True,
                        num_sms: int = 0) -> str:
    """The kernel pa_prefill runs for this shape (num_sms 0: the current device's)."""
    name = _lib.lib().pa_prefill_kernel_name(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                             block_size, max_q_len, int(bool(with_workspace)),
                                             int(num_sms))
    _need(name is not None, "pa_prefill_kernel_name rejected these sizes")
    return name.decode()


def prefill(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
            seq_lens: torch.Tensor, q_start: torch.Tensor, scale: float, *, max_q_len: int,
            out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
            k_scale: Optional[float] = None, v_scale: Optional[float] = None,
            workspace="auto") -> torch.Tensor:
    """Causal attention for several new tokens per sequence (chunked prefill,
    speculative verification): query row t of sequence s (rows q_start[s] ..
    q_start[s+1]) sits at position seq_lens[s] - n_s + (t - q_start[s]) and
    attends to positions 0 .. that position. The new tokens' K/V must already
    be in the cache. ``max_q_len`` bounds every n_s (it sizes the launch).
    E4M3 caches take the layer's ``k_scale`` and ``v_scale``. ``workspace``:
    a tensor from :func:`new_prefill_workspace`, "auto" (allocate one when the
    shape can use it) or None (run without, on the per-sequence kernels).
    """
    dev = _cuda(q, k_cache, v_cache, block_tables, seq_lens, q_start)
    _need(q.dim() == 3 and q.shape[2] == k_cache.shape[3], "q: [T, Hq, D] with the cache's D")
    _check_act(q, k_cache, "q")
    n = block_tables.shape[0]
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2, "block_tables: int32 [N, maxB]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.shape == (n,), "seq_lens: int32 [N]")
    _need(q_start.dtype == torch.int32 and q_start.shape == (n + 1,), "q_start: int32 [N + 1]")
    t_all, hq, d = q.shape
    if out is None:
        out = torch.empty((t_all, hq, d), dtype=out_dtype or q.dtype, device=dev)
    _cuda(out, q)
    _need(out.shape == q.shape and out.dtype in _DTYPES, "out: [T, Hq, D] of float16/bfloat16/float32")
    cache = make_cache(k_cache, v_cache, act_dtype=q.dtype, k_scale=k_scale, v_scale=v_scale)
    if isinstance(workspace, str):
        _need(workspace == "auto", 'workspace: a tensor, "auto" or None')
        workspace = new_prefill_workspace(n, hq, cache.num_kv_heads, d, cache.block_size,
                                          int(max_q_len), dev)
    if workspace is not None:
        _cuda(workspace, q)
    with _on(dev):
        st = _lib.lib().pa_prefill(_ptr(q), n, _ptr(q_start), int(max_q_len), hq, ctypes.byref(cache),
                               _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                               float(scale), _ptr(out), _DTYPES[out.dtype], _ptr(workspace),
                               0 if workspace is None else workspace.numel() * workspace.element_size(),
                               _stream(dev))
    _lib.check("pa_prefill", st)
    return out


def decode_static_workspace(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                            block_tables: torch.Tensor, seq_lens: torch.Tensor, scale: float, *,
                            max_seq_len: int, partition_tokens: int,
                            out: Optional[torch.Tensor] = None,
                            out_dtype: Optional[torch.dtype] = None, k_scale: Optional[float] = None,
                            v_scale: Optional[float] = None) -> torch.Tensor:
    """Decode like :func:`decode`, with the split-K partials kept in the library's
    fixed device array instead of a workspace from the caller.

    For callers that cannot allocate device memory. The array holds
    ``STATIC_WORKSPACE_BYTES``; larger workspaces raise. All calls share it, so
    calls that overlap on the GPU race. Only ``out`` (when not given) is
    allocated here, by torch, for convenience.
    """
    dev = _cuda(q, k_cache, v_cache, block_tables, seq_lens)
    _need(q.dim() == 3 and q.shape[2] == k_cache.shape[3], "q: [N, Hq, D] with the cache's D")
    _check_act(q, k_cache, "q")
    _need(block_tables.dtype == torch.int32 and block_tables.dim() == 2
          and block_tables.shape[0] == q.shape[0], "block_tables: int32 [N, maxB]")
    _need(seq_lens.dtype == torch.int32 and seq_lens.shape == (q.shape[0],), "seq_lens: int32 [N]")
    n, hq, d = q.shape
    if out is None:
        out = torch.empty((n, hq, d), dtype=out_dtype or q.dtype, device=dev)
    _cuda(out, q)
    _need(out.shape == q.shape and out.dtype in _DTYPES, "out: [N, Hq, D] of float16/bfloat16/float32")
    cache = make_cache(k_cache, v_cache, act_dtype=q.dtype, k_scale=k_scale, v_scale=v_scale)
    with _on(dev):
        st = _lib.lib().pa_decode_static_workspace(
        _ptr(q), n, hq, ctypes.byref(cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), int(max_seq_len), float(scale), _ptr(out), _DTYPES[out.dtype],
        int(partition_tokens), _stream(dev))
    _lib.check("pa_decode_static_workspace", st)
    return out


def get_device_error(device: Optional[torch.device] = None) -> int:
    """Synchronise the current stream, read and clear the device error word."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    v = ctypes.c_int32(0)
    with torch.cuda.device(dev):
        st = _lib.lib().pa_get_device_error(ctypes.byref(v), _stream(dev))
    _lib.check("pa_get_device_error", st)
    return int(v.value)
