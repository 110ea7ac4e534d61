"""A decode step bound to fixed buffers, for loops that run the same shapes.

A serving loop calls slot mapping, the KV write and decode on buffers whose
shapes do not change between steps. :class:`DecodeStep` checks those buffers
once, builds the C-ABI argument lists once, and then each :meth:`run` is three
pre-marshalled calls into libpagedkv on one stream. :meth:`run_from_host`
adds the per-step traffic a host-driven engine has: one host-to-device copy
of a pinned staging buffer holding all of the step's inputs, and one
device-to-host copy of the output.

Marshalling only: every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

import ctypes
from typing import Dict, Optional

import torch

from . import _lib
from .ops import _DTYPES, _cuda, _need, default_partition, is_fp8_cache, make_cache, new_workspace

_ALIGN = 256  # bytes; every packed input starts on a 256-byte boundary


def _vp(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


class DecodeStep:
    """slot_mapping -> write_kv -> decode over fixed device buffers.

    Device inputs are views into one staging buffer, laid out by
    :meth:`layout`: ``q [N, Hq, D]``, ``key``/``value [T, H_kv, D]`` (the cache
    dtype, or ``act_dtype`` for an E4M3 cache), ``seq_idx``/``positions`` int32
    ``[T]``, ``block_tables`` int32 ``[N, maxB]`` and ``seq_lens`` int32
    ``[N]``. The caches, the output (``[N, Hq, D]`` of ``out_dtype``) and the
    decode workspace are allocated or passed once. E4M3 caches also take the
    layer's ``k_scale`` and ``v_scale``.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, *, num_seqs: int,
                 num_q_heads: int, num_tokens: int, max_blocks_per_seq: int, max_seq_len: int,
                 scale: float, out_dtype: torch.dtype = torch.float32,
                 partition_tokens: Optional[int] = None, stream: Optional[torch.cuda.Stream] = None,
                 act_dtype: Optional[torch.dtype] = None, k_scale: Optional[float] = None,
                 v_scale: Optional[float] = None):
        dev = _cuda(k_cache, v_cache)
        self.device = dev
        self.k_cache, self.v_cache = k_cache, v_cache
        self.act_dtype = act_dtype if is_fp8_cache(k_cache) else k_cache.dtype
        nb, b, hkv, d = k_cache.shape
        self.num_blocks, self.block_size = int(nb), int(b)
        _need(num_q_heads % hkv == 0, "num_q_heads must be a multiple of the cache's KV heads")
        self.shape = dict(N=num_seqs, Hq=num_q_heads, Hkv=int(hkv), D=int(d), T=num_tokens,
                          maxB=max_blocks_per_seq)
        self.max_seq_len = int(max_seq_len)
        self.scale = float(scale)
        # Its own stream by default (graph capture needs a non-default one); it
        # starts after whatever the caller's stream has queued so far.
        self.stream = stream if stream is not None else torch.cuda.Stream(dev)
        self.stream.wait_stream(torch.cuda.current_stream(dev))
        # one staging buffer for every per-step input
        self.offsets, self.nbytes = self.layout(self.act_dtype, **self.shape)
        self.staging = torch.empty(self.nbytes, dtype=torch.uint8, device=dev)
        self.inputs = self._views(self.staging)
        self.slots = torch.empty(num_tokens, dtype=torch.int64, device=dev)
        self.out = torch.empty((num_seqs, num_q_heads, d), dtype=out_dtype, device=dev)
        _need(out_dtype in _DTYPES, "out_dtype: float16, bfloat16 or float32")
        if partition_tokens is None:
            partition_tokens = default_partition(num_seqs, int(hkv), self.max_seq_len, int(b))
        self.partition_tokens = int(partition_tokens)
        self.workspace = new_workspace(num_seqs, num_q_heads, int(hkv), int(d), self.max_seq_len,
                                       self.partition_tokens, dev)
        self._cache = make_cache(k_cache, v_cache, act_dtype=self.act_dtype, k_scale=k_scale,
                                 v_scale=v_scale)
        lib = _lib.lib()
        st = ctypes.c_void_p(self.stream.cuda_stream)
        i = self.inputs
        self._calls = (
            ("pa_slot_mapping", lib.pa_slot_mapping,
             (_vp(i["block_tables"]), num_seqs, max_blocks_per_seq, _vp(i["seq_idx"]),
              _vp(i["positions"]), num_tokens, self.block_size, self.num_blocks, _vp(self.slots), st)),
            ("pa_write_kv", lib.pa_write_kv,
             (_vp(i["key"]), _vp(i["value"]), _vp(self.slots), num_tokens,
              ctypes.byref(self._cache), st)),
            ("pa_decode", lib.pa_decode,
             (_vp(i["q"]), num_seqs, num_q_heads, ctypes.byref(self._cache), _vp(i["block_tables"]),
              max_blocks_per_seq, _vp(i["seq_lens"]), self.max_seq_len, ctypes.c_float(self.scale),
              _vp(self.out), _DTYPES[out_dtype], self.partition_tokens, _vp(self.workspace),
              0 if self.workspace is None else self.workspace.numel(), st)),
        )
        self._host_staging: Optional[torch.Tensor] = None
        self._host_out: Optional[torch.Tensor] = None
        self._graph: Optional[torch.cuda.CUDAGraph] = None

    # ------------------------------------------------------------------ layout

    @staticmethod
    def layout(act_dtype: torch.dtype, *, N: int, Hq: int, Hkv: int, D: int, T: int, maxB: int):
        """Byte offsets of each input in the staging buffer, and its size."""
        esz = torch.tensor([], dtype=act_dtype).element_size()
        sizes = [("q", N * Hq * D * esz), ("key", T * Hkv * D * esz), ("value", T * Hkv * D * esz),
                 ("seq_idx", T * 4), ("positions", T * 4), ("block_tables", N * maxB * 4),
                 ("seq_lens", N * 4)]
        offsets, pos = {}, 0
        for name, n in sizes:
            offsets[name] = (pos, n)
            pos += (n + _ALIGN - 1) // _ALIGN * _ALIGN
        return offsets, pos

    def _views(self, buf: torch.Tensor) -> Dict[str, torch.Tensor]:
        s, cdt = self.shape, self.act_dtype
        shapes = {"q": ((s["N"], s["Hq"], s["D"]), cdt), "key": ((s["T"], s["Hkv"], s["D"]), cdt),
                  "value": ((s["T"], s["Hkv"], s["D"]), cdt), "seq_idx": ((s["T"],), torch.int32),
                  "positions": ((s["T"],), torch.int32),
                  "block_tables": ((s["N"], s["maxB"]), torch.int32), "seq_lens": ((s["N"],), torch.int32)}
        out = {}
        for name, (off, n) in self.offsets.items():
            shape, dt = shapes[name]
            out[name] = buf[off:off + n].view(dt).view(shape)
        return out

    def host_buffers(self):
        """Pinned host staging buffer (same layout, as named views) and output."""
        if self._host_staging is None:
            self._host_staging = torch.empty(self.nbytes, dtype=torch.uint8).pin_memory()
            self._host_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
            self._host_views = self._views(self._host_staging)
        return self._host_views, self._host_out

    # ------------------------------------------------------------------ run

    def run(self, decode_events=None) -> torch.Tensor:
        """One step on the device buffers, enqueued on :attr:`stream` (the
        caller synchronises); returns the device output.

        ``decode_events``: optional (start, end) CUDA events recorded on the
        step's stream around the decode call alone.
        """
        for name, fn, args in self._calls:
            if decode_events is not None and name == "pa_decode":
                decode_events[0].record(self.stream)
            st = fn(*args)
            if st != 0:
                raise _lib.PagedKVError(name, st)
        if decode_events is not None:
            decode_events[1].record(self.stream)
        return self.out

    def _enqueue_from_host(self) -> None:
        self.staging.copy_(self._host_staging, non_blocking=True)
        self.run()
        self._host_out.copy_(self.out, non_blocking=True)

    def capture_graph(self) -> None:
        """Record copy-in, the three calls and copy-out as one CUDA graph that
        :meth:`run_from_host` then replays. Runs the step once first, on the
        step's stream, so every one-time set-up happens outside the capture.
        The graph bakes in this step's buffers, shapes and partition choice."""
        if self._host_staging is None:
            self.host_buffers()
        with torch.cuda.stream(self.stream):
            self._enqueue_from_host()
        self.stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=self.stream):
            self._enqueue_from_host()
        self._graph = graph

    def run_from_host(self) -> torch.Tensor:
        """Copy the pinned staging buffer in, run the step, copy the output out
        and wait for it; returns the pinned host output."""
        if self._host_staging is None:
            self.host_buffers()
        with torch.cuda.stream(self.stream):  # replay() launches on the current stream
            if self._graph is not None:
                self._graph.replay()
            else:
                self._enqueue_from_host()
        self.stream.synchronize()
        return self._host_out
