"""GB300-native paged KV-cache hot path.

The compute lives in ``libpagedkv.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/pa.h``); this package is its Python binding.

* :func:`slot_mapping` - pool slot of each new token;
* :func:`write_kv` - slot-mapped write of new K/V rows;
* :func:`copy_blocks` - whole-block copies for copy-on-write;
* :func:`swap_blocks` - block copies between the GPU pool and a pinned host
  pool, for preemption by swapping;
* :func:`prefix_hash` - prefix-cache keys of full blocks (SHA-256 chain), packed
  by :func:`prefix_key_offsets`;
* :func:`decode` - decode attention through block tables (single pass,
  split-K with a reduce, or a balanced split), GQA heads packed per KV head;
* :func:`prefill` - causal attention for several new tokens per sequence
  (chunked prefill, speculative verification); a few-token batch given a
  workspace (:func:`new_prefill_workspace`) may run on the balanced kernel;
* :class:`DecodeStep` - the three calls bound to fixed buffers for loops.
"""
from ._lib import (DEVERR_BLOCK_ID, DEVERR_POSITION, DEVERR_SEQ_LEN, DEVERR_SLOT, DEVERR_TIMEOUT,
                   EXPORTED, LIB_PATH, PagedKVError, lib)
from ._lib import PA_PARTITION_BALANCED, STATIC_WORKSPACE_BYTES
from .step import DecodeStep
from .ops import (check_copy_pairs, copy_blocks, decode, decode_kernel_name, decode_static_workspace,
                  decode_workspace_bytes, default_partition, get_device_error, make_cache,
                  new_prefill_workspace, new_workspace, prefill, prefill_kernel_name,
                  prefill_workspace_bytes, prefix_hash, prefix_key_offsets, slot_mapping,
                  swap_blocks, write_kv)

__all__ = [
    "DEVERR_BLOCK_ID", "DEVERR_POSITION", "DEVERR_SEQ_LEN", "DEVERR_SLOT", "DEVERR_TIMEOUT",
    "EXPORTED", "LIB_PATH", "PagedKVError", "lib", "check_copy_pairs", "copy_blocks", "decode",
    "decode_workspace_bytes", "default_partition", "get_device_error", "make_cache",
    "slot_mapping", "write_kv", "decode_static_workspace", "STATIC_WORKSPACE_BYTES",
    "PA_PARTITION_BALANCED", "new_workspace", "DecodeStep", "decode_kernel_name",
    "prefill", "prefill_workspace_bytes", "new_prefill_workspace", "prefill_kernel_name",
    "swap_blocks", "prefix_hash", "prefix_key_offsets",
]
