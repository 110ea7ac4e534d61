"""fp64 CPU oracle for the paged KV-cache hot path (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU baseline / reference
arm may import this package. The library never imports it.
"""
from .paged_attention import (attention, bits_to_f64, combine_partitions, copy_blocks, decode,
                              e4m3_to_f64, f32_to_e4m3, gather_kv, online_softmax_blocks,
                              partition_state, prefill, prefix_block_keys, quantize_e4m3, slot_mapping,
                              swap_blocks,
                              write_kv, write_kv_e4m3)

__all__ = ["attention", "bits_to_f64", "combine_partitions", "copy_blocks", "decode",
           "e4m3_to_f64", "f32_to_e4m3", "gather_kv", "online_softmax_blocks", "partition_state",
           "prefill", "prefix_block_keys", "quantize_e4m3", "slot_mapping", "swap_blocks", "write_kv", "write_kv_e4m3"]
