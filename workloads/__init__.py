"""Seeded synthetic inputs for the paged KV-cache hot path.

Shared by the tests, the benchmark and the oracle checks. It holds input
generation and host-side block bookkeeping only; no attention arithmetic and no
slot arithmetic live here.
"""
from .block_manager import BlockPool, PoolExhausted, SeqTable, kv_bytes_per_token
from .configs import (CONFIG_NAMES, PREFILL_NAMES, Workload, decode_step_tokens, f16_bits_to_f32,
                      make_config, make_config5_steps, make_prefill_case, make_prefill_config,
                      make_random_case, bf16_bits_to_f32)

__all__ = [
    "BlockPool", "PoolExhausted", "SeqTable", "kv_bytes_per_token",
    "CONFIG_NAMES", "PREFILL_NAMES", "Workload", "decode_step_tokens", "make_config",
    "make_config5_steps",
    "make_prefill_case", "make_prefill_config", "make_random_case",
    "f16_bits_to_f32", "bf16_bits_to_f32",
]
