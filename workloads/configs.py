"""Seeded synthetic workloads shaped like the pages' decode scenarios.

Every array is generated on the host with ``numpy.random.default_rng`` and a
fixed seed, so the GPU path and the oracle see identical bytes on any machine.
Half-precision tensors are carried as ``uint16`` bit patterns (fp16 or bf16).

Recipe (shared by every config):

* ``q`` and the K/V rows the scenario writes are drawn N(0,1) and rounded to
  the storage dtype (round-to-nearest-even).
* Pool blocks that hold a sequence's tokens are filled with N(0,1) values. Each
  block is a window, at a seeded random offset, into one 2**24-element N(0,1)
  sample (drawing >1e9 normals per workload on the host is too slow).
* Every slot that no sequence owns holds a quiet-NaN pattern: unused blocks and
  the tail rows of each sequence's last block. A kernel that lets any of them
  into its arithmetic produces NaN, so masking is checked at every size.
* Physical placement comes from :mod:`workloads.block_manager` with a seeded
  shuffle of the free list; block tables are zero padded to the longest table.
* FP8 (E4M3) caches (``kv_dtype="e4m3"``) hold uniformly drawn byte codes
  (every code but the two NaN codes, 0x7F and 0xFF) in owned rows and the NaN
  code elsewhere; q and the new K/V rows stay fp16/bf16 and the layer scales
  are FP8_K_SCALE / FP8_V_SCALE. The generator draws bytes only: it encodes
  nothing.

Five named configs follow the decode scenarios the pages discuss: a tiny case
holding the ten-token, b=4, table [7, 2, 11] example; a 7B/13B-style MHA batch;
the 70B GQA head shape (80 layers, 8 KV heads, head_dim 128) timed per layer;
a 32k-token long-context batch for split-K; and a shared 1000-token prefix with
copy-on-write.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional, Sequence

import numpy as np

from .block_manager import BlockPool, SeqTable

NAN_BITS = {"f16": np.uint16(0x7E00), "bf16": np.uint16(0x7FC0), "e4m3": np.uint8(0x7F)}
# Per-layer scales of E4M3 caches in the generated workloads: a stored code c
# stands for value(c) * scale. Uniform codes times these give K and V of rms
# about 0.8 and 0.65; N(0,1) inputs beyond |x| = 3 (K) and 2.5 (V) saturate.
FP8_K_SCALE = float(np.float32(3.0 / 448.0))
FP8_V_SCALE = float(np.float32(2.5 / 448.0))
_BASE_LEN = 1 << 24

CONFIG_NAMES = {
    1: "tiny_b4_fp16",
    2: "mha_7b13b_fp16_b16",
    3: "gqa_70b_bf16_b16",
    4: "long32k_splitk_bf16",
    5: "prefix_cow_fp16_b16",
}


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even) and return the bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))
    return ((u + rounding) >> np.uint32(16)).astype(np.uint16)


def f16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(np.float32)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f16":
        return f32_to_f16_bits(x)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclass
class Workload:
    """All host-side inputs of one scenario.

    Layouts: ``k_cache``/``v_cache`` are ``[num_blocks, block_size, num_kv_heads,
    head_dim]``; ``q`` is ``[num_seqs, num_q_heads, head_dim]``; ``key``/``value``
    are ``[num_tokens, num_kv_heads, head_dim]``; ``block_tables`` is
    ``int32[num_seqs, max_blocks_per_seq]``.

    The scenario is: block copies ``copy_pairs`` (copy-on-write), then the write
    of ``key``/``value`` for the tokens ``(seq_idx, positions)``, then decode of
    every sequence at length ``seq_lens``.
    """
    name: str
    dtype: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    scale: float
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    block_tables: np.ndarray
    seq_lens: np.ndarray
    key: np.ndarray
    value: np.ndarray
    seq_idx: np.ndarray
    positions: np.ndarray
    copy_pairs: np.ndarray
    partition_tokens: int = 0
    shared_blocks: List[int] = field(default_factory=list)
    meta: Dict[str, object] = field(default_factory=dict)
    # Multi-token cases: sequence s owns query rows q_start[s] .. q_start[s+1]
    # of q [T, H_q, D] (None: decode, one query row per sequence).
    q_start: Optional[np.ndarray] = None
    # E4M3 caches: "e4m3" (uint8 codes, K/V values code * k_scale / v_scale);
    # None: the cache holds ``dtype`` bit patterns.
    kv_dtype: Optional[str] = None
    k_scale: float = 1.0
    v_scale: float = 1.0

    @property
    def cache_dtype(self) -> str:
        return self.kv_dtype or self.dtype

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.seq_lens.size else 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def decode_step_tokens(w: Workload) -> np.ndarray:
    """Indices (into key/value) of each sequence's newest token, position L-1.

    A decode step writes exactly these rows and then attends over L tokens.
    """
    last = {}
    for i, (s, t) in enumerate(zip(w.seq_idx.tolist(), w.positions.tolist())):
        if t == int(w.seq_lens[s]) - 1:
            last[s] = i
    return np.array([last[s] for s in sorted(last)], dtype=np.int64)


# ----------------------------------------------------------------------------
# helpers


class _Filler:
    """Fills pool blocks with windows of one N(0,1) sample (fp16 / bf16), or of
    one sample of uniform non-NaN byte codes (e4m3)."""

    def __init__(self, rng: np.random.Generator, dtype: str) -> None:
        self.rng = rng
        if dtype == "e4m3":
            mag = rng.integers(0, 0x7F, size=_BASE_LEN, dtype=np.uint8)  # 0x00 .. 0x7E
            sign = rng.integers(0, 2, size=_BASE_LEN, dtype=np.uint8) << np.uint8(7)
            self.base = mag | sign
        else:
            self.base = to_bits(rng.standard_normal(_BASE_LEN, dtype=np.float32), dtype)

    def block(self, n: int) -> np.ndarray:
        off = int(self.rng.integers(0, _BASE_LEN - n))
        return self.base[off:off + n]


def _normal_bits(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    return to_bits(rng.standard_normal(shape, dtype=np.float32), dtype)


def _pad_tables(tables: Sequence[Sequence[int]], pad: int) -> np.ndarray:
    width = max(1, max((len(t) for t in tables), default=1))
    out = np.full((len(tables), width), pad, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out


def _fill_sequences(k: np.ndarray, v: np.ndarray, tables, lens, filler_k: _Filler,
                    filler_v: _Filler, nan: np.uint16, skip_blocks=()) -> None:
    """Give every block a sequence owns N(0,1) rows; NaN rows past the length."""
    b = k.shape[1]
    per_block = int(np.prod(k.shape[1:]))
    done = set(skip_blocks)
    for table, L in zip(tables, lens):
        nblk = -(-int(L) // b)
        for j in range(nblk):
            blk = int(table[j])
            if blk in done:
                continue
            done.add(blk)
            k[blk] = filler_k.block(per_block).reshape(k.shape[1:])
            v[blk] = filler_v.block(per_block).reshape(v.shape[1:])
            valid = int(L) - j * b
            if valid < b:
                k[blk, valid:] = nan
                v[blk, valid:] = nan


def _new_pool(nb: int, b: int, hkv: int, d: int, dtype: str):
    nan = NAN_BITS[dtype]
    k = np.full((nb, b, hkv, d), nan, dtype=nan.dtype)
    v = np.full((nb, b, hkv, d), nan, dtype=nan.dtype)
    return k, v, nan


def _fp8_fields(kv_dtype: Optional[str]) -> dict:
    if kv_dtype is None:
        return {}
    if kv_dtype != "e4m3":
        raise ValueError(f"unknown kv_dtype {kv_dtype!r}")
    return {"kv_dtype": "e4m3", "k_scale": FP8_K_SCALE, "v_scale": FP8_V_SCALE}


# ----------------------------------------------------------------------------
# generic random case (tests)


def make_random_case(seed: int, *, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                     head_dim: int, block_size: int, seq_lens: Sequence[int],
                     dtype: str = "f16", pool_factor: float = 1.25, pad: int = 0,
                     scale: Optional[float] = None, partition_tokens: int = 0,
                     name: str = "random", kv_dtype: Optional[str] = None) -> Workload:
    """A decode batch with given lengths and a shuffled pool.

    The scenario writes each sequence's newest token (position L-1) and decodes.
    Sequences of length 0 own no block and write nothing. ``kv_dtype="e4m3"``
    gives an FP8 pool (q and the new rows stay ``dtype``).
    """
    rng = np.random.default_rng(seed)
    b = block_size
    lens = [int(x) for x in seq_lens]
    assert len(lens) == num_seqs
    need = sum(-(-L // b) for L in lens)
    nb = max(1, int(np.ceil(pool_factor * need)))
    pool = BlockPool(nb, b, free_order=rng.permutation(nb))
    seqs = []
    for L in lens:
        s = SeqTable(pool)
        s.admit(L)
        seqs.append(s)
    tables = [s.table for s in seqs]
    cdt = kv_dtype or dtype
    k, v, nan = _new_pool(nb, b, num_kv_heads, head_dim, cdt)
    fk, fv = _Filler(rng, cdt), _Filler(rng, cdt)
    _fill_sequences(k, v, tables, lens, fk, fv, nan)
    q = _normal_bits(rng, (num_seqs, num_q_heads, head_dim), dtype)
    writers = [i for i, L in enumerate(lens) if L > 0]
    key = _normal_bits(rng, (len(writers), num_kv_heads, head_dim), dtype)
    value = _normal_bits(rng, (len(writers), num_kv_heads, head_dim), dtype)
    return Workload(
        name=name, dtype=dtype, num_seqs=num_seqs, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=b, num_blocks=nb,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_dim)),
        q=q, k_cache=k, v_cache=v, block_tables=_pad_tables(tables, pad),
        seq_lens=np.array(lens, dtype=np.int32), key=key, value=value,
        seq_idx=np.array(writers, dtype=np.int32),
        positions=np.array([lens[i] - 1 for i in writers], dtype=np.int32),
        copy_pairs=np.zeros((0, 2), dtype=np.int64), partition_tokens=partition_tokens,
        **_fp8_fields(kv_dtype))


def make_prefill_case(seed: int, *, num_seqs: int, num_q_heads: int, num_kv_heads: int,
                      head_dim: int, block_size: int, seq_lens: Sequence[int],
                      q_lens: Sequence[int], dtype: str = "f16", pool_factor: float = 1.25,
                      scale: Optional[float] = None, name: str = "prefill",
                      kv_dtype: Optional[str] = None) -> Workload:
    """A multi-token batch: sequence s ends with q_lens[s] new tokens.

    The pool holds the first L - n tokens of each sequence (n = q_lens[s]); the
    scenario writes the K/V of the n new tokens (positions L - n .. L - 1) and
    then runs causal attention for their n queries. Query rows are laid out
    sequence by sequence in ``q [sum(q_lens), H_q, D]``.
    """
    rng = np.random.default_rng(seed)
    b = block_size
    lens = [int(x) for x in seq_lens]
    qn = [int(x) for x in q_lens]
    assert len(lens) == num_seqs and len(qn) == num_seqs
    assert all(0 <= n <= L for n, L in zip(qn, lens))
    need = sum(-(-L // b) for L in lens)
    nb = max(1, int(np.ceil(pool_factor * need)))
    pool = BlockPool(nb, b, free_order=rng.permutation(nb))
    seqs = []
    for L in lens:
        s = SeqTable(pool)
        s.admit(L)
        seqs.append(s)
    tables = [s.table for s in seqs]
    cdt = kv_dtype or dtype
    k, v, nan = _new_pool(nb, b, num_kv_heads, head_dim, cdt)
    fk, fv = _Filler(rng, cdt), _Filler(rng, cdt)
    _fill_sequences(k, v, tables, lens, fk, fv, nan)
    t_all = sum(qn)
    q = _normal_bits(rng, (t_all, num_q_heads, head_dim), dtype)
    key = _normal_bits(rng, (t_all, num_kv_heads, head_dim), dtype)
    value = _normal_bits(rng, (t_all, num_kv_heads, head_dim), dtype)
    seq_idx = np.concatenate([np.full(n, i, dtype=np.int32) for i, n in enumerate(qn)] +
                             [np.zeros(0, dtype=np.int32)])
    positions = np.concatenate([np.arange(L - n, L, dtype=np.int32) for n, L in zip(qn, lens)] +
                               [np.zeros(0, dtype=np.int32)])
    q_start = np.concatenate([[0], np.cumsum(qn)]).astype(np.int32)
    return Workload(
        name=name, dtype=dtype, num_seqs=num_seqs, num_q_heads=num_q_heads,
        num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=b, num_blocks=nb,
        scale=float(scale if scale is not None else 1.0 / np.sqrt(head_dim)),
        q=q, k_cache=k, v_cache=v, block_tables=_pad_tables(tables, 0),
        seq_lens=np.array(lens, dtype=np.int32), key=key, value=value, seq_idx=seq_idx,
        positions=positions, copy_pairs=np.zeros((0, 2), dtype=np.int64), q_start=q_start,
        **_fp8_fields(kv_dtype))


# ----------------------------------------------------------------------------
# the five named configs


def _config1(rng: np.random.Generator) -> Workload:
    """Tiny: 4 sequences {10,1,16,33}, 4/4 heads, d=64, b=4, 64 blocks, fp16.

    Sequence 0 holds the ten-token example with block table [7, 2, 11]. The pool
    starts as NaN; one write of all 60 tokens fills it, then decode runs.
    """
    lens = [10, 1, 16, 33]
    n, hq, hkv, d, b, nb = 4, 4, 4, 64, 4, 64
    pool = BlockPool(nb, b, free_order=rng.permutation(nb))
    s0 = SeqTable(pool)
    s0.table = [pool.take(7), pool.take(2), pool.take(11)]
    s0.length = 10
    seqs = [s0]
    for L in lens[1:]:
        s = SeqTable(pool)
        s.admit(L)
        seqs.append(s)
    k, v, _ = _new_pool(nb, b, hkv, d, "f16")
    total = sum(lens)
    seq_idx = np.concatenate([np.full(L, i, dtype=np.int32) for i, L in enumerate(lens)])
    positions = np.concatenate([np.arange(L, dtype=np.int32) for L in lens])
    return Workload(
        name=CONFIG_NAMES[1], dtype="f16", num_seqs=n, num_q_heads=hq, num_kv_heads=hkv,
        head_dim=d, block_size=b, num_blocks=nb, scale=1.0 / np.sqrt(d),
        q=_normal_bits(rng, (n, hq, d), "f16"), k_cache=k, v_cache=v,
        block_tables=_pad_tables([s.table for s in seqs], 0),
        seq_lens=np.array(lens, dtype=np.int32),
        key=_normal_bits(rng, (total, hkv, d), "f16"),
        value=_normal_bits(rng, (total, hkv, d), "f16"),
        seq_idx=seq_idx, positions=positions,
        copy_pairs=np.zeros((0, 2), dtype=np.int64), partition_tokens=0)


def _decode_batch(rng, name, *, n, hq, hkv, d, b, dtype, lens, partition_tokens,
                  kv_dtype=None) -> Workload:
    w = make_random_case(int(rng.integers(0, 2**31)), num_seqs=n, num_q_heads=hq,
                         num_kv_heads=hkv, head_dim=d, block_size=b, seq_lens=lens,
                         dtype=dtype, partition_tokens=partition_tokens, name=name,
                         kv_dtype=kv_dtype)
    return w


def _config5(rng: np.random.Generator, kv_dtype: Optional[str] = None) -> Workload:
    """256 sequences sharing one 1000-token prefix, private suffixes U[16,512].

    The prefix fills 62 full blocks and 8 rows of a 63rd. Each sequence's first
    suffix token lands in that shared partial block, so all but the last writer
    copy it first (255 copy-on-write pairs). The scenario then writes every
    suffix token and decodes.
    """
    n, hq, hkv, d, b, dtype = 256, 32, 8, 128, 16, "f16"
    prefix = 1000
    suffix = rng.integers(16, 512, size=n, endpoint=True)
    need = 63 + sum(-(-(prefix + int(s)) // b) - 62 for s in suffix)
    nb = int(np.ceil(1.25 * need))
    pool = BlockPool(nb, b, free_order=rng.permutation(nb))
    root = SeqTable(pool)
    root.admit(prefix)
    prefix_blocks = list(root.table)
    seqs = [root.fork() for _ in range(n)]
    root.free()
    pairs = []
    seq_idx, positions = [], []
    for i, s in enumerate(seqs):
        for _ in range(int(suffix[i])):
            seq_idx.append(i)
            positions.append(s.length)
            p = s.append()
            if p is not None:
                pairs.append(p)
    cdt = kv_dtype or dtype
    k, v, nan = _new_pool(nb, b, hkv, d, cdt)
    fk, fv = _Filler(rng, cdt), _Filler(rng, cdt)
    _fill_sequences(k, v, [prefix_blocks], [prefix], fk, fv, nan)
    lens = [prefix + int(s) for s in suffix]
    total = len(seq_idx)
    return Workload(
        name=CONFIG_NAMES[5], dtype=dtype, num_seqs=n, num_q_heads=hq, num_kv_heads=hkv,
        head_dim=d, block_size=b, num_blocks=nb, scale=1.0 / np.sqrt(d),
        q=_normal_bits(rng, (n, hq, d), dtype), k_cache=k, v_cache=v,
        block_tables=_pad_tables([s.table for s in seqs], 0),
        seq_lens=np.array(lens, dtype=np.int32),
        key=_normal_bits(rng, (total, hkv, d), dtype),
        value=_normal_bits(rng, (total, hkv, d), dtype),
        seq_idx=np.array(seq_idx, dtype=np.int32), positions=np.array(positions, dtype=np.int32),
        copy_pairs=np.array(pairs, dtype=np.int64).reshape(-1, 2), partition_tokens=512,
        shared_blocks=prefix_blocks[:62],
        meta={"prefix_tokens": prefix, "suffix_tokens": suffix.astype(np.int64)},
        **_fp8_fields(kv_dtype))


def make_config5_steps(steps: int = 32, kv_dtype: Optional[str] = None, seed: int = 1005) -> dict:
    """Config 5 as a decode loop: 256 sequences share one 1000-token prefix
    (62 full blocks and 8 rows of a 63rd) and then take ``steps`` decode steps;
    in step i every sequence appends its token at position 1000 + i.

    Step 0's tokens land in the shared partial block, so every sequence but
    the last to write copies it first (255 copy-on-write pairs, in sequence
    order); steps 8 and 24 open a fresh block for every sequence. Returns the
    initial pools (prefix rows filled, every other slot NaN) and, per step, the
    copy pairs to apply before the write, the new tokens' (seq_idx, positions,
    key, value), the step's q, the block tables and the lengths after the
    write.
    """
    rng = np.random.default_rng(seed)
    n, hq, hkv, d, b, dtype = 256, 32, 8, 128, 16, "f16"
    prefix = 1000
    need = 63 + n * (-(-(prefix + steps) // b) - 62)
    nb = int(np.ceil(1.25 * need))
    pool = BlockPool(nb, b, free_order=rng.permutation(nb))
    root = SeqTable(pool)
    root.admit(prefix)
    prefix_blocks = list(root.table)
    seqs = [root.fork() for _ in range(n)]
    root.free()
    cdt = kv_dtype or dtype
    k, v, nan = _new_pool(nb, b, hkv, d, cdt)
    fk, fv = _Filler(rng, cdt), _Filler(rng, cdt)
    _fill_sequences(k, v, [prefix_blocks], [prefix], fk, fv, nan)
    out_steps = []
    for _ in range(steps):
        pairs, positions = [], []
        for sq in seqs:
            positions.append(sq.length)
            p = sq.append()
            if p is not None:
                pairs.append(p)
        out_steps.append({
            "pairs": np.array(pairs, dtype=np.int64).reshape(-1, 2),
            "seq_idx": np.arange(n, dtype=np.int32),
            "positions": np.array(positions, dtype=np.int32),
            "key": _normal_bits(rng, (n, hkv, d), dtype),
            "value": _normal_bits(rng, (n, hkv, d), dtype),
            "q": _normal_bits(rng, (n, hq, d), dtype),
            "block_tables": _pad_tables([sq.table for sq in seqs], 0),
            "seq_lens": np.array([sq.length for sq in seqs], dtype=np.int32),
        })
    return {"name": "prefix_cow_steps_fp16_b16", "dtype": dtype, "num_seqs": n, "num_q_heads": hq,
            "num_kv_heads": hkv, "head_dim": d, "block_size": b, "num_blocks": nb,
            "scale": float(1.0 / np.sqrt(d)), "k_cache": k, "v_cache": v,
            "shared_blocks": prefix_blocks, "steps": out_steps, **_fp8_fields(kv_dtype)}


PREFILL_NAMES = ("verify4_70b_bf16_b16", "chunk512_gqa_bf16_b16", "prompt2k_mha_fp16_b16",
                 "verify4_long_bf16_b16")


def make_prefill_config(name: str, kv_dtype: Optional[str] = None) -> Workload:
    """Named multi-token workloads (seeded like the decode configs):

    * ``verify4_70b_bf16_b16``: speculative verification of 4 draft tokens per
      sequence on the 70B head shape (128 sequences, 64 / 8 heads, d 128,
      bf16, b 16, lengths U[512, 8192]) - reads the whole cache, like decode.
    * ``chunk512_gqa_bf16_b16``: chunked prefill, a 512-token chunk after
      4096 cached tokens for 8 sequences (32 / 8 heads, d 128, bf16, b 16).
    * ``prompt2k_mha_fp16_b16``: whole 2048-token prompts of 16 sequences on
      the 7B/13B head shape (32 / 32 heads, d 128, fp16, b 16).
    * ``verify4_long_bf16_b16``: verification of 4 drafts per sequence at long
      context, the long-context decode shape (8 sequences of 32768 tokens,
      32 / 8 heads, d 128, bf16, b 16): few (sequence, KV head) units.

    ``kv_dtype="e4m3"`` gives the same shapes an FP8 pool.
    """
    seed = 2000 + PREFILL_NAMES.index(name)
    rng = np.random.default_rng(seed)
    if name == "verify4_70b_bf16_b16":
        lens = rng.integers(512, 8192, size=128, endpoint=True)
        return make_prefill_case(seed, num_seqs=128, num_q_heads=64, num_kv_heads=8, head_dim=128,
                                 block_size=16, seq_lens=lens, q_lens=[4] * 128, dtype="bf16",
                                 name=name, kv_dtype=kv_dtype)
    if name == "chunk512_gqa_bf16_b16":
        return make_prefill_case(seed, num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 block_size=16, seq_lens=[4096 + 512] * 8, q_lens=[512] * 8,
                                 dtype="bf16", name=name, kv_dtype=kv_dtype)
    if name == "prompt2k_mha_fp16_b16":
        return make_prefill_case(seed, num_seqs=16, num_q_heads=32, num_kv_heads=32, head_dim=128,
                                 block_size=16, seq_lens=[2048] * 16, q_lens=[2048] * 16,
                                 dtype="f16", name=name, kv_dtype=kv_dtype)
    if name == "verify4_long_bf16_b16":
        return make_prefill_case(seed, num_seqs=8, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                 block_size=16, seq_lens=[32768] * 8, q_lens=[4] * 8, dtype="bf16",
                                 name=name, kv_dtype=kv_dtype)
    raise ValueError(f"unknown prefill workload {name!r}")


def make_config(cid: int, *, block_size: Optional[int] = None,
                kv_dtype: Optional[str] = None) -> Workload:
    """Build named config ``cid`` (1..5). ``block_size`` overrides config 4's b;
    ``kv_dtype="e4m3"`` gives configs 2-5 an FP8 pool of the same shape and
    lengths (tables and values are drawn afresh)."""
    rng = np.random.default_rng(1000 + cid)
    if kv_dtype is not None and cid == 1:
        raise ValueError("config 1 (head_dim 64) has no FP8 variant")
    suffix = "_e4m3" if kv_dtype == "e4m3" else ""
    if cid == 1:
        return _config1(rng)
    if cid == 2:
        lens = rng.integers(128, 2048, size=64, endpoint=True)
        return _decode_batch(rng, CONFIG_NAMES[2] + suffix, n=64, hq=32, hkv=32, d=128, b=16,
                             dtype="f16", lens=lens, partition_tokens=512, kv_dtype=kv_dtype)
    if cid == 3:
        lens = rng.integers(512, 8192, size=128, endpoint=True)
        return _decode_batch(rng, CONFIG_NAMES[3] + suffix, n=128, hq=64, hkv=8, d=128, b=16,
                             dtype="bf16", lens=lens, partition_tokens=512, kv_dtype=kv_dtype)
    if cid == 4:
        b = 32 if block_size is None else int(block_size)
        name = CONFIG_NAMES[4] + f"_b{b}" + suffix
        return _decode_batch(rng, name, n=8, hq=32, hkv=8, d=128, b=b, dtype="bf16",
                             lens=[32768] * 8, partition_tokens=512, kv_dtype=kv_dtype)
    if cid == 5:
        w = _config5(rng, kv_dtype)
        w.name += suffix
        return w
    raise ValueError(f"unknown config {cid}")
