"""Plain fp64 CPU oracle for the paged KV-cache hot path.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline / reference arm may import this module; the library never does, and
it shares no code with the CUDA path.

Each function is the plain definition of one step, written from the pages:

* slot mapping: logical block floor(t/B), offset t mod B, physical id from the
  block table ("PagedAttention: Virtual-Memory KV Cache Management, Continuous
  Batching, and PyTorch Architecture", ailinkdeeptech.com, §1 Paged Virtual
  Memory Mapping; "PagedAttention: Manage the Cache Without Moving the
  Sequence", neelmishra.github.io, §Map a ten-token sequence into pages);
* KV write: the new token's k, v go to slot len % b of the last block
  ("PagedAttention: paging the KV cache", pofe.ai, §How it works and §Minimal
  implementation);
* block copy for copy-on-write: the whole block, K and V, every layer (pofe.ai
  §Sharing and copy-on-write; ailinkdeeptech.com §4, step 2);
* decode attention: gather the sequence's K and V through its block table, then
  textbook softmax attention (pofe.ai §Minimal implementation gather; "the math
  is unchanged; only the addresses are indirect", pofe.ai §How it works;
  ailinkdeeptech.com §3 standard attention softmax(QK^T/sqrt(d_k))V). Query
  head h reads KV head h // g with g = H_q / H_kv (repeat_interleave grouping,
  ailinkdeeptech.com Step 2 and pofe.ai §Minimal implementation).
* multi-token (chunked prefill / speculative verify) attention: the i-th of a
  sequence's n new queries sits at position L - n + i, its K/V and those of
  every earlier position already in the cache (pofe.ai §How it works: prefill
  writes into the blocks, then attention reads them), and attends to tokens
  0..L - n + i only: the causal mask describes the allowed attention edges,
  the block table only where the rows are stored (neelmishra.github.io §The
  kernel must understand the mapping). Same gather and textbook softmax as
  decode, which is the case n = 1.
* the blockwise online-softmax recurrence and the partition-combine rule of
  ailinkdeeptech.com §3 (running max m, normaliser l, unnormalised o), used to
  pin the split-K reduction.
* swap for preemption: a preempted sequence's blocks are copied, every layer,
  K and V, to a pool in host memory and later back, possibly to other block
  ids (pofe.ai §When memory runs out: swapping copies the evicted blocks to
  CPU memory and back; learn.pranaymahendrakar.com §Preemption: copy blocks
  to pinned host memory and back). A copy between two pools.
* prefix-cache keys: every full block of a sequence gets a content key that
  covers the whole block-aligned prefix ending with it, so a cache hit is an
  unbroken chain of matching keys and the first differing token ends the
  chain (firehose-demo "Paged Attention"; learn.pranaymahendrakar.com
  §Prefix caching: hash each block-aligned prefix of token ids; only full
  blocks are keyed, as in ailinkdeeptech.com's allocator). Reading taken:
  key_j = SHA-256(key_{j-1} || the block's token ids as little-endian int32),
  key_{-1} = a 32-byte root (zeros by default; a different root, e.g. one per
  adapter, keeps caches apart, pofe.ai §Fine-tuned models and adapters).
* an FP8 cache: the same pool with one byte per element, which "halves the
  bytes per block; nothing else about paging changes" (pofe.ai §Fine-tuned
  models and adapters, quantised caches). The pages fix no format or scale, so
  the reading taken is the OCP E4M3 encoding (1 sign, 4 exponent bits with
  bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN, largest finite
  448) with one float scale per layer for K and one for V: a stored code c
  stands for value(c) * scale. A write stores e4m3(x / scale), the quotient
  taken in float32 and rounded to the nearest code (ties to the even code),
  magnitudes above 448 saturating to 448.

Half-precision inputs arrive as uint16 bit patterns and are widened exactly to
fp64 before any arithmetic. Parity unpinned: none (every function is checked
against the pages' worked values, closed forms, library routines or
invariants by the CPU tests).
"""
from __future__ import annotations

import hashlib
import math
from typing import Iterable, List, Optional, Sequence, Tuple

import numpy as np


# ----------------------------------------------------------------------------
# exact widening of stored values


def bits_to_f64(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 value of fp16 / bf16 bit patterns (uint16) or of E4M3 codes
    (uint8, dtype "e4m3")."""
    if dtype == "e4m3":
        return e4m3_to_f64(bits)
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


# ----------------------------------------------------------------------------
# FP8 E4M3 codes (the reading of the pages' "FP8 cache")


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    """Exact value of E4M3 codes: sign bit 7, exponent bits 6..3 (bias 7),
    mantissa bits 2..0. Exponent 0 is subnormal, m / 8 * 2^-6; otherwise
    (1 + m / 8) * 2^(e - 7); exponent 15 with mantissa 7 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


_E4M3_MAX = 448.0


def _e4m3_grid() -> np.ndarray:
    """Values of the non-negative finite codes 0x00 .. 0x7E, in code order
    (which is also increasing value order)."""
    return e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))


def f32_to_e4m3(x: np.ndarray) -> np.ndarray:
    """Encode float32 values as E4M3 codes: nearest representable value, ties
    to the even code, magnitudes beyond 448 saturate to 448, NaN gives 0x7F.
    The sign is kept, so values that round to zero give +0 or -0."""
    v = np.asarray(x, dtype=np.float32).astype(np.float64)
    grid = _e4m3_grid()
    a = np.abs(v)
    hi = np.clip(np.searchsorted(grid, a, side="left"), 1, len(grid) - 1)  # grid[hi] >= a
    lo = hi - 1
    d_lo = a - grid[lo]
    d_hi = grid[hi] - a
    code = np.where(d_lo < d_hi, lo, hi)
    code = np.where(d_lo == d_hi, np.where(lo % 2 == 0, lo, hi), code)
    code = np.where(a == 0.0, 0, code)
    code = np.where(a >= _E4M3_MAX, 0x7E, code)
    out = (np.where(np.signbit(v), 0x80, 0) | code).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7F), out).astype(np.uint8)


def quantize_e4m3(bits: np.ndarray, dtype: str, scale: float) -> np.ndarray:
    """Codes a write stores for fp16 / bf16 inputs: e4m3(x / scale), the
    quotient rounded once to float32."""
    x = bits_to_f64(bits, dtype).astype(np.float32)
    return f32_to_e4m3(x / np.float32(scale))


def write_kv_e4m3(k_cache: np.ndarray, v_cache: np.ndarray, key: np.ndarray, value: np.ndarray,
                  slots: Sequence[int], dtype: str, k_scale: float, v_scale: float
                  ) -> Tuple[np.ndarray, np.ndarray]:
    """write_kv into E4M3 caches: each token's k, v rows (fp16 / bf16 bits of
    ``dtype``) are quantised with the layer's scale, then stored at the slot."""
    return write_kv(k_cache, v_cache, quantize_e4m3(key, dtype, k_scale),
                    quantize_e4m3(value, dtype, v_scale), slots)


# ----------------------------------------------------------------------------
# slot mapping (integer)


def slot_mapping(block_tables: np.ndarray, seq_idx: Sequence[int], positions: Sequence[int],
                 block_size: int) -> np.ndarray:
    """slot = table[s][t // B] * B + t % B for every (s, t) pair.

    Logical block i = floor(t / B), offset j = t mod B, physical block B(i) from
    the sequence's table; a slot numbers rows of the pool, block-major.
    """
    out = np.empty(len(positions), dtype=np.int64)
    for n, (s, t) in enumerate(zip(seq_idx, positions)):
        i, j = int(t) // block_size, int(t) % block_size
        out[n] = int(block_tables[int(s)][i]) * block_size + j
    return out


# ----------------------------------------------------------------------------
# KV write and block copy (bytes)


def write_kv(k_cache: np.ndarray, v_cache: np.ndarray, key: np.ndarray, value: np.ndarray,
             slots: Sequence[int]) -> Tuple[np.ndarray, np.ndarray]:
    """New caches with row ``slot`` of the pool set to each token's k and v.

    Caches are ``[num_blocks, B, H_kv, D]``; slot s is block s // B, row s % B.
    A slot of -1 marks a padding token and writes nothing.
    """
    k = k_cache.copy()
    v = v_cache.copy()
    b = k.shape[1]
    for n, s in enumerate(slots):
        s = int(s)
        if s < 0:
            continue
        k[s // b, s % b] = key[n]
        v[s // b, s % b] = value[n]
    return k, v


def copy_blocks(k_caches: Sequence[np.ndarray], v_caches: Sequence[np.ndarray],
                pairs: Iterable[Tuple[int, int]]) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    """New caches where block dst holds a copy of block src, for every layer."""
    ks = [k.copy() for k in k_caches]
    vs = [v.copy() for v in v_caches]
    for src, dst in pairs:
        for k, v in zip(ks, vs):
            k[int(dst)] = k[int(src)]
            v[int(dst)] = v[int(src)]
    return ks, vs


def swap_blocks(src_k: Sequence[np.ndarray], src_v: Sequence[np.ndarray],
                dst_k: Sequence[np.ndarray], dst_v: Sequence[np.ndarray],
                pairs: Iterable[Tuple[int, int]]) -> Tuple[List[np.ndarray], List[np.ndarray]]:
    """New destination pools where, for every (src, dst) pair and every layer,
    block dst of the destination holds a copy of block src of the source (K and
    V). The source pools are not changed; the two pools may differ in size."""
    ks = [k.copy() for k in dst_k]
    vs = [v.copy() for v in dst_v]
    for src, dst in pairs:
        for layer in range(len(ks)):
            ks[layer][int(dst)] = src_k[layer][int(src)]
            vs[layer][int(dst)] = src_v[layer][int(src)]
    return ks, vs



# ----------------------------------------------------------------------------
# prefix-cache keys (bytes)


def prefix_block_keys(tokens: Sequence[int], block_size: int,
                      root: Optional[bytes] = None) -> List[bytes]:
    """Content keys of a sequence's full blocks: key_j = SHA-256(key_{j-1} ||
    int32 little-endian token ids of block j), key_{-1} = ``root`` (32 zero
    bytes by default). A trailing partial block gets no key."""
    parent = bytes(32) if root is None else bytes(root)
    assert len(parent) == 32
    keys = []
    for j in range(len(tokens) // block_size):
        block = np.asarray(tokens[j * block_size:(j + 1) * block_size], dtype="<i4")
        parent = hashlib.sha256(parent + block.tobytes()).digest()
        keys.append(parent)
    return keys

# ----------------------------------------------------------------------------
# decode attention (fp64)


def gather_kv(cache: np.ndarray, table_row: Sequence[int], length: int, kv_head: int) -> np.ndarray:
    """The first ``length`` rows of one KV head, in logical order.

    Blocks ``table_row[:ceil(length / B)]`` are gathered, flattened to token
    rows and cut at the sequence length, so slots past the length are never
    read.
    """
    b = cache.shape[1]
    nblk = -(-length // b)
    idx = np.asarray(table_row[:nblk], dtype=np.int64)
    rows = cache[idx].reshape(nblk * b, cache.shape[2], cache.shape[3])
    return rows[:length, kv_head]


def attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for query rows q [g, D] over keys K, V [L, D]."""
    x = scale * (q @ K.T)
    x = x - x.max(axis=1, keepdims=True)
    p = np.exp(x)
    p = p / p.sum(axis=1, keepdims=True)
    return p @ V


def _cache_rows(cache: np.ndarray, table_row, length: int, kv_head: int, dtype: str,
                kv_dtype: Optional[str], kv_scale: float) -> np.ndarray:
    """fp64 K or V rows of one sequence and KV head: the gathered stored values,
    times the layer's scale for an E4M3 cache."""
    rows = gather_kv(cache, table_row, length, kv_head)
    if kv_dtype == "e4m3":
        return e4m3_to_f64(rows) * float(np.float32(kv_scale))
    return bits_to_f64(rows, dtype)


def decode(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray, block_tables: np.ndarray,
           seq_lens: Sequence[int], scale: float, dtype: str,
           pairs: Optional[Sequence[Tuple[int, int]]] = None, kv_dtype: Optional[str] = None,
           k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Decode attention for every (sequence, query head), or for ``pairs`` only.

    Returns fp64 ``[N, H_q, D]``; rows not in ``pairs`` are NaN. A sequence of
    length 0 attends to nothing and yields zeros. ``dtype`` is that of q (and of
    the cache unless ``kv_dtype`` is "e4m3", whose codes stand for
    value * k_scale and value * v_scale).
    """
    n, hq, d = q.shape
    hkv = k_cache.shape[2]
    g = hq // hkv
    out = np.full((n, hq, d), np.nan)
    if pairs is None:
        want = {(s, kvh): list(range(kvh * g, (kvh + 1) * g)) for s in range(n) for kvh in range(hkv)}
    else:
        want = {}
        for s, h in pairs:
            want.setdefault((int(s), int(h) // g), []).append(int(h))
    for (s, kvh), heads in want.items():
        L = int(seq_lens[s])
        if L == 0:
            out[s, heads] = 0.0
            continue
        K = _cache_rows(k_cache, block_tables[s], L, kvh, dtype, kv_dtype, k_scale)
        V = _cache_rows(v_cache, block_tables[s], L, kvh, dtype, kv_dtype, v_scale)
        Q = bits_to_f64(q[s, heads], dtype)
        out[s, heads] = attention(Q, K, V, scale)
    return out


def prefill(q: np.ndarray, q_start: Sequence[int], k_cache: np.ndarray, v_cache: np.ndarray,
            block_tables: np.ndarray, seq_lens: Sequence[int], scale: float, dtype: str,
            rows: Optional[Sequence[Tuple[int, int]]] = None, kv_dtype: Optional[str] = None,
            k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """Causal multi-token attention over the paged cache.

    ``q`` is ``[T, H_q, D]``; sequence s owns query rows ``q_start[s] ..
    q_start[s + 1]``. With n of them and L = seq_lens[s], query i sits at
    position L - n + i and attends to the tokens at positions 0 .. L - n + i,
    read through the block table. Returns fp64 ``[T, H_q, D]``; with ``rows``
    (a list of (query row, query head)) only those are computed and the rest
    are NaN. ``kv_dtype`` and the scales are those of :func:`decode`.
    """
    t_all, hq, d = q.shape
    hkv = k_cache.shape[2]
    g = hq // hkv
    out = np.full((t_all, hq, d), np.nan)
    owner = {}
    for s in range(len(seq_lens)):
        for t in range(int(q_start[s]), int(q_start[s + 1])):
            owner[t] = s
    if rows is None:
        want = {(t, kvh): list(range(kvh * g, (kvh + 1) * g)) for t in range(t_all) for kvh in range(hkv)}
    else:
        want = {}
        for t, h in rows:
            want.setdefault((int(t), int(h) // g), []).append(int(h))
    cache = {}
    for (t, kvh), heads in sorted(want.items(), key=lambda kv: (owner[kv[0][0]], kv[0][1], kv[0][0])):
        s = owner[t]
        L = int(seq_lens[s])
        n = int(q_start[s + 1]) - int(q_start[s])
        if n > L:
            raise ValueError(f"sequence {s}: {n} queries but only {L} tokens")
        pos = L - n + (t - int(q_start[s]))
        if (s, kvh) not in cache:
            cache = {(s, kvh): (_cache_rows(k_cache, block_tables[s], L, kvh, dtype, kv_dtype, k_scale),
                                _cache_rows(v_cache, block_tables[s], L, kvh, dtype, kv_dtype, v_scale))}
        K, V = cache[(s, kvh)]
        Q = bits_to_f64(q[t, heads], dtype)
        out[t, heads] = attention(Q, K[:pos + 1], V[:pos + 1], scale)
    return out


# ----------------------------------------------------------------------------
# blockwise online softmax and the partition combine


def online_softmax_blocks(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float,
                          block_size: int) -> np.ndarray:
    """The per-block recurrence: running max m, normaliser l, accumulator o.

    For each block of B keys: S = scale q K_b^T (masked to the sequence),
    m_new = max(m, max S), P = exp(S - m_new), l = l exp(m - m_new) + sum P,
    o = o exp(m - m_new) + P V_b, m = m_new; finally O = o / l.
    """
    L = K.shape[0]
    m = -math.inf
    l = 0.0
    o = np.zeros(V.shape[1])
    for start in range(0, L, block_size):
        S = scale * (K[start:start + block_size] @ q)
        m_new = max(m, float(S.max()))
        P = np.exp(S - m_new)
        alpha = math.exp(m - m_new) if m != -math.inf else 0.0
        l = l * alpha + float(P.sum())
        o = o * alpha + P @ V[start:start + block_size]
        m = m_new
    return o / l


def partition_state(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float
                    ) -> Tuple[float, float, np.ndarray]:
    """(m, l, o) of one token range: max logit, sum of exp(S - m), unnormalised output."""
    S = scale * (K @ q)
    m = float(S.max())
    P = np.exp(S - m)
    return m, float(P.sum()), P @ V


def combine_partitions(states: Sequence[Tuple[float, float, np.ndarray]]) -> np.ndarray:
    """Merge per-range (m, l, o) states with the rescale identity.

    M = max m_p, l = sum l_p exp(m_p - M), O = sum o_p exp(m_p - M) / l.
    """
    M = max(s[0] for s in states)
    l = sum(s[1] * math.exp(s[0] - M) for s in states)
    o = sum(s[2] * math.exp(s[0] - M) for s in states)
    return o / l
