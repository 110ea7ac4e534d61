// pa_decode.cuh - paged decode attention for sm_103a.
//
// Computes, for one sequence s and one KV head, the g query heads
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[t]) V[t],   t < L_s,
// reading K[t], V[t] through the block table (logical block t / b, row t % b)
// and accumulating stage by stage with a running maximum m, normaliser l and
// unnormalised output o ("PagedAttention: Virtual-Memory KV Cache Management,
// ...", 3. Non-Contiguous Online Softmax Attention Kernel).
//
// Building blocks shared by both kernels:
//  * A stage is 16 token rows of K and of V for one KV head, loaded by TMA
//    tensor copies straight from the scattered pool blocks (box = 64 head-dim
//    elements x 1 head x up to 16 tokens x 1 block, 128-byte swizzle). Lane j
//    of the issuing warp looks up and copies the j-th block piece of the stage.
//  * Each warp owns a private ring of NS stages in shared memory and both
//    issues and consumes them, so warps never wait on one another.
//  * QK^T and PV run on mma.sync m16n8k16 with fp32 accumulation in the
//    transposed orientation S^T = K Q^T (M = 16 tokens, N = 8 query heads of
//    the group, K = head_dim) and O^T = V^T P^T (M = 16 head-dim rows, N = 8
//    heads, K = 16 tokens). The group's heads fill N, so each K/V row is read
//    once per KV head whatever g is. P^T reaches the B-operand layout with
//    movmatrix; P is split into a 16-bit high and low part so the PV product
//    keeps ~16 bits of the fp32 weights.
//  * Slots past the length, pieces of blocks whose id is out of range and the
//    padding rows of blocks smaller than 8 tokens are masked: their logits are
//    -inf and their V rows are zeroed in shared memory before PV, so stale or
//    NaN bytes in the pool never enter the result.
//
// FP8 caches (E4M3 codes, one scale per layer for K and one for V): a stage
// row is D bytes instead of 2D, so one 128-byte swizzled line holds 128 head-dim
// elements. Codes are widened exactly to fp16 in registers (two conversions
// per 32-bit word) and every MMA runs in fp16. ldmatrix treats byte pairs as
// its 16-bit elements: for S^T each lane gets four consecutive codes of a
// row, so the MMA's reduction index k maps to head-dim elements four at a
// time (q is loaded in the same order); for O^T the transposing ldmatrix
// gives each lane two dims of two tokens, which a byte permute turns into
// (token, token+1) pairs per dim, the two dims landing in rows gid and gid+8
// of the tile (acc_dim gives each accumulator's dim). bf16 queries become fp16 times a per-head
// power of two that keeps the row's largest element below 2^14; the logit
// scale of each head column undoes it. k_scale folds into the logit scale,
// v_scale multiplies the output.
//
// decode_kernel: one CTA per (sequence, KV head, partition); its 4 warps take
// the partition's stages round-robin and merge through shared memory at the
// end; the CTA writes the output (one partition) or (m, l, o) partials that
// decode_reduce_kernel merges.
//
// decode_balanced_kernel: a persistent grid. The 16-token stages of all
// sequences are cut into equal contiguous ranges, one per group of H_kv warps
// (one warp per KV head), so every warp streams the same number of stages
// whatever the lengths, and a group reads whole pool blocks together. A warp
// writes each (sequence, KV head) piece it covers whole straight to the
// output; a piece cut across ranges leaves one (m, l, o) partial per warp, and
// the last warp to finish it (an atomicInc counter) merges them in order.
#pragma once

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

// Element layout of a cache: 16-bit values or 8-bit E4M3 codes. A "piece" is
// the run of head-dim elements in one 128-byte line (one TMA box column).
template <bool FP8>
struct KvLayout {
  static constexpr int kBytes = FP8 ? 1 : 2;
  static constexpr int kPieceElems = 128 / kBytes;
};

// Head-dim index of accumulator element r of O^T tile dm held by lane group
// gid (rows gid and gid + 8 of the m16 tile).
template <bool FP8>
__device__ __forceinline__ int acc_dim(int dm, int gid, int r) {
  if constexpr (FP8) return dm * 16 + (gid << 1) + (r >> 1);
  return dm * 16 + gid + ((r >> 1) << 3);
}

// Sequence length after range checks; out-of-range lengths are clamped and
// reported once.
__device__ __forceinline__ int decode_seq_len(const DecodeArgs& a, int s, bool report) {
  const int raw = a.seq_lens[s];
  const int64_t table_cap = static_cast<int64_t>(a.max_blocks) * a.block_size;
  const int cap = static_cast<int>(table_cap < a.max_seq_len ? table_cap : a.max_seq_len);
  if (raw < 0 || raw > cap) {
    if (report) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    return raw < 0 ? 0 : cap;
  }
  return raw;
}

// Tokens a sequence puts on the balanced kernels' stage line. Decode: its
// checked length. Multi-token rows (MULTI): L_s when the sequence has new
// rows that can be placed; 0 when it has none, and 0, flagged, when n_s > L_s
// or L_s exceeds its block table. n_s > max_q is flagged too; the rows past
// max_q are then skipped, the others computed.
template <bool MULTI>
__device__ __forceinline__ int line_len(const DecodeArgs& a, int s, bool report) {
  if constexpr (!MULTI) {
    return decode_seq_len(a, s, report);
  } else {
    const int n = __ldg(a.q_start + s + 1) - __ldg(a.q_start + s);
    const int L = __ldg(a.seq_lens + s);
    if (n <= 0) return 0;
    if (n > L || static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks) * a.block_size) {
      if (report) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
      return 0;
    }
    if (n > a.max_q && report) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    return L;
  }
}

__device__ __forceinline__ void store_out(const DecodeArgs& a, int64_t idx, float v) {
  if (a.out_dtype == PA_F32) {
    static_cast<float*>(a.out)[idx] = v;
  } else if (a.out_dtype == PA_BF16) {
    static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(a.out)[idx] = __float2half_rn(v);
  }
}

// ---------------------------------------------------------------- warp merges

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// E consecutive floats through L2 (bypassing L1, which is not coherent with
// other SMs' writes), E = 2, 4 or 8 with matching alignment.
template <int E>
__device__ __forceinline__ void ldcg_vec(const float* p, float (&v)[E]) {
  if constexpr (E == 2) {
    const float2 t = __ldcg(reinterpret_cast<const float2*>(p));
    v[0] = t.x; v[1] = t.y;
  } else {
#pragma unroll
    for (int i = 0; i < E; i += 4) {
      const float4 t = __ldcg(reinterpret_cast<const float4*>(p + i));
      v[i] = t.x; v[i + 1] = t.y; v[i + 2] = t.z; v[i + 3] = t.w;
    }
  }
}

// Merges the (m, l, o) partials of `ncols` output rows with the rescale
// identity M = max m_c, l = sum l_c 2^(m_c - M), out = sum o_c 2^(m_c - M) / l,
// in contributor order. slot(c) gives contributor c's partial index, or -1 for
// a contributor that holds none. For partial i and row j, (m, l) sit at
// ml[i * ml_stride + j * ml_col] (+1) and the output at o[i * o_stride +
// j * o_col .. + D); row j is written to out row out_row0 + j. Rows go four at
// a time: lanes scan 32 contributors for the maxima and normalisers of all
// four, then each lane accumulates D/32 consecutive outputs of the four rows
// with unrolled vector loads, so a merge costs a few rounds of L2 latency.
template <int D, typename SlotFn>
__device__ __forceinline__ void merge_rows(const DecodeArgs& a, int n, SlotFn slot, int ncols,
                                           const float* ml, int64_t ml_stride, int64_t ml_col,
                                           const float* o, int64_t o_stride, int64_t o_col,
                                           int64_t out_row0, int lane) {
  constexpr int E = D / 32;
  constexpr int CC = 4;
  for (int j0 = 0; j0 < ncols; j0 += CC) {
    float mmax[CC];
    float lsum[CC];
    float acc[CC][E];
#pragma unroll
    for (int j = 0; j < CC; ++j) {
      mmax[j] = -INFINITY;
      lsum[j] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[j][e] = 0.f;
    }
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int sid = c0 + lane < n ? slot(c0 + lane) : -1;
#pragma unroll
      for (int j = 0; j < CC; ++j) {
        const bool live = sid >= 0 && j0 + j < ncols;
        mmax[j] = fmaxf(mmax[j], warp_max(live ? __ldcg(ml + sid * ml_stride + (j0 + j) * ml_col)
                                              : -INFINITY));
      }
    }
    for (int c0 = 0; c0 < n; c0 += 32) {
      const int sid = c0 + lane < n ? slot(c0 + lane) : -1;
      float f[CC];
#pragma unroll
      for (int j = 0; j < CC; ++j) {
        const bool live = sid >= 0 && j0 + j < ncols && mmax[j] != -INFINITY;
        const float* p = ml + (live ? sid * ml_stride + (j0 + j) * ml_col : 0);
        f[j] = live ? exp2f(__ldcg(p) - mmax[j]) : 0.f;
        lsum[j] += warp_sum(live ? __ldcg(p + 1) * f[j] : 0.f);
      }
      const int nch = n - c0 < 32 ? n - c0 : 32;
      // Branch-free so the unrolled loads of several partials are in flight
      // together (eight contributors' rows per round: a merge is a few L2
      // round trips even while other SMs stream): a contributor or row without
      // a partial reads partial 0 of row 0 (always in bounds) and its weight 0
      // selects the value away.
#pragma unroll 8
      for (int c = 0; c < nch; ++c) {
        const int sc = __shfl_sync(0xffffffffu, sid, c);
#pragma unroll
        for (int j = 0; j < CC; ++j) {
          const float fc = __shfl_sync(0xffffffffu, f[j], c);
          const bool use = sc >= 0 && j0 + j < ncols;
          float v[E];
          ldcg_vec<E>(o + (use ? sc * o_stride + (j0 + j) * o_col : 0) + lane * E, v);
#pragma unroll
          for (int e = 0; e < E; ++e) acc[j][e] += fc != 0.f ? v[e] * fc : 0.f;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < CC; ++j) {
      if (j0 + j >= ncols) break;
#pragma unroll
      for (int e = 0; e < E; ++e)
        store_out(a, (out_row0 + j0 + j) * D + lane * E + e, lsum[j] > 0.f ? acc[j][e] / lsum[j] : 0.f);
    }
  }
}

template <int D, int NT, int NS, bool FP8>
struct DecodeSmem {
  static constexpr int kHalves = D / KvLayout<FP8>::kPieceElems;  // 128-byte column pieces of a row
  static constexpr int kHalfBytes = kStageRows * 128;     // one piece of 16 rows
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;  // K then V
  static constexpr int kRingBytes = kDecodeWarps * NS * kStageBytes;
  static constexpr int kCombineBytes = kDecodeWarps * NT * 8 * (D + 2) * 4;
  static constexpr int kDataBytes = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
  static constexpr int kBarOffset = kDataBytes;
  static constexpr int kMaskOffset = kBarOffset + kDecodeWarps * NS * 8;
  static constexpr int kPrefixOffset = kMaskOffset + kDecodeWarps * NS * 4;  // balanced kernel
  static constexpr int kTotal = kPrefixOffset + 1024;  // + base-alignment slack
};

// Logit multipliers of the S^T tile's columns, in log2 units: the scalar
// scale * log2(e) for 16-bit caches; per query head for E4M3 caches, whose
// fp16 copy of a bf16 query carries a per-head power of two (see load_q).
template <int NT, bool PER_HEAD>
struct LogitScale {
  float s[PER_HEAD ? NT : 1][PER_HEAD ? 2 : 1];
  __device__ __forceinline__ float operator()(int nt, int c) const {
    if constexpr (PER_HEAD) return s[nt][c];
    return s[0][0];
  }
};

// Per-warp online-softmax state for NT tiles of 8 query heads.
template <int D, int NT>
struct Acc {
  float m[NT][2];
  float l[NT][2];
  float o[D / 16][NT][4];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m[nt][0] = m[nt][1] = -INFINITY;
      l[nt][0] = l[nt][1] = 0.f;
#pragma unroll
      for (int dm = 0; dm < D / 16; ++dm) o[dm][nt][0] = o[dm][nt][1] = o[dm][nt][2] = o[dm][nt][3] = 0.f;
    }
  }
  // Sums the normaliser over the 8 lanes that share each head column.
  __device__ __forceinline__ void reduce_l() {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v = l[nt][c];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        l[nt][c] = v;
      }
    }
  }
};

// q rows as the B operand of S^T = K Q^T (k = head-dim index, n = column of
// the tile): column gid of n-tile nt holds q row qrow(nt) (in rows of D
// elements), or zeros when that is negative; plus the column logit scales.
// For FP8 caches, lane quad t takes dims 16kk + 4t .. + 3 of k-step kk, the
// order in which compute_stage reads the codes, and a bf16 query row is
// stored as fp16 times 2^(13 - e), e the exponent of its largest magnitude
// (exact for every element at or above 2^-14 of that scale; the column's
// logit scale carries 2^(e - 13)).
template <bool IS_BF16, int D, int NT, bool FP8, class RowFn>
__device__ __forceinline__ void load_q_rows(const DecodeArgs& a, RowFn qrow, int lane,
                                            uint32_t (&qb)[NT][D / 16][2],
                                            LogitScale<NT, FP8>& ls) {
  const int tig = lane & 3;
  const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int64_t qr = qrow(nt);
    const bool live = qr >= 0;
    const int64_t row = (live ? qr : 0) * D;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int64_t d0 = FP8 ? kk * 16 + tig * 4 : kk * 16 + tig * 2;
      const int64_t d1 = FP8 ? d0 + 2 : d0 + 8;
      qb[nt][kk][0] = live ? __ldg(q32 + ((row + d0) >> 1)) : 0u;
      qb[nt][kk][1] = live ? __ldg(q32 + ((row + d1) >> 1)) : 0u;
    }
    if constexpr (FP8 && IS_BF16) {
      float m = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 f = unpack2<true>(qb[nt][kk][i]);
          m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        }
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
      const int e = max(static_cast<int>((__float_as_uint(m) >> 23) & 0xFFu) - 127, -100);
      const float p = __uint_as_float(static_cast<uint32_t>(127 + 13 - e) << 23);    // 2^(13-e)
      const float inv = __uint_as_float(static_cast<uint32_t>(127 - 13 + e) << 23);  // 2^(e-13)
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const float2 f = unpack2<true>(qb[nt][kk][i]);
          qb[nt][kk][i] = pack2<false>(f.x * p, f.y * p);
        }
      }
      ls.s[nt][0] = a.scale_log2 * __shfl_sync(0xffffffffu, inv, tig * 8);
      ls.s[nt][1] = a.scale_log2 * __shfl_sync(0xffffffffu, inv, tig * 8 + 4);
    } else if constexpr (FP8) {
      ls.s[nt][0] = ls.s[nt][1] = a.scale_log2;
    }
  }
  if constexpr (!FP8) ls.s[0][0] = a.scale_log2;
}

// q of the g heads of KV head kvh for sequence s (one decode query); heads
// past g are zero columns.
template <bool IS_BF16, int D, int NT, bool FP8>
__device__ __forceinline__ void load_q(const DecodeArgs& a, int s, int kvh, int lane,
                                       uint32_t (&qb)[NT][D / 16][2], LogitScale<NT, FP8>& ls) {
  const int gid = lane >> 2;
  const int64_t row0 = static_cast<int64_t>(s) * a.num_q_heads + static_cast<int64_t>(kvh) * a.group;
  load_q_rows<IS_BF16, D, NT, FP8>(
      a, [&](int nt) -> int64_t { return nt * 8 + gid < a.group ? row0 + nt * 8 + gid : -1; }, lane,
      qb, ls);
}

// Pulls the q rows that load_q(s, kvh) will read (g contiguous rows of D
// 16-bit elements) into L1 ahead of time, one 128-byte line per lane. The
// streamed pool evicts q from L2, so without this a warp that starts a new
// piece waits a DRAM round trip for its q.
// prefetch_q_group takes the g rows that start at q row `row`.
template <int D>
__device__ __forceinline__ void prefetch_q_group(const DecodeArgs& a, int64_t row, int lane) {
  const char* base = static_cast<const char*>(a.q) + row * D * 2;
  const int lines = (a.group * D * 2 + 127) / 128;
  for (int i = lane; i < lines; i += 32)
    asm volatile("prefetch.global.L1 [%0];" ::"l"(base + static_cast<int64_t>(i) * 128));
}

template <int D>
__device__ __forceinline__ void prefetch_q(const DecodeArgs& a, int s, int kvh, int lane) {
  prefetch_q_group<D>(
      a, static_cast<int64_t>(s) * a.num_q_heads + static_cast<int64_t>(kvh) * a.group, lane);
}

// Issues the TMA copies of one stage - tokens [t0, t0 + tt) of the sequence
// whose table row starts at `table_row`, KV head kvh, clipped at tok_end -
// into the stage at shared address `stage`, completing on mbarrier `bar`.
// Stores the stage's valid-row mask (bit r = row r holds a token < tok_end of
// a block with a valid id) to *mask. Called by the whole warp.
template <int D, bool FP8>
__device__ __forceinline__ void issue_stage(const DecodeArgs& a, const CUtensorMap* tmk,
                                            const CUtensorMap* tmv, int64_t table_row, int kvh,
                                            int t0, int tok_end, uint32_t stage, uint32_t bar,
                                            uint32_t* mask, int lane) {
  constexpr int PE = KvLayout<FP8>::kPieceElems;
  constexpr int HALVES = D / PE;
  constexpr int HB = kStageRows * 128;
  int blk = 0;
  int off = 0;
  bool ok = false;
  if (lane < a.ops_per_stage) {
    const int t = t0 + lane * a.tok_per_op;
    if (t < tok_end) {
      const int j = t / a.block_size;
      off = t - j * a.block_size;
      blk = __ldg(a.block_tables + table_row + j);
      ok = blk >= 0 && blk < a.num_blocks;
      if (!ok) atomicOr(a.err, PA_DEVERR_BLOCK_ID);
    }
  }
  const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
  bool rv = false;
  if (lane < kStageRows) {
    const int jr = lane / a.slot_rows;
    const int o = lane - jr * a.slot_rows;
    const int tok = t0 + jr * a.tok_per_op + o;
    rv = o < a.tok_per_op && tok < tok_end && ((okmask >> jr) & 1u);
  }
  const uint32_t rowmask = __ballot_sync(0xffffffffu, rv) & ((1u << kStageRows) - 1u);
  if (lane == 0) {
    *mask = rowmask;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(okmask)) * a.tok_per_op * D * 2u *
                                   KvLayout<FP8>::kBytes);
  }
  __syncwarp();
  if (ok) {
    const uint32_t dk = stage + lane * a.slot_rows * 128;
    const uint32_t dv = dk + HALVES * HB;
#pragma unroll
    for (int c = 0; c < HALVES; ++c) {
      tma_load_4d(dk + c * HB, tmk, bar, c * PE, kvh, off, blk);
      tma_load_4d(dv + c * HB, tmv, bar, c * PE, kvh, off, blk);
    }
  }
}

// Where one KV head's rows of a loaded stage sit in shared memory. Views
// give the shared addresses of K and V (column half 0), the bytes between
// 64-element column halves, and the offset of row r. Rows sit in groups of
// 8 or 16 contiguous 128-byte lines, each group starting on a 1024-byte
// boundary, so the 128-byte swizzle of row r is r & 7. The layout constants
// are compile-time so the compiler schedules ldmatrix/mma freely.

// Per-warp stage: 16 consecutive lines, halves kStageRows * 128 bytes apart.
struct WarpView {
  uint32_t k, v;
  static constexpr uint32_t half_stride = kStageRows * 128u;
  __device__ __forceinline__ uint32_t row(int r) const { return static_cast<uint32_t>(r) * 128u; }
};

__device__ __forceinline__ WarpView warp_stage_view(uint32_t stage, int halves) {
  return WarpView{stage, stage + halves * WarpView::half_stride};
}

// Head-grouped stage of ST token rows (box of 64 x TPO tokens x HG heads per
// column half): per token group, HG heads of TPO lines each; this head's lines
// at head_off.
template <int HG, int TPO, int ST = kStageRows>
struct GroupView {
  uint32_t k, v, head_off;
  static constexpr uint32_t half_stride = HG * ST * 128u;
  static constexpr uint32_t op_stride = HG * TPO * 128u;
  __device__ __forceinline__ uint32_t row(int r) const {
    return static_cast<uint32_t>(r / TPO) * op_stride + head_off + static_cast<uint32_t>(r % TPO) * 128u;
  }
};

// Causal limits of the S^T tile's columns. Decode: every valid token row of
// a stage is admitted. Multi-token rows (ColLimit): this lane's column c of
// n-tile nt (tile column 2 * tig + c) admits the stage's token rows
// 0 .. rel[nt][c] only.
struct NoColLimit {
  __device__ __forceinline__ bool ok(int, int, int) const { return true; }
};

template <int NT>
struct ColLimit {
  int rel[NT][2];
  __device__ __forceinline__ bool ok(int nt, int c, int row) const { return row <= rel[nt][c]; }
};

// Folds one loaded stage into the warp's softmax state. `sv` (a WarpView or
// GroupView) places the warp's rows; `smem_base` / `smem_base_ptr` are one shared address and its
// generic pointer, used to zero masked V rows; `lim` masks (token, column)
// pairs past a column's causal limit. LAZY raises the running maximum only
// when a logit exceeds it by more than 8 (E4M3 caches always); VOTE (with
// LAZY) first asks the warp whether any logit does, and reduces the column
// maxima only then; QK2 splits the 16-bit S^T product into two independent
// MMA chains (even and odd k-steps).
template <bool IS_BF16, int D, int NT, bool SPLIT_P, bool FP8, class View, class Lim = NoColLimit,
          bool LAZY = FP8, bool QK2 = false, bool VOTE = false>
__device__ __forceinline__ void compute_stage(const View sv, uint32_t smem_base,
                                              uint8_t* smem_base_ptr, uint32_t rowmask,
                                              const uint32_t (&qb)[NT][D / 16][2],
                                              Acc<D, NT>& acc, const LogitScale<NT, FP8>& ls,
                                              int lane, const Lim& lim = Lim()) {
  constexpr bool MB = IS_BF16 && !FP8;  // MMA operand type: E4M3 caches run in fp16
  constexpr int TS = kStageRows;
  constexpr int KD = D / 16;
  constexpr int HALVES = D / KvLayout<FP8>::kPieceElems;
  const int gid = lane >> 2;

  if (rowmask != (1u << TS) - 1u) {  // zero V rows that must not contribute
    for (int idx = lane; idx < TS * HALVES * 8; idx += 32) {
      const int row = idx / (HALVES * 8);
      const int rem = idx - row * (HALVES * 8);
      if (!((rowmask >> row) & 1u)) {
        const uint32_t a = sv.v + (rem >> 3) * View::half_stride + sv.row(row) + (rem & 7) * 16;
        *reinterpret_cast<uint4*>(smem_base_ptr + (a - smem_base)) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    __syncwarp();
  }

  // S^T = K Q^T over head_dim.
  float sacc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
  if constexpr (FP8) {
    // ldmatrix over byte-pair rows: matrix j holds rows 8(j & 1) .. + 7 of
    // 16-byte chunk kk + (j >> 1), and lane (gid, tig) receives bytes 4tig ..
    // 4tig + 3 of its row: dims 16kk + 4tig .. + 3, the order load_q uses. Even
    // and odd k-steps accumulate separately, two independent MMA chains.
    const int i = lane >> 3;
    const int row = ((i & 1) << 3) + (lane & 7);
    float sodd[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sodd[nt][0] = sodd[nt][1] = sodd[nt][2] = sodd[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KD; kk += 2) {
      const int chunk = (kk & 7) + (i >> 1);
      uint32_t w[4];
      ldsm_x4(sv.k + (kk >> 3) * View::half_stride + sv.row(row) + ((chunk ^ (row & 7)) << 4), w);
      uint32_t a0[4];
      uint32_t a1[4];
      e4m3x4_to_f16(w[0], a0[0], a0[2]);
      e4m3x4_to_f16(w[1], a0[1], a0[3]);
      e4m3x4_to_f16(w[2], a1[0], a1[2]);
      e4m3x4_to_f16(w[3], a1[1], a1[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816<MB>(sacc[nt], a0, qb[nt][kk][0], qb[nt][kk][1]);
        mma16816<MB>(sodd[nt], a1, qb[nt][kk + 1][0], qb[nt][kk + 1][1]);
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) sacc[nt][r] += sodd[nt][r];
    }
  } else if constexpr (QK2) {
    const int i = lane >> 3;
    const int row = ((i & 1) << 3) + (lane & 7);
    float sodd[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sodd[nt][0] = sodd[nt][1] = sodd[nt][2] = sodd[nt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KD; ++kk) {
      const int chunk = ((kk & 3) << 1) + (i >> 1);
      uint32_t af[4];
      ldsm_x4(sv.k + (kk >> 2) * View::half_stride + sv.row(row) + ((chunk ^ (row & 7)) << 4), af);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
        mma16816<MB>((kk & 1) ? sodd[nt] : sacc[nt], af, qb[nt][kk][0], qb[nt][kk][1]);
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) sacc[nt][r] += sodd[nt][r];
    }
  } else {
    const int i = lane >> 3;
    const int row = ((i & 1) << 3) + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < KD; ++kk) {
      const int chunk = ((kk & 3) << 1) + (i >> 1);
      uint32_t af[4];
      ldsm_x4(sv.k + (kk >> 2) * View::half_stride + sv.row(row) + ((chunk ^ (row & 7)) << 4), af);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) mma16816<MB>(sacc[nt], af, qb[nt][kk][0], qb[nt][kk][1]);
    }
  }

  // Online softmax update (log2 domain). LAZY (E4M3 caches, multi-token
  // rows): the running maximum is raised only when a logit exceeds it by more
  // than 8 (a factor of 2^8), so most stages keep it and skip rescaling the
  // output; p then stays below 2^8, and o / l is unchanged.
  const bool v0 = (rowmask >> gid) & 1u;
  const bool v1 = (rowmask >> (gid + 8)) & 1u;
  float p[NT][4];
  float lazy_alpha[NT][2];
  bool grew = false;
  bool quiet = false;  // VOTE: no logit of the stage passes its column's maximum + 8
  if constexpr (VOTE) {
    static_assert(LAZY, "the vote decides the lazy maximum");
    float x[NT][4];
    bool need = false;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      x[nt][0] = v0 && lim.ok(nt, 0, gid) ? sacc[nt][0] * ls(nt, 0) : -INFINITY;
      x[nt][1] = v0 && lim.ok(nt, 1, gid) ? sacc[nt][1] * ls(nt, 1) : -INFINITY;
      x[nt][2] = v1 && lim.ok(nt, 0, gid + 8) ? sacc[nt][2] * ls(nt, 0) : -INFINITY;
      x[nt][3] = v1 && lim.ok(nt, 1, gid + 8) ? sacc[nt][3] * ls(nt, 1) : -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c)
        need |= fmaxf(x[nt][c], x[nt][c + 2]) > acc.m[nt][c] + 8.f;
    }
    quiet = !__any_sync(0xffffffffu, need);
    if (quiet) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const float m_use = acc.m[nt][c] == -INFINITY ? 0.f : acc.m[nt][c];
          p[nt][c] = exp2f(x[nt][c] - m_use);
          p[nt][c + 2] = exp2f(x[nt][c + 2] - m_use);
          acc.l[nt][c] += p[nt][c] + p[nt][c + 2];
        }
      }
    }
  }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if (quiet) break;
    float x[4];
    x[0] = v0 && lim.ok(nt, 0, gid) ? sacc[nt][0] * ls(nt, 0) : -INFINITY;
    x[1] = v0 && lim.ok(nt, 1, gid) ? sacc[nt][1] * ls(nt, 1) : -INFINITY;
    x[2] = v1 && lim.ok(nt, 0, gid + 8) ? sacc[nt][2] * ls(nt, 0) : -INFINITY;
    x[3] = v1 && lim.ok(nt, 1, gid + 8) ? sacc[nt][3] * ls(nt, 1) : -INFINITY;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float mx = fmaxf(x[c], x[c + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      if constexpr (LAZY) {
        const bool grow = mx > acc.m[nt][c] + 8.f;
        const float m_new = grow ? mx : acc.m[nt][c];
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = grow ? exp2f(acc.m[nt][c] - m_use) : 1.f;
        acc.m[nt][c] = m_new;
        p[nt][c] = exp2f(x[c] - m_use);
        p[nt][c + 2] = exp2f(x[c + 2] - m_use);
        acc.l[nt][c] = acc.l[nt][c] * alpha + p[nt][c] + p[nt][c + 2];
        lazy_alpha[nt][c] = alpha;
        grew |= grow;
        continue;
      }
      const float m_new = fmaxf(acc.m[nt][c], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = exp2f(acc.m[nt][c] - m_use);
      acc.m[nt][c] = m_new;
      p[nt][c] = exp2f(x[c] - m_use);
      p[nt][c + 2] = exp2f(x[c + 2] - m_use);
      acc.l[nt][c] = acc.l[nt][c] * alpha + p[nt][c] + p[nt][c + 2];
#pragma unroll
      for (int dm = 0; dm < KD; ++dm) {
        acc.o[dm][nt][c] *= alpha;
        acc.o[dm][nt][c + 2] *= alpha;
      }
    }
  }
  if constexpr (LAZY) {
    if (__any_sync(0xffffffffu, grew)) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int dm = 0; dm < KD; ++dm) {
          acc.o[dm][nt][0] *= lazy_alpha[nt][0];
          acc.o[dm][nt][1] *= lazy_alpha[nt][1];
          acc.o[dm][nt][2] *= lazy_alpha[nt][0];
          acc.o[dm][nt][3] *= lazy_alpha[nt][1];
        }
      }
    }
  }

  // P^T as the B operand (k = token, n = head): transpose the 8x8 halves.
  uint32_t bh[NT][2];
  uint32_t bl[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t h01 = pack2<MB>(p[nt][0], p[nt][1]);
    const uint32_t h23 = pack2<MB>(p[nt][2], p[nt][3]);
    bh[nt][0] = movmatrix_trans(h01);
    bh[nt][1] = movmatrix_trans(h23);
    if constexpr (SPLIT_P) {
      const float2 f01 = unpack2<MB>(h01);
      const float2 f23 = unpack2<MB>(h23);
      bl[nt][0] = movmatrix_trans(pack2<MB>(p[nt][0] - f01.x, p[nt][1] - f01.y));
      bl[nt][1] = movmatrix_trans(pack2<MB>(p[nt][2] - f23.x, p[nt][3] - f23.y));
    }
  }

  // O^T += V^T P^T over the 16 tokens of the stage.
  if constexpr (FP8) {
    // ldmatrix.trans over byte-pair rows: matrix j holds tokens 8(j & 1) .. + 7
    // of 16-byte chunk c + (j >> 1), and lane (gid, tig) receives dims 16c +
    // 2gid, + 1 of tokens 2tig and 2tig + 1. A byte permute pairs the two
    // tokens per dim: tile c of O^T holds dim 16c + 2gid in row gid and
    // 16c + 2gid + 1 in row gid + 8 (acc_dim).
    const int i = lane >> 3;
    const int row = ((i & 1) << 3) + (lane & 7);
#pragma unroll
    for (int dm = 0; dm < KD; dm += 2) {
      const int chunk = (dm & 7) + (i >> 1);
      uint32_t x[4];
      ldsm_x4_trans(sv.v + (dm >> 3) * View::half_stride + sv.row(row) + ((chunk ^ (row & 7)) << 4),
                    x);
      uint32_t fa[4];
      uint32_t fb[4];
      e4m3x4_to_f16(prmt(x[0], x[0], 0x3120u), fa[0], fa[1]);
      e4m3x4_to_f16(prmt(x[1], x[1], 0x3120u), fa[2], fa[3]);
      e4m3x4_to_f16(prmt(x[2], x[2], 0x3120u), fb[0], fb[1]);
      e4m3x4_to_f16(prmt(x[3], x[3], 0x3120u), fb[2], fb[3]);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816<MB>(acc.o[dm][nt], fa, bh[nt][0], bh[nt][1]);
        mma16816<MB>(acc.o[dm + 1][nt], fb, bh[nt][0], bh[nt][1]);
        if constexpr (SPLIT_P) {
          mma16816<MB>(acc.o[dm][nt], fa, bl[nt][0], bl[nt][1]);
          mma16816<MB>(acc.o[dm + 1][nt], fb, bl[nt][0], bl[nt][1]);
        }
      }
    }
  } else {
    const int i = lane >> 3;
    const int row = ((i >> 1) << 3) + (lane & 7);
#pragma unroll
    for (int dm = 0; dm < KD; ++dm) {
      const int chunk = ((dm & 3) << 1) + (i & 1);
      uint32_t af[4];
      ldsm_x4_trans(sv.v + (dm >> 2) * View::half_stride + sv.row(row) + ((chunk ^ (row & 7)) << 4),
                    af);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        mma16816<MB>(acc.o[dm][nt], af, bh[nt][0], bh[nt][1]);
        if constexpr (SPLIT_P) mma16816<MB>(acc.o[dm][nt], af, bl[nt][0], bl[nt][1]);
      }
    }
  }
}

// ============================================================================
// One CTA per (sequence, KV head, partition).

template <bool IS_BF16, int D, int NT, int NS, bool SPLIT_P, bool FP8>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  using S = DecodeSmem<D, NT, NS, FP8>;
  constexpr int W = kDecodeWarps;
  constexpr int KD = D / 16;
  extern __shared__ __align__(16) uint8_t smem_raw[];

  const int kvh = blockIdx.x;
  const int part = blockIdx.y;
  const int s = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tig = lane & 3;

  const int L = decode_seq_len(a, s, kvh == 0 && part == 0 && threadIdx.x == 0);
  const int PT = a.part_tokens > 0 ? a.part_tokens : (L > 0 ? L : 1);
  const int tok_begin = part * PT;
  if (part > 0 && tok_begin >= L) return;  // uniform across the CTA
  const int tok_end = min(L, tok_begin + PT);
  const int ntok = max(tok_end - tok_begin, 0);
  const bool direct = (a.part_tokens == 0) || (L <= PT);

  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sm_base = smem_u32(sm);
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + S::kMaskOffset) + warp * NS;

  const int tt = a.ops_per_stage * a.tok_per_op;  // tokens per stage
  const int nst = (ntok + tt - 1) / tt;
  const int my_n = nst > warp ? (nst - warp - 1) / W + 1 : 0;

  uint32_t qb[NT][KD][2];
  LogitScale<NT, FP8> ls;
  load_q<IS_BF16, D, NT, FP8>(a, s, kvh, lane, qb, ls);

  const uint32_t bar0 = sm_base + S::kBarOffset + warp * NS * 8;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();

  const uint32_t ring = sm_base + warp * NS * S::kStageBytes;
  uint8_t* const ring_ptr = sm + warp * NS * S::kStageBytes;
  const int64_t table_row = static_cast<int64_t>(s) * a.max_blocks;
  int n_issued = 0;  // stages 0 .. n_issued - 1 have their copies issued
  auto issue = [&](int it) {
    if (a.test_stop_stage >= 0 && it >= a.test_stop_stage) return;
    const int slot = it % NS;
    issue_stage<D, FP8>(a, &tmk, &tmv, table_row, kvh, tok_begin + (warp + it * W) * tt, tok_end,
                        ring + slot * S::kStageBytes, bar0 + 8 * slot, masks + slot, lane);
    n_issued = it + 1;
  };
  const uint64_t wait_ns = PA_STAGE_WAIT_NS(a, kWaitLimitNs);

  Acc<D, NT> acc;
  acc.reset();
  const int pro = my_n < NS ? my_n : NS;
  for (int i = 0; i < pro; ++i) issue(i);

  bool aborted = false;
  int it = 0;
  for (; it < my_n; ++it) {
    const int slot = it % NS;
    const bool got = mbar_wait_bounded(bar0 + 8 * slot, (it / NS) & 1, wait_ns);
    if (__any_sync(0xffffffffu, !got)) {
      aborted = true;
      break;
    }
    compute_stage<IS_BF16, D, NT, SPLIT_P, FP8>(
        warp_stage_view(ring + slot * S::kStageBytes, S::kHalves), ring + slot * S::kStageBytes,
        ring_ptr + slot * S::kStageBytes, masks[slot], qb, acc, ls, lane);
    fence_proxy_async_smem();  // our generic reads/writes of this slot precede the next TMA into it
    __syncwarp();
    if (it + NS < my_n) issue(it + NS);
  }

  if (aborted) {
    if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    // copies this warp issued and has not consumed complete before it moves on
    for (int j = it; j < n_issued; ++j) mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, kWaitLimitNs);
    acc.reset();
  }
  acc.reduce_l();

  // Merge the warps' states through shared memory (the rings are free now).
  __syncthreads();
  constexpr int COLS = NT * 8;
  float* c_o = reinterpret_cast<float*>(sm);  // [W][COLS][D]
  float* c_m = c_o + W * COLS * D;            // [W][COLS]
  float* c_l = c_m + W * COLS;                // [W][COLS]
#pragma unroll
  for (int dm = 0; dm < KD; ++dm) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = acc_dim<FP8>(dm, gid, r);
        const int col = nt * 8 + tig * 2 + (r & 1);
        c_o[(warp * COLS + col) * D + d] = FP8 ? acc.o[dm][nt][r] * a.v_scale : acc.o[dm][nt][r];
      }
    }
  }
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = nt * 8 + tig * 2 + c;
        c_m[warp * COLS + col] = acc.m[nt][c];
        c_l[warp * COLS + col] = acc.l[nt][c];
      }
    }
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < a.group * D; idx += W * 32) {
    const int col = idx / D;
    const int d = idx - col * D;
    float mmax = -INFINITY;
#pragma unroll
    for (int w = 0; w < W; ++w) mmax = fmaxf(mmax, c_m[w * COLS + col]);
    float o = 0.f;
    float lsum = 0.f;
    if (mmax != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = exp2f(c_m[w * COLS + col] - mmax);
        o += c_o[(w * COLS + col) * D + d] * f;
        lsum += c_l[w * COLS + col] * f;
      }
    }
    const int64_t head = static_cast<int64_t>(kvh) * a.group + col;
    const int64_t sh = static_cast<int64_t>(s) * a.num_q_heads + head;
    if (direct) {
      store_out(a, sh * D + d, lsum > 0.f ? o / lsum : 0.f);
    } else {
      const int64_t pidx = sh * a.max_parts + part;
      a.part_o[pidx * D + d] = o;
      if (d == 0) {
        a.part_ml[pidx * 2] = mmax;
        a.part_ml[pidx * 2 + 1] = lsum;
      }
    }
  }
}

// ============================================================================
// Balanced: persistent warps, equal stage ranges per group of H_kv warps.
//
// The 16-token stages of all sequences, in sequence order, form one line of
// S "head-stages" (pre[s] = stages before sequence s). The line is cut into
// G = floor(warps / H_kv) equal ranges; warp grp*H_kv + h streams KV head h of
// range grp. The H_kv warps of a range read the same token rows of every
// head at the same time, so each pool block is consumed whole, as in the
// per-partition grid, while every warp gets the same amount of work.

// Position of one warp's stream on the line: sequence s, stage j of it.
struct Cursor {
  int s;     // sequence
  int j;     // stage within the sequence
  int n;     // stages of this sequence
  int ps;    // line index of the sequence's first stage
  int len;   // sequence length (tokens)
};

template <bool MULTI = false>
__device__ __forceinline__ Cursor cursor_at(const DecodeArgs& a, const int32_t* pre, int g) {
  int lo = 0;
  int hi = a.num_seqs - 1;  // largest s with pre[s] <= g: a non-empty sequence
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= g) lo = mid; else hi = mid - 1;
  }
  Cursor c;
  c.s = lo;
  c.n = pre[lo + 1] - pre[lo];
  c.j = g - pre[lo];
  c.ps = pre[lo];
  c.len = line_len<MULTI>(a, lo, false);
  return c;
}

template <bool MULTI = false>
__device__ __forceinline__ void cursor_next(const DecodeArgs& a, const int32_t* pre, Cursor& c) {
  if (++c.j < c.n) return;
  c.j = 0;
  do {
    ++c.s;
  } while (c.s < a.num_seqs && pre[c.s + 1] == pre[c.s]);
  if (c.s < a.num_seqs) {
    c.n = pre[c.s + 1] - pre[c.s];
    c.ps = pre[c.s];
    c.len = line_len<MULTI>(a, c.s, false);
  }
}

// Range owning line index g when S stages are cut into R ranges, range r taking
// [r*S/R, (r+1)*S/R). Ranges can be empty when R > S.
__device__ __forceinline__ int64_t stage_owner(int64_t g, int64_t S, int64_t R) {
  return ((g + 1) * R - 1) / S;
}

__device__ __forceinline__ int64_t range_start(int64_t r, int64_t S, int64_t R) {
  return (r * S) / R;
}

// pre[s] = number of 16-token stages of sequences before s (line_len tokens
// each), pre[N] = all of them; built by the whole CTA (nwarps warps, nwarps <= 16).
template <bool MULTI = false>
__device__ __forceinline__ void build_line_prefix(const DecodeArgs& a, int32_t* pre, int tt,
                                                  int* warp_tot, int nwarps) {
  const int N = a.num_seqs;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int per = (N + blockDim.x - 1) / blockDim.x;
  const int beg = min(N, static_cast<int>(threadIdx.x) * per);
  const int end = min(N, beg + per);
  int local = 0;
  for (int s = beg; s < end; ++s) local += (line_len<MULTI>(a, s, blockIdx.x == 0) + tt - 1) / tt;
  int x = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  int run = x - local;
  int total = 0;
  for (int w = 0; w < nwarps; ++w) {
    if (w < warp) run += warp_tot[w];
    total += warp_tot[w];
  }
  for (int s = beg; s < end; ++s) {
    pre[s] = run;
    run += (line_len<MULTI>(a, s, false) + tt - 1) / tt;
  }
  if (threadIdx.x == 0) pre[N] = total;
  __syncthreads();
}

// A warp finished its share of piece (sequence s, KV head kvh), which covers
// line stages [ps, pe); its own stages are [g0, g1), range `range` of `ranges`
// cut from the line of stot stages. A piece the warp covered whole is
// normalised and written; otherwise the warp leaves an (m, l, o) partial in
// slot (range * H_kv + kvh) * 2 + (0: its first piece, 1: its last) and the
// last contributor to arrive merges the piece. DEFER: the warp only leaves
// its partial; decode_piece_merge_kernel merges every cut piece once the
// stream kernel has finished, so no piece end waits on a fence, an atomic or
// a merge.
template <int D, int NT, bool FP8, bool DEFER = false>
__device__ __forceinline__ void finish_piece(const DecodeArgs& a, Acc<D, NT>& acc, int s, int ps,
                                             int pe, int g0, int g1, int64_t stot, int64_t ranges,
                                             int64_t range, int kvh, int lane) {
  constexpr int KD = D / 16;
  const int gid = lane >> 2;
  const int tig = lane & 3;
  const int hkv = a.num_kv_heads;
  acc.reduce_l();
  const int64_t row0 = static_cast<int64_t>(s) * a.num_q_heads + static_cast<int64_t>(kvh) * a.group;
  if (ps >= g0 && pe <= g1) {
    // whole piece: normalise and write, one reciprocal per column (v_scale
    // folded in for E4M3) rather than a division per element
    float inv[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float l = acc.l[nt][c];
        inv[nt][c] = l > 0.f ? (FP8 ? a.v_scale : 1.f) / l : 0.f;
      }
    }
#pragma unroll
    for (int dm = 0; dm < KD; ++dm) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = nt * 8 + tig * 2 + (r & 1);
          if (col < a.group)
            store_out(a, (row0 + col) * D + acc_dim<FP8>(dm, gid, r), acc.o[dm][nt][r] * inv[nt][r & 1]);
        }
      }
    }
  } else {
    // cut piece: leave a partial, the last contributor merges
    const int64_t slot_id = (range * hkv + kvh) * 2 + (ps <= g0 ? 0 : 1);
    float* po = a.part_o + slot_id * a.group * D;
    float* pml = a.part_ml + slot_id * a.group * 2;
#pragma unroll
    for (int dm = 0; dm < KD; ++dm) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int col = nt * 8 + tig * 2 + (r & 1);
          if (col < a.group)
            po[col * D + acc_dim<FP8>(dm, gid, r)] =
                FP8 ? acc.o[dm][nt][r] * a.v_scale : acc.o[dm][nt][r];
        }
      }
    }
    if (gid == 0) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int col = nt * 8 + tig * 2 + c;
          if (col < a.group) {
            pml[col * 2] = acc.m[nt][c];
            pml[col * 2 + 1] = acc.l[nt][c];
          }
        }
      }
    }
    if constexpr (DEFER) return;
    __threadfence();
    __syncwarp();
    // Contributors: the warps of head kvh in the non-empty ranges ra..rb that
    // meet [ps, pe). Ranges in between are empty only when there are more
    // ranges than stages.
    const int64_t ra = stage_owner(ps, stot, ranges);
    const int64_t rb = stage_owner(pe - 1, stot, ranges);
    const int span = static_cast<int>(rb - ra + 1);
    auto nonempty = [&](int64_t r) {
      return range_start(r, stot, ranges) < range_start(r + 1, stot, ranges);
    };
    int contrib = 0;
    for (int c0 = 0; c0 < span; c0 += 32)
      contrib += __popc(__ballot_sync(0xffffffffu, c0 + lane < span && nonempty(ra + c0 + lane)));
    unsigned int old = 0;
    if (lane == 0)
      old = atomicInc(a.counters + static_cast<int64_t>(s) * hkv + kvh,
                      static_cast<unsigned int>(contrib - 1));
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old == static_cast<unsigned int>(contrib - 1)) {
      __threadfence();
      const bool ra_first = range_start(ra, stot, ranges) == ps;  // piece is ra's first
      auto slot = [&](int c) -> int {
        const int64_t r = ra + c;
        if (!nonempty(r)) return -1;
        return static_cast<int>((r * hkv + kvh) * 2 + ((c == 0 && !ra_first) ? 1 : 0));
      };
      merge_rows<D>(a, span, slot, a.group, a.part_ml, a.group * 2, 2, a.part_o,
                    static_cast<int64_t>(a.group) * D, D, row0, lane);
    }
  }

}

template <bool IS_BF16, int D, int NT, int NS, bool SPLIT_P, bool FP8>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_balanced_kernel(const __grid_constant__ CUtensorMap tmk,
                           const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  using S = DecodeSmem<D, NT, NS, FP8>;
  constexpr int W = kDecodeWarps;
  constexpr int KD = D / 16;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int warp_tot[16];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = a.num_seqs;
  const int hkv = a.num_kv_heads;
  const int tt = a.ops_per_stage * a.tok_per_op;

  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sm_base = smem_u32(sm);
  int32_t* pre = reinterpret_cast<int32_t*>(sm + S::kPrefixOffset);  // [N + 1]

  // ---- line offset of every sequence: pre[s] = sum_{s'<s} ceil(L_s'/tt)
  build_line_prefix(a, pre, tt, warp_tot, W);

  // ---- zero the output rows of empty sequences (CTA c takes s = c mod grid)
  for (int s = blockIdx.x; s < N; s += gridDim.x) {
    if (pre[s + 1] != pre[s]) continue;
    const int64_t base = static_cast<int64_t>(s) * a.num_q_heads * D;
    for (int i = threadIdx.x; i < a.num_q_heads * D; i += W * 32) store_out(a, base + i, 0.f);
  }

  // ---- this warp's KV head and range of the line
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * W + warp;
  const int64_t ranges = static_cast<int64_t>(gridDim.x) * W / hkv;
  const int kvh = static_cast<int>(wid % hkv);
  const int64_t grp = wid / hkv;
  const int64_t stot = pre[N];
  if (grp >= ranges) return;  // no CTA-wide barrier follows
  const int g0 = static_cast<int>(range_start(grp, stot, ranges));
  const int g1 = static_cast<int>(range_start(grp + 1, stot, ranges));
  if (g0 >= g1) return;
  const int count = g1 - g0;

  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + S::kMaskOffset) + warp * NS;
  const uint32_t bar0 = sm_base + S::kBarOffset + warp * NS * 8;
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < NS; ++i) mbar_init(bar0 + 8 * i, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t ring = sm_base + warp * NS * S::kStageBytes;
  uint8_t* const ring_ptr = sm + warp * NS * S::kStageBytes;

  Cursor ic = cursor_at(a, pre, g0);  // next stage to issue
  Cursor cc = ic;                     // stage being computed
  int n_issued = 0;  // stages 0 .. n_issued - 1 have their copies issued
  auto issue = [&](int it) {
    if (a.test_stop_stage >= 0 && it >= a.test_stop_stage) return;
    const int slot = it % NS;
    issue_stage<D, FP8>(a, &tmk, &tmv, static_cast<int64_t>(ic.s) * a.max_blocks, kvh, ic.j * tt,
                        ic.len, ring + slot * S::kStageBytes, bar0 + 8 * slot, masks + slot, lane);
    cursor_next(a, pre, ic);
    n_issued = it + 1;
  };
  const uint64_t wait_ns = PA_STAGE_WAIT_NS(a, kWaitLimitNs);
  const int pro = count < NS ? count : NS;
  for (int i = 0; i < pro; ++i) issue(i);

  uint32_t qb[NT][KD][2];
  LogitScale<NT, FP8> ls;
  load_q<IS_BF16, D, NT, FP8>(a, cc.s, kvh, lane, qb, ls);
  Acc<D, NT> acc;
  acc.reset();
  bool aborted = false;

  for (int it = 0; it < count; ++it) {
    const int slot = it % NS;
    if (!aborted) {
      const bool got = mbar_wait_bounded(bar0 + 8 * slot, (it / NS) & 1, wait_ns);
      if (__any_sync(0xffffffffu, !got)) {
        aborted = true;
        if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
        for (int j = it; j < n_issued; ++j)
          mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, kWaitLimitNs);
      }
    }
    if (!aborted) {
      compute_stage<IS_BF16, D, NT, SPLIT_P, FP8>(
          warp_stage_view(ring + slot * S::kStageBytes, S::kHalves), ring, ring_ptr, masks[slot],
          qb, acc, ls, lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (it + NS < count) issue(it + NS);
    }

    const bool piece_end = (cc.j == cc.n - 1) || (it == count - 1);
    if (!piece_end) {
      cursor_next(a, pre, cc);
      continue;
    }

    // ---- the warp is done with its share of piece (cc.s, kvh)
    if (aborted) acc.reset();  // contribute nothing, but still take part
    finish_piece<D, NT, FP8>(a, acc, cc.s, cc.ps, cc.ps + cc.n, g0, g1, stot, ranges, grp, kvh,
                             lane);

    if (it + 1 < count) {
      cursor_next(a, pre, cc);
      load_q<IS_BF16, D, NT, FP8>(a, cc.s, kvh, lane, qb, ls);
      acc.reset();
    }
  }
}

// ============================================================================
// launch helpers

// Stages per warp: keeps 2 CTAs (8 warps) resident per SM for D <= 128. FP8
// stages are half the bytes, so twice as many keep the same bytes in flight.
template <int D, bool FP8>
constexpr int decode_stages() {
  return (D == 64 ? 6 : (D == 128 ? 3 : 2)) * (FP8 ? 2 : 1);
}

template <bool IS_BF16, int D, int NT, bool FP8>
cudaError_t launch_decode_tiles(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                dim3 grid, bool balanced, cudaStream_t st) {
  constexpr int NS = decode_stages<D, FP8>();
  using S = DecodeSmem<D, NT, NS, FP8>;
  if (balanced) {
    auto kern = decode_balanced_kernel<IS_BF16, D, NT, NS, true, FP8>;
    const int smem = S::kTotal + (a.num_seqs + 1) * 4;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, kDecodeWarps * 32, smem, st>>>(tk, tv, a);
    return cudaGetLastError();
  }
  auto kern = decode_kernel<IS_BF16, D, NT, NS, true, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecodeWarps * 32, S::kTotal, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <bool IS_BF16, int D, bool FP8>
cudaError_t launch_decode_dispatch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                   int group_tiles, dim3 grid, bool balanced, cudaStream_t st) {
  if (group_tiles == 1) return launch_decode_tiles<IS_BF16, D, 1, FP8>(tk, tv, a, grid, balanced, st);
  if (group_tiles == 2) return launch_decode_tiles<IS_BF16, D, 2, FP8>(tk, tv, a, grid, balanced, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
