// pa_verify.cuh - balanced, head-grouped attention for a few new tokens per
// sequence (speculative verification of a handful of drafts, short chunks).
//
// pa_prefill's query i of a sequence with n new tokens sits at position
// L - n + i and attends to positions 0 .. L - n + i ("PagedAttention: paging
// the KV cache", How it works: prefill writes into the blocks). With n * g of
// at most 32 (query, head) rows per KV head the work is that of decode: every
// row reads the whole cache once, so HBM bounds it. This kernel is the grouped
// decode kernel's stream (pa_decode_grouped.cuh) with (query, head) rows in
// place of heads:
//  * The rows of a KV head are numbered r = i * g + j (query i, head j) and cut
//    into R tiles of 8 * NT columns of the S^T = K Q^T tile. One consumer warp
//    owns one (KV head, tile); HG * R = 8 warps share each stage of HG heads.
//  * Column r admits the stage rows up to position L - n + r / g (ColLimit).
//  * The stage line carries each sequence with new rows, whole; ranges,
//    pieces, partials and last-arriver merges are the balanced decode ones,
//    with a (KV head, tile) pair as the column group of a partial.
//  * No producer warp: a ninth warp would leave three warps on one SM
//    sub-partition and cap every thread at 168 registers, too few for two
//    n-tiles of accumulators. The consumer that releases a slot last (a
//    shared counter per slot, acquire-release) issues the slot's next stage.
//    Every consumer reads that stage's block id a stage ahead, in a lane other
//    than the one that releases (the release orders only that lane's own
//    accesses), so the issue does not wait for the table.
#pragma once

#include "pa_decode_grouped.cuh"

namespace pa {

// Output rows of a tile's columns: column c is row r = tb + c of its KV head
// (query i = r / g, head r - i * g), stored at q/out row
// (q0 + i) * hq + head0 + r - i * g. The first n columns hold rows (queries
// past n_s or max_q hold none); run_end(c) ends the run of columns from c
// whose rows are consecutive (one query's heads).
struct QueryRows {
  int64_t q0;     // first q row of the sequence
  int64_t hq;     // query heads
  int64_t head0;  // kvh * g
  int tb;
  int g;
  int n;
  __device__ __forceinline__ int64_t row(int c) const {
    const int r = tb + c;
    const int i = r / g;
    return (q0 + i) * hq + head0 + (r - i * g);
  }
  __device__ __forceinline__ int run_end(int c) const {
    const int e = ((tb + c) / g + 1) * g - tb;
    return e < n ? e : n;
  }
};

// A warp finished its share of the piece (sequence s, column group vh of nvh)
// covering line stages [ps, pe); its own stages are [g0, g1), range `range` of
// `ranges` cut from the line of stot stages. A piece covered whole is
// normalised and written; otherwise the warp leaves the (m, l, o) partial of
// its 8 * NT columns in slot (range * nvh + vh) * 2 + (0: its first piece,
// 1: its last), and the last contributor to arrive merges the piece, one run
// of consecutive output rows at a time (decode's finish_piece with rows
// placed by QueryRows).
template <int D, int NT, bool FP8>
__device__ __forceinline__ void finish_piece_rows(const DecodeArgs& a, Acc<D, NT>& acc, int s,
                                                  int ps, int pe, int g0, int g1, int64_t stot,
                                                  int64_t ranges, int64_t range, int vh, int nvh,
                                                  const QueryRows& rows, int lane) {
  constexpr int KD = D / 16;
  constexpr int TC = 8 * NT;
  const int gid = lane >> 2;
  const int tig = lane & 3;
  acc.reduce_l();
  if (ps >= g0 && pe <= g1) {
    float inv[NT][2];
    int64_t orow[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const float l = acc.l[nt][c];
        inv[nt][c] = l > 0.f ? (FP8 ? a.v_scale : 1.f) / l : 0.f;
        const int col = nt * 8 + tig * 2 + c;
        orow[nt][c] = col < rows.n ? rows.row(col) : -1;
      }
    }
#pragma unroll
    for (int dm = 0; dm < KD; ++dm) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          if (orow[nt][r & 1] >= 0)
            store_out(a, orow[nt][r & 1] * D + acc_dim<FP8>(dm, gid, r),
                      acc.o[dm][nt][r] * inv[nt][r & 1]);
        }
      }
    }
    return;
  }
  const int64_t slot_id = (range * nvh + vh) * 2 + (ps <= g0 ? 0 : 1);
  float* po = a.part_o + slot_id * TC * D;
  float* pml = a.part_ml + slot_id * TC * 2;
#pragma unroll
  for (int dm = 0; dm < KD; ++dm) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int col = nt * 8 + tig * 2 + (r & 1);
        po[col * D + acc_dim<FP8>(dm, gid, r)] = FP8 ? acc.o[dm][nt][r] * a.v_scale : acc.o[dm][nt][r];
      }
    }
  }
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = nt * 8 + tig * 2 + c;
        pml[col * 2] = acc.m[nt][c];
        pml[col * 2 + 1] = acc.l[nt][c];
      }
    }
  }
  __threadfence();
  __syncwarp();
  // contributors: the warps of column group vh in the non-empty ranges
  // ra .. rb that meet [ps, pe)
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
    old = atomicInc(a.counters + static_cast<int64_t>(s) * nvh + vh,
                    static_cast<unsigned int>(contrib - 1));
  old = __shfl_sync(0xffffffffu, old, 0);
  if (old != static_cast<unsigned int>(contrib - 1)) return;
  __threadfence();
  const bool ra_first = range_start(ra, stot, ranges) == ps;  // the piece is ra's first
  auto slot = [&](int c) -> int {
    const int64_t r = ra + c;
    if (!nonempty(r)) return -1;
    return static_cast<int>((r * nvh + vh) * 2 + ((c == 0 && !ra_first) ? 1 : 0));
  };
  for (int c0 = 0; c0 < rows.n;) {
    const int c1 = rows.run_end(c0);
    merge_rows<D>(a, span, slot, c1 - c0, a.part_ml + c0 * 2, TC * 2, 2, a.part_o + c0 * D,
                  static_cast<int64_t>(TC) * D, D, rows.row(c0), lane);
    c0 = c1;
  }
}

// One stage of HG heads for blocks of 16 or more tokens: one box per column
// half covers the stage's 16 tokens of every head. The block id `blk` is
// already read; lane 0 issues the K and V boxes on `bar` and stores the
// stage's valid-row mask to *mask (no rows for an id out of range).
template <int D, bool FP8>
__device__ __forceinline__ void issue_group_stage16(const DecodeArgs& a, const CUtensorMap* tmk,
                                                    const CUtensorMap* tmv, int blk, int head0,
                                                    int hg, int t0, int tok_end, uint32_t stage,
                                                    uint32_t half_bytes, uint32_t bar,
                                                    uint32_t* mask, int lane) {
  constexpr int PE = KvLayout<FP8>::kPieceElems;
  constexpr int HALVES = D / PE;
  if (lane != 0) return;
  const int off = t0 % a.block_size;
  const bool ok = blk >= 0 && blk < a.num_blocks;
  if (!ok) atomicOr(a.err, PA_DEVERR_BLOCK_ID);
  const int rows = tok_end - t0;
  *mask = ok ? (rows >= kStageRows ? (1u << kStageRows) - 1u : (1u << rows) - 1u) : 0u;
  mbar_arrive_expect_tx(
      bar, ok ? static_cast<uint32_t>(kStageRows * hg * D * 2 * KvLayout<FP8>::kBytes) : 0u);
  if (ok) {
    const uint32_t dv = stage + HALVES * half_bytes;
#pragma unroll
    for (int c = 0; c < HALVES; ++c) {
      tma_load_4d(stage + c * half_bytes, tmk, bar, c * PE, off, head0, blk);
      tma_load_4d(dv + c * half_bytes, tmv, bar, c * PE, off, head0, blk);
    }
  }
}

// Shared-memory atomic add, acquire-release at CTA scope; returns the old value.
__device__ __forceinline__ uint32_t atom_add_acq_rel_smem(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(addr), "r"(v)
               : "memory");
  return old;
}

// Grid: ranges x (H_kv / HG) CTAs of HG * R warps (one per SM); CTA c takes
// range c / nhg and head group c % nhg. Warp w owns KV head head0 + w / R and
// row tile w % R.
template <bool IS_BF16, int NT, int NS, int HG, int R, bool FP8>
__global__ void __launch_bounds__(HG * R * 32, 1)
    multi_grouped_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  constexpr int D = 128;
  constexpr int TPO = kStageRows;
  using S = GroupedSmem<D, NS, FP8>;
  constexpr int KD = D / 16;
  constexpr int HALVES = S::kHalves;
  constexpr int CW = HG * R;  // warps, all consumers
  constexpr int TC = 8 * NT;  // columns of one tile
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int warp_tot[16];
  __shared__ uint32_t released[NS];  // releases per slot, over all its uses
  __shared__ int last_issued[NS];    // latest stage issued into each slot
  __shared__ int any_abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tig = lane & 3;
  const int N = a.num_seqs;
  const int hkv = a.num_kv_heads;
  const int g = a.group;
  const int tt = kStageRows;
  const uint32_t half_bytes = S::half_bytes(HG);
  const uint32_t stage_bytes = S::stage_bytes(HG);

  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sm_base = smem_u32(sm);
  int32_t* pre = reinterpret_cast<int32_t*>(sm + S::prefix_offset(HG));
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + S::mask_offset(HG));
  const uint32_t full0 = sm_base + S::bar_offset(HG);

  build_line_prefix<true>(a, pre, tt, warp_tot, CW);

  const int nhg = hkv / HG;
  const int64_t ranges = gridDim.x / nhg;
  if (blockIdx.x >= ranges * nhg) return;  // uniform across the CTA; no barrier follows
  const int64_t range = blockIdx.x / nhg;
  const int head0 = static_cast<int>(blockIdx.x % nhg) * HG;
  const int64_t stot = pre[N];
  const int g0 = static_cast<int>(range_start(range, stot, ranges));
  const int g1 = static_cast<int>(range_start(range + 1, stot, ranges));
  if (g0 >= g1) return;
  const int count = g1 - g0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      released[i] = 0u;
      last_issued[i] = -1;
    }
    any_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---- ring prologue: lane i of warp 0 reads stage i's block id, lane 0
  // issues the stages in order
  const int pro = count < NS ? count : NS;
  if (warp == 0) {
    const Cursor c = cursor_at<true>(a, pre, g0 + (lane < pro ? lane : pro - 1));
    const int blk = lane < pro ? __ldg(a.block_tables + static_cast<int64_t>(c.s) * a.max_blocks +
                                       (c.j * tt) / a.block_size)
                               : 0;
    for (int i = 0; i < pro; ++i) {
      const int b_i = __shfl_sync(0xffffffffu, blk, i);
      const int t0_i = __shfl_sync(0xffffffffu, c.j * tt, i);
      const int len_i = __shfl_sync(0xffffffffu, c.len, i);
      issue_group_stage16<D, FP8>(a, &tmk, &tmv, b_i, head0, HG, t0_i, len_i,
                                  sm_base + i * stage_bytes, half_bytes, full0 + 8 * i, masks + i,
                                  lane);
      if (lane == 0) last_issued[i] = i;
    }
  }

  const int hw = warp / R;         // KV head within the group
  const int tile = warp - hw * R;  // row tile of that head
  const int kvh = head0 + hw;
  const int vh = kvh * R + tile;   // column group of the partials
  const int nvh = hkv * R;
  GroupView<HG, TPO> sv;
  sv.head_off = static_cast<uint32_t>(hw * TPO * 128);

  // The stage NS ahead of the current one (a release of the current slot may
  // issue it) and its block id, read by lane 1 while the current stage
  // computes, apart from lane 0's release.
  Cursor ic{};
  if (pro < count) ic = cursor_at<true>(a, pre, g0 + pro);
  int next_blk = 0;

  // The current piece's rows: output placement, each column's last admitted
  // position, q.
  QueryRows rows{};
  ColLimit<NT> lim_pos;
  uint32_t qb[NT][KD][2];
  LogitScale<NT, FP8> ls;
  auto start_piece = [&](const Cursor& c) {
    const int qa = __ldg(a.q_start + c.s);
    const int n = __ldg(a.q_start + c.s + 1) - qa;
    const int n_live = n < a.max_q ? n : a.max_q;
    rows.q0 = qa;
    rows.hq = a.num_q_heads;
    rows.head0 = static_cast<int64_t>(kvh) * g;
    rows.tb = tile * TC;
    rows.g = g;
    const int live = n_live * g - tile * TC;  // columns holding rows
    rows.n = live < 0 ? 0 : (live < TC ? live : TC);
    const int first_pos = c.len - n;  // position of query 0
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int k = 0; k < 2; ++k)
        lim_pos.rel[nt][k] = first_pos + (tile * TC + nt * 8 + tig * 2 + k) / g;
    }
    if (rows.n > 0)
      load_q_rows<IS_BF16, D, NT, FP8>(
          a,
          [&](int nt) -> int64_t {
            const int col = nt * 8 + gid;
            return col < rows.n ? rows.row(col) : -1;
          },
          lane, qb, ls);
  };
  // q of the piece after c, when that piece starts inside this range
  auto prefetch_next = [&](const Cursor& c) {
    if (c.ps + c.n >= g1) return;
    int s2 = c.s + 1;
    while (s2 < N && pre[s2 + 1] == pre[s2]) ++s2;  // sequences without rows have no piece
    if (s2 >= N) return;
    const int qa = __ldg(a.q_start + s2);
    int n2 = __ldg(a.q_start + s2 + 1) - qa;
    n2 = n2 < a.max_q ? n2 : a.max_q;
    const int i1 = min(n2, (tile * TC + TC - 1) / g + 1);
    for (int i = (tile * TC) / g; i < i1; ++i)
      prefetch_q_group<D>(a, (static_cast<int64_t>(qa) + i) * a.num_q_heads +
                                 static_cast<int64_t>(kvh) * g, lane);
  };

  Cursor cc = cursor_at<true>(a, pre, g0);
  start_piece(cc);
  prefetch_next(cc);
  Acc<D, NT> acc;
  acc.reset();
  bool aborted = false;

  for (int it = 0; it < count; ++it) {
    const int slot = it % NS;
    const bool refill = it + NS < count;  // a later stage goes into this slot
    if (refill && !aborted && lane == 1)
      next_blk = __ldg(a.block_tables + static_cast<int64_t>(ic.s) * a.max_blocks +
                       (ic.j * tt) / a.block_size);
    if (!aborted) {
      const bool got = mbar_wait_bounded(full0 + 8 * slot, (it / NS) & 1, kWaitLimitNs);
      if (__any_sync(0xffffffffu, !got)) {
        aborted = true;
        if (lane == 0) {
          atomicOr(a.err, PA_DEVERR_TIMEOUT);
          atomicOr(&any_abort, 1);
        }
      }
    }
    if (!aborted) {
      if (rows.n > 0) {
        sv.k = sm_base + slot * stage_bytes;
        sv.v = sv.k + HALVES * half_bytes;
        ColLimit<NT> rel;  // limits relative to this stage's first token
        const int t0 = cc.j * tt;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          rel.rel[nt][0] = lim_pos.rel[nt][0] - t0;
          rel.rel[nt][1] = lim_pos.rel[nt][1] - t0;
        }
        compute_stage<IS_BF16, D, NT, true, FP8, GroupView<HG, TPO>, ColLimit<NT>, true, true, true>(
            sv, sm_base, sm, masks[slot], qb, acc, ls, lane, rel);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (refill) {  // the last of the CW releases of this use of the slot refills it
        uint32_t old = 0;
        if (lane == 0) old = atom_add_acq_rel_smem(smem_u32(released + slot), 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        if (old == static_cast<uint32_t>(CW * (it / NS + 1) - 1)) {
          const int blk = __shfl_sync(0xffffffffu, next_blk, 1);
          issue_group_stage16<D, FP8>(a, &tmk, &tmv, blk, head0, HG, ic.j * tt, ic.len,
                                      sm_base + slot * stage_bytes, half_bytes, full0 + 8 * slot,
                                      masks + slot, lane);
          if (lane == 0) last_issued[slot] = it + NS;
        }
      }
    }
    if (refill) cursor_next<true>(a, pre, ic);

    const bool piece_end = (cc.j == cc.n - 1) || (it == count - 1);
    if (!piece_end) {
      cursor_next<true>(a, pre, cc);
      continue;
    }
    if (aborted) acc.reset();  // contribute nothing, but still take part
    // A tile without rows of this sequence has none in any range covering the
    // piece, so none of its contributors takes part.
    if (rows.n > 0)
      finish_piece_rows<D, NT, FP8>(a, acc, cc.s, cc.ps, cc.ps + cc.n, g0, g1, stot, ranges, range,
                                    vh, nvh, rows, lane);
    if (it + 1 < count) {
      cursor_next<true>(a, pre, cc);
      start_piece(cc);
      prefetch_next(cc);
      acc.reset();
    }
  }

  // After a timeout some issued stages were never awaited: their copies land
  // before the CTA and its shared memory go away. Each slot's earlier stages
  // completed before it was refilled.
  __syncthreads();
  if (any_abort && threadIdx.x == 0) {
    for (int k = 0; k < NS; ++k) {
      const int j = last_issued[k];
      if (j >= 0) mbar_wait_bounded(full0 + 8 * k, (j / NS) & 1, kWaitLimitNs);
    }
  }
}

// Eight warps (HG KV heads x R tiles of 8 NT columns), one CTA per SM with
// 192 KB of stages. (NT, R, HG) = (1, 1, 8) serves up to 8 rows per KV head,
// (2, 1, 8) up to 16 and (2, 2, 4) up to 32.
template <bool IS_BF16, int NT, int R, int HG, bool FP8>
cudaError_t launch_multi_grouped(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                 dim3 grid, cudaStream_t st) {
  constexpr int NS = static_cast<int>((192u * 1024u) / GroupedSmem<128, 1, FP8>::stage_bytes(HG));
  using S = GroupedSmem<128, NS, FP8>;
  static_assert(HG * R == 8, "eight warps");
  auto kern = multi_grouped_kernel<IS_BF16, NT, NS, HG, R, FP8>;
  const int smem = static_cast<int>(S::total(HG, a.num_seqs));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, HG * R * 32, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <bool IS_BF16, bool FP8>
cudaError_t launch_multi_rows(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                              int nt, int row_tiles, int head_group, dim3 grid, cudaStream_t st) {
  if (a.tok_per_op != kStageRows || a.q_start == nullptr) return cudaErrorInvalidValue;
  if (nt == 1 && row_tiles == 1 && head_group == 8)
    return launch_multi_grouped<IS_BF16, 1, 1, 8, FP8>(tk, tv, a, grid, st);
  if (nt == 2 && row_tiles == 1 && head_group == 8)
    return launch_multi_grouped<IS_BF16, 2, 1, 8, FP8>(tk, tv, a, grid, st);
  if (nt == 2 && row_tiles == 2 && head_group == 4)
    return launch_multi_grouped<IS_BF16, 2, 2, 4, FP8>(tk, tv, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
