// pa_decode_grouped.cuh - balanced decode with head-grouped TMA loads.
//
// HBM streams scattered pool blocks at full speed only when each block is
// fetched as a few large requests. Loading one KV head's 16 rows at a time
// (one box per warp) leaves HBM at about 90% of the rate a box covering the
// rows of several heads reaches, so here one box carries all HG heads of a
// CTA's head group.
//
// A CTA = one producer warp + HG consumer warps (one per KV head of its group)
// and owns one range of the stage line (the same equal-range split as the
// balanced kernel, now per range x head group). The producer fills a shared
// ring of NS stages: per stage, block piece and 64-element column half, one
// TMA box of 64 x 16 tokens x HG heads for K and one for V. Its tensor map lists the
// cache as (head_dim, token, head, block) - token before head - so the box
// lands head-major in shared memory, [head][token][64]: each consumer's rows
// are 16 contiguous 128-byte lines, read with the same conflict-free swizzled
// ldmatrix addressing as the per-warp kernels. Consumers release a slot on an
// "empty" mbarrier (HG arrivals); the producer refills it.
//
// Partials are those of the balanced kernel (warp slot range * H_kv + kv_head),
// but a piece end only stores: no fence, no arrival counter, no merge. While
// HBM is saturated every global round trip waits behind the stream (several
// microseconds), so those steps cost a warp that is as fast as the stream
// time it never makes up. decode_piece_merge_kernel, launched right after on
// the same stream as a programmatic dependent, merges every cut piece.
//
// FP8 caches: a 128-byte line holds 128 head-dim codes, so a box is 128 x 16
// tokens x HG heads; a stage holds 32 tokens (ST = 32, two boxes per 16-token
// half) to carry the same bytes as a 16-bit stage, and consumers run their
// 16-row step twice per stage.
#pragma once

#include "pa_decode.cuh"

namespace pa {

// Shared-memory plan of the grouped kernel for head group HG (runtime) and
// stages of ST token rows.
template <int D, int NS, bool FP8, int ST = kStageRows>
struct GroupedSmem {
  static constexpr int kHalves = D / KvLayout<FP8>::kPieceElems;
  __host__ __device__ static constexpr uint32_t half_bytes(int hg) { return hg * ST * 128u; }
  __host__ __device__ static constexpr uint32_t stage_bytes(int hg) { return 2u * kHalves * half_bytes(hg); }
  __host__ __device__ static constexpr uint32_t bar_offset(int hg) { return NS * stage_bytes(hg); }
  __host__ __device__ static constexpr uint32_t mask_offset(int hg) { return bar_offset(hg) + 2u * NS * 8u; }
  __host__ __device__ static constexpr uint32_t prefix_offset(int hg) { return mask_offset(hg) + NS * 4u; }
  // + (N + 1) * 4 prefix bytes + 1024 base-alignment slack
  __host__ __device__ static constexpr uint32_t total(int hg, int n) {
    return prefix_offset(hg) + (n + 1) * 4u + 1024u;
  }
};

// The producer's issue of one stage (tokens [t0, t0 + ST) of the sequence at
// table_row, clipped at tok_end) for KV heads [head0, head0 + hg): one box per
// block piece and column half, for K and for V, all completing on `bar`.
// Lane j handles the j-th block piece. Stores the valid-row mask to *mask.
template <int D, bool FP8, int ST = kStageRows>
__device__ __forceinline__ void issue_group_stage(const DecodeArgs& a, const CUtensorMap* tmk,
                                                  const CUtensorMap* tmv, int64_t table_row,
                                                  int head0, int hg, int t0, int tok_end,
                                                  uint32_t stage, uint32_t half_bytes, uint32_t bar,
                                                  uint32_t* mask, int lane) {
  constexpr int PE = KvLayout<FP8>::kPieceElems;
  constexpr int HALVES = D / PE;
  const int tpo = a.tok_per_op;  // 8 or 16 here: a multiple of 8, no padding rows
  int blk = 0;
  int off = 0;
  bool ok = false;
  if (lane < ST / tpo) {
    const int t = t0 + lane * tpo;
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
  if (lane < ST) {
    const int jr = lane / tpo;
    const int tok = t0 + lane;
    rv = tok < tok_end && ((okmask >> jr) & 1u);
  }
  static_assert(ST == 16 || ST == 32, "stage rows");
  const uint32_t rowmask = __ballot_sync(0xffffffffu, rv) & (ST == 32 ? 0xffffffffu : (1u << ST) - 1u);
  if (lane == 0) {
    *mask = rowmask;
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(okmask)) * tpo * hg * D * 2u *
                                   KvLayout<FP8>::kBytes);
  }
  __syncwarp();
  if (ok) {
    const uint32_t dk = stage + lane * static_cast<uint32_t>(hg * tpo * 128);
    const uint32_t dv = dk + HALVES * half_bytes;
#pragma unroll
    for (int c = 0; c < HALVES; ++c) {
      tma_load_4d(dk + c * half_bytes, tmk, bar, c * PE, off, head0, blk);
      tma_load_4d(dv + c * half_bytes, tmv, bar, c * PE, off, head0, blk);
    }
  }
}

// Largest head group per instantiation: 8, or 4 where a consumer warp holds
// more registers (head_dim 256, or more than 8 query heads per KV head), so the
// CTA's register budget covers every warp without spills.
__host__ __device__ constexpr int max_head_group(int d, int nt) { return (d > 128 || nt > 1) ? 4 : 8; }

// Grid: ranges x (H_kv / HG) CTAs of HG + 1 warps; CTA c takes range c / nhg
// and head group c % nhg, so the head groups of one range run side by side.
template <bool IS_BF16, int D, int NT, int NS, int HG, int TPO, bool SPLIT_P, bool FP8, int ST>
__global__ void __launch_bounds__((HG + 1) * 32, 1)
    decode_grouped_kernel(const __grid_constant__ CUtensorMap tmk,
                          const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  using S = GroupedSmem<D, NS, FP8, ST>;
  constexpr int KD = D / 16;
  constexpr int HALVES = S::kHalves;
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int warp_tot[16];

  constexpr int hg = HG;  // consumer warps = KV heads per CTA
  const int nwarps = HG + 1;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int N = a.num_seqs;
  const int hkv = a.num_kv_heads;
  const int tt = ST;  // tokens per stage of the line
  const uint32_t half_bytes = S::half_bytes(hg);
  const uint32_t stage_bytes = S::stage_bytes(hg);

  // the merge kernel may be scheduled now; it waits for this grid to finish
  // before it reads a partial
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sm_base = smem_u32(sm);
  int32_t* pre = reinterpret_cast<int32_t*>(sm + S::prefix_offset(hg));
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + S::mask_offset(hg));
  const uint32_t full0 = sm_base + S::bar_offset(hg);
  const uint32_t empty0 = full0 + NS * 8;

  build_line_prefix(a, pre, tt, warp_tot, nwarps);

  for (int s = blockIdx.x; s < N; s += gridDim.x) {  // zero rows of empty sequences
    if (pre[s + 1] != pre[s]) continue;
    const int64_t base = static_cast<int64_t>(s) * a.num_q_heads * D;
    for (int i = threadIdx.x; i < a.num_q_heads * D; i += blockDim.x) store_out(a, base + i, 0.f);
  }

  const int nhg = hkv / hg;
  const int64_t ranges = gridDim.x / nhg;
  if (blockIdx.x >= ranges * nhg) return;  // uniform across the CTA; no barrier follows
  const int64_t range = blockIdx.x / nhg;
  const int head0 = static_cast<int>(blockIdx.x % nhg) * hg;
  const int64_t stot = pre[N];
  const int g0 = static_cast<int>(range_start(range, stot, ranges));
  const int g1 = static_cast<int>(range_start(range + 1, stot, ranges));
  if (g0 >= g1) return;
  const int count = g1 - g0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, hg);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == hg) {
    // ------------------------------------------------------------ producer
    Cursor ic = cursor_at(a, pre, g0);
    int issued = 0;
    const int stop = a.test_stop_stage >= 0 && a.test_stop_stage < count ? a.test_stop_stage : count;
    for (; issued < stop; ++issued) {
      const int slot = issued % NS;
      if (issued >= NS) {  // every consumer released this slot's previous stage
        const bool got = mbar_wait_bounded(empty0 + 8 * slot, ((issued / NS) - 1) & 1, kWaitLimitNs);
        if (__any_sync(0xffffffffu, !got)) {
          if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
          break;
        }
      }
      issue_group_stage<D, FP8, ST>(a, &tmk, &tmv, static_cast<int64_t>(ic.s) * a.max_blocks, head0,
                                hg, ic.j * tt, ic.len, sm_base + slot * stage_bytes, half_bytes,
                                full0 + 8 * slot, masks + slot, lane);
      cursor_next(a, pre, ic);
    }
    // the last stages' copies complete before the producer leaves
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
      mbar_wait_bounded(full0 + 8 * (j % NS), (j / NS) & 1, kWaitLimitNs);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int kvh = head0 + warp;
  GroupView<HG, TPO, ST> sv;
  sv.head_off = static_cast<uint32_t>(warp * TPO * 128);

  Cursor cc = cursor_at(a, pre, g0);
  // q of the piece after c, when that piece starts inside this range
  auto prefetch_next = [&](const Cursor& c) {
    if (c.ps + c.n >= g1) return;
    int s2 = c.s + 1;
    while (s2 < N && pre[s2 + 1] == pre[s2]) ++s2;  // empty sequences have no piece
    if (s2 < N) prefetch_q<D>(a, s2, kvh, lane);
  };
  uint32_t qb[NT][KD][2];
  LogitScale<NT, FP8> ls;
  load_q<IS_BF16, D, NT, FP8>(a, cc.s, kvh, lane, qb, ls);
  prefetch_next(cc);
  Acc<D, NT> acc;
  acc.reset();
  bool aborted = false;

  const uint64_t wait_ns = PA_STAGE_WAIT_NS(a, kWaitLimitNs);
  for (int it = 0; it < count; ++it) {
    const int slot = it % NS;
    if (!aborted) {
      const bool got = mbar_wait_bounded(full0 + 8 * slot, (it / NS) & 1, wait_ns);
      if (__any_sync(0xffffffffu, !got)) {
        aborted = true;
        if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
      }
    }
    if (!aborted) {
      // a stage holds ST / 16 tiles of 16 token rows; each goes through the
      // 16-row step (rows 16h .. 16h + 15 start (16h / TPO) boxes in)
#pragma unroll
      for (int h = 0; h < ST / kStageRows; ++h) {
        const uint32_t rm = (masks[slot] >> (kStageRows * h)) & ((1u << kStageRows) - 1u);
        if (h > 0 && rm == 0u) break;  // the rest of the stage lies past the sequence
        sv.k = sm_base + slot * stage_bytes + h * (kStageRows / TPO) * GroupView<HG, TPO, ST>::op_stride;
        sv.v = sv.k + HALVES * half_bytes;
        // E4M3: lazy maximum, and a warp vote skips its reduction on the
        // stages where no logit passes it by more than 8 (most of them)
        compute_stage<IS_BF16, D, NT, SPLIT_P, FP8, GroupView<HG, TPO, ST>, NoColLimit, FP8, false, FP8>(
            sv, sm_base, sm, rm, qb, acc, ls, lane);
      }
      static_assert(GroupView<HG, TPO, ST>::half_stride == S::half_bytes(HG), "layout");
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    }

    const bool piece_end = (cc.j == cc.n - 1) || (it == count - 1);
    if (!piece_end) {
      cursor_next(a, pre, cc);
      continue;
    }
    if (aborted) acc.reset();  // contribute nothing, but still take part
    finish_piece<D, NT, FP8, true>(a, acc, cc.s, cc.ps, cc.ps + cc.n, g0, g1, stot, ranges, range,
                                   kvh, lane);

    if (it + 1 < count) {
      cursor_next(a, pre, cc);
      load_q<IS_BF16, D, NT, FP8>(a, cc.s, kvh, lane, qb, ls);
      prefetch_next(cc);
      acc.reset();
    }
  }
}

// Stages in the shared ring: 16-token stages of 64 KB for HG = 8 at D = 128
// (HG = 4 at D = 256), three of them. E4M3 stages hold 32 tokens, so they
// carry the same bytes and each stage's fixed costs (the producer's block-id
// read and issue, the consumers' wait and release) are paid once per 64 KB.
template <int D, bool FP8>
constexpr int grouped_stages() {
  return 3;
}


template <bool IS_BF16, int D, int NT, int HG, int TPO, bool FP8>
cudaError_t launch_grouped(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                           dim3 grid, cudaStream_t st) {
  constexpr int NS = grouped_stages<D, FP8>();
  constexpr int ST = grouped_line_tokens(FP8);
  using S = GroupedSmem<D, NS, FP8, ST>;
  auto kern = decode_grouped_kernel<IS_BF16, D, NT, NS, HG, TPO, true, FP8, ST>;
  const int smem = static_cast<int>(S::total(HG, a.num_seqs));
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, (HG + 1) * 32, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

// Head groups of 8 (4 where max_head_group says so) and of 4; boxes of 16
// tokens (blocks of 16 or more) or 8 (blocks of 8).
template <bool IS_BF16, int D, int NT, bool FP8>
cudaError_t launch_grouped_tiles(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                 int head_group, dim3 grid, cudaStream_t st) {
  if (head_group > max_head_group(D, NT)) return cudaErrorInvalidValue;
  if constexpr (max_head_group(D, NT) >= 8) {
    if (head_group == 8) {
      return a.tok_per_op == 16 ? launch_grouped<IS_BF16, D, NT, 8, 16, FP8>(tk, tv, a, grid, st)
                                : launch_grouped<IS_BF16, D, NT, 8, 8, FP8>(tk, tv, a, grid, st);
    }
  }
  if (head_group == 4) {
    return a.tok_per_op == 16 ? launch_grouped<IS_BF16, D, NT, 4, 16, FP8>(tk, tv, a, grid, st)
                              : launch_grouped<IS_BF16, D, NT, 4, 8, FP8>(tk, tv, a, grid, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace pa
