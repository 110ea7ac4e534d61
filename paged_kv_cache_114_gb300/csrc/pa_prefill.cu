// pa_prefill.cu - multi-token paged attention with a causal mask (chunked
// prefill, speculative verification, recompute after preemption) for sm_103a.
//
// Sequence s has n new queries in rows q_start[s] .. q_start[s+1] of q; their
// K/V are already in the cache ("PagedAttention: paging the KV cache", How it
// works: prefill writes into the blocks). Query i sits at position
// p = L - n + i and attends to the tokens at positions 0 .. p, read through
// the block table; the block table says where rows are stored, the mask which
// attention edges exist ("PagedAttention: Manage the Cache Without Moving the
// Sequence", The kernel must understand the mapping). Decode is the case n = 1.
//
// Layout of the work: the (query, head) rows of one (sequence, KV head) are
// numbered r = i * g + j (query i, head j of the group), so the g heads that
// share a KV head share every K/V load. A CTA takes 64 such rows in 4 warps of
// 16 rows. The sequence's K and V stream, 64 tokens a stage, into a shared
// ring of TMA tensor copies (one box of 64 head-dim elements x tpo tokens per
// block piece and column half, 128-byte swizzle), up to the CTA's last query
// position; warp 0 refills a slot once all four warps have released it (a
// separate producer warp would put three warps on some SM sub-partitions and
// cap every thread at 168 registers). Each warp computes, per stage,
//   S = Q K^T   (mma.sync m16n8k16: M = its 16 rows, N = 8 tokens, K = head dim)
//   online softmax per row in the log2 domain, causal mask per element,
//   O += P V    (M = 16 rows, N = 8 head-dim columns, K = 16 tokens),
// with the P operand built straight from the S accumulators and split into a
// 16-bit high and low part so the PV product keeps ~16 bits of the weights.
// Rows of a stage that hold no valid token (past the CTA's last position, or
// of a block whose id is out of range) have their V rows zeroed before PV, so
// stale or NaN bytes never reach the output.
//
// Few rows (verifying a few drafts: g * n rows per KV head, often 32 or less):
// the warps without rows of their own take a share of each stage's tokens,
// keep their own softmax state, and fold it into the first part through the
// freed ring at the end, so all four warps compute. Batches of up to 256
// sequences run longest first (CTA z takes the sequence of rank z by length).
//
// FP8 (E4M3) caches: a stage row is D bytes, one 128-byte swizzled line per
// 128 head-dim codes. ldmatrix treats byte pairs as its 16-bit elements: for
// S = Q K^T each lane gets four consecutive codes of a token, so the MMA's
// reduction index runs over head-dim elements four at a time (q is loaded in
// that order); for O = P V the transposing ldmatrix gives two dims of two
// tokens, and one byte permute pairs the tokens per dim, the two dims landing
// in two n-tiles of O. Codes widen exactly to fp16 (cvt.rn.f16x2.e4m3x2) and
// every MMA runs in fp16; a bf16 query row becomes fp16 times a power of two
// that keeps its largest element below 2^14, undone in the row's logit scale.
// k_scale folds into the logit scale, v_scale multiplies the output.
#include <cuda.h>
#include <cuda_runtime.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kRows = 64;        // query rows per CTA
constexpr int kTok = 64;         // tokens per stage
constexpr int kWarps = 4;        // consumer warps
constexpr int kOrderMax = 256;   // batches up to this size run longest sequence first
constexpr int kIdsCap = 512;     // block ids staged in shared memory per CTA
constexpr uint64_t kLimitNs = 2000000000ull;  // 2 s per bounded wait

template <int D>
constexpr int prefill_stages() {
  return D == 64 ? 4 : (D == 128 ? 3 : 2);
}

template <int D, int NS, bool FP8>
struct PrefillSmem {
  static constexpr int kHalves = D / (FP8 ? 128 : 64);
  static constexpr uint32_t kPlane = kTok * 128;               // 64 rows of one column half
  static constexpr uint32_t kStage = 2 * kHalves * kPlane;     // K planes then V planes
  static constexpr uint32_t kBar = NS * kStage;                // full[NS], empty[NS]
  static constexpr uint32_t kMask = kBar + 2 * NS * 8;         // uint64 valid-row mask per stage
  static constexpr uint32_t kIds = kMask + NS * 8;             // the sequence's first block ids
  static constexpr uint32_t kTotal = kIds + kIdsCap * 4 + 1024; // + base-alignment slack
};

__device__ __forceinline__ void store_val(const PrefillArgs& a, int64_t idx, float v) {
  if (a.out_dtype == PA_F32) {
    static_cast<float*>(a.out)[idx] = v;
  } else if (a.out_dtype == PA_F16) {
    static_cast<__half*>(a.out)[idx] = __float2half_rn(v);
  } else {
    static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
  }
}

// Shared address of (token row t, 16-byte chunk c8 of the head dim) in a
// stage's K or V planes: plane c8 / 8, 128-byte swizzle of chunk c8 % 8.
__device__ __forceinline__ uint32_t swz(uint32_t planes, int t, int c8) {
  return planes + (c8 >> 3) * (kTok * 128u) + t * 128u + ((((c8 & 7) ^ (t & 7))) << 4);
}

// Warp-wide issue of stage `it` (tokens it*64 ..) into ring slot `slot`: lane
// j < ops_per_stage copies block piece j if it starts at or before max_pos.
// Lane 0 records the stage's valid-row mask and arms the full barrier.
template <int D, int NS, bool FP8>
__device__ __forceinline__ void issue_prefill_stage(const PrefillArgs& a, const CUtensorMap* tmk,
                                                    const CUtensorMap* tmv, int64_t table_row,
                                                    int kvh, int it, int max_pos, uint32_t base,
                                                    uint32_t full0, uint64_t* masks,
                                                    const int32_t* ids, int lane) {
  using S = PrefillSmem<D, NS, FP8>;
  constexpr int PE = FP8 ? 128 : 64;  // head-dim elements per 128-byte line
  const int slot = it % NS;
  const int tpo = a.tok_per_op;
  const int t0 = it * kTok;
  int blk = 0;
  int off = 0;
  bool ok = false;
  if (lane < a.ops_per_stage) {
    const int t = t0 + lane * tpo;
    if (t <= max_pos) {
      const int j = t / a.block_size;
      off = t - j * a.block_size;
      blk = j < kIdsCap ? ids[j] : __ldg(a.block_tables + table_row + j);
      ok = blk >= 0 && blk < a.num_blocks;
      if (!ok) atomicOr(a.err, PA_DEVERR_BLOCK_ID);
    }
  }
  const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
  if (lane == 0) {
    // valid rows: loaded, and at a position some row of the CTA may see
    uint64_t m = 0;
    for (int j = 0; j < a.ops_per_stage; ++j)
      if ((okmask >> j) & 1u) m |= ((tpo >= 64) ? ~0ull : ((1ull << tpo) - 1ull)) << (j * tpo);
    const int last = max_pos - t0;  // rows 0 .. last are at or before max_pos
    if (last < kTok - 1) m &= (1ull << (last + 1)) - 1ull;
    masks[slot] = m;
    mbar_arrive_expect_tx(full0 + 8 * slot,
                          static_cast<uint32_t>(__popc(okmask)) * tpo * D * (FP8 ? 2u : 4u));
  }
  __syncwarp();
  if (ok) {
    const uint32_t dk = base + slot * S::kStage + lane * tpo * 128u;
    const uint32_t dv = dk + S::kHalves * S::kPlane;
#pragma unroll
    for (int c = 0; c < S::kHalves; ++c) {
      tma_load_4d(dk + c * S::kPlane, tmk, full0 + 8 * slot, c * PE, kvh, off, blk);
      tma_load_4d(dv + c * S::kPlane, tmv, full0 + 8 * slot, c * PE, kvh, off, blk);
    }
  }
}

// MINB: CTAs per SM the register budget is cut for (2 for D <= 128, 1 for
// 256; 3 for the thin launch of CTAs with few rows, with a shorter ring).
template <bool IS_BF16, int D, int NS, bool FP8, int MINB>
__global__ void __launch_bounds__(kWarps * 32, MINB)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const PrefillArgs a) {
  using S = PrefillSmem<D, NS, FP8>;
  constexpr bool MB = IS_BF16 && !FP8;  // MMA operand type: E4M3 caches run in fp16
  constexpr int KD = D / 16;   // k-steps of QK^T
  constexpr int ND = D / 8;    // n-tiles of O
  extern __shared__ __align__(16) uint8_t smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int gid = lane >> 2;
  const int tig = lane & 3;
  // CTA z takes the sequence of rank z by length, longest first (ties by
  // index), so the long sequences start in the first wave and the short ones
  // fill the tail. The ranks of all lengths are a permutation of 0 .. N-1.
  int s = blockIdx.z;
  if (a.num_seqs <= kOrderMax && static_cast<int>(gridDim.z) == a.num_seqs) {
    __shared__ int lens_sm[kOrderMax];
    __shared__ int pick;
    const int N = a.num_seqs;
    for (int i = threadIdx.x; i < N; i += blockDim.x) lens_sm[i] = __ldg(a.seq_lens + i);
    __syncthreads();
    for (int i = threadIdx.x; i < N; i += blockDim.x) {
      const int li = lens_sm[i];
      int rank = 0;
      for (int u = 0; u < N; ++u) {
        const int lu = lens_sm[u];
        rank += (lu > li || (lu == li && u < i)) ? 1 : 0;
      }
      if (rank == static_cast<int>(blockIdx.z)) pick = i;
    }
    __syncthreads();
    s = pick;
  }
  const int kvh = blockIdx.y;
  const int g = a.group;

  const int q0 = __ldg(a.q_start + s);
  const int nq = __ldg(a.q_start + s + 1) - q0;
  const int L = __ldg(a.seq_lens + s);
  const int rows_total = nq * g;
  const int row_base = blockIdx.x * kRows;
  if (nq <= 0 || row_base >= rows_total) return;  // uniform: no barrier has been used
  if (nq > L || static_cast<int64_t>(L) > static_cast<int64_t>(a.max_blocks) * a.block_size) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && kvh == 0) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    return;
  }
  if (blockIdx.x == gridDim.x - 1 && rows_total > row_base + kRows && threadIdx.x == 0 && kvh == 0)
    atomicOr(a.err, PA_DEVERR_SEQ_LEN);  // more queries than the launch covers

  const int row_end = min(row_base + kRows, rows_total);
  const int first_pos = L - nq;                                   // position of query 0
  const int max_pos = first_pos + (row_end - 1) / g;              // last position any row sees
  const int n_stages = max_pos / kTok + 1;

  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t base = smem_u32(sm);
  const uint32_t full0 = base + S::kBar;
  const uint32_t empty0 = full0 + NS * 8;
  uint64_t* masks = reinterpret_cast<uint64_t*>(sm + S::kMask);
  int32_t* ids = reinterpret_cast<int32_t*>(sm + S::kIds);
  const int64_t table_row = static_cast<int64_t>(s) * a.max_blocks;

  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kWarps);
    }
    fence_mbar_init();
  }
  // the block ids up to the CTA's last position, read once by every thread
  // together, so refilling a stage never waits on the table
  const int n_ids = min(max_pos / a.block_size + 1, kIdsCap);
  for (int j = threadIdx.x; j < n_ids; j += blockDim.x) ids[j] = __ldg(a.block_tables + table_row + j);
  __syncthreads();

  int issued = 0;  // stages warp 0 has issued
  if (warp == 0) {
    for (; issued < NS && issued < n_stages; ++issued)
      issue_prefill_stage<D, NS, FP8>(a, &tmk, &tmv, table_row, kvh, issued, max_pos, base, full0,
                                      masks, ids, lane);
  }

  // -------------------------------------------------------------- consumers
  // A warp computes 16 rows. With fewer than 64 rows (e.g. verifying a few
  // draft tokens), the warps left over split each stage's tokens instead:
  // warp w takes row group w % row_warps and token part w / row_warps of every
  // stage, and the parts' softmax states are merged at the end.
  const int row_warps = (row_end - row_base + 15) / 16;
  const int split = row_warps == 1 ? 4 : (row_warps == 2 ? 2 : 1);
  const int pcount = 4 / split;               // 16-token groups per stage and warp
  const int tpart = warp / row_warps;         // token part of this warp
  const int pg0 = tpart * pcount;             // its first 16-token group
  const int wrow = row_base + (warp % row_warps) * 16;  // this warp's first row
  const bool active = tpart < split;
  const int r0 = wrow + gid;                   // the lane's two rows
  const int r1 = r0 + 8;
  const bool v0 = r0 < row_end;
  const bool v1 = r1 < row_end;
  const int pos0 = first_pos + r0 / g;
  const int pos1 = first_pos + r1 / g;
  const int min_pos = first_pos + wrow / g;   // smallest position in the warp

  // Q rows as A fragments (row = query row, k = head dim), zero past the rows
  uint32_t qa[KD][4];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
    const int64_t b0 = v0 ? ((static_cast<int64_t>(q0) + r0 / g) * a.num_q_heads + kvh * g + r0 % g) * D : 0;
    const int64_t b1 = v1 ? ((static_cast<int64_t>(q0) + r1 / g) * a.num_q_heads + kvh * g + r1 % g) * D : 0;
#pragma unroll
    for (int kk = 0; kk < KD; ++kk) {
      const int d = kk * 16 + tig * 2;
      // E4M3: lane quad t takes dims 16kk + 4t .. + 3, the order the codes arrive in
      const int da = FP8 ? kk * 16 + tig * 4 : d;
      const int db = FP8 ? da + 2 : d + 8;
      qa[kk][0] = v0 ? __ldg(q32 + ((b0 + da) >> 1)) : 0u;
      qa[kk][1] = v1 ? __ldg(q32 + ((b1 + da) >> 1)) : 0u;
      qa[kk][2] = v0 ? __ldg(q32 + ((b0 + db) >> 1)) : 0u;
      qa[kk][3] = v1 ? __ldg(q32 + ((b1 + db) >> 1)) : 0u;
    }
  }
  // logit scale per row (log2 units); E4M3 with bf16 q: q rows become fp16
  // times 2^(13 - e), e the exponent of the row's largest magnitude
  float sl0 = a.scale_log2, sl1 = a.scale_log2;
  if constexpr (FP8 && IS_BF16) {
    float mx0 = 0.f, mx1 = 0.f;
#pragma unroll
    for (int kk = 0; kk < KD; ++kk) {
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const float2 f0 = unpack2<true>(qa[kk][i]);
        const float2 f1 = unpack2<true>(qa[kk][i + 1]);
        mx0 = fmaxf(mx0, fmaxf(fabsf(f0.x), fabsf(f0.y)));
        mx1 = fmaxf(mx1, fmaxf(fabsf(f1.x), fabsf(f1.y)));
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const int e0 = max(static_cast<int>((__float_as_uint(mx0) >> 23) & 0xFFu) - 127, -100);
    const int e1 = max(static_cast<int>((__float_as_uint(mx1) >> 23) & 0xFFu) - 127, -100);
    const float p0 = __uint_as_float(static_cast<uint32_t>(127 + 13 - e0) << 23);
    const float p1 = __uint_as_float(static_cast<uint32_t>(127 + 13 - e1) << 23);
#pragma unroll
    for (int kk = 0; kk < KD; ++kk) {
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const float2 f0 = unpack2<true>(qa[kk][i]);
        const float2 f1 = unpack2<true>(qa[kk][i + 1]);
        qa[kk][i] = pack2<false>(f0.x * p0, f0.y * p0);
        qa[kk][i + 1] = pack2<false>(f1.x * p1, f1.y * p1);
      }
    }
    sl0 *= __uint_as_float(static_cast<uint32_t>(127 - 13 + e0) << 23);
    sl1 *= __uint_as_float(static_cast<uint32_t>(127 - 13 + e1) << 23);
  }

  float o[ND][4];
#pragma unroll
  for (int n = 0; n < ND; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  bool aborted = false;

  for (int it = 0; it < n_stages; ++it) {
    const int slot = it % NS;
    const bool got = mbar_wait_bounded(full0 + 8 * slot, (it / NS) & 1, kLimitNs);
    if (__any_sync(0xffffffffu, !got)) {
      if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
      aborted = true;
      break;
    }
    const uint32_t kp = base + slot * S::kStage;
    const uint32_t vp = kp + S::kHalves * S::kPlane;
    const uint64_t vmask = masks[slot];
    const int t0 = it * kTok;
    if (vmask != ~0ull) {
      // Zero the V rows that hold no valid token. Every warp does it for
      // itself (the same zeros, so the warps need not wait for one another);
      // the slot is refilled only after all four have released it.
      uint8_t* vrow = sm + slot * S::kStage + S::kHalves * S::kPlane;
      for (int i = lane; i < kTok * S::kHalves * 8; i += 32) {
        const int r = i / (S::kHalves * 8);
        const int c = i - r * (S::kHalves * 8);
        if (!((vmask >> r) & 1ull))
          *reinterpret_cast<uint4*>(vrow + (c >> 3) * S::kPlane + r * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      __syncwarp();
    }

    if (active) {
      // ---- S = Q K^T over the stage's 64 tokens (8 n-tiles)
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      if constexpr (FP8) {
        // matrix j: tokens 16p + 8(j & 1) .. + 7 of 16-byte chunk kk + (j >> 1);
        // lane (gid, tig) gets codes 4tig .. 4tig + 3 of its token
#pragma unroll
        for (int kk = 0; kk < KD; kk += 2) {
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            if (p >= pcount) break;
            const int mi = lane >> 3;
            const int t = (pg0 + p) * 16 + ((mi & 1) << 3) + (lane & 7);
            uint32_t r[4];
            ldsm_x4(swz(kp, t, kk + (mi >> 1)), r);
            uint32_t b[4][2];
#pragma unroll
            for (int j = 0; j < 4; ++j) e4m3x4_to_f16(r[j], b[j][0], b[j][1]);
            mma16816<false>(sc[2 * p], qa[kk], b[0][0], b[0][1]);
            mma16816<false>(sc[2 * p + 1], qa[kk], b[1][0], b[1][1]);
            mma16816<false>(sc[2 * p], qa[kk + 1], b[2][0], b[2][1]);
            mma16816<false>(sc[2 * p + 1], qa[kk + 1], b[3][0], b[3][1]);
          }
        }
      } else {
#pragma unroll
        for (int kk = 0; kk < KD; ++kk) {
#pragma unroll
          for (int p = 0; p < 4; ++p) {  // tokens 16(pg0 + p) .. + 15
            if (p >= pcount) break;
            const int mi = lane >> 3;
            const int t = (pg0 + p) * 16 + ((mi >> 1) << 3) + (lane & 7);
            uint32_t r[4];
            ldsm_x4(swz(kp, t, kk * 2 + (mi & 1)), r);
            mma16816<IS_BF16>(sc[2 * p], qa[kk], r[0], r[1]);
            mma16816<IS_BF16>(sc[2 * p + 1], qa[kk], r[2], r[3]);
          }
        }
      }
      // ---- scale, mask, online softmax (log2 domain)
      const bool need_mask = (t0 + kTok - 1 > min_pos) || vmask != ~0ull;
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int tl = pg0 * 16 + n * 8 + tig * 2 + c;
          const int t = t0 + tl;
          float x0 = sc[n][c] * sl0;
          float x1 = sc[n][2 + c] * sl1;
          if (n >= 2 * pcount) {  // not this warp's tokens
            x0 = -INFINITY;
            x1 = -INFINITY;
          } else if (need_mask) {
            const bool ok = (vmask >> tl) & 1ull;
            x0 = (ok && t <= pos0) ? x0 : -INFINITY;
            x1 = (ok && t <= pos1) ? x1 : -INFINITY;
          }
          sc[n][c] = x0;
          sc[n][2 + c] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0);
      const float mn1 = fmaxf(m1, mx1);
      const float sub0 = mn0 == -INFINITY ? 0.f : mn0;  // a row with nothing seen yet
      const float sub1 = mn1 == -INFINITY ? 0.f : mn1;
      const float al0 = exp2f(m0 - sub0);
      const float al1 = exp2f(m1 - sub1);
      m0 = mn0;
      m1 = mn1;
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        sc[n][0] = exp2f(sc[n][0] - sub0);
        sc[n][1] = exp2f(sc[n][1] - sub0);
        sc[n][2] = exp2f(sc[n][2] - sub1);
        sc[n][3] = exp2f(sc[n][3] - sub1);
        ps0 += sc[n][0] + sc[n][1];
        ps1 += sc[n][2] + sc[n][3];
      }
      l0 = l0 * al0 + ps0;
      l1 = l1 * al1 + ps1;
#pragma unroll
      for (int n = 0; n < ND; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      // ---- O += P V, 16 tokens per k-step, P split into high and low parts
#pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        if (k2 >= pcount) break;
        uint32_t hi[4], lo[4];
        const float* pa = sc[2 * k2];
        const float* pb = sc[2 * k2 + 1];
        const float pv[4][2] = {{pa[0], pa[1]}, {pa[2], pa[3]}, {pb[0], pb[1]}, {pb[2], pb[3]}};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          hi[i] = pack2<MB>(pv[i][0], pv[i][1]);
          const float2 h = unpack2<MB>(hi[i]);
          lo[i] = pack2<MB>(pv[i][0] - h.x, pv[i][1] - h.y);
        }
        if constexpr (FP8) {
          // matrix j: tokens 16k2 + 8(j & 1) .. + 7 of 16-byte chunk c + (j >> 1);
          // lane (gid, tig) gets dims 16c + 2gid, + 1 of tokens 2tig, 2tig + 1
#pragma unroll
          for (int c = 0; c < D / 16; c += 2) {
            const int mi = lane >> 3;
            const int t = (pg0 + k2) * 16 + ((mi & 1) << 3) + (lane & 7);
            uint32_t r[4];
            ldsm_x4_trans(swz(vp, t, c + (mi >> 1)), r);
            uint32_t b[4][2];  // [matrix][dim + 0 / dim + 1]
#pragma unroll
            for (int j = 0; j < 4; ++j) e4m3x4_to_f16(prmt(r[j], r[j], 0x3120u), b[j][0], b[j][1]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {  // chunk c + h
#pragma unroll
              for (int e = 0; e < 2; ++e) {  // n-tile of dims 16(c + h) + 2n + e
                auto& acc = o[2 * (c + h) + e];
                mma16816<false>(acc, hi, b[2 * h][e], b[2 * h + 1][e]);
                mma16816<false>(acc, lo, b[2 * h][e], b[2 * h + 1][e]);
              }
            }
          }
        } else {
#pragma unroll
          for (int dn = 0; dn < D / 16; ++dn) {  // head-dim columns 16dn .. 16dn + 15
            const int mi = lane >> 3;
            const int t = (pg0 + k2) * 16 + ((mi & 1) << 3) + (lane & 7);
            uint32_t r[4];
            ldsm_x4_trans(swz(vp, t, dn * 2 + (mi >> 1)), r);
            mma16816<IS_BF16>(o[2 * dn], hi, r[0], r[1]);
            mma16816<IS_BF16>(o[2 * dn], lo, r[0], r[1]);
            mma16816<IS_BF16>(o[2 * dn + 1], hi, r[2], r[3]);
            mma16816<IS_BF16>(o[2 * dn + 1], lo, r[2], r[3]);
          }
        }
      }
    }
    // release the slot: this warp's reads of it are done
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * slot);
    if (warp == 0 && it + NS < n_stages) {
      // refill once every warp has released it
      const bool freed = mbar_wait_bounded(empty0 + 8 * slot, (it / NS) & 1, kLimitNs);
      if (__any_sync(0xffffffffu, !freed)) {
        if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
        aborted = true;
        break;
      }
      issue_prefill_stage<D, NS, FP8>(a, &tmk, &tmv, table_row, kvh, it + NS, max_pos, base, full0,
                                      masks, ids, lane);
      ++issued;
    }
  }
  if (warp == 0) {
    // copies still in flight land before the CTA can leave
    for (int j = (issued > NS ? issued - NS : 0); j < issued; ++j)
      mbar_wait_bounded(full0 + 8 * (j % NS), (j / NS) & 1, kLimitNs);
  }
  // ---- merge the token parts of a split row group (uniform across the CTA,
  // so every thread takes both barriers). The ring is free by now: the other
  // parts park (m, l, O) there, lane-major, and part 0 folds them in.
  if (split > 1) {
    constexpr int kF = 4 + ND * 4;  // floats of state per lane
    static_assert(kWarps * kF * 32 * 4 <= S::kBar, "the parked states fit in the ring");
    float* park = reinterpret_cast<float*>(sm);
    __syncthreads();  // every copy has landed and every warp is done with the ring
    if (tpart > 0) {
      float* my = park + warp * kF * 32 + lane;
      my[0] = m0;
      my[32] = m1;
      my[64] = l0;
      my[96] = l1;
#pragma unroll
      for (int n = 0; n < ND; ++n) {
#pragma unroll
        for (int e = 0; e < 4; ++e) my[(4 + n * 4 + e) * 32] = o[n][e];
      }
    }
    __syncthreads();
    if (tpart == 0) {
      for (int pt = 1; pt < split; ++pt) {
        const float* ot = park + (warp + pt * row_warps) * kF * 32 + lane;
        const float om0 = ot[0], om1 = ot[32];
        const float nm0 = fmaxf(m0, om0), nm1 = fmaxf(m1, om1);
        const float u0 = nm0 == -INFINITY ? 0.f : nm0;
        const float u1 = nm1 == -INFINITY ? 0.f : nm1;
        const float a0 = exp2f(m0 - u0), b0 = exp2f(om0 - u0);
        const float a1 = exp2f(m1 - u1), b1 = exp2f(om1 - u1);
        l0 = l0 * a0 + ot[64] * b0;
        l1 = l1 * a1 + ot[96] * b1;
#pragma unroll
        for (int n = 0; n < ND; ++n) {
          o[n][0] = o[n][0] * a0 + ot[(4 + n * 4 + 0) * 32] * b0;
          o[n][1] = o[n][1] * a0 + ot[(4 + n * 4 + 1) * 32] * b0;
          o[n][2] = o[n][2] * a1 + ot[(4 + n * 4 + 2) * 32] * b1;
          o[n][3] = o[n][3] * a1 + ot[(4 + n * 4 + 3) * 32] * b1;
        }
        m0 = nm0;
        m1 = nm1;
      }
    }
  }
  if (!active || tpart > 0 || aborted) return;

  // ---- normalise and store
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float vs = FP8 ? a.v_scale : 1.f;
  const float inv0 = l0 > 0.f ? vs / l0 : 0.f;
  const float inv1 = l1 > 0.f ? vs / l1 : 0.f;
  const int64_t ob0 = ((static_cast<int64_t>(q0) + r0 / g) * a.num_q_heads + kvh * g + r0 % g) * D;
  const int64_t ob1 = ((static_cast<int64_t>(q0) + r1 / g) * a.num_q_heads + kvh * g + r1 % g) * D;
#pragma unroll
  for (int n = 0; n < ND; ++n) {
    // 16-bit: columns 2tig, 2tig + 1 of n-tile n are dims 8n + 2tig, + 1; E4M3:
    // n-tile 2c + e holds dim 16c + 2col + e, so its columns are dims
    // 16c + 4tig + e and 16c + 4tig + 2 + e
    const int d = FP8 ? (n >> 1) * 16 + tig * 4 + (n & 1) : n * 8 + tig * 2;
    const int dd = FP8 ? 2 : 1;
    if (v0) {
      store_val(a, ob0 + d, o[n][0] * inv0);
      store_val(a, ob0 + d + dd, o[n][1] * inv0);
    }
    if (v1) {
      store_val(a, ob1 + d, o[n][2] * inv1);
      store_val(a, ob1 + d + dd, o[n][3] * inv1);
    }
  }
}

// THIN (head_dim 128, at most 32 rows per CTA): two stages instead of three
// and three CTAs per SM, the same bytes in flight per SM with half again as
// many warps to hide the latency.
template <bool IS_BF16, int D, bool FP8 = false, bool THIN = false>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a, dim3 grid,
                   cudaStream_t st) {
  constexpr int NS = (THIN ? 2 : prefill_stages<D>()) * (FP8 ? 2 : 1);  // same bytes per stage
  constexpr int MINB = THIN ? 3 : (D <= 128 ? 2 : 1);
  auto kern = prefill_kernel<IS_BF16, D, NS, FP8, MINB>;
  const int smem = static_cast<int>(PrefillSmem<D, NS, FP8>::kTotal);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kWarps * 32, smem, st>>>(tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                           int head_dim, bool bf16, bool fp8, bool thin, dim3 grid,
                           cudaStream_t st) {
  if (thin && head_dim == 128) {
    if (fp8) return bf16 ? launch<true, 128, true, true>(tk, tv, a, grid, st)
                         : launch<false, 128, true, true>(tk, tv, a, grid, st);
    return bf16 ? launch<true, 128, false, true>(tk, tv, a, grid, st)
                : launch<false, 128, false, true>(tk, tv, a, grid, st);
  }
  if (fp8) {  // E4M3 caches: head_dim 128 or 256
    if (head_dim == 128) return bf16 ? launch<true, 128, true>(tk, tv, a, grid, st)
                                     : launch<false, 128, true>(tk, tv, a, grid, st);
    if (head_dim == 256) return bf16 ? launch<true, 256, true>(tk, tv, a, grid, st)
                                     : launch<false, 256, true>(tk, tv, a, grid, st);
    return cudaErrorInvalidValue;
  }
  if (bf16) {
    return head_dim == 64 ? launch<true, 64>(tk, tv, a, grid, st)
           : head_dim == 128 ? launch<true, 128>(tk, tv, a, grid, st)
                             : launch<true, 256>(tk, tv, a, grid, st);
  }
  return head_dim == 64 ? launch<false, 64>(tk, tv, a, grid, st)
         : head_dim == 128 ? launch<false, 128>(tk, tv, a, grid, st)
                           : launch<false, 256>(tk, tv, a, grid, st);
}

}  // namespace pa
