// pa_decode.cuh - paged decode attention for sm_103a.
//
// Computes, for one sequence s and one KV head, the g query heads
//   out[s][h] = sum_t softmax_t(scale * q[s][h] . K[t]) V[t],   t < L_s,
// reading K[t], V[t] through the block table (logical block t / b, row t % b)
// and accumulating block by block with a running maximum m, normaliser l and
// unnormalised output o ("PagedAttention: Virtual-Memory KV Cache Management,
// ...", 3. Non-Contiguous Online Softmax Attention Kernel).
//
// Design (one CTA = one (sequence, KV head, partition)):
//  * 4 warps; each warp owns a private ring of NS shared-memory stages. A stage
//    is 16 token rows of K and of V for this KV head, loaded by TMA tensor
//    copies straight from the scattered pool blocks (box = 64 head-dim
//    elements x 1 head x up to 16 tokens x 1 block, 128-byte swizzle). Lane j
//    issues the copies of the j-th block piece of the stage, so block-table
//    lookups and copy issue are spread over the warp. Warps take stages
//    round-robin, so the CTA streams consecutive tokens.
//  * QK^T and PV run on mma.sync m16n8k16 with fp32 accumulation, in the
//    transposed orientation S^T = K Q^T (M = 16 tokens, N = 8 query heads of
//    the group, K = head_dim) and O^T = V^T P^T (M = 16 head-dim rows, N = 8
//    heads, K = 16 tokens). The group's heads fill N, so each K/V row is read
//    once per KV head whatever g is. P^T reaches the B-operand layout with
//    movmatrix; P is split into a 16-bit high and low part so the PV product
//    keeps ~16 bits of the fp32 weights.
//  * Softmax state per head lives in registers; warps merge at the end through
//    shared memory with the rescale identity, then the CTA writes either the
//    normalised output (one partition) or (m, l, o) partials for the reduce.
//  * Slots past the length, pieces of blocks whose id is out of range and the
//    padding rows of blocks smaller than 8 tokens are masked: their logits are
//    -inf and their V rows are zeroed in shared memory before PV, so stale or
//    NaN bytes in the pool never enter the result.
#pragma once

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per bounded wait

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

__device__ __forceinline__ void store_out(const DecodeArgs& a, int64_t idx, float v) {
  if (a.out_dtype == PA_F32) {
    static_cast<float*>(a.out)[idx] = v;
  } else if (a.out_dtype == PA_BF16) {
    static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
  } else {
    static_cast<__half*>(a.out)[idx] = __float2half_rn(v);
  }
}

template <int D, int NT, int NS>
struct DecodeSmem {
  static constexpr int kHalves = D / 64;                  // 128-byte column pieces of a row
  static constexpr int kHalfBytes = kStageRows * 128;     // one piece of 16 rows
  static constexpr int kStageBytes = 2 * kHalves * kHalfBytes;  // K then V
  static constexpr int kRingBytes = kDecodeWarps * NS * kStageBytes;
  static constexpr int kCombineBytes = kDecodeWarps * NT * 8 * (D + 2) * 4;
  static constexpr int kDataBytes = kRingBytes > kCombineBytes ? kRingBytes : kCombineBytes;
  static constexpr int kBarOffset = kDataBytes;
  static constexpr int kMaskOffset = kBarOffset + kDecodeWarps * NS * 8;
  static constexpr int kTotal = kMaskOffset + kDecodeWarps * NS * 4 + 1024;  // + alignment slack
};

template <bool IS_BF16, int D, int NT, int NS, bool SPLIT_P>
__global__ void __launch_bounds__(kDecodeWarps * 32)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  using S = DecodeSmem<D, NT, NS>;
  constexpr int W = kDecodeWarps;
  constexpr int TS = kStageRows;
  constexpr int KD = D / 16;
  constexpr int HALVES = S::kHalves;
  constexpr int HB = S::kHalfBytes;
  constexpr uint32_t kAllRows = (1u << TS) - 1u;
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
  uint32_t* masks = reinterpret_cast<uint32_t*>(sm + S::kMaskOffset);

  const int tt = a.ops_per_stage * a.tok_per_op;  // tokens per stage
  const int nst = (ntok + tt - 1) / tt;
  const int my_n = nst > warp ? (nst - warp - 1) / W + 1 : 0;

  // q as the B operand of S^T = K Q^T: k = head-dim index, n = head in tile.
  uint32_t qb[NT][KD][2];
  {
    const uint32_t* q32 = static_cast<const uint32_t*>(a.q);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int head = nt * 8 + gid;
      const bool live = head < a.group;
      const int64_t row =
          (static_cast<int64_t>(s) * a.num_q_heads + static_cast<int64_t>(kvh) * a.group + head) * D;
#pragma unroll
      for (int kk = 0; kk < KD; ++kk) {
        qb[nt][kk][0] = live ? __ldg(q32 + ((row + kk * 16 + tig * 2) >> 1)) : 0u;
        qb[nt][kk][1] = live ? __ldg(q32 + ((row + kk * 16 + 8 + tig * 2) >> 1)) : 0u;
      }
    }
  }

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

  // Issue the TMA copies of this warp's it-th stage into slot it % NS.
  auto issue = [&](int it) {
    const int slot = it % NS;
    const int t0 = tok_begin + (warp + it * W) * tt;
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
    if (lane < TS) {
      const int jr = lane / a.slot_rows;
      const int o = lane - jr * a.slot_rows;
      const int tok = t0 + jr * a.tok_per_op + o;
      rv = o < a.tok_per_op && tok < tok_end && ((okmask >> jr) & 1u);
    }
    const uint32_t rowmask = __ballot_sync(0xffffffffu, rv) & kAllRows;
    const uint32_t bar = bar0 + 8 * slot;
    if (lane == 0) {
      masks[warp * NS + slot] = rowmask;
      mbar_arrive_expect_tx(bar, static_cast<uint32_t>(__popc(okmask)) * a.tok_per_op * D * 4u);
    }
    __syncwarp();
    if (ok) {
      const uint32_t dk = ring + slot * S::kStageBytes + lane * a.slot_rows * 128;
      const uint32_t dv = dk + HALVES * HB;
#pragma unroll
      for (int c = 0; c < HALVES; ++c) {
        tma_load_4d(dk + c * HB, &tmk, bar, c * 64, kvh, off, blk);
        tma_load_4d(dv + c * HB, &tmv, bar, c * 64, kvh, off, blk);
      }
    }
  };

  float m_run[NT][2];
  float l_run[NT][2];
  float o[KD][NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -INFINITY;
    l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
    for (int dm = 0; dm < KD; ++dm) o[dm][nt][0] = o[dm][nt][1] = o[dm][nt][2] = o[dm][nt][3] = 0.f;
  }

  const int pro = my_n < NS ? my_n : NS;
  for (int i = 0; i < pro; ++i) issue(i);

  bool aborted = false;
  int it = 0;
  for (; it < my_n; ++it) {
    const int slot = it % NS;
    const bool got = mbar_wait_bounded(bar0 + 8 * slot, (it / NS) & 1, kWaitLimitNs);
    if (__any_sync(0xffffffffu, !got)) {
      aborted = true;
      break;
    }
    const uint32_t kb = ring + slot * S::kStageBytes;
    const uint32_t vb = kb + HALVES * HB;
    const uint32_t rowmask = masks[warp * NS + slot];

    if (rowmask != kAllRows) {  // zero V rows that must not contribute
      uint8_t* vp = ring_ptr + slot * S::kStageBytes + HALVES * HB;
      for (int idx = lane; idx < TS * HALVES * 8; idx += 32) {
        const int row = idx / (HALVES * 8);
        const int rem = idx - row * (HALVES * 8);
        if (!((rowmask >> row) & 1u)) {
          *reinterpret_cast<uint4*>(vp + (rem >> 3) * HB + row * 128 + (rem & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
      }
      __syncwarp();
    }

    // S^T = K Q^T over head_dim.
    float sacc[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    {
      const int i = lane >> 3;
      const int row = ((i & 1) << 3) + (lane & 7);
#pragma unroll
      for (int kk = 0; kk < KD; ++kk) {
        const int chunk = ((kk & 3) << 1) + (i >> 1);
        uint32_t af[4];
        ldsm_x4(kb + (kk >> 2) * HB + row * 128 + ((chunk ^ (row & 7)) << 4), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816<IS_BF16>(sacc[nt], af, qb[nt][kk][0], qb[nt][kk][1]);
      }
    }

    // Online softmax update (log2 domain).
    const bool v0 = (rowmask >> gid) & 1u;
    const bool v1 = (rowmask >> (gid + 8)) & 1u;
    float p[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      float x[4];
      x[0] = v0 ? sacc[nt][0] * a.scale_log2 : -INFINITY;
      x[1] = v0 ? sacc[nt][1] * a.scale_log2 : -INFINITY;
      x[2] = v1 ? sacc[nt][2] * a.scale_log2 : -INFINITY;
      x[3] = v1 ? sacc[nt][3] * a.scale_log2 : -INFINITY;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float mx = fmaxf(x[c], x[c + 2]);
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float m_new = fmaxf(m_run[nt][c], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m_run[nt][c] - m_use);
        m_run[nt][c] = m_new;
        p[nt][c] = exp2f(x[c] - m_use);
        p[nt][c + 2] = exp2f(x[c + 2] - m_use);
        l_run[nt][c] = l_run[nt][c] * alpha + p[nt][c] + p[nt][c + 2];
#pragma unroll
        for (int dm = 0; dm < KD; ++dm) {
          o[dm][nt][c] *= alpha;
          o[dm][nt][c + 2] *= alpha;
        }
      }
    }

    // P^T as the B operand (k = token, n = head): transpose the 8x8 halves.
    uint32_t bh[NT][2];
    uint32_t bl[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const uint32_t h01 = pack2<IS_BF16>(p[nt][0], p[nt][1]);
      const uint32_t h23 = pack2<IS_BF16>(p[nt][2], p[nt][3]);
      bh[nt][0] = movmatrix_trans(h01);
      bh[nt][1] = movmatrix_trans(h23);
      if constexpr (SPLIT_P) {
        const float2 f01 = unpack2<IS_BF16>(h01);
        const float2 f23 = unpack2<IS_BF16>(h23);
        bl[nt][0] = movmatrix_trans(pack2<IS_BF16>(p[nt][0] - f01.x, p[nt][1] - f01.y));
        bl[nt][1] = movmatrix_trans(pack2<IS_BF16>(p[nt][2] - f23.x, p[nt][3] - f23.y));
      }
    }

    // O^T += V^T P^T over the 16 tokens of the stage.
    {
      const int i = lane >> 3;
      const int row = ((i >> 1) << 3) + (lane & 7);
#pragma unroll
      for (int dm = 0; dm < KD; ++dm) {
        const int chunk = ((dm & 3) << 1) + (i & 1);
        uint32_t af[4];
        ldsm_x4_trans(vb + (dm >> 2) * HB + row * 128 + ((chunk ^ (row & 7)) << 4), af);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          mma16816<IS_BF16>(o[dm][nt], af, bh[nt][0], bh[nt][1]);
          if constexpr (SPLIT_P) mma16816<IS_BF16>(o[dm][nt], af, bl[nt][0], bl[nt][1]);
        }
      }
    }

    fence_proxy_async_smem();  // our generic reads/writes of this slot precede the next TMA into it
    __syncwarp();
    if (it + NS < my_n) issue(it + NS);
  }

  if (aborted) {
    if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    const int last = (it + NS < my_n) ? it + NS : my_n;
    for (int j = it; j < last; ++j) mbar_wait_bounded(bar0 + 8 * (j % NS), (j / NS) & 1, kWaitLimitNs);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int dm = 0; dm < KD; ++dm) o[dm][nt][0] = o[dm][nt][1] = o[dm][nt][2] = o[dm][nt][3] = 0.f;
    }
  }

  // Per-head normaliser: sum the 8 lanes that share a head column.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float v = l_run[nt][c];
      v += __shfl_xor_sync(0xffffffffu, v, 4);
      v += __shfl_xor_sync(0xffffffffu, v, 8);
      v += __shfl_xor_sync(0xffffffffu, v, 16);
      l_run[nt][c] = v;
    }
  }

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
        const int d = dm * 16 + gid + ((r >> 1) << 3);
        const int col = nt * 8 + tig * 2 + (r & 1);
        c_o[(warp * COLS + col) * D + d] = o[dm][nt][r];
      }
    }
  }
  if (gid == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int col = nt * 8 + tig * 2 + c;
        c_m[warp * COLS + col] = m_run[nt][c];
        c_l[warp * COLS + col] = l_run[nt][c];
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
    float acc = 0.f;
    float lsum = 0.f;
    if (mmax != -INFINITY) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float f = exp2f(c_m[w * COLS + col] - mmax);
        acc += c_o[(w * COLS + col) * D + d] * f;
        lsum += c_l[w * COLS + col] * f;
      }
    }
    const int64_t head = static_cast<int64_t>(kvh) * a.group + col;
    const int64_t sh = static_cast<int64_t>(s) * a.num_q_heads + head;
    if (direct) {
      store_out(a, sh * D + d, lsum > 0.f ? acc / lsum : 0.f);
    } else {
      const int64_t pidx = sh * a.max_parts + part;
      a.part_o[pidx * D + d] = acc;
      if (d == 0) {
        a.part_ml[pidx * 2] = mmax;
        a.part_ml[pidx * 2 + 1] = lsum;
      }
    }
  }
}

// Stages per warp: keeps 2 CTAs (8 warps) resident per SM for D <= 128.
template <int D>
constexpr int decode_stages() {
  return D == 64 ? 6 : (D == 128 ? 3 : 2);
}

template <bool IS_BF16, int D, int NT>
cudaError_t launch_decode_tiles(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                dim3 grid, cudaStream_t st) {
  constexpr int NS = decode_stages<D>();
  using S = DecodeSmem<D, NT, NS>;
  auto kern = decode_kernel<IS_BF16, D, NT, NS, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kTotal);
  if (e != cudaSuccess) return e;
  kern<<<grid, kDecodeWarps * 32, S::kTotal, st>>>(tk, tv, a);
  return cudaGetLastError();
}

template <bool IS_BF16, int D>
cudaError_t launch_decode_dispatch(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                   int group_tiles, dim3 grid, cudaStream_t st) {
  if (group_tiles == 1) return launch_decode_tiles<IS_BF16, D, 1>(tk, tv, a, grid, st);
  if (group_tiles == 2) return launch_decode_tiles<IS_BF16, D, 2>(tk, tv, a, grid, st);
  return cudaErrorInvalidValue;
}

}  // namespace pa
