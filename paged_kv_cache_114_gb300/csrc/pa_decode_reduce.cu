// pa_decode_reduce.cu - merge of split-K decode partials.
//
// Partition p of a sequence left (m_p, l_p, o_p): its largest logit (log2
// units), sum of 2^(x - m_p) and the unnormalised output. The merge is the
// rescale identity of the online softmax ("PagedAttention: Virtual-Memory KV
// Cache Management, ...", 3. Non-Contiguous Online Softmax Attention Kernel):
//   M = max_p m_p,  l = sum_p l_p 2^(m_p - M),  out = sum_p o_p 2^(m_p - M) / l,
// taken in partition order, so results are deterministic.
#include "pa_decode.cuh"

namespace pa {
namespace {

// One CTA per (sequence, query head), one thread per output element; rows the
// partition kernel finished itself (one partition) are skipped. Partition
// maxima and normalisers are broadcast loads; the partition loop is unrolled
// so the coalesced partial rows of several partitions are in flight at once.
__global__ void decode_reduce_kernel(const DecodeArgs a, int head_dim) {
  const int64_t sh = blockIdx.x;  // s * Hq + h
  const int s = static_cast<int>(sh / a.num_q_heads);
  const int L = decode_seq_len(a, s, false);
  const int nparts = (L + a.part_tokens - 1) / a.part_tokens;
  if (nparts <= 1) return;
  const int64_t base = sh * a.max_parts;
  const float* ml = a.part_ml + base * 2;
  float mmax = -INFINITY;
#pragma unroll 8
  for (int p = 0; p < nparts; ++p) mmax = fmaxf(mmax, __ldg(ml + 2 * p));
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    const float* po = a.part_o + base * head_dim + d;
    float acc = 0.f;
    float lsum = 0.f;
    if (mmax != -INFINITY) {
#pragma unroll 8
      for (int p = 0; p < nparts; ++p) {
        const float f = exp2f(__ldg(ml + 2 * p) - mmax);
        acc += __ldg(po + static_cast<int64_t>(p) * head_dim) * f;
        lsum += __ldg(ml + 2 * p + 1) * f;
      }
    }
    store_out(a, sh * head_dim + d, lsum > 0.f ? acc / lsum : 0.f);
  }
}

constexpr int kMergeThreads = 256;
constexpr int kMergeRangeRuns = 8;  // ranges one thread examines per pass

// Merge of the cut pieces decode_grouped_kernel leaves as partials. The
// equal-range split of the stage line (stage_tokens tokens a stage, as the
// stream kernel cut it) follows from the lengths alone, so the
// kernel finds the cut pieces before griddepcontrol.wait, while the stream
// kernel's last CTAs still run: it builds the stage prefix, and for each
// range r takes its last piece - the sequence s holding stage g1(r) - 1. That
// piece is cut and starts in r when pre[s] >= g0(r) and pre[s + 1] > g1(r);
// every cut piece is the last piece of the range it starts in, so this lists
// each exactly once (the same for every KV head). Its contributors are the
// non-empty ranges r .. rb, rb the owner of its last stage; range r'
// holds its partial in slot (r' * H_kv + kvh) * 2, + 1 for r itself when the
// piece does not start r (then it is r's last piece, not its first).
// Past the wait the (piece, KV head, R query rows) tasks are spread over every
// warp of the grid - cut pieces cluster in few ranges when sequences are
// long. A task loads the contributors' (m, l) (lane c holds contributor c)
// and the first CB contributors' output rows (D / 32 values per lane and row)
// together, branch-free, before it uses any of them - the weights are not
// needed to fetch the rows - so a piece of at most CB contributors costs one
// round trip. Pieces of a few contributors (many pieces): CB = 4 and R = 4
// (R = 1 below 4 query heads per KV head); long pieces (few pieces, many
// contributors): R = 1, CB = 32. Contributors go 32 at a time with the
// rescale identity between chunks; up to 32 it is the same arithmetic, in the
// same contributor order, as the last-arriver merge of the other balanced
// kernels.
template <int D, int R, int CB>
__global__ void __launch_bounds__(kMergeThreads, 1)
    decode_piece_merge_kernel(const DecodeArgs a, int64_t ranges, int stage_tokens) {
  constexpr int E = D / 32;
  constexpr int W = kMergeThreads / 32;
  extern __shared__ __align__(16) unsigned char merge_smem[];
  __shared__ int warp_tot[16];
  const int N = a.num_seqs;
  int32_t* pre = reinterpret_cast<int32_t*>(merge_smem);                    // [N + 1]
  int4* cut = reinterpret_cast<int4*>(merge_smem + ((N + 1) * 4 + 15) / 16 * 16);  // [ranges]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- before the wait: the cut pieces, from the lengths alone
  build_line_prefix(a, pre, stage_tokens, warp_tot, W);
  const int64_t stot = pre[N];
  int ncut = 0;
  for (int64_t r0 = 0; r0 < ranges; r0 += static_cast<int64_t>(kMergeThreads) * kMergeRangeRuns) {
    const int64_t left = ranges - r0;
    const int n = left < kMergeThreads * kMergeRangeRuns ? static_cast<int>(left)
                                                         : kMergeThreads * kMergeRangeRuns;
    const int run = (n + kMergeThreads - 1) / kMergeThreads;
    const int64_t i0 = r0 + static_cast<int64_t>(threadIdx.x) * run;
    int4 cv[kMergeRangeRuns];
    int mine = 0;
#pragma unroll
    for (int k = 0; k < kMergeRangeRuns; ++k) {
      cv[k] = make_int4(-1, 0, 0, 0);
      const int64_t r = i0 + k;
      if (k < run && r < r0 + n) {
        const int64_t g0 = range_start(r, stot, ranges);
        const int64_t g1 = range_start(r + 1, stot, ranges);
        if (g0 < g1) {
          int lo = 0;
          int hi = N - 1;  // the sequence holding stage g1 - 1
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= g1 - 1) lo = mid; else hi = mid - 1;
          }
          if (pre[lo] >= g0 && pre[lo + 1] > g1)
            cv[k] = make_int4(lo, static_cast<int>(stage_owner(pre[lo + 1] - 1, stot, ranges)),
                              pre[lo] == g0 ? 0 : 1, static_cast<int>(r));
        }
      }
      mine += cv[k].x >= 0 ? 1 : 0;
    }
    int incl = mine;  // inclusive scan over the warp, then over the warps
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int pos = ncut + incl - mine;
    int total = 0;
#pragma unroll
    for (int w2 = 0; w2 < W; ++w2) {
      pos += w2 < warp ? warp_tot[w2] : 0;
      total += warp_tot[w2];
    }
#pragma unroll
    for (int k = 0; k < kMergeRangeRuns; ++k)
      if (cv[k].x >= 0) cut[pos++] = cv[k];
    ncut += total;
    __syncthreads();  // the list is complete; warp_tot is rewritten next pass
  }

  // every partial of the stream kernel is written and visible past this point
  asm volatile("griddepcontrol.wait;" ::: "memory");

  // ---- tasks (valid piece, R rows), spread over all warps of the grid
  const int hkv = a.num_kv_heads;
  const int g = a.group;
  const int rgroups = (g + R - 1) / R;
  const int ntasks = ncut * hkv * rgroups;
  for (int t = warp * static_cast<int>(gridDim.x) + static_cast<int>(blockIdx.x); t < ntasks;
       t += static_cast<int>(gridDim.x) * W) {
    const int4 d = cut[t / (hkv * rgroups)];  // {sequence, last range, slot bit, first range}
    const int rest = t - (t / (hkv * rgroups)) * (hkv * rgroups);
    const int kvh = rest / rgroups;
    const int j0 = (rest - kvh * rgroups) * R;
    const int64_t ra = d.w;
    const int span = static_cast<int>(d.y - ra + 1);
    const int64_t first = (ra * hkv + kvh) * 2 + d.z;  // range ra's partial of the piece
    float M[R];
    float L[R];
    float acc[R][E];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      M[r] = -INFINITY;
      L[r] = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    }
    for (int c0 = 0; c0 < span; c0 += 32) {
      const int64_t rr = ra + c0 + lane;
      int sid = -1;
      if (c0 + lane < span && range_start(rr, stot, ranges) < range_start(rr + 1, stot, ranges))
        sid = static_cast<int>((rr * hkv + kvh) * 2 + (c0 + lane == 0 ? d.z : 0));
      // Loads are branch-free so that all of them are in flight together: a
      // contributor or row without a partial reads the first contributor's
      // row j0 (this task's own data, always written), and its weight 0
      // selects the value away.
      float2 ml[R];
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const bool use = sid >= 0 && j0 + r < g;
        ml[r] = __ldcg(reinterpret_cast<const float2*>(a.part_ml) +
                       (use ? static_cast<int64_t>(sid) * g + j0 + r : first * g + j0));
      }
      const int nch = span - c0 < 32 ? span - c0 : 32;
      float w[R];
      for (int b0 = 0; b0 < nch; b0 += CB) {
        float v[CB][R][E];
#pragma unroll
        for (int c = 0; c < CB; ++c) {
          const int sc = __shfl_sync(0xffffffffu, sid, (b0 + c) & 31);
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const bool use = b0 + c < nch && sc >= 0 && j0 + r < g;
            ldcg_vec<E>(a.part_o + (use ? static_cast<int64_t>(sc) * g + j0 + r : first * g + j0) * D +
                            lane * E,
                        v[c][r]);
          }
        }
        if (b0 == 0) {  // the chunk's weights, while its rows are in flight
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const bool use = sid >= 0 && j0 + r < g;
            const float m = use ? ml[r].x : -INFINITY;
            ml[r].y = use ? ml[r].y : 0.f;
            const float mnew = fmaxf(M[r], warp_max(m));
            // what earlier chunks summed, rescaled to the new maximum (0 when
            // nothing came before; a row with no logit yet keeps zeros)
            const float alpha = M[r] == -INFINITY ? 0.f : exp2f(M[r] - mnew);
            w[r] = m == -INFINITY ? 0.f : exp2f(m - mnew);
            L[r] = L[r] * alpha + warp_sum(w[r] * ml[r].y);
#pragma unroll
            for (int e = 0; e < E; ++e) acc[r][e] *= alpha;
            M[r] = mnew;
          }
        }
#pragma unroll
        for (int c = 0; c < CB; ++c) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const float wc = __shfl_sync(0xffffffffu, w[r], (b0 + c) & 31);
            if (b0 + c < nch) {
#pragma unroll
              for (int e = 0; e < E; ++e) acc[r][e] += wc != 0.f ? v[c][r][e] * wc : 0.f;
            }
          }
        }
      }
    }
    const int64_t row0 = static_cast<int64_t>(d.x) * a.num_q_heads + static_cast<int64_t>(kvh) * g + j0;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      if (j0 + r >= g) break;
#pragma unroll
      for (int e = 0; e < E; ++e)
        store_out(a, (row0 + r) * D + lane * E + e, L[r] > 0.f ? acc[r][e] / L[r] : 0.f);
    }
  }
}

template <int D, int R, int CB>
cudaError_t launch_merge(const DecodeArgs& a, int64_t ranges, int stage_tokens, int sms,
                         cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(sms), 1, 1);  // one CTA per SM
  cfg.blockDim = dim3(kMergeThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(a.num_seqs + 1 + 3) / 4 * 16 +
                         static_cast<size_t>(ranges) * sizeof(int4);
  cfg.stream = st;
  // a programmatic dependent of the stream kernel: it is scheduled while that
  // kernel runs and waits for it in griddepcontrol.wait
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto kern = decode_piece_merge_kernel<D, R, CB>;
  if (cfg.dynamicSmemBytes > 48 * 1024) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(cfg.dynamicSmemBytes));
    if (e != cudaSuccess) return e;
  }
  return cudaLaunchKernelEx(&cfg, kern, a, ranges, stage_tokens);
}

template <int D>
cudaError_t launch_merge_for(const DecodeArgs& a, int64_t ranges, int stage_tokens, int sms,
                             cudaStream_t st) {
  constexpr int E = D / 32;
  // a piece spans about ranges / N + 1 ranges when the lengths are alike
  if (ranges >= 4LL * a.num_seqs)
    return launch_merge<D, 1, (E > 4 ? 16 : 32)>(a, ranges, stage_tokens, sms, st);
  if (a.group < 4) return launch_merge<D, 1, (E > 4 ? 2 : 4)>(a, ranges, stage_tokens, sms, st);
  return launch_merge<D, 4, (E > 4 ? 2 : 4)>(a, ranges, stage_tokens, sms, st);
}

}  // namespace

cudaError_t launch_decode_piece_merge(const DecodeArgs& a, int head_dim, int64_t ranges,
                                      int stage_tokens, int sms, cudaStream_t st) {
  switch (head_dim) {
    case 64: return launch_merge_for<64>(a, ranges, stage_tokens, sms, st);
    case 128: return launch_merge_for<128>(a, ranges, stage_tokens, sms, st);
    case 256: return launch_merge_for<256>(a, ranges, stage_tokens, sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(a.num_seqs) * a.num_q_heads);
  decode_reduce_kernel<<<blocks, head_dim < 256 ? head_dim : 256, 0, st>>>(a, head_dim);
  return cudaGetLastError();
}

}  // namespace pa
