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

}  // namespace

cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(a.num_seqs) * a.num_q_heads);
  decode_reduce_kernel<<<blocks, head_dim < 256 ? head_dim : 256, 0, st>>>(a, head_dim);
  return cudaGetLastError();
}

}  // namespace pa
