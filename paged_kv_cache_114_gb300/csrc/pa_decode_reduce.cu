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

__global__ void decode_reduce_kernel(const DecodeArgs a, int head_dim) {
  const int64_t sh = blockIdx.x;  // s * Hq + h
  const int s = static_cast<int>(sh / a.num_q_heads);
  const int L = decode_seq_len(a, s, false);
  const int nparts = (L + a.part_tokens - 1) / a.part_tokens;
  if (nparts <= 1) return;  // the partition kernel wrote this row already
  const int64_t base = sh * a.max_parts;
  float mmax = -INFINITY;
  for (int p = 0; p < nparts; ++p) mmax = fmaxf(mmax, a.part_ml[(base + p) * 2]);
  for (int d = threadIdx.x; d < head_dim; d += blockDim.x) {
    float acc = 0.f;
    float lsum = 0.f;
    if (mmax != -INFINITY) {
      for (int p = 0; p < nparts; ++p) {
        const float f = exp2f(a.part_ml[(base + p) * 2] - mmax);
        acc += a.part_o[(base + p) * head_dim + d] * f;
        lsum += a.part_ml[(base + p) * 2 + 1] * f;
      }
    }
    store_out(a, sh * head_dim + d, lsum > 0.f ? acc / lsum : 0.f);
  }
}

}  // namespace

cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t st) {
  const unsigned blocks = static_cast<unsigned>(static_cast<int64_t>(a.num_seqs) * a.num_q_heads);
  decode_reduce_kernel<<<blocks, head_dim < 128 ? head_dim : 128, 0, st>>>(a, head_dim);
  return cudaGetLastError();
}

}  // namespace pa
