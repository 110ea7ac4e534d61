// pa_cache_ops.cu - slot mapping, slot-mapped KV write and block copy.
//
// All three are integer indexing plus byte movement; results are bit-exact.
// Out-of-range indices never fault: the row is skipped and a bit is OR-ed
// into the device error word.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// slot = table[s][t / b] * b + t % b  (logical block floor(t/B), offset t mod B;
// "PagedAttention: Virtual-Memory KV Cache Management, ...", 1. Paged Virtual
// Memory Mapping).
__global__ void slot_mapping_kernel(const int32_t* __restrict__ tables, int32_t num_seqs,
                                    int32_t max_blocks, const int32_t* __restrict__ seq_idx,
                                    const int32_t* __restrict__ positions, int64_t num_tokens,
                                    int32_t block_size, int64_t num_blocks,
                                    int64_t* __restrict__ slots, int* err) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= num_tokens) return;
  const int32_t s = seq_idx[i];
  const int32_t t = positions[i];
  int64_t slot = -1;
  if (s < 0 || s >= num_seqs || t < 0 || t / block_size >= max_blocks) {
    atomicOr(err, PA_DEVERR_POSITION);
  } else {
    const int32_t blk = tables[static_cast<int64_t>(s) * max_blocks + t / block_size];
    if (blk < 0 || blk >= num_blocks) {
      atomicOr(err, PA_DEVERR_BLOCK_ID);
    } else {
      slot = static_cast<int64_t>(blk) * block_size + t % block_size;
    }
  }
  slots[i] = slot;
}

// One CTA per token: the token's K row and V row (H_kv * D elements each, one
// contiguous run on both sides) move as 16-byte vectors.
__global__ void write_kv_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                const int64_t* __restrict__ slots, uint4* __restrict__ k_cache,
                                uint4* __restrict__ v_cache, int64_t num_slots,
                                int64_t row_vecs, int* err) {
  const int64_t tok = blockIdx.x;
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) {
    if (slot != -1 && threadIdx.x == 0) atomicOr(err, PA_DEVERR_SLOT);
    return;
  }
  const uint4* ks = key + tok * row_vecs;
  const uint4* vs = value + tok * row_vecs;
  uint4* kd = k_cache + slot * row_vecs;
  uint4* vd = v_cache + slot * row_vecs;
  for (int64_t c = threadIdx.x; c < row_vecs; c += blockDim.x) {
    const uint4 kx = __ldg(ks + c);
    const uint4 vx = __ldg(vs + c);
    kd[c] = kx;
    vd[c] = vx;
  }
}

// E4M3 caches: one CTA per token quantises its K and V rows (H_kv * D fp16 or
// bf16 values) to codes e4m3(x / scale) - the quotient rounded once to float32
// (IEEE division), then to the nearest code, ties to even, saturating at +-448 -
// and stores them at the slot; 8 values per thread and step (16-byte loads,
// 8-byte stores). This is the "FP8 cache" of "PagedAttention: paging the KV
// cache" (Fine-tuned models and adapters) read as E4M3 with per-layer scales.
template <bool IS_BF16>
__device__ __forceinline__ uint2 quantize8(const uint4 x, float scale) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
  uint32_t out[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float2 a = unpack2<IS_BF16>(w[2 * i]);
    const float2 b = unpack2<IS_BF16>(w[2 * i + 1]);
    const uint32_t lo = e4m3x2_encode(__fdiv_rn(a.x, scale), __fdiv_rn(a.y, scale));
    const uint32_t hi = e4m3x2_encode(__fdiv_rn(b.x, scale), __fdiv_rn(b.y, scale));
    out[i] = lo | (hi << 16);
  }
  return make_uint2(out[0], out[1]);
}

template <bool IS_BF16>
__global__ void write_kv_e4m3_kernel(const uint4* __restrict__ key, const uint4* __restrict__ value,
                                     const int64_t* __restrict__ slots, uint2* __restrict__ k_cache,
                                     uint2* __restrict__ v_cache, int64_t num_slots,
                                     int64_t row_vecs, float k_scale, float v_scale, int* err) {
  const int64_t tok = blockIdx.x;
  const int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) {
    if (slot != -1 && threadIdx.x == 0) atomicOr(err, PA_DEVERR_SLOT);
    return;
  }
  const uint4* ks = key + tok * row_vecs;
  const uint4* vs = value + tok * row_vecs;
  uint2* kd = k_cache + slot * row_vecs;
  uint2* vd = v_cache + slot * row_vecs;
  for (int64_t c = threadIdx.x; c < row_vecs; c += blockDim.x) {
    const uint4 kx = __ldg(ks + c);
    const uint4 vx = __ldg(vs + c);
    kd[c] = quantize8<IS_BF16>(kx, k_scale);
    vd[c] = quantize8<IS_BF16>(vx, v_scale);
  }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
constexpr int64_t kCopyPieceVecs = kCopyThreads * kCopyUnroll;  // 16 KiB per CTA

// grid.x = pair * pieces + piece, grid.y = layer * 2 + (0: K, 1: V).
__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(const CopyLayers layers, const int64_t* __restrict__ pairs,
                       int64_t num_blocks, int64_t block_vecs, int64_t pieces, int* err) {
  const int64_t pair = blockIdx.x / pieces;
  const int64_t piece = blockIdx.x - pair * pieces;
  const int64_t src = pairs[2 * pair];
  const int64_t dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && piece == 0 && blockIdx.y == 0) atomicOr(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  const int layer = blockIdx.y >> 1;
  uint4* base = static_cast<uint4*>((blockIdx.y & 1) ? layers.v[layer] : layers.k[layer]);
  const uint4* from = base + src * block_vecs + piece * kCopyPieceVecs;
  uint4* to = base + dst * block_vecs + piece * kCopyPieceVecs;
  const int64_t n = min(kCopyPieceVecs, block_vecs - piece * kCopyPieceVecs);
  uint4 buf[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(u) * kCopyThreads;
    if (c < n) buf[u] = from[c];
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(u) * kCopyThreads;
    if (c < n) to[c] = buf[u];
  }
}

// Swap for preemption: block src of one pool -> block dst of another, for
// every pair, layer, K and V ("PagedAttention: paging the KV cache", When
// memory runs out: swapping copies the evicted blocks to CPU memory and back).
// On GB300 the host pool is Grace memory that the SMs read and write directly
// over NVLink-C2C through the unified address space, so one launch gathers or
// scatters any set of scattered blocks. A CTA moves a 32 KiB piece with 8
// 16-byte vectors per thread in flight, enough to cover the link's latency.
constexpr int kSwapUnroll = 8;
constexpr int64_t kSwapPieceVecs = kCopyThreads * kSwapUnroll;  // 32 KiB per CTA

// grid.x = pair * pieces + piece, grid.y = layer * 2 + (0: K, 1: V).
__global__ void __launch_bounds__(kCopyThreads)
    swap_blocks_kernel(const SwapLayers layers, const int64_t* __restrict__ pairs,
                       int64_t src_blocks, int64_t dst_blocks, int64_t block_vecs, int64_t pieces,
                       int* err) {
  const int64_t pair = blockIdx.x / pieces;
  const int64_t piece = blockIdx.x - pair * pieces;
  const int64_t src = pairs[2 * pair];
  const int64_t dst = pairs[2 * pair + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && piece == 0 && blockIdx.y == 0) atomicOr(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  const int layer = blockIdx.y >> 1;
  const bool is_v = blockIdx.y & 1;
  const uint4* from = static_cast<const uint4*>(is_v ? layers.src_v[layer] : layers.src_k[layer]) +
                      src * block_vecs + piece * kSwapPieceVecs;
  uint4* to = static_cast<uint4*>(is_v ? layers.dst_v[layer] : layers.dst_k[layer]) +
              dst * block_vecs + piece * kSwapPieceVecs;
  const int64_t n = min(kSwapPieceVecs, block_vecs - piece * kSwapPieceVecs);
  uint4 buf[kSwapUnroll];
#pragma unroll
  for (int u = 0; u < kSwapUnroll; ++u) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(u) * kCopyThreads;
    if (c < n) buf[u] = from[c];
  }
#pragma unroll
  for (int u = 0; u < kSwapUnroll; ++u) {
    const int64_t c = threadIdx.x + static_cast<int64_t>(u) * kCopyThreads;
    if (c < n) to[c] = buf[u];
  }
}

}  // namespace

cudaError_t launch_swap_blocks(const SwapLayers& layers, int32_t num_layers, const int64_t* pairs,
                               int64_t num_pairs, int64_t src_blocks, int64_t dst_blocks,
                               int64_t block_bytes, int* err, cudaStream_t st) {
  const int64_t block_vecs = block_bytes / 16;
  const int64_t pieces = (block_vecs + kSwapPieceVecs - 1) / kSwapPieceVecs;
  dim3 grid(static_cast<unsigned>(num_pairs * pieces), static_cast<unsigned>(2 * num_layers));
  swap_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(layers, pairs, src_blocks, dst_blocks,
                                                    block_vecs, pieces, err);
  return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                                const int32_t* seq_idx, const int32_t* positions, int64_t num_tokens,
                                int32_t block_size, int64_t num_blocks, int64_t* slots, int* err,
                                cudaStream_t st) {
  const int threads = 256;
  const int64_t blocks = (num_tokens + threads - 1) / threads;
  slot_mapping_kernel<<<static_cast<unsigned>(blocks), threads, 0, st>>>(
      block_tables, num_seqs, max_blocks, seq_idx, positions, num_tokens, block_size, num_blocks,
      slots, err);
  return cudaGetLastError();
}

cudaError_t launch_write_kv(const void* key, const void* value, const int64_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                            int32_t block_size, int64_t row_bytes, int* err, cudaStream_t st) {
  const int64_t row_vecs = row_bytes / 16;
  int threads = static_cast<int>(row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256);
  write_kv_kernel<<<static_cast<unsigned>(num_tokens), threads, 0, st>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), slots,
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), num_blocks * block_size,
      row_vecs, err);
  return cudaGetLastError();
}

cudaError_t launch_write_kv_e4m3(const void* key, const void* value, bool bf16,
                                 const int64_t* slots, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_blocks, int32_t block_size,
                                 int64_t row_elems, float k_scale, float v_scale, int* err,
                                 cudaStream_t st) {
  const int64_t row_vecs = row_elems / 8;
  const int threads = static_cast<int>(row_vecs < 256 ? ((row_vecs + 31) / 32) * 32 : 256);
  auto kern = bf16 ? write_kv_e4m3_kernel<true> : write_kv_e4m3_kernel<false>;
  kern<<<static_cast<unsigned>(num_tokens), threads, 0, st>>>(
      static_cast<const uint4*>(key), static_cast<const uint4*>(value), slots,
      static_cast<uint2*>(k_cache), static_cast<uint2*>(v_cache), num_blocks * block_size,
      row_vecs, k_scale, v_scale, err);
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const CopyLayers& layers, int32_t num_layers,
                               const int64_t* pairs, int64_t num_pairs, int64_t num_blocks,
                               int64_t block_bytes, int* err, cudaStream_t st) {
  const int64_t block_vecs = block_bytes / 16;
  const int64_t pieces = (block_vecs + kCopyPieceVecs - 1) / kCopyPieceVecs;
  dim3 grid(static_cast<unsigned>(num_pairs * pieces), static_cast<unsigned>(2 * num_layers));
  copy_blocks_kernel<<<grid, kCopyThreads, 0, st>>>(layers, pairs, num_blocks, block_vecs, pieces,
                                                    err);
  return cudaGetLastError();
}

}  // namespace pa
