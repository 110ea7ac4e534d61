// pa_internal.h - host-side launchers shared between the translation units of
// libpagedkv. Not part of the public ABI (include/pa.h is).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"  // from include/, on the compiler include path

namespace pa {

// Kernel arguments of the decode kernels (plain data, passed by value).
struct DecodeArgs {
  const void* q;                 // [N][Hq][D]
  void* out;                     // [N][Hq][D] of out_dtype
  float* part_o;                 // [N][Hq][max_parts][D]   (split-K only)
  float* part_ml;                // [N][Hq][max_parts][2]   (max in log2 units, normaliser)
  unsigned int* counters;        // balanced mode: [N][H_kv] arrival counters, cleared by each call
  const int32_t* block_tables;   // [N][max_blocks]
  const int32_t* seq_lens;       // [N]
  int* err;                      // device error word
  int64_t num_blocks;
  int32_t num_seqs, num_q_heads, num_kv_heads, group;
  int32_t block_size, max_blocks, max_seq_len;
  int32_t part_tokens;           // 0 = single pass
  int32_t max_parts;             // partitions per sequence held in the workspace
  int32_t tok_per_op;            // tokens one TMA box covers: min(block_size, 16)
  int32_t slot_rows;             // shared-memory rows reserved per box: max(tok_per_op, 8)
  int32_t ops_per_stage;         // boxes per 16-row stage
  int32_t out_dtype;             // pa_dtype
  float scale_log2;              // scale * log2(e) (times k_scale for E4M3 caches)
  float v_scale;                 // E4M3 caches: V code c stands for value(c) * v_scale
  // Multi-token rows (pa_prefill on the grouped kernel); unused by decode.
  const int32_t* q_start;        // [N + 1] query rows of each sequence
  int32_t max_q;                 // bound of every n_s; rows past it are not computed
  // Stall hook for tests of the bounded waits (pa_test_set_stall): when
  // test_stop_stage >= 0, each TMA ring issues only its first test_stop_stage
  // stages, and a consumer waits test_wait_ns (not the 2 s bound) for a stage
  // before giving up with PA_DEVERR_TIMEOUT. Copies already issued are still
  // drained under the full bound, so no copy is in flight when a CTA exits.
  int32_t test_stop_stage = -1;  // < 0: off
  uint32_t test_wait_ns = 0;
};

// The bound a consumer's wait for a TMA stage uses (the test hook can shorten it).
#define PA_STAGE_WAIT_NS(args, full_ns) \
  ((args).test_stop_stage >= 0 && (args).test_wait_ns > 0 ? static_cast<uint64_t>((args).test_wait_ns) : (full_ns))

// Rows of shared memory one pipeline stage holds (one m16 tile of tokens).
constexpr int kStageRows = 16;
// Warps per decode CTA; each owns a private ring of stages.
constexpr int kDecodeWarps = 4;

// Which decode kernel a launch runs.
enum DecodeKernel { kPerPartition = 0, kPerWarpRanges = 1, kGroupedRanges = 2 };

// Decode launchers, one per (dtype, head_dim) translation unit.
// group_tiles = ceil(group / 8) in {1, 2}; `kernel` is a DecodeKernel and
// head_group the KV heads per CTA of the grouped kernel (8 or 4).
cudaError_t launch_decode_f16_64(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                 int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
cudaError_t launch_decode_f16_128(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
cudaError_t launch_decode_f16_256(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
cudaError_t launch_decode_bf16_64(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                  int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
cudaError_t launch_decode_bf16_128(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                   int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
cudaError_t launch_decode_bf16_256(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a,
                                   int group_tiles, int head_group, dim3 grid, int kernel,
                                  cudaStream_t st);
// E4M3 caches (q and outputs fp16 or bf16), head_dim 128 and 256.
cudaError_t launch_decode_e4m3_f16_128(const CUtensorMap& tk, const CUtensorMap& tv,
                                       const DecodeArgs& a, int group_tiles, int head_group,
                                       dim3 grid, int kernel, cudaStream_t st);
cudaError_t launch_decode_e4m3_f16_256(const CUtensorMap& tk, const CUtensorMap& tv,
                                       const DecodeArgs& a, int group_tiles, int head_group,
                                       dim3 grid, int kernel, cudaStream_t st);
cudaError_t launch_decode_e4m3_bf16_128(const CUtensorMap& tk, const CUtensorMap& tv,
                                        const DecodeArgs& a, int group_tiles, int head_group,
                                        dim3 grid, int kernel, cudaStream_t st);
cudaError_t launch_decode_e4m3_bf16_256(const CUtensorMap& tk, const CUtensorMap& tv,
                                        const DecodeArgs& a, int group_tiles, int head_group,
                                        dim3 grid, int kernel, cudaStream_t st);

// Multi-token rows on the grouped balanced kernel (pa_verify_inst.cu): head_dim
// 128, blocks of 16 or more tokens, a.q_start / a.max_q set; (nt, row_tiles,
// head_group) is (1, 1, 8), (2, 1, 8) or (2, 2, 4): at most 8, 16 or 32
// (query, head) rows per KV head. Grid: one CTA per SM (a multiple of
// H_kv / head_group); the workspace is the balanced one with column groups of
// 8 * nt rows, H_kv * row_tiles of them per sequence.
#define PA_DECLARE_MULTI(name)                                                               \
  cudaError_t name(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeArgs& a, int nt, \
                   int row_tiles, int head_group, dim3 grid, cudaStream_t st);
PA_DECLARE_MULTI(launch_multi_f16)
PA_DECLARE_MULTI(launch_multi_bf16)
PA_DECLARE_MULTI(launch_multi_e4m3_f16)
PA_DECLARE_MULTI(launch_multi_e4m3_bf16)
#undef PA_DECLARE_MULTI

// Balanced mode: resident CTAs per SM of the per-warp-range kernel, the
// largest batch whose per-sequence offsets fit shared memory, and the partial
// slots per SM either balanced kernel may use (the workspace is sized by it).
constexpr int balanced_ctas_per_sm(int head_dim) { return head_dim > 128 ? 1 : 2; }
constexpr int kMaxBalancedSeqs = 2048;
constexpr int kBalancedSlotsPerSm = 16;

// Multi-token causal attention (pa_prefill.cu).
struct PrefillArgs {
  const void* q;                 // [T][Hq][D]
  void* out;                     // [T][Hq][D] of out_dtype
  const int32_t* q_start;        // [N + 1] query rows of each sequence
  const int32_t* block_tables;   // [N][max_blocks]
  const int32_t* seq_lens;       // [N]
  int* err;                      // device error word
  int64_t num_blocks;
  int32_t num_seqs, num_q_heads, num_kv_heads, group;
  int32_t block_size, max_blocks;
  int32_t tok_per_op;            // tokens one TMA box covers: min(block_size, 64)
  int32_t ops_per_stage;         // boxes per 64-token stage
  int32_t out_dtype;             // pa_dtype
  float scale_log2;              // scale * log2(e) (times k_scale for E4M3 caches)
  float v_scale;                 // E4M3 caches: V code c stands for value(c) * v_scale
  int32_t test_stop_stage = -1;  // stall hook, as in DecodeArgs (tcgen05 kernel)
  uint32_t test_wait_ns = 0;
};
// Grid: (ceil(max_q_len * g / 64), H_kv, N). bf16: q/out MMA type (the act
// dtype for E4M3 caches); fp8: E4M3 cache (head_dim 128 or 256); thin: head
// dim 128 with at most 32 rows per CTA (three CTAs per SM, a two-stage ring).
cudaError_t launch_prefill(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                           int head_dim, bool bf16, bool fp8, bool thin, dim3 grid,
                           cudaStream_t st);
// tcgen05/TMEM kernels for head_dim 128. Grid: (ceil(max_q_len * g / 256), H_kv, N);
// q and out 16-byte aligned. fp16 / bf16 caches: 128-key tiles (pa_prefill_tc128.cu);
// E4M3 caches: 64-key tiles with converter warps (pa_prefill_tc.cu), bf16 = q / out type.
cudaError_t launch_prefill_tc128(const CUtensorMap& tk, const CUtensorMap& tv, const PrefillArgs& a,
                                 bool bf16, dim3 grid, cudaStream_t st);
cudaError_t launch_prefill_tc_e4m3(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const PrefillArgs& a, bool bf16, dim3 grid, cudaStream_t st);

// Merges split-K partials into out (pa_decode_reduce.cu).
cudaError_t launch_decode_reduce(const DecodeArgs& a, int head_dim, cudaStream_t st);
// Merges the cut pieces decode_grouped_kernel left as partials (it stores them
// without a merge); `ranges` and `stage_tokens` are that launch's range count
// and tokens per stage of the line. Launched right after it on the same
// stream, as a programmatic dependent.
cudaError_t launch_decode_piece_merge(const DecodeArgs& a, int head_dim, int64_t ranges,
                                      int stage_tokens, int sms, cudaStream_t st);
// Tokens per stage of the head-grouped decode kernel's line: 32 for E4M3
// caches (64 KB stages at 8 heads), 16 otherwise.
constexpr int grouped_line_tokens(bool fp8) { return fp8 ? 32 : kStageRows; }

// Cache operations (pa_cache_ops.cu).
cudaError_t launch_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                                const int32_t* seq_idx, const int32_t* positions, int64_t num_tokens,
                                int32_t block_size, int64_t num_blocks, int64_t* slots, int* err,
                                cudaStream_t st);
cudaError_t launch_write_kv(const void* key, const void* value, const int64_t* slots,
                            int64_t num_tokens, void* k_cache, void* v_cache, int64_t num_blocks,
                            int32_t block_size, int64_t row_bytes, int* err, cudaStream_t st);
// Quantising write into E4M3 caches; row_elems = H_kv * D, a multiple of 8.
cudaError_t launch_write_kv_e4m3(const void* key, const void* value, bool bf16,
                                 const int64_t* slots, int64_t num_tokens, void* k_cache,
                                 void* v_cache, int64_t num_blocks, int32_t block_size,
                                 int64_t row_elems, float k_scale, float v_scale, int* err,
                                 cudaStream_t st);

constexpr int kMaxCopyLayers = 64;
struct CopyLayers {
  void* k[kMaxCopyLayers];
  void* v[kMaxCopyLayers];
};
cudaError_t launch_copy_blocks(const CopyLayers& layers, int32_t num_layers,
                               const int64_t* pairs, int64_t num_pairs, int64_t num_blocks,
                               int64_t block_bytes, int* err, cudaStream_t st);

// Swap between two pools (either may be pinned host memory reached through
// the unified address space).
struct SwapLayers {
  const void* src_k[kMaxCopyLayers];
  const void* src_v[kMaxCopyLayers];
  void* dst_k[kMaxCopyLayers];
  void* dst_v[kMaxCopyLayers];
};
cudaError_t launch_swap_blocks(const SwapLayers& layers, int32_t num_layers, const int64_t* pairs,
                               int64_t num_pairs, int64_t src_blocks, int64_t dst_blocks,
                               int64_t block_bytes, int* err, cudaStream_t st);

// Prefix-cache keys (pa_prefix_hash.cu): SHA-256 constants of FIPS 180-4
// (derived from the primes at first use) and a 32-byte root as 8 big-endian
// words.
struct Sha256Consts {
  uint32_t k[64];
  uint32_t h0[8];
};
struct Sha256Root {
  uint32_t w[8];
};
const Sha256Consts& sha256_consts();
cudaError_t launch_key_offsets(const int64_t* tok_off, int32_t num_seqs, int32_t block_size,
                               int64_t* key_off, int* err, cudaStream_t st);
cudaError_t launch_prefix_hash(const int32_t* tokens, const int64_t* tok_off, const int64_t* key_off,
                               int32_t num_seqs, int32_t block_size, const Sha256Root& root,
                               uint8_t* keys, int* err, cudaStream_t st);

}  // namespace pa
