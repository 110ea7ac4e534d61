/*
 * pa.h - C ABI of libpagedkv: the device hot path of PagedAttention on one GB300.
 *
 * A sequence's KV cache lives in fixed-size blocks of a shared pool; a block
 * table maps its logical block floor(t/b) to a physical block id and token t
 * sits at row t mod b of that block ("PagedAttention: paging the KV cache",
 * pofe.ai, section "How it works"; "PagedAttention: Virtual-Memory KV Cache
 * Management, Continuous Batching, and PyTorch Architecture", ailinkdeeptech.com,
 * section "Mathematical Foundations", 1. Paged Virtual Memory Mapping).
 *
 * Conventions for every call:
 *  - All buffers are caller-owned. Pointers documented as "device" must be CUDA
 *    device memory of the current device; "host" pointers are ordinary memory.
 *    The library allocates no device memory and keeps only one static device
 *    error word per device. Its address (and the device's SM count) is looked
 *    up on the first call made with that device current and kept until the
 *    process exits, so a device that went through cudaDeviceReset must not be
 *    used with the library again.
 *  - Every call enqueues work on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and returns without synchronising, except pa_get_device_error.
 *  - Return value: PA_OK (0) or a negative PA_ERR_* status. A negative status
 *    means nothing was launched. Problems only the device can see (a block id
 *    out of range, a bad length or slot) never trap: the offending row is
 *    skipped and a PA_DEVERR_* bit is OR-ed into the device error word, which
 *    pa_get_device_error reads and clears.
 *
 * Cache layout (per layer): k and v are each [num_blocks][block_size]
 * [num_kv_heads][head_dim], row-major, fp16, bf16 or FP8 E4M3 codes; element
 * (blk, off, h, d) is at ((blk*block_size + off)*num_kv_heads + h)*head_dim + d.
 * A "slot" numbers pool rows: slot = blk*block_size + off. Layers are separate
 * pools that share block ids.
 *
 * FP8 caches ("PagedAttention: paging the KV cache", section "Fine-tuned models
 * and adapters": an FP8 cache halves the bytes per block and nothing else about
 * paging changes). The pages fix no format, so this library takes OCP E4M3
 * (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no infinities,
 * 0x7F/0xFF NaN, largest finite 448) with one float scale per layer for K and
 * one for V: a stored code c stands for value(c) * k_scale (or v_scale).
 * Writes store e4m3(x / scale): the quotient rounded once to float32, then to
 * the nearest code, ties to even, magnitudes past 448 saturating to 448.
 * q, the new key/value rows and the outputs stay fp16/bf16 (act_dtype).
 */
#ifndef PAGED_KV_CACHE_114_GB300_PA_H
#define PAGED_KV_CACHE_114_GB300_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_ABI_VERSION 4

typedef enum { PA_F16 = 0, PA_BF16 = 1, PA_F32 = 2, PA_FP8_E4M3 = 3 } pa_dtype;

enum {
  PA_OK = 0,
  PA_ERR_NULL = -1,       /* a required pointer is NULL */
  PA_ERR_DTYPE = -2,      /* unsupported or mismatched dtype */
  PA_ERR_SHAPE = -3,      /* unsupported head_dim, block_size, head grouping or size */
  PA_ERR_ALIGN = -4,      /* a pointer is not aligned as documented */
  PA_ERR_WORKSPACE = -5,  /* workspace missing or smaller than pa_decode_workspace_bytes */
  PA_ERR_ARG = -6,        /* other invalid argument */
  PA_ERR_CUDA = -7,       /* a CUDA runtime call failed */
  PA_ERR_PAIRS = -8       /* copy pairs violate the distinct-destination rule */
};

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID 1  /* a block id outside [0, num_blocks) in a table or pair */
#define PA_DEVERR_SEQ_LEN 2   /* seq_len < 0 or above max_seq_len or the table's capacity */
#define PA_DEVERR_SLOT 4      /* a slot outside [-1, num_blocks*block_size) */
#define PA_DEVERR_POSITION 8  /* slot mapping: seq index or position outside the table */
#define PA_DEVERR_TIMEOUT 16  /* a bounded wait for an asynchronous copy gave up */

/* One layer's paged cache. k and v: device, 16-byte aligned, layout above. */
typedef struct {
  void* k;
  void* v;
  int64_t num_blocks;   /* blocks in the pool, < 2^31 */
  int32_t block_size;   /* tokens per block b */
  int32_t num_kv_heads; /* H_kv */
  int32_t head_dim;     /* D */
  pa_dtype dtype;       /* element type of k and v: PA_F16, PA_BF16 or PA_FP8_E4M3 */
  pa_dtype act_dtype;   /* PA_FP8_E4M3 caches: dtype of q, key and value (PA_F16 or
                           PA_BF16); ignored for 16-bit caches, whose q, key and
                           value have the cache's own dtype */
  float k_scale;        /* PA_FP8_E4M3 caches: K code c stands for value(c) * k_scale;
                           finite and > 0. Ignored for 16-bit caches. */
  float v_scale;        /* the same for V */
} pa_cache;

/*
 * pa_slot_mapping - pool slot of each new token.
 * slot[i] = block_tables[seq_idx[i]][positions[i] / block_size] * block_size
 *           + positions[i] % block_size
 * (ailinkdeeptech.com, 1. Paged Virtual Memory Mapping: logical block
 * floor(t/B), offset t mod B; neelmishra.github.io "PagedAttention: Manage the
 * Cache Without Moving the Sequence", section "Map a ten-token sequence into
 * pages").
 *   block_tables  device int32 [num_seqs][max_blocks_per_seq]
 *   seq_idx       device int32 [num_tokens]  sequence of each token
 *   positions     device int32 [num_tokens]  logical position t of each token
 *   num_blocks    pool size, used to range-check table entries
 *   slot_mapping  device int64 [num_tokens]  output
 * Errors: a seq index, position or table entry out of range writes slot -1 and
 * sets PA_DEVERR_POSITION or PA_DEVERR_BLOCK_ID. num_tokens == 0 is a no-op.
 */
int pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                    const int32_t* seq_idx, const int32_t* positions, int64_t num_tokens,
                    int32_t block_size, int64_t num_blocks, int64_t* slot_mapping, void* stream);

/*
 * pa_write_kv - store each new token's key and value rows at its slot.
 * k_cache[slot / b][slot % b][h][:] = key[i][h][:], same for v (pofe.ai,
 * sections "How it works", "write k, v of the new token into slot len(s) % b of
 * block table[s][-1]", and "Minimal implementation", Sequence.append).
 *   key, value    device [num_tokens][num_kv_heads][head_dim], 16-byte aligned,
 *                 of the cache's dtype (16-bit caches) or of act_dtype (FP8
 *                 caches, whose rows are quantised: code = e4m3(x / k_scale)
 *                 for K and e4m3(x / v_scale) for V, see the FP8 note above)
 *   slot_mapping  device int64 [num_tokens]; -1 marks a padding token (skipped)
 *   cache         host pointer to one pa_cache
 * Errors: a slot outside [-1, num_blocks*block_size) skips the token and sets
 * PA_DEVERR_SLOT. Two tokens with the same slot race (last writer unspecified).
 */
int pa_write_kv(const void* key, const void* value, const int64_t* slot_mapping,
                int64_t num_tokens, const pa_cache* cache, void* stream);

/*
 * pa_copy_blocks - copy-on-write block copies: for every (src, dst) pair and
 * every layer, block dst of k and v becomes a copy of block src (pofe.ai,
 * section "Sharing and copy-on-write" and Sequence.append in "Minimal
 * implementation"; ailinkdeeptech.com section 4, Copy-on-Write step 2).
 *   caches         host array of num_layers pa_cache (same geometry and dtype;
 *                  FP8 blocks are copied code for code, scales play no part)
 *   src_dst_pairs  device int64 [num_pairs][2]
 * Destinations must be distinct and no destination may also be a source
 * (copy-on-write always copies into a fresh block); pa_check_copy_pairs checks
 * this on a host copy. Violations race. An id outside [0, num_blocks) skips the
 * pair and sets PA_DEVERR_BLOCK_ID.
 */
int pa_copy_blocks(const pa_cache* caches, int32_t num_layers, const int64_t* src_dst_pairs,
                   int64_t num_pairs, void* stream);

/*
 * pa_swap_blocks - swap for preemption: for every (src, dst) pair and every
 * layer, block dst of the destination pool becomes a copy of block src of the
 * source pool, K and V. Swapping out copies a preempted sequence's blocks to
 * host memory, swapping in copies them back, possibly to other block ids, after
 * which the caller remaps the sequence's table ("PagedAttention: paging the KV
 * cache", section "When memory runs out"; learn.pranaymahendrakar.com
 * "PagedAttention", section "Preemption": copy blocks to pinned host memory and
 * back). On GB300 the host pool is Grace memory that the kernel reads or
 * writes directly over NVLink-C2C, so one launch moves any set of scattered
 * blocks.
 *   src, dst       host arrays of num_layers pa_cache; each k / v pointer is
 *                  device memory of the current device, managed memory, or
 *                  pinned host memory (cudaHostAlloc / cudaHostRegister).
 *                  Every layer and both sides share dtype, block_size,
 *                  num_kv_heads and head_dim; num_blocks may differ between
 *                  the source and the destination. FP8 blocks move as codes.
 *   src_dst_pairs  int64 [num_pairs][2] in device or pinned host memory
 * Destinations must be distinct. When src and dst are the same pool, no
 * destination may also be a source (as pa_copy_blocks). Pageable host memory
 * returns PA_ERR_ARG before anything is launched. An id outside its pool skips
 * the pair and sets PA_DEVERR_BLOCK_ID.
 */
int pa_swap_blocks(const pa_cache* src, const pa_cache* dst, int32_t num_layers,
                   const int64_t* src_dst_pairs, int64_t num_pairs, void* stream);

/*
 * pa_prefix_hash - prefix-cache keys of every full block of a batch of
 * sequences, for automatic prefix caching: a cached block is found again by
 * its key, a hit needs an unbroken chain of matching keys from position zero,
 * and the first differing token ends the chain (firehose-demo "Paged
 * Attention"; learn.pranaymahendrakar.com "PagedAttention", section "Prefix
 * caching": hash each block-aligned prefix of token ids). The pages fix no
 * function; this library computes
 *   key_j = SHA-256(key_{j-1} || token ids of block j as int32 little-endian),
 *   key_{-1} = root,
 * SHA-256 as FIPS 180-4 defines it. A trailing partial block gets no key.
 *   token_ids      device int32, the sequences' ids back to back
 *   token_offsets  device int64 [num_seqs + 1]: sequence s owns ids
 *                  token_offsets[s] .. token_offsets[s+1] - 1
 *   key_offsets    device int64 [num_seqs + 1]: sequence s writes keys
 *                  key_offsets[s] .. key_offsets[s+1] - 1, which must number
 *                  floor(length_s / block_size) (pa_prefix_key_offsets
 *                  computes the packed layout on the device)
 *   root           host, 32 bytes, or NULL for 32 zero bytes (a distinct root,
 *                  e.g. per adapter, keeps caches apart)
 *   keys           device [key_offsets[num_seqs]][32] bytes (digest byte
 *                  order), 16-byte aligned
 * Errors (device): a negative length or a key range of the wrong size sets
 * PA_DEVERR_SEQ_LEN and the sequence writes nothing.
 */
int pa_prefix_hash(const int32_t* token_ids, const int64_t* token_offsets,
                   const int64_t* key_offsets, int32_t num_seqs, int32_t block_size,
                   const uint8_t* root, uint8_t* keys, void* stream);

/*
 * pa_prefix_key_offsets - where pa_prefix_hash writes each sequence's keys
 * when they are packed back to back: key_offsets[0] = 0 and
 * key_offsets[s + 1] = key_offsets[s] + floor(length_s / block_size), with
 * length_s = token_offsets[s + 1] - token_offsets[s] (only full blocks get a
 * key: "PagedAttention: Virtual-Memory KV Cache Management, Continuous
 * Batching, and PyTorch Architecture", ailinkdeeptech.com, Step 1). One
 * device scan; the result can be passed straight to pa_prefix_hash, and
 * key_offsets[num_seqs] is the number of keys.
 *   token_offsets  device int64 [num_seqs + 1], as for pa_prefix_hash
 *   key_offsets    device int64 [num_seqs + 1], output
 * Errors (device): a negative length counts as zero keys and sets
 * PA_DEVERR_SEQ_LEN. num_seqs == 0 writes key_offsets[0] = 0.
 */
int pa_prefix_key_offsets(const int64_t* token_offsets, int32_t num_seqs, int32_t block_size,
                          int64_t* key_offsets, void* stream);

/* Host-side check of copy pairs: ids in range, distinct destinations, no
 * destination used as a source. Returns PA_OK or PA_ERR_PAIRS / PA_ERR_NULL. */
int pa_check_copy_pairs(const int64_t* host_pairs, int64_t num_pairs, int64_t num_blocks);

/*
 * pa_decode - single-query (decode) attention through block tables.
 * For sequence s and query head h (KV head h / g, g = num_q_heads/num_kv_heads):
 *   out[s][h] = sum_{t < L_s} softmax_t(scale * q[s][h] . K_s[t]) V_s[t]
 * where K_s[t], V_s[t] are gathered at slot(s, t). The sum runs block by block
 * with a running maximum and normaliser (ailinkdeeptech.com section 3,
 * Non-Contiguous Online Softmax Attention Kernel; learn.pranaymahendrakar.com
 * "PagedAttention", section "The kernel consequence"); the g query heads of a
 * KV head share each loaded block (ailinkdeeptech.com Step 2, grouped-query
 * ratio). Slots at t >= L_s are never part of the result.
 *   q              device [num_seqs][num_q_heads][head_dim], of the cache's
 *                  dtype (16-bit caches) or of act_dtype (FP8 caches)
 *   cache          host pointer to one pa_cache; head_dim 64, 128 or 256
 *                  (128 or 256 for FP8 caches); block_size a divisor of 16 or
 *                  a multiple of 16. With an FP8 cache, K[t] and V[t] are the
 *                  stored codes' values times k_scale and v_scale.
 *   block_tables   device int32 [num_seqs][max_blocks_per_seq]; entries past
 *                  ceil(L_s/b) are never read
 *   seq_lens       device int32 [num_seqs]; 0 gives a zero output row
 *   max_seq_len    host upper bound of seq_lens (sizes the launch)
 *   scale          softmax scale, usually 1/sqrt(head_dim)
 *   out            device [num_seqs][num_q_heads][head_dim] of out_dtype
 *   partition_tokens  0: one pass per (sequence, KV head); a multiple of 16:
 *                  split-K, each sequence cut into partitions of that many
 *                  tokens whose (max, normaliser, unnormalised output)
 *                  partials a second kernel merges with the rescale identity;
 *                  PA_PARTITION_BALANCED: a persistent grid in which every warp
 *                  streams an equal share of all sequences' 16-token stages;
 *                  a (sequence, KV head) cut between warps is merged by a
 *                  second kernel on `stream` (head-grouped kernel) or by the
 *                  last warp to finish its share (per-warp kernel)
 *                  (num_seqs <= 2048)
 *   workspace      device, >= pa_decode_workspace_bytes(...) bytes; 16-byte
 *                  aligned (256-byte in balanced mode); unused (may be NULL)
 *                  when no sequence needs more than one partition. Its prior
 *                  contents do not matter: the per-warp balanced kernel's
 *                  arrival counters are cleared (a memset on `stream`) at the
 *                  start of each call
 * Errors (device): L_s outside [0, min(max_seq_len, max_blocks_per_seq*b)]
 * sets PA_DEVERR_SEQ_LEN and is clamped; a table entry out of range sets
 * PA_DEVERR_BLOCK_ID and its tokens are left out.
 */
int pa_decode(const void* q, int32_t num_seqs, int32_t num_q_heads, const pa_cache* cache,
              const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
              int32_t max_seq_len, float scale, void* out, pa_dtype out_dtype,
              int32_t partition_tokens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill - causal attention for several new tokens per sequence over the
 * paged cache: a prefill chunk, the draft tokens of speculative decoding, or
 * the re-run prompt of a preempted sequence ("PagedAttention: paging the KV
 * cache", How it works: prefill writes into the blocks; When memory runs out:
 * recomputation re-runs prompt and generated tokens as one prefill).
 * Sequence s owns query rows q_start[s] .. q_start[s+1] - 1 (n_s of them). With
 * L_s = seq_lens[s], its query i sits at position L_s - n_s + i and attends to
 * the tokens at positions 0 .. L_s - n_s + i: the mask gives the attention
 * edges, the block table only where each row is stored ("PagedAttention:
 * Manage the Cache Without Moving the Sequence", The kernel must understand
 * the mapping). For query row t of sequence s and query head h (KV head
 * h / g):
 *   out[t][h] = sum_{u <= p} softmax_u(scale * q[t][h] . K_s[u]) V_s[u],
 *   p = L_s - n_s + (t - q_start[s]).
 * The K/V of all L_s positions, the new ones included, must already be in
 * the cache (pa_slot_mapping + pa_write_kv first). Decode is the case n_s = 1.
 *   q            device [q_start[num_seqs]][num_q_heads][head_dim], cache dtype
 *                (act_dtype for FP8 caches)
 *   q_start      device int32 [num_seqs + 1], non-decreasing, q_start[0] = 0
 *   max_q_len    host upper bound of every n_s (sizes the launch)
 *   cache        host pointer to one pa_cache; head_dim 64, 128 or 256 (128
 *                or 256 for FP8 caches, whose q is act_dtype and whose K/V
 *                rows are the codes' values times k_scale / v_scale);
 *                block_size >= 8 and a divisor or a multiple of 64
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]
 *   seq_lens     device int32 [num_seqs]
 *   out          device [q_start[num_seqs]][num_q_heads][head_dim] of out_dtype
 *   workspace    device, pa_prefill_workspace_bytes() bytes or more, 256-byte
 *                aligned, owned by the caller and not used by another call
 *                in flight; or NULL with workspace_bytes 0. Batches of a few
 *                new tokens per sequence (at most 32 (query, head) rows per KV
 *                head, head_dim 128, blocks of 16 or more tokens, at most 2048
 *                sequences; over 16 rows only while the batch has fewer than
 *                4 (sequence, KV head) pairs per SM) use it to run on the
 *                balanced head-grouped kernel, whose per-SM ranges of the
 *                cache need partials and arrival counters (cleared by each
 *                call); without one they run one CTA per (sequence, KV head,
 *                64 rows). Other shapes never use it.
 * num_seqs <= 65535 and num_kv_heads <= 65535.
 * Errors (host): a workspace of workspace_bytes > 0 but fewer bytes than the
 * shape needs, or NULL, returns PA_ERR_WORKSPACE; misaligned, PA_ERR_ALIGN.
 * Errors (device): n_s > L_s, L_s above the table's capacity or n_s above
 * max_q_len set PA_DEVERR_SEQ_LEN and the sequence's rows (or those past
 * max_q_len) are not written; a table entry out of range sets
 * PA_DEVERR_BLOCK_ID and its tokens are left out.
 */
int pa_prefill(const void* q, int32_t num_seqs, const int32_t* q_start, int32_t max_q_len,
               int32_t num_q_heads, const pa_cache* cache, const int32_t* block_tables,
               int32_t max_blocks_per_seq, const int32_t* seq_lens, float scale, void* out,
               pa_dtype out_dtype, void* workspace, size_t workspace_bytes, void* stream);

/* Workspace bytes pa_prefill can use for these sizes on the current device
 * (0 when the shape runs on a kernel that needs none). */
size_t pa_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t max_q_len);

/* Name of the kernel pa_prefill launches for this shape, given a workspace
 * (with_workspace != 0) or not, on a device of num_sms SMs (0: the current
 * device): "multi_grouped_kernel", "prefill_tc_kernel" (tcgen05; with an
 * E4M3 cache its variant "prefill_tc_e4m3_kernel" runs) or "prefill_kernel";
 * NULL for sizes it rejects (or num_sms 0 without a device). pa_prefill makes
 * the same choice from the same helper, and two more inputs that this call
 * takes as met: q and out 16-byte aligned (otherwise "prefill_tc_kernel"
 * becomes "prefill_kernel"), and num_seqs * ceil(max_blocks_per_seq *
 * block_size / 16) below 2^31 (otherwise "multi_grouped_kernel" becomes one
 * of the other two). */
const char* pa_prefill_kernel_name(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_q_len,
                                   int32_t with_workspace, int32_t num_sms);

/* Workspace bytes pa_decode needs for these sizes (0 when one partition covers
 * max_seq_len or partition_tokens == 0). The balanced mode's size depends on
 * the current device's SM count. */
size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_seq_len, int32_t partition_tokens);

/* partition_tokens value selecting pa_decode's balanced split. */
#define PA_PARTITION_BALANCED (-1)

/* A partition_tokens value for pa_decode chosen from the batch shape and the
 * current device's SM count: 0 (single pass; always for max_seq_len <= 256),
 * PA_PARTITION_BALANCED, or a partition size. Returns a negative status (other
 * than -1) on error. */
int32_t pa_decode_default_partition(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                    int32_t block_size);

/* Name of the kernel(s) pa_decode launches for this shape and partition_tokens:
 * "decode_kernel" (single pass), "decode_kernel+decode_reduce_kernel" (fixed
 * split with more than one partition), "decode_grouped_kernel+
 * decode_piece_merge_kernel" (balanced, one TMA box per stage for a group of
 * KV heads, then the merge of cut pieces) or "decode_balanced_kernel"
 * (balanced, per-warp boxes). NULL when pa_decode would reject the shape.
 * Host only: reads no device state. */
const char* pa_decode_kernel_name(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t max_seq_len,
                                  int32_t partition_tokens);

/*
 * pa_decode_static_workspace - pa_decode for callers that cannot allocate
 * device memory. The pages have no counterpart; this call is a library
 * convenience. Some callers cannot cudaMalloc a workspace: code inside a host
 * application whose own pool owns all device memory, latency-critical paths
 * where cudaMalloc/cudaFree may synchronise the device, and bindings from
 * runtimes without a device allocator. This call takes the same arguments as
 * pa_decode minus the workspace, and keeps the split-K partials in a
 * fixed array of PA_STATIC_WORKSPACE_BYTES compiled into the library (held by
 * every GPU that loads it until the process exits). The caller still passes q,
 * the cache, the tables, the lengths and out.
 *   - Sizes whose workspace (pa_decode_workspace_bytes) exceeds
 *     PA_STATIC_WORKSPACE_BYTES return PA_ERR_WORKSPACE and launch nothing.
 *     The balanced mode (PA_PARTITION_BALANCED, the default for most batches)
 *     needs 16 * SMs * g * (head_dim + 2) * 4 bytes of partials plus 4 bytes
 *     per (sequence, KV head), g = num_q_heads / num_kv_heads, whatever the
 *     batch: on a 152-SM GB300 that fits while g * (head_dim + 2) <= 1,700 or
 *     so, e.g. g <= 13 at head_dim 128 and g <= 6 at head_dim 256. Larger
 *     groups (g = 16 at head_dim 128, g = 8 at head_dim 256) are refused in
 *     that mode even for one sequence; a fixed partition size may still fit.
 *   - The call allocates nothing. The first call on a device looks up the
 *     array's device address (once per device, with that device current); make
 *     that first call before any stream capture. Like the error word's, that
 *     address is kept for the life of the process: after cudaDeviceReset on a
 *     device, do not call the library on that device again.
 *   - Every call shares the one array, which keeps the previous call's
 *     partials. Nothing in it needs to start at zero: each call writes every
 *     partial before reading it, and clears the per-warp balanced kernel's arrival
 *     counters itself. Calls that overlap on the GPU (other streams, other
 *     threads) race on the array: serialise them.
 * Other arguments, errors and results are those of pa_decode.
 */
#define PA_STATIC_WORKSPACE_BYTES (16u * 1024u * 1024u)
int pa_decode_static_workspace(const void* q, int32_t num_seqs, int32_t num_q_heads,
                               const pa_cache* cache, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                               int32_t max_seq_len, float scale, void* out, pa_dtype out_dtype,
                               int32_t partition_tokens, void* stream);

/*
 * pa_test_set_stall - test hook for the bounded waits; not for production use.
 * With stop_stage >= 0, every later pa_decode call, and pa_prefill on the
 * tcgen05 kernel, runs with each TMA ring issuing only its first stop_stage
 * stages of K/V copies, and a consumer's wait for a stage bounded by wait_us
 * microseconds (1 .. 1,000,000) instead of 2 s. The consumers of the stages
 * that never arrive give up, set PA_DEVERR_TIMEOUT and finish without them;
 * the copies that were issued are still waited for (under the full bound), so
 * no copy is in flight when a CTA exits and the context stays usable. Rows
 * that lost stages hold unspecified values. stop_stage < 0 turns the hook off
 * (the default). The setting is process-wide; calls made while it changes may
 * see either value. Returns PA_ERR_ARG for a wait_us out of range.
 */
int pa_test_set_stall(int32_t stop_stage, uint32_t wait_us);

/* Synchronise `stream`, copy the current device's error word to *err_out and
 * clear it. */
int pa_get_device_error(int32_t* err_out, void* stream);

/* Human-readable name of a status code. */
const char* pa_status_string(int status);

/* PA_ABI_VERSION of the loaded library. */
int pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_114_GB300_PA_H */
