// pa_api.cu - the extern "C" entry points of libpagedkv (declared in
// include/pa.h): argument checks, TMA tensor maps, launches on the caller's
// stream, and the per-device error word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <atomic>
#include <mutex>
#include <unordered_set>

#include "pa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// One word per device; kernels OR PA_DEVERR_* bits into it.
__device__ int g_device_error;

struct DeviceInfo {
  int* err = nullptr;
  int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_info[kMaxDevices];

// pa_test_set_stall: copied into the kernels' arguments by every later call.
std::atomic<int32_t> g_stall_stage{-1};
std::atomic<uint32_t> g_stall_wait_ns{0};

// The device address of g_device_error and the SM count of the current device.
// The address comes from cudaGetSymbolAddress once per device: in host code
// the symbol itself only names a host-side shadow.
bool device_info(DeviceInfo* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& di = g_info[dev];
  if (di.err == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return false;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    di.err = static_cast<int*>(p);
    di.sms = sms;
  }
  *out = di;
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

bool is_fp8(const pa_cache& c) { return c.dtype == PA_FP8_E4M3; }

// Bytes per stored element of a cache.
cuuint64_t elem_bytes(const pa_cache& c) { return is_fp8(c) ? 1 : 2; }

// Element type of the tensor maps; a box's inner extent is one 128-byte line.
CUtensorMapDataType map_type(const pa_cache& c) {
  if (is_fp8(c)) return CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return c.dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Tensor map over one cache [num_blocks][b][H_kv][D] viewed as 4-D
// (D, H_kv, b, num_blocks), box = (128 bytes of D) x 1 x tok_per_op x 1,
// 128-byte swizzle.
bool encode_cache_map(CUtensorMap* m, const void* base, const pa_cache& c, int tok_per_op) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t e = elem_bytes(c);
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(c.head_dim), static_cast<cuuint64_t>(c.num_kv_heads),
                        static_cast<cuuint64_t>(c.block_size), static_cast<cuuint64_t>(c.num_blocks)};
  cuuint64_t strides[3] = {dims[0] * e, dims[0] * dims[1] * e, dims[0] * dims[1] * dims[2] * e};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / e), 1u, static_cast<cuuint32_t>(tok_per_op), 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType dt = map_type(c);
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cache(const pa_cache* c) {
  if (c == nullptr || c->k == nullptr || c->v == nullptr) return PA_ERR_NULL;
  if (c->dtype != PA_F16 && c->dtype != PA_BF16 && c->dtype != PA_FP8_E4M3) return PA_ERR_DTYPE;
  if (c->num_blocks <= 0 || c->num_blocks > 0x7fffffffLL || c->block_size <= 0 ||
      c->num_kv_heads <= 0 || c->head_dim <= 0 || c->head_dim % 8 != 0)
    return PA_ERR_SHAPE;
  if (is_fp8(*c)) {
    if (c->act_dtype != PA_F16 && c->act_dtype != PA_BF16) return PA_ERR_DTYPE;
    if (!(std::isfinite(c->k_scale) && c->k_scale > 0.f && std::isfinite(c->v_scale) &&
          c->v_scale > 0.f))
      return PA_ERR_ARG;
    if (c->head_dim % 16 != 0) return PA_ERR_SHAPE;  // 16-byte rows for the vector copies
  }
  if (!aligned(c->k, 16) || !aligned(c->v, 16)) return PA_ERR_ALIGN;
  return PA_OK;
}


int64_t decode_parts(int32_t max_seq_len, int32_t partition_tokens) {
  if (partition_tokens <= 0 || max_seq_len <= partition_tokens) return 1;
  return (static_cast<int64_t>(max_seq_len) + partition_tokens - 1) / partition_tokens;
}

// Balanced-mode workspace: arrival counters [N][H_kv] (cleared by every call),
// then kBalancedSlotsPerSm * SMs partial slots of (m, l) and o for the g query
// heads of a KV head. Both balanced kernels stay within that many slots.
struct BalancedLayout {
  size_t ml_offset, o_offset, total;
};

BalancedLayout balanced_layout(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int sms) {
  BalancedLayout l{};
  const int64_t g = num_q_heads / num_kv_heads;
  const int64_t slots = static_cast<int64_t>(pa::kBalancedSlotsPerSm) * sms;
  const size_t counters = static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(unsigned int);
  l.ml_offset = (counters + 255) / 256 * 256;
  l.o_offset = l.ml_offset + static_cast<size_t>(slots * g * 2) * sizeof(float);
  l.total = l.o_offset + static_cast<size_t>(slots * g * head_dim) * sizeof(float);
  return l;
}

// Which balanced kernel runs, on how many CTAs. The head-grouped kernel needs
// blocks of at least 8 tokens (no padding rows in its boxes) and a divisor HG
// HG of H_kv, 8 or 4, whose 64 KB-or-smaller stages fit three to a CTA; it runs
// 8 / HG CTAs per SM (8 consumer warps). Otherwise each warp issues its own
// per-head boxes (2 or 1 CTAs of 4 warps per SM).
struct BalancedPlan {
  int kernel;
  int head_group;
  unsigned ctas;
};

BalancedPlan balanced_plan(int32_t num_kv_heads, int32_t group, int32_t head_dim, int32_t block_size,
                          int sms) {
  BalancedPlan p{pa::kPerWarpRanges, 1,
                 static_cast<unsigned>(pa::balanced_ctas_per_sm(head_dim) * sms)};
  if (block_size < 8) return p;
  // mirrors max_head_group(): 4 when a consumer warp needs more registers
  const int limit = (head_dim > 128 || group > 8) ? 4 : 8;
  int hg = 0;
  for (int c = limit; c >= 4; c /= 2) {  // the grouped kernel is built for HG = 8 and 4
    if (num_kv_heads % c == 0 && c * head_dim <= 1024) {
      hg = c;
      break;
    }
  }
  if (hg == 0) return p;
  p.kernel = pa::kGroupedRanges;
  p.head_group = hg;
  p.ctas = static_cast<unsigned>((8 / hg) * sms);
  return p;
}

// Tensor map for the grouped kernel: the cache viewed as (D, token, head,
// block) - token before head, strides permuted - with box (128 bytes of D) x
// tok_per_op x HG x 1, so one box lands head-major in shared memory.
bool encode_grouped_map(CUtensorMap* m, const void* base, const pa_cache& c, int tok_per_op,
                        int hg) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t e = elem_bytes(c);
  const cuuint64_t D = c.head_dim, H = c.num_kv_heads, B = c.block_size;
  cuuint64_t dims[4] = {D, B, H, static_cast<cuuint64_t>(c.num_blocks)};
  cuuint64_t strides[3] = {D * H * e, D * e, D * H * B * e};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / e), static_cast<cuuint32_t>(tok_per_op),
                       static_cast<cuuint32_t>(hg), 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapDataType dt = map_type(c);
  CUresult r = enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// pa_prefill on the grouped balanced kernel (few new tokens per sequence):
// head_dim 128, blocks of 16 or more tokens, at most 32 (query, head) rows
// per KV head, at most kMaxBalancedSeqs sequences. Eight warps per CTA: HG
// KV heads x R tiles of 8 * NT rows, one CTA per SM. It is chosen over the
// per-sequence kernel (3 CTAs of (sequence, KV head) per SM at these sizes)
// for up to 16 rows per KV head, and for more while the batch has fewer than
// 4 (sequence, KV head) pairs per SM: below that the per-sequence kernel is
// bound by its longest sequence, which one CTA streams. Measured on GB300 with
// 64 / 8 heads, 4 drafts, lengths U[512, 8192] (balanced vs per-sequence):
// 16 sequences 118 vs 357 us, 48: 265 vs 392, 64: 349 vs 406, 80: 410 vs 414,
// 96: 483 vs 423, 128: 634 vs 535; with 2 drafts, 128 sequences 368 vs 477 us.
struct MultiPlan {
  bool ok;
  int nt, row_tiles, head_group;
  unsigned ctas;
};

MultiPlan multi_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int32_t max_q_len, int sms) {
  MultiPlan p{false, 0, 0, 0, 0};
  if (head_dim != 128 || block_size < pa::kStageRows || block_size % pa::kStageRows != 0) return p;
  if (num_seqs <= 0 || num_seqs > pa::kMaxBalancedSeqs || num_kv_heads <= 0 ||
      num_q_heads <= 0 || num_q_heads % num_kv_heads != 0)
    return p;
  const int64_t rows = static_cast<int64_t>(max_q_len) * (num_q_heads / num_kv_heads);
  if (rows <= 0 || rows > 32) return p;
  if (rows <= 8) {
    p.nt = 1; p.row_tiles = 1; p.head_group = 8;
  } else if (rows <= 16) {
    p.nt = 2; p.row_tiles = 1; p.head_group = 8;
  } else {
    p.nt = 2; p.row_tiles = 2; p.head_group = 4;
  }
  if (num_kv_heads % p.head_group != 0 || num_kv_heads / p.head_group > sms) return p;
  if (rows > 16 && static_cast<int64_t>(num_seqs) * num_kv_heads >= 4LL * sms) return p;
  p.ctas = static_cast<unsigned>(sms);
  p.ok = true;
  return p;
}

// Which kernel pa_prefill runs. The balanced grouped kernel needs its plan,
// a workspace and a stage line whose per-sequence offsets fit int32; the
// tcgen05 kernels need head_dim 128, 128 to 2^30 (query, head) rows per KV
// head (rows are numbered in int32) and 16-byte aligned q and out (its rows
// move as 16-byte vectors);
// everything else runs on the mma.sync kernel.
enum PrefillKernel { kPrefillMulti, kPrefillTc, kPrefillMma };

PrefillKernel route_prefill(bool multi_ok, bool have_workspace, bool line_fits, int32_t head_dim,
                            int64_t rows_per_kv_head, bool vec_aligned) {
  if (multi_ok && have_workspace && line_fits) return kPrefillMulti;
  if (head_dim == 128 && rows_per_kv_head >= 128 && rows_per_kv_head <= (1LL << 30) &&
      vec_aligned)
    return kPrefillTc;
  return kPrefillMma;
}

// Its workspace: arrival counters [N][H_kv * R], then kBalancedSlotsPerSm * SMs
// partial slots of 8 * NT rows ((m, l), then o).
BalancedLayout multi_layout(int32_t num_seqs, int32_t num_kv_heads, const MultiPlan& p, int sms) {
  BalancedLayout l{};
  const int64_t cols = 8LL * p.nt;
  const int64_t slots = static_cast<int64_t>(pa::kBalancedSlotsPerSm) * sms;
  const size_t counters =
      static_cast<size_t>(num_seqs) * num_kv_heads * p.row_tiles * sizeof(unsigned int);
  l.ml_offset = (counters + 255) / 256 * 256;
  l.o_offset = l.ml_offset + static_cast<size_t>(slots * cols * 2) * sizeof(float);
  l.total = l.o_offset + static_cast<size_t>(slots * cols * 128) * sizeof(float);
  return l;
}

}  // namespace

extern "C" {

int pa_abi_version(void) { return PA_ABI_VERSION; }

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_NULL: return "null pointer";
    case PA_ERR_DTYPE: return "unsupported or mismatched dtype";
    case PA_ERR_SHAPE: return "unsupported shape";
    case PA_ERR_ALIGN: return "misaligned pointer";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_ARG: return "invalid argument";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_PAIRS: return "copy pairs violate the distinct-destination rule";
    default: return "unknown status";
  }
}

int pa_test_set_stall(int32_t stop_stage, uint32_t wait_us) {
  if (stop_stage >= 0 && (wait_us == 0 || wait_us > 1000000u)) return PA_ERR_ARG;
  g_stall_wait_ns.store(stop_stage >= 0 ? wait_us * 1000u : 0u);
  g_stall_stage.store(stop_stage >= 0 ? stop_stage : -1);
  return PA_OK;
}

int pa_get_device_error(int32_t* err_out, void* stream) {
  if (err_out == nullptr) return PA_ERR_NULL;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, di.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpy(di.err, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return PA_ERR_CUDA;
  *err_out = v;
  return PA_OK;
}

int pa_slot_mapping(const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks_per_seq,
                    const int32_t* seq_idx, const int32_t* positions, int64_t num_tokens,
                    int32_t block_size, int64_t num_blocks, int64_t* slot_mapping, void* stream) {
  if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 0) return PA_ERR_ARG;
  if (num_tokens == 0) return PA_OK;
  if (!block_tables || !seq_idx || !positions || !slot_mapping) return PA_ERR_NULL;
  if (block_size <= 0 || num_blocks <= 0 || num_blocks > 0x7fffffffLL) return PA_ERR_SHAPE;
  if (num_tokens > 0x7fffffffLL * 256) return PA_ERR_SHAPE;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  cudaError_t e = pa::launch_slot_mapping(block_tables, num_seqs, max_blocks_per_seq, seq_idx,
                                          positions, num_tokens, block_size, num_blocks,
                                          slot_mapping, di.err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_write_kv(const void* key, const void* value, const int64_t* slot_mapping,
                int64_t num_tokens, const pa_cache* cache, void* stream) {
  if (num_tokens < 0) return PA_ERR_ARG;
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping) return PA_ERR_NULL;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(slot_mapping, 8)) return PA_ERR_ALIGN;
  if (num_tokens > 0x7fffffffLL) return PA_ERR_SHAPE;
  const int64_t row_elems = static_cast<int64_t>(cache->num_kv_heads) * cache->head_dim;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  cudaError_t e;
  if (is_fp8(*cache)) {
    e = pa::launch_write_kv_e4m3(key, value, cache->act_dtype == PA_BF16, slot_mapping, num_tokens,
                                 cache->k, cache->v, cache->num_blocks, cache->block_size,
                                 row_elems, cache->k_scale, cache->v_scale, di.err,
                                 static_cast<cudaStream_t>(stream));
  } else {
    e = pa::launch_write_kv(key, value, slot_mapping, num_tokens, cache->k, cache->v,
                            cache->num_blocks, cache->block_size, row_elems * 2, di.err,
                            static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_check_copy_pairs(const int64_t* host_pairs, int64_t num_pairs, int64_t num_blocks) {
  if (num_pairs < 0) return PA_ERR_ARG;
  if (num_pairs == 0) return PA_OK;
  if (host_pairs == nullptr) return PA_ERR_NULL;
  std::unordered_set<int64_t> dsts;
  std::unordered_set<int64_t> srcs;
  for (int64_t i = 0; i < num_pairs; ++i) {
    const int64_t s = host_pairs[2 * i];
    const int64_t d = host_pairs[2 * i + 1];
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) return PA_ERR_PAIRS;
    if (!dsts.insert(d).second) return PA_ERR_PAIRS;
    srcs.insert(s);
  }
  for (int64_t d : dsts)
    if (srcs.count(d)) return PA_ERR_PAIRS;
  return PA_OK;
}

int pa_copy_blocks(const pa_cache* caches, int32_t num_layers, const int64_t* src_dst_pairs,
                   int64_t num_pairs, void* stream) {
  if (num_layers <= 0 || num_pairs < 0) return PA_ERR_ARG;
  if (caches == nullptr) return PA_ERR_NULL;
  for (int32_t l = 0; l < num_layers; ++l) {
    int rc = check_cache(&caches[l]);
    if (rc != PA_OK) return rc;
    const pa_cache& c0 = caches[0];
    const pa_cache& c = caches[l];
    if (c.dtype != c0.dtype) return PA_ERR_DTYPE;
    if (c.num_blocks != c0.num_blocks || c.block_size != c0.block_size ||
        c.num_kv_heads != c0.num_kv_heads || c.head_dim != c0.head_dim)
      return PA_ERR_SHAPE;
  }
  if (num_pairs == 0) return PA_OK;
  if (src_dst_pairs == nullptr) return PA_ERR_NULL;
  if (!aligned(src_dst_pairs, 8)) return PA_ERR_ALIGN;
  const int64_t block_bytes = static_cast<int64_t>(caches[0].block_size) * caches[0].num_kv_heads *
                              caches[0].head_dim * static_cast<int64_t>(elem_bytes(caches[0]));
  if (num_pairs * ((block_bytes + 16383) / 16384) > 0x7fffffffLL) return PA_ERR_SHAPE;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  for (int32_t l0 = 0; l0 < num_layers; l0 += pa::kMaxCopyLayers) {
    const int32_t n = (num_layers - l0) < pa::kMaxCopyLayers ? (num_layers - l0) : pa::kMaxCopyLayers;
    pa::CopyLayers layers{};
    for (int32_t i = 0; i < n; ++i) {
      layers.k[i] = caches[l0 + i].k;
      layers.v[i] = caches[l0 + i].v;
    }
    cudaError_t e = pa::launch_copy_blocks(layers, n, src_dst_pairs, num_pairs, caches[0].num_blocks,
                                           block_bytes, di.err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

// A pointer the current device can read and write at the same address:
// device memory of this device, managed memory, or pinned (registered) host
// memory mapped into the unified address space.
bool device_reachable(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // a failed query leaves its error behind: clear it
    return false;
  }
  if (at.devicePointer != p) return false;
  if (at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged) return true;
  if (at.type != cudaMemoryTypeDevice) return false;
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && at.device == dev;
}

int pa_swap_blocks(const pa_cache* src, const pa_cache* dst, int32_t num_layers,
                   const int64_t* src_dst_pairs, int64_t num_pairs, void* stream) {
  if (num_layers <= 0 || num_pairs < 0) return PA_ERR_ARG;
  if (src == nullptr || dst == nullptr) return PA_ERR_NULL;
  for (int32_t l = 0; l < num_layers; ++l) {
    for (const pa_cache* c : {&src[l], &dst[l]}) {
      const int rc = check_cache(c);
      if (rc != PA_OK) return rc;
      if (c->dtype != src[0].dtype) return PA_ERR_DTYPE;
      if (c->block_size != src[0].block_size || c->num_kv_heads != src[0].num_kv_heads ||
          c->head_dim != src[0].head_dim)
        return PA_ERR_SHAPE;
    }
    if (src[l].num_blocks != src[0].num_blocks || dst[l].num_blocks != dst[0].num_blocks)
      return PA_ERR_SHAPE;
  }
  if (num_pairs == 0) return PA_OK;
  if (src_dst_pairs == nullptr) return PA_ERR_NULL;
  if (!aligned(src_dst_pairs, 8)) return PA_ERR_ALIGN;
  const int64_t block_bytes = static_cast<int64_t>(src[0].block_size) * src[0].num_kv_heads *
                              src[0].head_dim * static_cast<int64_t>(elem_bytes(src[0]));
  if (num_pairs * ((block_bytes + 32767) / 32768) > 0x7fffffffLL) return PA_ERR_SHAPE;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  // every pool and the pairs must be reachable from this device: no pageable memory
  if (!device_reachable(src_dst_pairs)) return PA_ERR_ARG;
  for (int32_t l = 0; l < num_layers; ++l) {
    if (!device_reachable(src[l].k) || !device_reachable(src[l].v) ||
        !device_reachable(dst[l].k) || !device_reachable(dst[l].v))
      return PA_ERR_ARG;
  }
  for (int32_t l0 = 0; l0 < num_layers; l0 += pa::kMaxCopyLayers) {
    const int32_t n = (num_layers - l0) < pa::kMaxCopyLayers ? (num_layers - l0) : pa::kMaxCopyLayers;
    pa::SwapLayers layers{};
    for (int32_t i = 0; i < n; ++i) {
      layers.src_k[i] = src[l0 + i].k;
      layers.src_v[i] = src[l0 + i].v;
      layers.dst_k[i] = dst[l0 + i].k;
      layers.dst_v[i] = dst[l0 + i].v;
    }
    const cudaError_t e = pa::launch_swap_blocks(layers, n, src_dst_pairs, num_pairs,
                                                 src[0].num_blocks, dst[0].num_blocks, block_bytes,
                                                 di.err, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

int pa_prefix_hash(const int32_t* token_ids, const int64_t* token_offsets,
                   const int64_t* key_offsets, int32_t num_seqs, int32_t block_size,
                   const uint8_t* root, uint8_t* keys, void* stream) {
  if (num_seqs < 0) return PA_ERR_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!token_ids || !token_offsets || !key_offsets || !keys) return PA_ERR_NULL;
  if (block_size <= 0 || block_size > 4096) return PA_ERR_SHAPE;
  if (!aligned(token_ids, 4) || !aligned(token_offsets, 8) || !aligned(key_offsets, 8) ||
      !aligned(keys, 16))
    return PA_ERR_ALIGN;
  pa::Sha256Root r{};
  for (int i = 0; i < 8; ++i) {  // the root's bytes, read as big-endian words
    uint32_t w = 0;
    for (int j = 0; j < 4; ++j) w = (w << 8) | (root ? root[4 * i + j] : 0u);
    r.w[i] = w;
  }
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_prefix_hash(token_ids, token_offsets, key_offsets, num_seqs,
                                               block_size, r, keys, di.err,
                                               static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_prefix_key_offsets(const int64_t* token_offsets, int32_t num_seqs, int32_t block_size,
                          int64_t* key_offsets, void* stream) {
  if (num_seqs < 0) return PA_ERR_ARG;
  if (!token_offsets || !key_offsets) return PA_ERR_NULL;
  if (block_size <= 0 || block_size > 4096) return PA_ERR_SHAPE;
  if (!aligned(token_offsets, 8) || !aligned(key_offsets, 8)) return PA_ERR_ALIGN;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  const cudaError_t e = pa::launch_key_offsets(token_offsets, num_seqs, block_size, key_offsets,
                                               di.err, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

size_t pa_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t max_seq_len, int32_t partition_tokens) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  if (partition_tokens == PA_PARTITION_BALANCED) {
    DeviceInfo di;
    if (!device_info(&di)) return 0;
    const BalancedLayout lay = balanced_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, di.sms);
    return lay.total;
  }
  const int64_t parts = decode_parts(max_seq_len, partition_tokens);
  if (parts <= 1) return 0;
  return static_cast<size_t>(num_seqs) * num_q_heads * parts * (head_dim + 2) * sizeof(float);
}

const char* pa_decode_kernel_name(int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t max_seq_len,
                                  int32_t partition_tokens) {
  if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return nullptr;
  if (head_dim != 64 && head_dim != 128 && head_dim != 256) return nullptr;
  if (block_size <= 0 || !(block_size % pa::kStageRows == 0 || pa::kStageRows % block_size == 0))
    return nullptr;
  if (max_seq_len < 0 || partition_tokens < PA_PARTITION_BALANCED) return nullptr;
  if (partition_tokens == PA_PARTITION_BALANCED) {
    const BalancedPlan plan =
        balanced_plan(num_kv_heads, num_q_heads / num_kv_heads, head_dim, block_size, 1);
    return plan.kernel == pa::kGroupedRanges ? "decode_grouped_kernel+decode_piece_merge_kernel"
                                             : "decode_balanced_kernel";
  }
  if (partition_tokens != 0 && partition_tokens % pa::kStageRows != 0) return nullptr;
  return decode_parts(max_seq_len, partition_tokens) > 1 ? "decode_kernel+decode_reduce_kernel"
                                                         : "decode_kernel";
}

int32_t pa_decode_default_partition(int32_t num_seqs, int32_t num_kv_heads, int32_t max_seq_len,
                                    int32_t block_size) {
  if (num_seqs < 0 || num_kv_heads <= 0 || max_seq_len < 0 || block_size <= 0) return PA_ERR_ARG;
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  // Whole (sequence, KV head) units, scheduled by the hardware, balance well
  // once there are many of them per SM; below that, ragged lengths leave SMs
  // idle at the end and the balanced split (equal stage ranges per warp) wins.
  const int64_t units = static_cast<int64_t>(num_seqs) * num_kv_heads;
  // Short contexts: one CTA streams a (sequence, KV head) of at most 16 stages
  // in about the balanced split's fixed cost (its line prefix, counter memset
  // and persistent grid; measured on GB300: 4 sequences of up to 33 tokens
  // decode in 8.5 us single pass, 35.3 us balanced).
  if (units == 0 || max_seq_len <= 256) return 0;
  const int64_t tt = block_size < pa::kStageRows ? 2LL * block_size : pa::kStageRows;
  const bool balanced_fits = num_seqs <= pa::kMaxBalancedSeqs &&
                             num_kv_heads <= 2LL * di.sms * pa::kDecodeWarps &&
                             units * ((max_seq_len + tt - 1) / tt) <= 0x7fffffffLL;
  if (balanced_fits && units < 64LL * di.sms) return PA_PARTITION_BALANCED;
  if (units >= 8LL * di.sms || max_seq_len <= 512) return 0;
  // few units but no balanced split: fixed partitions, ~16 CTAs per SM
  const int64_t parts = (16LL * di.sms + units - 1) / units;
  int64_t pt = (max_seq_len + parts - 1) / parts;
  pt = ((pt + 255) / 256) * 256;
  pt = pt < 512 ? 512 : (pt > 2048 ? 2048 : pt);
  return pt >= max_seq_len ? 0 : static_cast<int32_t>(pt);
}

size_t pa_prefill_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int32_t max_q_len) {
  DeviceInfo di;
  if (!device_info(&di)) return 0;
  const MultiPlan p = multi_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                                 max_q_len, di.sms);
  return p.ok ? multi_layout(num_seqs, num_kv_heads, p, di.sms).total : 0;
}

const char* pa_prefill_kernel_name(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t block_size, int32_t max_q_len,
                                   int32_t with_workspace, int32_t num_sms) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_q_len <= 0 ||
      num_q_heads % num_kv_heads != 0 || num_sms < 0)
    return nullptr;
  if (num_sms == 0) {
    DeviceInfo di;
    if (!device_info(&di)) return nullptr;
    num_sms = di.sms;
  }
  const bool multi_ok =
      multi_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_q_len, num_sms).ok;
  const int64_t rows = static_cast<int64_t>(max_q_len) * (num_q_heads / num_kv_heads);
  switch (route_prefill(multi_ok, with_workspace != 0, true, head_dim, rows, true)) {
    case kPrefillMulti: return "multi_grouped_kernel";
    case kPrefillTc: return "prefill_tc_kernel";
    default: return "prefill_kernel";
  }
}

int pa_prefill(const void* q, int32_t num_seqs, const int32_t* q_start, int32_t max_q_len,
               int32_t num_q_heads, const pa_cache* cache, const int32_t* block_tables,
               int32_t max_blocks_per_seq, const int32_t* seq_lens, float scale, void* out,
               pa_dtype out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  const bool fp8 = is_fp8(*cache);
  if (num_seqs < 0 || num_q_heads <= 0 || max_q_len < 0 || max_blocks_per_seq <= 0)
    return PA_ERR_ARG;
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (!q || !q_start || !block_tables || !seq_lens || !out) return PA_ERR_NULL;
  if (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32) return PA_ERR_DTYPE;
  const int D = cache->head_dim;
  const int b = cache->block_size;
  const int hkv = cache->num_kv_heads;
  if (D != 64 && D != 128 && D != 256) return PA_ERR_SHAPE;
  if (fp8 && D == 64) return PA_ERR_SHAPE;
  if (b < 8 || !(64 % b == 0 || b % 64 == 0)) return PA_ERR_SHAPE;
  if (num_q_heads % hkv != 0) return PA_ERR_SHAPE;
  if (num_seqs > 65535 || hkv > 65535) return PA_ERR_SHAPE;
  if (!std::isfinite(scale)) return PA_ERR_ARG;
  if (!aligned(q, 4) || !aligned(out, 4)) return PA_ERR_ALIGN;
  const int g = num_q_heads / hkv;
  const int64_t tiles = (static_cast<int64_t>(max_q_len) * g + 63) / 64;
  if (tiles > 0x7fffffffLL) return PA_ERR_SHAPE;

  pa::PrefillArgs a{};
  a.q = q;
  a.out = out;
  a.q_start = q_start;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.num_blocks = cache->num_blocks;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = hkv;
  a.group = g;
  a.block_size = b;
  a.max_blocks = max_blocks_per_seq;
  a.tok_per_op = b < 64 ? b : 64;
  a.ops_per_stage = 64 / a.tok_per_op;
  a.out_dtype = out_dtype;
  // E4M3: the logit of code row c is scale * k_scale * (q . value(c))
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) *
                                    (fp8 ? static_cast<double>(cache->k_scale) : 1.0) *
                                    1.4426950408889634);
  a.v_scale = fp8 ? cache->v_scale : 1.f;
  a.test_stop_stage = g_stall_stage.load();
  a.test_wait_ns = g_stall_wait_ns.load();
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  a.err = di.err;
  cudaError_t e;
  const bool act_bf16 = (fp8 ? cache->act_dtype : cache->dtype) == PA_BF16;
  const MultiPlan mp = multi_plan(num_seqs, num_q_heads, hkv, D, b, max_q_len, di.sms);
  // the stage line's per-sequence offsets are int32 in the kernel
  const int64_t line_cap = static_cast<int64_t>(num_seqs) *
                           ((static_cast<int64_t>(max_blocks_per_seq) * b + pa::kStageRows - 1) /
                            pa::kStageRows);
  const PrefillKernel route =
      route_prefill(mp.ok, workspace_bytes > 0, line_cap <= 0x7fffffffLL, D,
                    static_cast<int64_t>(max_q_len) * g, aligned(q, 16) && aligned(out, 16));
  if (route == kPrefillMulti) {
    // A few new tokens per sequence: the balanced, head-grouped stream with
    // (query, head) rows as the MMA columns.
    const BalancedLayout lay = multi_layout(num_seqs, hkv, mp, di.sms);
    if (workspace == nullptr || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
    if (!aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(q_start, 4))
      return PA_ERR_ALIGN;
    pa::DecodeArgs d{};
    d.q = q;
    d.out = out;
    d.block_tables = block_tables;
    d.seq_lens = seq_lens;
    d.err = di.err;
    d.num_blocks = cache->num_blocks;
    d.num_seqs = num_seqs;
    d.num_q_heads = num_q_heads;
    d.num_kv_heads = hkv;
    d.group = g;
    d.block_size = b;
    d.max_blocks = max_blocks_per_seq;
    d.max_seq_len = 0x7fffffff;
    d.max_parts = 1;
    d.tok_per_op = pa::kStageRows;
    d.slot_rows = pa::kStageRows;
    d.ops_per_stage = 1;
    d.out_dtype = out_dtype;
    d.scale_log2 = a.scale_log2;
    d.v_scale = a.v_scale;
    d.q_start = q_start;
    d.max_q = max_q_len;
    char* ws = static_cast<char*>(workspace);
    d.counters = reinterpret_cast<unsigned int*>(ws);
    d.part_ml = reinterpret_cast<float*>(ws + lay.ml_offset);
    d.part_o = reinterpret_cast<float*>(ws + lay.o_offset);
    CUtensorMap gk, gv;
    if (!encode_grouped_map(&gk, cache->k, *cache, pa::kStageRows, mp.head_group) ||
        !encode_grouped_map(&gv, cache->v, *cache, pa::kStageRows, mp.head_group))
      return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // arrival counters start each call at zero, whatever the workspace held
    e = cudaMemsetAsync(d.counters, 0,
                        static_cast<size_t>(num_seqs) * hkv * mp.row_tiles * sizeof(unsigned int), st);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    const dim3 grid(mp.ctas, 1, 1);
    if (fp8) {
      e = act_bf16 ? pa::launch_multi_e4m3_bf16(gk, gv, d, mp.nt, mp.row_tiles, mp.head_group, grid, st)
                   : pa::launch_multi_e4m3_f16(gk, gv, d, mp.nt, mp.row_tiles, mp.head_group, grid, st);
    } else {
      e = act_bf16 ? pa::launch_multi_bf16(gk, gv, d, mp.nt, mp.row_tiles, mp.head_group, grid, st)
                   : pa::launch_multi_f16(gk, gv, d, mp.nt, mp.row_tiles, mp.head_group, grid, st);
    }
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  CUtensorMap tk, tv;
  if (!encode_cache_map(&tk, cache->k, *cache, a.tok_per_op) ||
      !encode_cache_map(&tv, cache->v, *cache, a.tok_per_op))
    return PA_ERR_CUDA;
  if (route == kPrefillTc) {
    // 5th-generation tensor cores: 256 (query, head) rows per CTA, S and O in
    // TMEM. Batches of fewer rows per KV head (speculative verification of a few
    // drafts) stay on the 64-row kernel, whose tiles they fill.
    const int64_t tiles256 = (static_cast<int64_t>(max_q_len) * g + 255) / 256;
    const dim3 grid(static_cast<unsigned>(tiles256), static_cast<unsigned>(hkv),
                    static_cast<unsigned>(num_seqs));
    e = fp8 ? pa::launch_prefill_tc_e4m3(tk, tv, a, act_bf16, grid, static_cast<cudaStream_t>(stream))
            : pa::launch_prefill_tc128(tk, tv, a, act_bf16, grid, static_cast<cudaStream_t>(stream));
  } else {
    const dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(hkv),
                    static_cast<unsigned>(num_seqs));
    const bool thin = D == 128 && static_cast<int64_t>(max_q_len) * g <= 32;
    e = pa::launch_prefill(tk, tv, a, D, act_bf16, fp8, thin, grid,
                           static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode(const void* q, int32_t num_seqs, int32_t num_q_heads, const pa_cache* cache,
              const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
              int32_t max_seq_len, float scale, void* out, pa_dtype out_dtype,
              int32_t partition_tokens, void* workspace, size_t workspace_bytes, void* stream) {
  int rc = check_cache(cache);
  if (rc != PA_OK) return rc;
  if (num_seqs < 0 || num_q_heads <= 0) return PA_ERR_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!q || !block_tables || !seq_lens || !out) return PA_ERR_NULL;
  if (out_dtype != PA_F16 && out_dtype != PA_BF16 && out_dtype != PA_F32) return PA_ERR_DTYPE;
  const int D = cache->head_dim;
  const int b = cache->block_size;
  const int hkv = cache->num_kv_heads;
  const bool fp8 = is_fp8(*cache);
  if (D != 64 && D != 128 && D != 256) return PA_ERR_SHAPE;
  if (fp8 && D == 64) return PA_ERR_SHAPE;
  if (!(b % pa::kStageRows == 0 || pa::kStageRows % b == 0)) return PA_ERR_SHAPE;
  if (num_q_heads % hkv != 0) return PA_ERR_SHAPE;
  const int g = num_q_heads / hkv;
  if (g > 16) return PA_ERR_SHAPE;
  if (max_blocks_per_seq <= 0 || max_seq_len < 0) return PA_ERR_ARG;
  const bool balanced = partition_tokens == PA_PARTITION_BALANCED;
  if (!balanced && (partition_tokens < 0 || partition_tokens % pa::kStageRows != 0)) return PA_ERR_ARG;
  if (!std::isfinite(scale)) return PA_ERR_ARG;
  if (!aligned(q, 4) || !aligned(out, 4) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
    return PA_ERR_ALIGN;
  const int64_t parts = balanced ? 1 : decode_parts(max_seq_len, partition_tokens);
  if (parts > 65535 || num_seqs > 65535 || hkv > 65535) return PA_ERR_SHAPE;
  // partial indices (row * partitions + partition) are 32-bit in the merges
  if (static_cast<int64_t>(num_seqs) * num_q_heads * parts > 0x7fffffffLL) return PA_ERR_SHAPE;
  if (balanced) {
    // every per-sequence stage offset must fit the kernel's int32 prefix sums
    const int64_t tt = b < pa::kStageRows ? 2LL * b : pa::kStageRows;
    const int64_t max_stages = static_cast<int64_t>(num_seqs) * hkv * ((max_seq_len + tt - 1) / tt);
    if (num_seqs > pa::kMaxBalancedSeqs || max_stages > 0x7fffffffLL) return PA_ERR_SHAPE;
  }

  pa::DecodeArgs a{};
  a.q = q;
  a.out = out;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.num_blocks = cache->num_blocks;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = hkv;
  a.group = g;
  a.block_size = b;
  a.max_blocks = max_blocks_per_seq;
  a.max_seq_len = max_seq_len;
  a.part_tokens = parts > 1 ? partition_tokens : 0;
  a.max_parts = static_cast<int32_t>(parts);
  a.tok_per_op = b < pa::kStageRows ? b : pa::kStageRows;
  a.slot_rows = a.tok_per_op < 8 ? 8 : a.tok_per_op;
  a.ops_per_stage = pa::kStageRows / a.slot_rows;
  a.out_dtype = out_dtype;
  // E4M3: the logit of code row c is scale * k_scale * (q . value(c))
  const double kscale = fp8 ? static_cast<double>(cache->k_scale) : 1.0;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * kscale * 1.4426950408889634);
  a.v_scale = fp8 ? cache->v_scale : 1.f;
  a.test_stop_stage = g_stall_stage.load();
  a.test_wait_ns = g_stall_wait_ns.load();
  dim3 grid(static_cast<unsigned>(hkv), static_cast<unsigned>(parts),
            static_cast<unsigned>(num_seqs));
  if (!balanced && parts > 1) {
    const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, hkv, D, max_seq_len,
                                                  partition_tokens);
    if (workspace == nullptr || workspace_bytes < need) return PA_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return PA_ERR_ALIGN;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = a.part_o + static_cast<int64_t>(num_seqs) * num_q_heads * parts * D;
  }
  DeviceInfo di;
  if (!device_info(&di)) return PA_ERR_CUDA;
  a.err = di.err;
  int kernel = pa::kPerPartition;
  int head_group = 1;
  if (balanced) {
    const BalancedLayout lay = balanced_layout(num_seqs, num_q_heads, hkv, D, di.sms);
    const BalancedPlan plan = balanced_plan(hkv, g, D, b, di.sms);
    // every range needs one warp per KV head (or one CTA per head group)
    const int64_t units = plan.kernel == pa::kGroupedRanges
                              ? static_cast<int64_t>(plan.ctas) / (hkv / plan.head_group)
                              : static_cast<int64_t>(plan.ctas) * pa::kDecodeWarps / hkv;
    if (units < 1) return PA_ERR_SHAPE;
    if (workspace == nullptr || workspace_bytes < lay.total) return PA_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PA_ERR_ALIGN;
    char* ws = static_cast<char*>(workspace);
    a.counters = reinterpret_cast<unsigned int*>(ws);
    a.part_ml = reinterpret_cast<float*>(ws + lay.ml_offset);
    a.part_o = reinterpret_cast<float*>(ws + lay.o_offset);
    head_group = plan.head_group;
    kernel = plan.kernel;
    grid = dim3(plan.ctas, 1, 1);
  }

  CUtensorMap tk, tv;
  const bool grouped = kernel == pa::kGroupedRanges;
  if (grouped ? (!encode_grouped_map(&tk, cache->k, *cache, a.tok_per_op, head_group) ||
                 !encode_grouped_map(&tv, cache->v, *cache, a.tok_per_op, head_group))
              : (!encode_cache_map(&tk, cache->k, *cache, a.tok_per_op) ||
                 !encode_cache_map(&tv, cache->v, *cache, a.tok_per_op)))
    return PA_ERR_CUDA;

  const int tiles = (g + 7) / 8;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (balanced && !grouped) {
    // arrival counters start each call at zero, whatever the workspace held
    // (the grouped kernel counts nothing: its merge is a kernel of its own)
    static_assert(pa::kPerWarpRanges == 1, "kernel ids");
    e = cudaMemsetAsync(a.counters, 0, static_cast<size_t>(num_seqs) * hkv * sizeof(unsigned int), st);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  if (fp8) {
    if (cache->act_dtype == PA_F16) {
      e = D == 128 ? pa::launch_decode_e4m3_f16_128(tk, tv, a, tiles, head_group, grid, kernel, st)
                   : pa::launch_decode_e4m3_f16_256(tk, tv, a, tiles, head_group, grid, kernel, st);
    } else {
      e = D == 128 ? pa::launch_decode_e4m3_bf16_128(tk, tv, a, tiles, head_group, grid, kernel, st)
                   : pa::launch_decode_e4m3_bf16_256(tk, tv, a, tiles, head_group, grid, kernel, st);
    }
  } else if (cache->dtype == PA_F16) {
    e = D == 64 ? pa::launch_decode_f16_64(tk, tv, a, tiles, head_group, grid, kernel, st)
        : D == 128 ? pa::launch_decode_f16_128(tk, tv, a, tiles, head_group, grid, kernel, st)
                   : pa::launch_decode_f16_256(tk, tv, a, tiles, head_group, grid, kernel, st);
  } else {
    e = D == 64 ? pa::launch_decode_bf16_64(tk, tv, a, tiles, head_group, grid, kernel, st)
        : D == 128 ? pa::launch_decode_bf16_128(tk, tv, a, tiles, head_group, grid, kernel, st)
                   : pa::launch_decode_bf16_256(tk, tv, a, tiles, head_group, grid, kernel, st);
  }
  if (e != cudaSuccess) return PA_ERR_CUDA;
  if (!balanced && parts > 1) {
    e = pa::launch_decode_reduce(a, D, st);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  if (grouped) {
    const int64_t ranges = static_cast<int64_t>(grid.x) / (hkv / head_group);
    e = pa::launch_decode_piece_merge(a, D, ranges, pa::grouped_line_tokens(fp8), di.sms, st);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // extern "C"
