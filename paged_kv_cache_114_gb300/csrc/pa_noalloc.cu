// pa_noalloc.cu - split-K decode for callers that cannot allocate device memory.
//
// pa_decode's split-K path needs a workspace for its per-partition partials,
// and normally the caller allocates it. Some callers cannot do that: code that
// lives inside a host application owning every byte of device memory through
// its own pool (a side cudaMalloc would break its budget or fail mid-serving),
// latency-critical paths where cudaMalloc/cudaFree may synchronise the device
// and stall other streams, and thin bindings from runtimes that expose no
// device allocator at all. For them, pa_decode_static_workspace keeps the
// workspace in a fixed array compiled into this library.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds PA_STATIC_WORKSPACE_BYTES of it until the process exits. In
// host code the symbol names only a host-side stand-in; its device address
// comes from cudaGetSymbolAddress, taken once per device, with that device
// current, on the first call made on it.
#include <cuda_runtime.h>

#include <mutex>

#include "pa_internal.h"

namespace {

constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

std::mutex g_ws_mu;
void* g_ws_addr[kMaxDevices] = {};

// Device address of g_static_workspace on the current device, or nullptr.
void* static_workspace_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_ws_mu);
  if (g_ws_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess) return nullptr;
    g_ws_addr[dev] = p;
  }
  return g_ws_addr[dev];
}

}  // namespace

extern "C" int pa_decode_static_workspace(const void* q, int32_t num_seqs, int32_t num_q_heads,
                                          const pa_cache* cache, const int32_t* block_tables,
                                          int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                          int32_t max_seq_len, float scale, void* out,
                                          pa_dtype out_dtype, int32_t partition_tokens,
                                          void* stream) {
  if (cache == nullptr) return PA_ERR_NULL;
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, cache->num_kv_heads,
                                                cache->head_dim, max_seq_len, partition_tokens);
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0) {
    ws = static_workspace_address();
    if (ws == nullptr) return PA_ERR_CUDA;
  }
  return pa_decode(q, num_seqs, num_q_heads, cache, block_tables, max_blocks_per_seq, seq_lens,
                   max_seq_len, scale, out, out_dtype, partition_tokens, ws,
                   need > 0 ? static_cast<size_t>(PA_STATIC_WORKSPACE_BYTES) : 0, stream);
}
