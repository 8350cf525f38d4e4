// forward_noalloc.cu — pa_forward_noalloc: pa_forward with its split-KV
// scratch taken from a fixed array that the library itself holds in device
// memory, so the caller never has to allocate a workspace.
//
// Who needs it: code that may not call cudaMalloc (or any allocator) at the
// point where it runs attention — for example a plugin inside a host runtime
// that has already reserved the device memory through its own pool and hands
// plugins no allocator, or a serving loop that bans allocation after start-up
// because cudaMalloc can synchronise the device and stall other streams.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds PA_NOALLOC_SCRATCH_BYTES of it until the process exits. Host
// code cannot use the symbol as a pointer (on the host it only names a
// stand-in), so its device address is looked up once per device with
// cudaGetSymbolAddress and cached. The cache is never invalidated: after
// cudaDeviceReset the address is stale, and the library must not be called
// on that device again in the same process.
#include <mutex>

#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up on the
// first call per device), or nullptr if the lookup failed.
void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" pa_status pa_forward_noalloc(const void* q, void* out, const int32_t* query_start_loc,
                                        const int32_t* seq_lens, const int32_t* qsl_host,
                                        const int32_t* seq_lens_host,
                                        const int32_t* block_tables, int32_t max_blocks,
                                        int32_t num_reqs, int32_t num_tokens,
                                        int32_t num_q_heads, const pa_kv_pool* pool,
                                        float scale, int32_t causal, int32_t max_splits,
                                        pa_stream_t stream) {
  if (!pool || max_splits < 0) return PA_ERR_INVALID;
  const size_t need =
      max_splits > 0 ? pa_forward_workspace_size(num_reqs, num_q_heads, pool->head_dim, max_splits)
                     : 0;
  if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_UNSUPPORTED;
  void* scratch = scratch_address();
  if (!scratch) return PA_ERR_CUDA;
  // Every scratch cell that the merge reads is written earlier in the same
  // call, so nothing needs clearing between calls.
  return pa_forward(q, out, query_start_loc, seq_lens, qsl_host, seq_lens_host, block_tables,
                    max_blocks, num_reqs, num_tokens, num_q_heads, pool, scale, causal,
                    need ? scratch : nullptr, need, stream);
}
