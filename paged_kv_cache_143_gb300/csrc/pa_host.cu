// pa_host.cu — per-device error word, status strings, shared host checks.
#include <atomic>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {
__device__ unsigned g_error_word;  // sticky bits: pa::kErrBounds | pa::kErrTimeout
__device__ unsigned g_error_taken;  // where pa_get_error's exchange leaves the bits

constexpr int kMaxDevices = 64;
unsigned* g_word_addr[kMaxDevices];
int g_sms[kMaxDevices];
std::mutex g_mu;
std::atomic<unsigned long long> g_launches{0};

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

namespace pa {

unsigned* error_word() {
  int dev = current_device();
  if (dev < 0) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_word_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    g_word_addr[dev] = static_cast<unsigned*>(p);
  }
  return g_word_addr[dev];
}

int num_sms() {
  int dev = current_device();
  if (dev < 0) return 1;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
void uncount_launches(unsigned n) { g_launches.fetch_sub(n, std::memory_order_relaxed); }
unsigned long long launches_so_far() { return g_launches.load(std::memory_order_relaxed); }

pa_status check_pool(const pa_kv_pool* pool) {
  if (!pool || !pool->k_pool || !pool->v_pool) return PA_ERR_INVALID;
  if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool)) return PA_ERR_INVALID;
  if (pool->num_blocks < 0 || pool->num_kv_heads <= 0) return PA_ERR_INVALID;
  if (pool->head_dim != 64 && pool->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (pool->block_size != 16 && pool->block_size != 32 && pool->block_size != 64)
    return PA_ERR_UNSUPPORTED;
  if (pool->dtype != PA_KV_BF16 && pool->dtype != PA_KV_FP8_E4M3) return PA_ERR_UNSUPPORTED;
  if (pool->dtype == PA_KV_FP8_E4M3 &&
      !(pool->k_scale > 0.0f && pool->v_scale > 0.0f && pool->k_scale < 3.0e38f &&
        pool->v_scale < 3.0e38f))
    return PA_ERR_INVALID;
  return PA_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace pa

namespace {
// Reads and clears the error word in one atomic exchange, so that a bit set
// by a kernel on another stream is either returned now or kept for the next
// call, never cleared unseen.
__global__ void take_error_kernel(unsigned* word, unsigned* taken) {
  *taken = atomicExch(word, 0u);
}
std::mutex g_take_mu;  // one taker at a time per process (they share g_error_taken)
}  // namespace

extern "C" pa_status pa_get_error(pa_stream_t stream) {
  cudaStream_t s = pa::as_stream(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return PA_ERR_CUDA;
  unsigned* w = pa::error_word();
  if (!w) return PA_ERR_CUDA;
  unsigned bits = 0;
  {
    std::lock_guard<std::mutex> lock(g_take_mu);
    void* taken = nullptr;
    if (cudaGetSymbolAddress(&taken, g_error_taken) != cudaSuccess) return PA_ERR_CUDA;
    take_error_kernel<<<1, 1, 0, s>>>(w, static_cast<unsigned*>(taken));
    if (pa::launch_status() != PA_OK) return PA_ERR_CUDA;
    if (cudaMemcpyAsync(&bits, taken, sizeof bits, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  if (bits & 2u) return PA_ERR_TIMEOUT;
  if (bits & 1u) return PA_ERR_DEVICE_BOUNDS;
  return PA_OK;
}

extern "C" const char* pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: unsupported shape or dtype";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime error";
    case PA_ERR_DEVICE_BOUNDS: return "PA_ERR_DEVICE_BOUNDS: device index out of range";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: device wait gave up";
  }
  return "unknown pa_status";
}

extern "C" uint64_t pa_kernel_launches(void) {
  return g_launches.load(std::memory_order_relaxed);
}

namespace {
// Waits on a barrier that nothing completes, through the bounded wait every
// kernel of the library uses: it gives up after pa::kWaitLimitNs, records
// kErrTimeout and returns.
__global__ void wait_timeout_kernel(unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pa::mbar_init(&bar, 1);
    pa::fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) pa::mbar_wait(&bar, 0, err);
}
}  // namespace

extern "C" pa_status pa_selftest_wait_timeout(pa_stream_t stream) {
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, pa::as_stream(stream)>>>(err);
  return pa::launch_status();
}
