// pa_internal.h — host-side helpers shared by the libpa translation units.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pa.h"

namespace pa {

// Device address of the sticky error word of the current device (set up once
// per device); nullptr if the runtime call failed.
unsigned* error_word();

// Number of SMs of the current device (cached per device).
int num_sms();

inline cudaStream_t as_stream(pa_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Counts `n` kernel launches made by the library (reported by
// pa_kernel_launches).
void count_launches(unsigned n);
// Takes back launches counted while a stream was being captured (they run
// when the graph is launched), and reads the running count.
void uncount_launches(unsigned n);
unsigned long long launches_so_far();

// Maps the result of a launch (cudaGetLastError after <<<>>>) to a status and
// counts the launch when it succeeded.
inline pa_status launch_status() {
  if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA;
  count_launches(1);
  return PA_OK;
}

// Shape checks shared by every entry point that takes a pool.
pa_status check_pool(const pa_kv_pool* pool);

// The driver's cuTensorMapEncodeTiled (looked up once); nullptr if the driver
// does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

}  // namespace pa
