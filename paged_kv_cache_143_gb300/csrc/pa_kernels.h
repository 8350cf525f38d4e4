// pa_kernels.h — launch interfaces between the pa_forward planner and the
// attention kernels (internal to libpa).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

struct DecodeParams {
  const __nv_bfloat16* q;      // [T][Hq][D]
  __nv_bfloat16* out;          // [T][Hq][D]
  const int32_t* qsl;          // [R+1]
  const int32_t* seq_lens;     // [R]
  const int32_t* block_tables; // [R][max_blocks]
  int32_t max_blocks;
  int32_t Hq, Hkv, g;
  const uint8_t* k_pool;       // [num_blocks][Hkv][B][D] elements of 1 or 2 bytes
  const uint8_t* v_pool;
  int32_t num_blocks, B;
  float q_scale;               // softmax scale * log2(e) * k_scale (FP8) or * 1
  float v_scale;               // v_scale (FP8) or 1
  int32_t split_tokens;        // keys per split (multiple of 16)
  int32_t ws_splits;           // split stride of the workspace arrays
  float* ws_o;                 // [R][Hq][ws_splits][D] unnormalised partial outputs
  float2* ws_ml;               // [R][Hq][ws_splits] (max in log2 units, sum)
  unsigned* err;
};

constexpr int kMaxOrderedPrefill = 256;

struct PrefillParams {
  __nv_bfloat16* out;          // [T][Hq][D]
  const int32_t* qsl;          // [R+1]
  const int32_t* seq_lens;     // [R]
  const int32_t* block_tables; // [R][max_blocks]
  int32_t max_blocks;
  int32_t Hq, Hkv, g;
  int32_t num_blocks, B;
  int32_t causal;
  float scale_log2;            // softmax scale * log2(e) (* k_scale for E4M3 pools)
  float v_scale;               // v_scale for E4M3 pools, else 1
  unsigned* err;
  // prefill requests in launch order (most work first); n_order == 0 means
  // grid.z walks every request in batch order
  int32_t n_order;
  int32_t order[kMaxOrderedPrefill];
};

struct PrefillLaunch {
  PrefillParams p;
  const void* q;               // bf16 [T][Hq][D]
  const void* k_pool;          // [num_blocks][Hkv][B][D]
  const void* v_pool;
  int32_t T, R, D;
  bool fp8;                    // E4M3 pools
  int32_t max_q_tiles;         // max over prefill requests of ceil(q_len * g / 128)
};

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s);

cudaError_t launch_decode(const DecodeParams& p, int D, bool fp8, int R, int max_splits,
                          cudaStream_t s);
cudaError_t launch_merge(const DecodeParams& p, int D, int R, cudaStream_t s);

}  // namespace pa
