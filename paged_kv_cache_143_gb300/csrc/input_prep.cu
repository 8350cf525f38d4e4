// input_prep.cu — pa_prepare_inputs: one step's query_start_loc, seq_lens,
// positions and slot mapping built on the device from per-slot state.
//
// [MRV2 "재설계 1"]: a live request keeps a fixed persistent slot and the step's
// order is idx_mapping (entry i is slot idx_mapping[i]). [MRV2 "재설계 4"]: the
// running sum of the per-request token counts (query_start_loc), positions,
// seq_lens and the slot mapping are prepared on the GPU, so the host sends
// only the step's (slot, token count) list and the block-table diffs.
// [vLLM-wiki "블록 테이블"]: position p of a request is logical block p / B,
// offset p % B; its pool slot is physical_block * B + offset.
//
// One CTA of 1024 threads (the work is a few thousand integers):
//  1. block-wide scan of the counts (chunks of 1024 entries, carried), which
//     writes query_start_loc and seq_lens = num_computed[slot] + count;
//  2. one warp per entry writes that entry's positions and slots;
//  3. num_computed[slot] = seq_lens.
// A NULL count array means one token per entry (a decode step).
// Integer work, bit-exact. Bad input (slot outside [0, max_reqs), negative
// count, total past the output capacity, a position past the table row or a
// block outside the pool) sets PA_ERR_DEVICE_BOUNDS; the offending slots are
// written as -1 and nothing is written outside the given buffers.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads) prepare_inputs_kernel(
    int32_t* __restrict__ num_computed, int32_t max_reqs, const int32_t* __restrict__ table,
    int32_t max_blocks, int32_t B, int32_t num_blocks, const int32_t* __restrict__ idx_mapping,
    const int32_t* __restrict__ num_scheduled, int32_t R, int32_t T_cap,
    int32_t* __restrict__ qsl, int32_t* __restrict__ seq_lens, int32_t* __restrict__ positions,
    int64_t* __restrict__ slot_mapping, unsigned* err) {
  __shared__ int32_t warp_sums[32];
  __shared__ int32_t carry;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid == 0) {
    carry = 0;
    qsl[0] = 0;
  }
  __syncthreads();
  // ---- 1. scan of the counts; seq_lens from the slot state
  for (int base = 0; base < R; base += kThreads) {
    const int i = base + tid;
    int q = 0;
    if (i < R) {
      q = num_scheduled ? num_scheduled[i] : 1;
      const int s = idx_mapping[i];
      const bool bad = q < 0 || s < 0 || s >= max_reqs;
      if (bad) {
        pa::raise_error(err, pa::kErrBounds);
        q = 0;
      }
      seq_lens[i] = (bad ? 0 : num_computed[s]) + q;
    }
    int x = q;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int incl = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + x;
    if (i < R) qsl[i + 1] = incl;
    __syncthreads();
    if (tid == kThreads - 1) carry = incl;
    __syncthreads();
  }
  if (tid == 0 && carry > T_cap) pa::raise_error(err, pa::kErrBounds);
  // ---- 2. positions and slots, one warp per entry
  for (int i = warp; i < R; i += kThreads / 32) {
    const int s = idx_mapping[i];
    const int q = num_scheduled ? num_scheduled[i] : 1;
    if (q <= 0 || s < 0 || s >= max_reqs) continue;
    const int t0 = qsl[i];
    const int start = seq_lens[i] - q;
    const int32_t* row = table + (int64_t)s * max_blocks;
    for (int j = lane; j < q; j += 32) {
      const int t = t0 + j;
      if (t >= T_cap) break;
      const int pos = start + j;
      const int lb = pos / B;
      int64_t slot = -1;
      if (lb < max_blocks) {
        const int blk = row[lb];
        if (blk >= 0 && blk < num_blocks) slot = (int64_t)blk * B + pos % B;
      }
      if (slot < 0) pa::raise_error(err, pa::kErrBounds);
      positions[t] = pos;
      slot_mapping[t] = slot;
    }
  }
  __syncthreads();
  // ---- 3. the slots' stored-token counts after the step
  for (int i = tid; i < R; i += kThreads) {
    const int s = idx_mapping[i];
    const int q = num_scheduled ? num_scheduled[i] : 1;
    if (q >= 0 && s >= 0 && s < max_reqs) num_computed[s] = seq_lens[i];
  }
}

}  // namespace

extern "C" pa_status pa_prepare_inputs(int32_t* num_computed, int32_t max_reqs,
                                       const int32_t* table, int32_t max_blocks,
                                       int32_t block_size, int32_t num_blocks,
                                       const int32_t* idx_mapping, const int32_t* num_scheduled,
                                       int32_t num_reqs, int32_t token_capacity,
                                       int32_t* query_start_loc, int32_t* seq_lens,
                                       int32_t* positions, int64_t* slot_mapping,
                                       pa_stream_t stream) {
  if (num_reqs < 0 || max_reqs <= 0 || max_blocks < 0 || block_size <= 0 || num_blocks < 0 ||
      token_capacity < 0)
    return PA_ERR_INVALID;
  if (!query_start_loc) return PA_ERR_INVALID;
  if (num_reqs > 0 && (!num_computed || !table || !idx_mapping || !seq_lens))
    return PA_ERR_INVALID;
  if (token_capacity > 0 && (!positions || !slot_mapping)) return PA_ERR_INVALID;
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  prepare_inputs_kernel<<<1, kThreads, 0, pa::as_stream(stream)>>>(
      num_computed, max_reqs, table, max_blocks, block_size, num_blocks, idx_mapping,
      num_scheduled, num_reqs, token_capacity, query_start_loc, seq_lens, positions,
      slot_mapping, err);
  return pa::launch_status();
}
