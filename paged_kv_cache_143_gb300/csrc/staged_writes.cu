// staged_writes.cu — pa_apply_staged_writes.
//
// [MRV2 "재설계 3: 큰 block table은 staged diff만 보낸다"]: the device block table
// is the reference copy; the host sends only (row, start, values) diffs in one
// small staging buffer and one kernel applies them; the rows needed this step
// are then gathered by idx_mapping ([MRV2 "재설계 1"]).
//
// One launch, two kinds of CTA that never touch the same cell:
//  - writer CTAs apply value k of diff w to table[row_w][start_w + k] unless a
//    later diff also covers that cell (so the result is last-writer-wins in
//    record order, independent of thread timing). One warp per diff: it first
//    collects the later diffs of the same row (one coalesced pass over the
//    later records' rows, O(W) per diff, not per value), then each lane checks
//    its cells against only those;
//  - gather CTA i builds gathered[i][c] directly: the value of the latest diff
//    that covers (idx_mapping[i], c), else the untouched table cell. Covered
//    cells are never read, uncovered cells are never written: no race.
// Integer work, bit-exact.
#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kWriterWarps = kThreads / 32;
constexpr int kLaterCap = 64;     // later overlapping diffs a writer warp keeps per diff
constexpr int kRowDiffCap = 512;  // diffs of one row kept in shared memory

struct Diffs {
  const int32_t* rows;
  const int32_t* starts;
  const int32_t* offs;  // [W+1]
  const int32_t* vals;
  int32_t W;
};

__device__ __forceinline__ bool diff_valid(const Diffs& d, int32_t w, int32_t max_reqs,
                                           int32_t max_blocks) {
  const int32_t row = d.rows[w], start = d.starts[w];
  const int32_t len = d.offs[w + 1] - d.offs[w];
  return row >= 0 && row < max_reqs && start >= 0 && len >= 0 &&
         (int64_t)start + len <= max_blocks && d.offs[w] >= 0 && d.offs[w + 1] <= d.offs[d.W];
}

__device__ __forceinline__ bool diff_covers(const Diffs& d, int32_t w, int32_t row, int32_t col) {
  if (d.rows[w] != row) return false;
  const int32_t start = d.starts[w];
  return col >= start && col < start + (d.offs[w + 1] - d.offs[w]);
}

__global__ void __launch_bounds__(kThreads) staged_writes_kernel(
    int32_t* __restrict__ table, int32_t max_reqs, int32_t max_blocks, Diffs d,
    const int32_t* __restrict__ idx_mapping, int32_t R, int32_t* __restrict__ gathered,
    int32_t n_writer_ctas, unsigned* err) {
  __shared__ int32_t row_diffs[kRowDiffCap];
  __shared__ int32_t n_row_diffs;

  if ((int32_t)blockIdx.x < n_writer_ctas) {
    // ------------------------------------------------------------- writers
    __shared__ int2 later[kWriterWarps][kLaterCap];  // [start, end) of later same-row diffs
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned full = 0xffffffffu;
    const int32_t n_warps = n_writer_ctas * kWriterWarps;
    for (int32_t w = blockIdx.x * kWriterWarps + warp; w < d.W; w += n_warps) {
      if (!diff_valid(d, w, max_reqs, max_blocks)) {
        if (lane == 0) pa::raise_error(err, pa::kErrBounds);
        continue;
      }
      const int32_t row = d.rows[w], start = d.starts[w];
      const int32_t len = d.offs[w + 1] - d.offs[w];
      if (len == 0) continue;
      // the later diffs of this row that overlap [start, start + len)
      int n_later = 0;
      bool spilled = false;
      for (int32_t b = w + 1; b < d.W; b += 32) {
        const int32_t w2 = b + lane;
        bool hit = false;
        int2 iv = make_int2(0, 0);
        if (w2 < d.W && d.rows[w2] == row && diff_valid(d, w2, max_reqs, max_blocks)) {
          iv.x = d.starts[w2];
          iv.y = iv.x + (d.offs[w2 + 1] - d.offs[w2]);
          hit = iv.x < start + len && iv.y > start;
        }
        const unsigned m = __ballot_sync(full, hit);
        const int k = n_later + __popc(m & ((1u << lane) - 1u));
        if (hit && k < kLaterCap) later[warp][k] = iv;
        n_later += __popc(m);
      }
      if (n_later > kLaterCap) {
        spilled = true;
        n_later = kLaterCap;
      }
      __syncwarp();
      for (int32_t k = lane; k < len; k += 32) {
        const int32_t col = start + k;
        bool overwritten = false;
        for (int i = 0; i < n_later && !overwritten; ++i)
          overwritten = col >= later[warp][i].x && col < later[warp][i].y;
        // more overlapping later diffs than the list holds: check the rest
        for (int32_t w2 = w + 1; spilled && w2 < d.W && !overwritten; ++w2)
          overwritten = diff_covers(d, w2, row, col) && diff_valid(d, w2, max_reqs, max_blocks);
        if (!overwritten) table[(int64_t)row * max_blocks + col] = d.vals[d.offs[w] + k];
      }
      __syncwarp();
    }
    return;
  }

  // --------------------------------------------------------------- gather
  const int32_t i = blockIdx.x - n_writer_ctas;
  if (i >= R) return;
  const int32_t slot = idx_mapping[i];
  if (slot < 0 || slot >= max_reqs) {
    if (threadIdx.x == 0) pa::raise_error(err, pa::kErrBounds);
    return;
  }
  if (threadIdx.x == 0) n_row_diffs = 0;
  __syncthreads();
  for (int32_t w = threadIdx.x; w < d.W; w += kThreads) {
    if (d.rows[w] == slot && diff_valid(d, w, max_reqs, max_blocks)) {
      const int32_t k = atomicAdd(&n_row_diffs, 1);
      if (k < kRowDiffCap) row_diffs[k] = w;
    }
  }
  __syncthreads();
  const int32_t nd = n_row_diffs;
  const int32_t* src_row = table + (int64_t)slot * max_blocks;
  int32_t* out_row = gathered + (int64_t)i * max_blocks;
  for (int32_t c = threadIdx.x; c < max_blocks; c += kThreads) {
    int32_t best = -1;
    if (nd <= kRowDiffCap) {
      for (int32_t k = 0; k < nd; ++k) {
        const int32_t w = row_diffs[k];
        if (w > best && diff_covers(d, w, slot, c)) best = w;
      }
    } else {  // more diffs on this row than fit in shared memory: scan all
      for (int32_t w = d.W - 1; w >= 0 && best < 0; --w)
        if (diff_covers(d, w, slot, c) && diff_valid(d, w, max_reqs, max_blocks)) best = w;
    }
    out_row[c] = best >= 0 ? d.vals[d.offs[best] + (c - d.starts[best])] : src_row[c];
  }
}

}  // namespace

extern "C" pa_status pa_apply_staged_writes(int32_t* table, int32_t max_reqs, int32_t max_blocks,
                                            const int32_t* rows, const int32_t* starts,
                                            const int32_t* val_offsets, const int32_t* vals,
                                            int32_t W, const int32_t* idx_mapping, int32_t R,
                                            int32_t* gathered, pa_stream_t stream) {
  if (W < 0 || R < 0 || max_reqs < 0 || max_blocks < 0) return PA_ERR_INVALID;
  if ((W > 0 || R > 0) && (!table || max_blocks <= 0 || max_reqs <= 0)) return PA_ERR_INVALID;
  if (W > 0 && (!rows || !starts || !val_offsets || !vals)) return PA_ERR_INVALID;
  if (R > 0 && (!idx_mapping || !gathered)) return PA_ERR_INVALID;
  if (W == 0 && R == 0) return PA_OK;
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  // Writer CTAs: one warp per diff, capped; they grid-stride over the diffs.
  int64_t writers = 0;
  if (W > 0) {
    writers = ((int64_t)W + kWriterWarps - 1) / kWriterWarps;
    const int64_t cap = (int64_t)pa::num_sms() * 4;
    if (writers > cap) writers = cap;
  }
  const int64_t grid = writers + R;
  if (grid > 0x7FFFFFFF) return PA_ERR_INVALID;
  Diffs d{rows, starts, val_offsets, vals, W};
  staged_writes_kernel<<<(unsigned)grid, kThreads, 0, pa::as_stream(stream)>>>(
      table, max_reqs, max_blocks, d, idx_mapping, R, gathered, (int32_t)writers, err);
  return pa::launch_status();
}
