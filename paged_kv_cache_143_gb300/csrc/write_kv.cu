// write_kv.cu — pa_write_kv (scatter new K/V by slot_mapping, bf16 copy or
// FP8 E4M3 store), pa_copy_blocks (whole-block copy for copy-on-write) and
// pa_gather_rows (rows of a device array gathered by index).
//
// [vLLM-wiki "블록 테이블"]: token t goes to slot s = block * B + offset.
// [vLLM-wiki "엔진 구조와 주요 기능"], [V1-blog "FP8 KV 캐시 양자화의 네이티브 통합"]:
// the cache may be stored as 8-bit floats with a per-tensor scale.
// [vLLM-wiki "블록 공유와 쓰기 시 복사"]: a shared block is copied before a write.
//
// The kernels are HBM scatter/copy/gather work: every thread moves one 16-byte
// vector; consecutive threads cover consecutive bytes of one (token, head) row
// so loads and stores are coalesced.
#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"

namespace {

using pa::kErrBounds;

// E4M3 store of two fp32 values: round to nearest even, saturate finite
// overflow to +-448 (hardware satfinite); NaN is stored as the canonical 0x7F.
__device__ __forceinline__ uint16_t store_e4m3x2(float a, float b) {
  __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  uint16_t lo = c & 0xFF, hi = c >> 8;
  if (a != a) lo = 0x7F;
  if (b != b) hi = 0x7F;
  return static_cast<uint16_t>(lo | (hi << 8));
}

// One thread per 16 bytes of bf16 input (8 elements) of K or V.
// Grid-stride over T * Hkv * (D / 8) * 2 vectors.
template <bool kFp8>
__global__ void __launch_bounds__(256) write_kv_kernel(
    void* __restrict__ k_pool, void* __restrict__ v_pool, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int64_t* __restrict__ slots, int64_t n_vec,
    int32_t Hkv, int32_t D, int32_t B, int64_t num_slots, float k_scale, float v_scale, unsigned* err) {
  const int32_t vec_per_row = D / 8;                 // 16-byte vectors per (token, head)
  const int64_t per_tensor = n_vec / 2;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const bool is_v = i >= per_tensor;
    const int64_t j = is_v ? i - per_tensor : i;
    const int64_t row = j / vec_per_row;              // token * Hkv + head
    const int32_t c = static_cast<int32_t>(j - row * vec_per_row);
    const int64_t t = row / Hkv;
    const int32_t h = static_cast<int32_t>(row - t * Hkv);
    const int64_t s = slots[t];
    if (s < 0) continue;
    if (s >= num_slots) {
      pa::raise_error(err, kErrBounds);
      continue;
    }
    const int64_t blk = s / B, off = s - blk * B;
    const int64_t dst_elem = ((blk * Hkv + h) * B + off) * D + (int64_t)c * 8;
    const uint4 v = is_v ? v_new[j] : k_new[j];
    if (!kFp8) {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(is_v ? v_pool : k_pool) + dst_elem);
      *dst = v;
    } else {
      const float scale = is_v ? v_scale : k_scale;
      float f[8];
      pa::bf16x8_to_f32(v, f);
      uint2 out;
      out.x = store_e4m3x2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale)) |
              (static_cast<uint32_t>(store_e4m3x2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale))) << 16);
      out.y = store_e4m3x2(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale)) |
              (static_cast<uint32_t>(store_e4m3x2(__fdiv_rn(f[6], scale), __fdiv_rn(f[7], scale))) << 16);
      uint2* dst = reinterpret_cast<uint2*>(static_cast<uint8_t*>(is_v ? v_pool : k_pool) + dst_elem);
      *dst = out;
    }
  }
}

// One CTA per (pair, tensor K/V): copies block src[i] to dst[i] with 16-byte
// vectors.
__global__ void __launch_bounds__(256) copy_blocks_kernel(
    uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, int32_t num_blocks, int64_t block_bytes, unsigned* err) {
  const int32_t i = blockIdx.x;
  const int32_t s = src[i], d = dst[i];
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) pa::raise_error(err, kErrBounds);
    return;
  }
  uint8_t* pool = blockIdx.y == 0 ? k_pool : v_pool;
  const uint4* from = reinterpret_cast<const uint4*>(pool + s * block_bytes);
  uint4* to = reinterpret_cast<uint4*>(pool + d * block_bytes);
  const int64_t n = block_bytes / 16;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) to[j] = from[j];
}

}  // namespace

extern "C" pa_status pa_write_kv(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, int32_t T, pa_stream_t stream) {
  pa_status st = pa::check_pool(pool);
  if (st != PA_OK) return st;
  if (T < 0) return PA_ERR_INVALID;
  if (T == 0) return PA_OK;
  if (!k_new || !v_new || !slot_mapping || !pa::aligned16(k_new) || !pa::aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID;
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t n_vec = 2 * (int64_t)T * pool->num_kv_heads * (pool->head_dim / 8);
  const int64_t num_slots = (int64_t)pool->num_blocks * pool->block_size;
  const int threads = 256;
  int64_t blocks = (n_vec + threads - 1) / threads;
  const int64_t cap = (int64_t)pa::num_sms() * 8;
  if (blocks > cap) blocks = cap;
  cudaStream_t s = pa::as_stream(stream);
  if (pool->dtype == PA_KV_BF16)
    write_kv_kernel<false><<<(unsigned)blocks, threads, 0, s>>>(
        pool->k_pool, pool->v_pool, static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), slot_mapping, n_vec, pool->num_kv_heads,
        pool->head_dim, pool->block_size, num_slots, 1.f, 1.f, err);
  else
    write_kv_kernel<true><<<(unsigned)blocks, threads, 0, s>>>(
        pool->k_pool, pool->v_pool, static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), slot_mapping, n_vec, pool->num_kv_heads,
        pool->head_dim, pool->block_size, num_slots, pool->k_scale, pool->v_scale, err);
  return pa::launch_status();
}

extern "C" pa_status pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src,
                                    const int32_t* dst, int32_t n, pa_stream_t stream) {
  pa_status st = pa::check_pool(pool);
  if (st != PA_OK) return st;
  if (n < 0) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  if (!src || !dst) return PA_ERR_INVALID;
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t elt = pool->dtype == PA_KV_BF16 ? 2 : 1;
  const int64_t block_bytes =
      (int64_t)pool->num_kv_heads * pool->block_size * pool->head_dim * elt;
  dim3 grid((unsigned)n, 2);
  copy_blocks_kernel<<<grid, 256, 0, pa::as_stream(stream)>>>(
      static_cast<uint8_t*>(pool->k_pool), static_cast<uint8_t*>(pool->v_pool), src, dst,
      pool->num_blocks, block_bytes, err);
  return pa::launch_status();
}

namespace {

// dst row i = src row rows[i]; one thread per 16-byte vector (grid-stride).
__global__ void gather_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                   const int32_t* __restrict__ rows, int64_t n_vec,
                                   int64_t vec_per_row, int64_t src_rows, unsigned* err) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = i / vec_per_row, v = i - row * vec_per_row;
    const int32_t r = __ldg(rows + row);
    if (r < 0 || r >= src_rows) {
      if (v == 0) pa::raise_error(err, kErrBounds);
      continue;
    }
    dst[i] = src[(int64_t)r * vec_per_row + v];
  }
}

}  // namespace

extern "C" pa_status pa_gather_rows(const void* src, int64_t src_rows, int64_t row_bytes,
                                    const int32_t* rows, int32_t n, void* dst,
                                    pa_stream_t stream) {
  if (n < 0 || src_rows < 0 || row_bytes <= 0 || row_bytes % 16 != 0) return PA_ERR_INVALID;
  if (n == 0) return PA_OK;
  if (!src || !dst || !rows || !pa::aligned16(src) || !pa::aligned16(dst)) return PA_ERR_INVALID;
  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  const int64_t vec_per_row = row_bytes / 16, n_vec = (int64_t)n * vec_per_row;
  const int threads = 256;
  int64_t blocks = (n_vec + threads - 1) / threads;
  const int64_t cap = (int64_t)pa::num_sms() * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<(unsigned)blocks, threads, 0, pa::as_stream(stream)>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), rows, n_vec, vec_per_row,
      src_rows, err);
  return pa::launch_status();
}
