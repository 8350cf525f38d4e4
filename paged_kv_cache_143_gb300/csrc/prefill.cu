// prefill.cu — prefill-chunk paged attention (q_len > 1) on the 5th-generation
// tensor cores (tcgen05.mma, accumulators in tensor memory).
//
// [vLLM-wiki "블록 단위 어텐션 계산"]: o_i = sum_j V_j A_ij^T, the softmax taken
// across every visible key of every block (causal: keys up to the query's own
// position); the kernel walks the request's block table and fetches the
// scattered physical blocks one by one. [V1-blog "고정 예산 기반 청크 분할
// 알고리즘"]: a prefill chunk of q_len tokens follows P = seq_len - q_len cached
// tokens, so query j of the chunk sits at absolute position P + j.
//
// One CTA = one tile of 128 query rows x one kv head. The rows are the
// (token, head) pairs of the GQA group that shares the kv head, packed token
// major (row = token * g + head), so K/V are read once per group.
//   warp 0     TMA producer: the Q tile once (a 4-D tensor map over
//              [T][Hkv][g][D]), then per 128-key tile one 2-D box per physical
//              block (coordinates from the block table) for K and for V,
//              into a 3-stage ring, 128-byte swizzled (K of a stage is
//              released after its S MMA, V after its PV MMA);
//   warp 1     allocates 512 TMEM columns and issues the MMAs from one thread:
//              S_j = Q K_j^T (M 128, N 128, K = D; both operands K-major) into
//              one of two S buffers, and O += P_j V_j (M 128, N = D, K 128; P
//              read from TMEM, V MN-major from shared memory) into O;
//   warps 2-5  softmax, one TMEM lane (= one query row) per thread: read S,
//              mask, online max/sum in log2 units, write P as bf16 pairs into
//              one of two TMEM P buffers; O is rescaled in TMEM
//              only when the running max grows by more than 2^8 (the stale
//              max is otherwise kept, which is exact algebra); epilogue O/l.
// Every wait is bounded; a timeout sets the error word and the CTA unwinds
// (waits for its copies and MMAs, frees TMEM) without writing output.
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_kernels.h"
#include "tc_ptx.cuh"

namespace pa {
namespace {

constexpr int kM = 128;        // query rows per tile
constexpr int kN = 128;        // keys per KV tile
constexpr int kStages = 3;     // KV tiles in flight
constexpr int kThreads = 192;  // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct Smem {
  static constexpr int kChunkBytes = kN * 128;          // 128 rows x 64 bf16 (one swizzle column)
  static constexpr int kChunks = D / 64;
  static constexpr int kQBytes = kM * D * 2;
  static constexpr int kKVBytes = kN * D * 2;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffBar = kOffV + kStages * kKVBytes;
  static constexpr int kBytes = kOffBar + 256;
  static constexpr int kAlloc = kBytes + 1024;  // the base is rounded up to 1024 B
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t k_empty[kStages];  // K of a stage is free once its S MMA is done
  uint64_t v_empty[kStages];  // V of a stage is free once its PV MMA is done
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t final_mma;
  uint32_t tmem_base;
  int abort;
};

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool aborted(Bars* b) {
  return *reinterpret_cast<volatile int*>(&b->abort) != 0;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, PrefillParams p) {
  using S = Smem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + S::kOffBar);

  const int r = p.n_order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int q_begin = p.qsl[r];
  const int q_len = p.qsl[r + 1] - q_begin;
  if (q_len <= 1) return;  // decode requests and empty requests are not ours
  const int g = p.g;
  const int tpt = kM / g;  // tokens per tile
  const int ntq = (q_len + tpt - 1) / tpt;
  if ((int)blockIdx.x >= ntq) return;
  const int tile = ntq - 1 - (int)blockIdx.x;  // heaviest (latest) tiles start first
  const int q0 = tile * tpt;
  const int kvh = blockIdx.y;
  const int seq = p.seq_lens[r];
  if (seq < q_len || seq > p.max_blocks * p.B) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int P = seq - q_len;
  const int last_tok = min(q_len, q0 + tpt) - 1;
  const int n_kv = p.causal ? min(seq, P + last_tok + 1) : seq;
  const int ntk = (n_kv + kN - 1) / kN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->k_full[s], 1);
      mbar_init(&bars->v_full[s], 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 4);  // one arrival per softmax warp
      mbar_init(&bars->pv_done[b], 1);
    }
    mbar_init(&bars->final_mma, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars->tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tmem_o = tmem + 2 * kN;  // columns [256, 256 + D)
  const uint32_t tmem_p = tmem + 3 * kN;  // P_b (bf16 pairs) at columns [384 + 64 b, +64)

  if (warp == 0) {
    // ----------------------------------------------------------- TMA producer
    // The whole warp walks the tiles: lane i fetches the block id of entry i
    // of the next tile (one coalesced load, in flight while this tile waits);
    // lane 0 issues the copies with the ids broadcast by shuffle.
    const unsigned full = 0xffffffffu;
    if (lane == 0) {
      tc::prefetch_tensormap(&tmap_q);
      tc::prefetch_tensormap(&tmap_k);
      tc::prefetch_tensormap(&tmap_v);
      mbar_arrive_expect_tx(&bars->q_full, S::kQBytes);
      for (int c = 0; c < S::kChunks; ++c)
        tc::tma_load_4d(smem + S::kOffQ + c * S::kChunkBytes, &tmap_q, c * 64, 0, kvh,
                        q_begin + q0, &bars->q_full);
    }
    const int32_t* table = p.block_tables + (int64_t)r * p.max_blocks;
    const int nbt = kN / p.B;  // blocks per KV tile (<= 8)
    auto fetch = [&](int j) -> int {
      const int lb = j * nbt + lane;
      return (j < ntk && lane < nbt && lb * p.B < n_kv) ? __ldg(table + lb) : 0;
    };
    int ids = fetch(0);
    int issued = 0;
    // lane -> one box of the tile: tensor (K, V), block i, 64-column chunk c
    const int box_tensor = lane >> 4;
    const int box_block = (lane & 15) / S::kChunks;
    const int box_chunk = (lane & 15) % S::kChunks;
    for (int j = 0; j < ntk; ++j) {
      const int next = fetch(j + 1);
      const int st = j % kStages;
      bool ok = true;
      if (lane == 0 && j >= kStages)
        ok = mbar_wait(&bars->k_empty[st], ((j / kStages) - 1) & 1, p.err) &&
             mbar_wait(&bars->v_empty[st], ((j / kStages) - 1) & 1, p.err);
      ok = __shfl_sync(full, ok ? 1 : 0, 0) && !aborted(bars);
      if (!ok) {
        if (lane == 0) bars->abort = 1;
        break;
      }
      int nload = 0;
      while (nload < nbt && (j * nbt + nload) * p.B < n_kv) ++nload;
      const bool bad = lane < nload && (ids < 0 || ids >= p.num_blocks);
      if (__any_sync(full, bad) && lane == 0) raise_error(p.err, kErrBounds);
      const int blk_lane = bad ? 0 : ids;  // a valid block; the output is then unspecified
      const int blk = __shfl_sync(full, blk_lane, box_block & 7);
      const uint32_t bytes = (uint32_t)(nload * p.B * D * 2);
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars->k_full[st], bytes);
        mbar_arrive_expect_tx(&bars->v_full[st], bytes);
      }
      __syncwarp();
      if (box_block < nload) {
        const int row = (blk * p.Hkv + kvh) * p.B;
        uint8_t* dst = smem + (box_tensor ? S::kOffV : S::kOffK) + st * S::kKVBytes +
                       box_chunk * S::kChunkBytes + box_block * p.B * 128;
        tc::tma_load_2d(dst, box_tensor ? &tmap_v : &tmap_k, box_chunk * 64, row,
                        box_tensor ? &bars->v_full[st] : &bars->k_full[st]);
      }
      issued = j + 1;
      ids = next;
    }
    // every issued copy lands before the CTA may leave
    if (lane == 0) {
      mbar_wait(&bars->q_full, 0, p.err);
      for (int j = issued - kStages > 0 ? issued - kStages : 0; j < issued; ++j) {
        mbar_wait(&bars->k_full[j % kStages], (j / kStages) & 1, p.err);
        mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, p.err);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kM, kN, false, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kM, D, false, true);
      const uint8_t* qs = smem + S::kOffQ;
      auto issue_pv = [&](int jj) -> bool {
        const int bb = jj & 1, st = jj % kStages;
        if (!mbar_wait(&bars->p_full[bb], (jj >> 1) & 1, p.err)) return false;
        if (!mbar_wait(&bars->v_full[st], (jj / kStages) & 1, p.err)) return false;
        if (aborted(bars)) return false;
        tc::fence_after_sync();
        const uint8_t* vs = smem + S::kOffV + st * S::kKVBytes;
#pragma unroll
        for (int ks = 0; ks < kN / 16; ++ks) {
          const uint64_t b = tc::smem_desc_sw128(vs + ks * 16 * 128, S::kChunkBytes, 1024);
          tc::mma_bf16_ts(tmem_o, tmem_p + bb * (kN / 2) + ks * 8, b, idesc_o, jj > 0 || ks > 0);
        }
        tc::mma_commit(&bars->pv_done[bb]);
        tc::mma_commit(&bars->v_empty[st]);
        return true;
      };
      bool ok = mbar_wait(&bars->q_full, 0, p.err);
      for (int j = 0; ok && j < ntk; ++j) {
        const int st = j % kStages, b = j & 1;
        if (!mbar_wait(&bars->k_full[st], (j / kStages) & 1, p.err) || aborted(bars)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint8_t* ks_ = smem + S::kOffK + st * S::kKVBytes;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t a =
              tc::smem_desc_sw128(qs + (ks >> 2) * S::kChunkBytes + (ks & 3) * 32, 16, 1024);
          const uint64_t bd =
              tc::smem_desc_sw128(ks_ + (ks >> 2) * S::kChunkBytes + (ks & 3) * 32, 16, 1024);
          tc::mma_bf16_ss(tmem + b * kN, a, bd, idesc_s, ks > 0);
        }
        tc::mma_commit(&bars->s_full[b]);
        tc::mma_commit(&bars->k_empty[st]);
        if (j >= 1 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) ok = issue_pv(ntk - 1);
      if (!ok) bars->abort = 1;
      tc::mma_commit(&bars->final_mma);
      mbar_wait(&bars->final_mma, 0, p.err);
    }
  } else {
    // -------------------------------------------------------------- softmax
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int tok = q0 + row / g;
    const int head = row % g;
    const bool valid_row = tok < q_len;
    const int limit = !valid_row ? 0 : (p.causal ? min(P + tok + 1, seq) : seq);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < ntk; ++j) {
      const int b = j & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[b], (j >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      float s[kN];
      {
        uint32_t raw[kN / 32][32];
#pragma unroll
        for (int c = 0; c < kN / 32; ++c) tc::tmem_ld32(tmem + b * kN + c * 32 + lane_off, raw[c]);
        tc::tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kN / 32; ++c)
#pragma unroll
          for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(raw[c][k]);
      }
      const int key0 = j * kN;
      if (key0 + kN > limit) {
#pragma unroll
        for (int k = 0; k < kN; ++k)
          if (key0 + k >= limit) s[k] = -INFINITY;
      }
      // raw scores; the log2-domain max is max * scale_log2 (scale > 0).
      // Eight independent partial maxima keep the reduction off one long
      // dependency chain (one softmax warp per SM sub-partition has no other
      // warp to hide latency with).
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mx[u] = s[u];
#pragma unroll
      for (int k = 8; k < kN; k += 8)
#pragma unroll
        for (int u = 0; u < 8; ++u) mx[u] = fmaxf(mx[u], s[k + u]);
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                       fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      mt *= p.scale_log2;
      float m_use = m_run, alpha = 1.f;
      bool rescale = false;
      if (m_run == -INFINITY) {
        m_use = mt;
        alpha = 0.f;
      } else if (mt > m_run + kRescaleLog2) {
        m_use = mt;
        alpha = fast_exp2(m_run - mt);
        rescale = true;
      }
      const float m_sub = m_use == -INFINITY ? 0.f : m_use;
      float sum[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) sum[u] = 0.f;
#pragma unroll
      for (int k = 0; k < kN; k += 8)
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          s[k + u] = fast_exp2(fmaf(s[k + u], p.scale_log2, -m_sub));
          sum[u] += s[k + u];
        }
      const float rs = ((sum[0] + sum[1]) + (sum[2] + sum[3])) +
                       ((sum[4] + sum[5]) + (sum[6] + sum[7]));
      l_run = l_run * alpha + rs;
      m_run = m_use;

      // the P buffer b is free once PV(j-2) has finished
      if (j >= 2 &&
          !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[b], ((j - 2) >> 1) & 1, p.err))) {
        ok = false;
        break;
      }
      // P as bf16 pairs into this row's TMEM lane (the A operand of PV)
#pragma unroll
      for (int c = 0; c < kN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          __nv_bfloat162 h = __floats2bfloat162_rn(s[c * 64 + 2 * k], s[c * 64 + 2 * k + 1]);
          w[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        tc::tmem_st32(tmem_p + b * (kN / 2) + c * 32 + lane_off, w);
      }
      tc::tmem_wait_st();

      // rescale O (rare): needs PV(j-1) complete
      if (__any_sync(0xffffffffu, rescale)) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->pv_done[(j - 1) & 1], ((j - 1) >> 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tmem_o + c * 32 + lane_off, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * a);
          tc::tmem_st32(tmem_o + c * 32 + lane_off, o);
        }
        tc::tmem_wait_st();
      }

      // the last tile may hold keys past n_kv (unloaded blocks, unwritten
      // cells): zero those V rows so that P = 0 never meets a NaN
      if (j == ntk - 1 && key0 + kN > n_kv) {
        const int st = j % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (j / kStages) & 1, p.err))) {
          ok = false;
          break;
        }
        if (key0 + row >= n_kv) {
          uint8_t* vs = smem + S::kOffV + st * S::kKVBytes;
#pragma unroll
          for (int c = 0; c < S::kChunks; ++c)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vs + c * S::kChunkBytes + row * 128 + q * 16) =
                  make_uint4(0, 0, 0, 0);
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[b]);
    }

    // epilogue: O / l once the last PV has landed
    if (ok && !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[(ntk - 1) & 1],
                                                 ((ntk - 1) >> 1) & 1, p.err)))
      ok = false;
    if (!ok) bars->abort = 1;
    if (ok && !aborted(bars)) {
      tc::fence_after_sync();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow =
          p.out + ((int64_t)(q_begin + tok) * p.Hq + kvh * g + head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem_o + c * 32 + lane_off, o);
        tc::tmem_wait_ld();
        if (valid_row) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            uint32_t* w = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(o[q * 8 + 2 * e]) * inv_l,
                                                       __uint_as_float(o[q * 8 + 2 * e + 1]) * inv_l);
              w[e] = *reinterpret_cast<uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(orow + c * 32 + q * 8) = v;
          }
        }
      }
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------- host launch

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

template <int D>
cudaError_t launch_prefill_t(const PrefillLaunch& L, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const PrefillParams& p = L.p;
  CUtensorMap tq, tk, tv;
  // Q as [T][Hkv][g][D]: box = 64 dims x g heads x 1 kv head x 128/g tokens
  {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.g, (cuuint64_t)p.Hkv, (cuuint64_t)L.T};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)p.g * D * 2,
                             (cuuint64_t)p.Hq * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)p.g, 1, (cuuint32_t)(kM / p.g)};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode(&tq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(L.q), dims, strides,
               box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // K and V as rows [(block * Hkv + head) * B + offset][D]: box = 64 dims x B rows
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.num_blocks * p.Hkv * p.B};
    cuuint64_t strides[1] = {(cuuint64_t)D * 2};
    cuuint32_t box[2] = {64, (cuuint32_t)p.B};
    cuuint32_t es[2] = {1, 1};
    if (encode(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(L.k_pool), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(L.v_pool), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  constexpr int smem = Smem<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(L.max_q_tiles, p.Hkv, p.n_order ? p.n_order : L.R);
  prefill_kernel<D><<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s) {
  if (L.D == 128) return launch_prefill_t<128>(L, s);
  return launch_prefill_t<64>(L, s);
}

}  // namespace pa
