// decode.cu — decode (q_len = 1) paged attention with split-KV, and the
// log-sum-exp merge of the splits.
//
// [vLLM-wiki "블록 단위 어텐션 계산"]: o_i = sum_j V_j A_ij^T with the softmax
// taken over every key of every block, the blocks fetched one by one through
// the block table. A decode query sees all seq_len keys of its request.
// Splitting the key range and merging by log-sum-exp is exact algebra on that
// cross-block denominator:  with per-split max m_s, sum l_s and unnormalised
// o_s,  o = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s,  M = max_s m_s.
//
// Design (HBM-bound by construction):
//  - one CTA per (key split, kv head [x head group], request): the GH query
//    heads of a GQA group that share the kv head read the KV once;
//  - warp 4 is a producer: one lane walks the block table and issues a 1-D
//    bulk async copy (cp.async.bulk, completes on an mbarrier) per 16-key chunk
//    of K and of V into an 8-stage shared-memory ring; a (block, kv head) is
//    contiguous in the pool, so every chunk is one contiguous 16*D*elt copy;
//  - warps 0..3 each own every 4th chunk and keep their own online-softmax
//    state; lane (a, b) = (lane/8, lane%8) handles keys a, a+4, a+8, a+12 of the
//    chunk and a fixed 1/8 of the head dimension, so a quarter-warp reads 128
//    contiguous bytes of one key row (no bank conflicts); the dot product is
//    finished with 3 xor-shuffles; P*V accumulates in registers and is reduced
//    across the key lanes once per split;
//  - the four warps merge through shared memory; one split writes bf16 output
//    directly, several write fp32 partials (o, m, l) for the merge kernel.
// FP8 E4M3 codes are widened in registers (exact); k_scale is folded into the
// query scale and v_scale into the output.
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_kernels.h"

namespace pa {
namespace {

constexpr int kChunk = 16;         // keys per pipeline stage
constexpr int kConsumerWarps = 4;  // warps 0..3 compute, warp 4 produces
constexpr int kStages = 8;         // ring depth (a multiple of kConsumerWarps)
constexpr int kThreads = (kConsumerWarps + 1) * 32;

template <int D, bool FP8>
struct Geo {
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;                  // one key row
  static constexpr int kPieceBytes = kRowBytes / 8 >= 16 ? 16 : kRowBytes / 8;
  static constexpr int kPieces = kRowBytes / (8 * kPieceBytes);
  static constexpr int kPieceElems = kPieceBytes / kElt;
  static constexpr int kDimsPerLane = kPieces * kPieceElems;  // = D / 8
  static constexpr int kChunkBytes = kChunk * kRowBytes;
  static constexpr int kStageBytes = 2 * kChunkBytes;         // K then V
  static_assert(kDimsPerLane * 8 == D, "lane split must cover the head");
  // first dimension of piece p of lane b
  __device__ static constexpr int dim0(int p, int b) { return (p * 8 + b) * kPieceElems; }
};

template <int D, bool FP8>
__device__ __forceinline__ void load_piece(const uint8_t* src, float* f) {
  using G = Geo<D, FP8>;
  if constexpr (!FP8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    bf16x8_to_f32(v, f);
  } else if constexpr (G::kPieceBytes == 16) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    e4m3x16_to_f32(v, f);
  } else {
    const uint2 v = *reinterpret_cast<const uint2*>(src);
    e4m3x8_to_f32(v, f);
  }
}

struct SmemTail {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int abort;
};

template <int D, bool FP8, int GH>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeParams p) {
  using G = Geo<D, FP8>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                               // kStages stages
  float* comb_o = reinterpret_cast<float*>(smem + kStages * G::kStageBytes);  // [4][GH][D]
  float* comb_m = comb_o + kConsumerWarps * GH * D;                   // [4][GH]
  float* comb_l = comb_m + kConsumerWarps * GH;                       // [4][GH]
  SmemTail* tail = reinterpret_cast<SmemTail*>(comb_l + kConsumerWarps * GH);

  const int r = blockIdx.z;
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return;  // not a decode request
  const int seq = p.seq_lens[r];
  if (seq < 1 || seq > p.max_blocks * p.B) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int nsplit = (seq + p.split_tokens - 1) / p.split_tokens;
  if (nsplit > (int)gridDim.x) {  // device seq_lens disagree with the host mirror
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int split = blockIdx.x;
  if (split >= nsplit) return;
  const int k_begin = split * p.split_tokens;
  const int k_end = min(seq, k_begin + p.split_tokens);
  const int nch = (k_end - k_begin + kChunk - 1) / kChunk;
  const int groups_per_kv = p.g / GH;
  const int kvh = blockIdx.y / groups_per_kv;
  const int h0 = kvh * p.g + (blockIdx.y % groups_per_kv) * GH;  // first query head

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&tail->full[i], 1);
      mbar_init(&tail->empty[i], 1);
    }
    tail->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    // The warp fetches the block ids of 32 chunks at a time (lane i: chunk
    // base + i, one coalesced load); lane 0 issues the bulk copies.
    const unsigned full = 0xffffffffu;
    const int32_t* table = p.block_tables + (int64_t)r * p.max_blocks;
    const int64_t head_stride = (int64_t)p.B * G::kRowBytes;  // one (block, head)
    int issued = 0;
    bool ok = true;
    for (int base = 0; base < nch && ok; base += 32) {
      const int c_lane = base + lane;
      const int key_lane = k_begin + c_lane * kChunk;
      int blk_lane = c_lane < nch ? __ldg(table + key_lane / p.B) : 0;
      const bool bad = c_lane < nch && (blk_lane < 0 || blk_lane >= p.num_blocks);
      if (__any_sync(full, bad) && lane == 0) raise_error(p.err, kErrBounds);
      if (bad) blk_lane = 0;  // read a valid block; the call's output is then unspecified
      const int n = min(32, nch - base);
      for (int i = 0; i < n; ++i) {
        const int c = base + i;
        const int blk = __shfl_sync(full, blk_lane, i);
        if (lane == 0) {
          const int stage = c % kStages, round = c / kStages;
          if (round > 0 && !mbar_wait(&tail->empty[stage], (round - 1) & 1, p.err)) {
            tail->abort = 1;
            ok = false;
          } else if (*reinterpret_cast<volatile int*>(&tail->abort)) {
            ok = false;
          } else {
            const int key0 = k_begin + c * kChunk;
            const int64_t off = ((int64_t)blk * p.Hkv + kvh) * head_stride +
                                (int64_t)(key0 % p.B) * G::kRowBytes;
            uint8_t* dst = ring + stage * G::kStageBytes;
            mbar_arrive_expect_tx(&tail->full[stage], G::kStageBytes);
            bulk_g2s(dst, p.k_pool + off, G::kChunkBytes, &tail->full[stage]);
            bulk_g2s(dst + G::kChunkBytes, p.v_pool + off, G::kChunkBytes, &tail->full[stage]);
            issued = c + 1;
          }
        }
        ok = __shfl_sync(full, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
    }
    // drain: every issued copy has landed before the CTA may exit
    if (lane == 0)
      for (int c = issued - kStages > 0 ? issued - kStages : 0; c < issued; ++c)
        mbar_wait(&tail->full[c % kStages], (c / kStages) & 1, p.err);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int a = lane >> 3, b = lane & 7;
  float qf[GH][G::kDimsPerLane];
  {
    const __nv_bfloat16* qrow = p.q + ((int64_t)qs * p.Hq + h0) * D;
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc)
#pragma unroll
        for (int e = 0; e < G::kPieceElems; e += 8) {
          const uint4 v =
              __ldg(reinterpret_cast<const uint4*>(qrow + h * D + G::dim0(pc, b) + e));
          float f[8];
          bf16x8_to_f32(v, f);
#pragma unroll
          for (int x = 0; x < 8; ++x) qf[h][pc * G::kPieceElems + e + x] = f[x] * p.q_scale;
        }
  }
  float o[GH][G::kDimsPerLane];
  float m[GH], l[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < G::kDimsPerLane; ++d) o[h][d] = 0.f;
  }

  bool ok = true;
  for (int c = warp; c < nch && ok; c += kConsumerWarps) {
    const int stage = c % kStages, round = c / kStages;
    // every lane waits; the warp proceeds only if all lanes saw the data
    if (!__all_sync(0xffffffffu, mbar_wait(&tail->full[stage], round & 1, p.err))) {
      tail->abort = 1;
      ok = false;
      break;
    }
    const uint8_t* Ks = ring + stage * G::kStageBytes;
    const uint8_t* Vs = Ks + G::kChunkBytes;
    const int key0 = k_begin + c * kChunk;

    float s[4][GH];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint8_t* krow = Ks + (a + 4 * i) * G::kRowBytes;
#pragma unroll
      for (int h = 0; h < GH; ++h) s[i][h] = 0.f;
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc) {
        float kf[G::kPieceElems];
        load_piece<D, FP8>(krow + (pc * 8 + b) * G::kPieceBytes, kf);
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
          for (int e = 0; e < G::kPieceElems; ++e)
            s[i][h] = fmaf(qf[h][pc * G::kPieceElems + e], kf[e], s[i][h]);
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        s[i][h] += __shfl_xor_sync(0xffffffffu, s[i][h], 1);
        s[i][h] += __shfl_xor_sync(0xffffffffu, s[i][h], 2);
        s[i][h] += __shfl_xor_sync(0xffffffffu, s[i][h], 4);
      }
    bool valid[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      valid[i] = key0 + a + 4 * i < k_end;
      if (!valid[i])
#pragma unroll
        for (int h = 0; h < GH; ++h) s[i][h] = -INFINITY;
    }
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float mx = fmaxf(fmaxf(s[0][h], s[1][h]), fmaxf(s[2][h], s[3][h]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m[h], mx);
      const float alpha = exp2f(m[h] - m_new);
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        s[i][h] = exp2f(s[i][h] - m_new);  // now p
        psum += s[i][h];
      }
      l[h] = l[h] * alpha + psum;
      m[h] = m_new;
#pragma unroll
      for (int d = 0; d < G::kDimsPerLane; ++d) o[h][d] *= alpha;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!valid[i]) continue;  // unwritten cells may hold NaN: never touch them
      const uint8_t* vrow = Vs + (a + 4 * i) * G::kRowBytes;
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc) {
        float vf[G::kPieceElems];
        load_piece<D, FP8>(vrow + (pc * 8 + b) * G::kPieceBytes, vf);
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
          for (int e = 0; e < G::kPieceElems; ++e)
            o[h][pc * G::kPieceElems + e] = fmaf(s[i][h], vf[e], o[h][pc * G::kPieceElems + e]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[stage]);
  }

  // reduce l and o over the four key-lane groups (lanes differing in bits 3, 4)
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 8);
    l[h] += __shfl_xor_sync(0xffffffffu, l[h], 16);
#pragma unroll
    for (int d = 0; d < G::kDimsPerLane; ++d) {
      o[h][d] += __shfl_xor_sync(0xffffffffu, o[h][d], 8);
      o[h][d] += __shfl_xor_sync(0xffffffffu, o[h][d], 16);
    }
  }
  if (a == 0) {
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc)
#pragma unroll
        for (int e = 0; e < G::kPieceElems; ++e)
          comb_o[(warp * GH + h) * D + G::dim0(pc, b) + e] = o[h][pc * G::kPieceElems + e];
  }
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      comb_m[warp * GH + h] = m[h];
      comb_l[warp * GH + h] = l[h];
    }
  named_bar_sync(1, kConsumerWarps * 32);
  if (*reinterpret_cast<volatile int*>(&tail->abort)) return;

  const int t = threadIdx.x;  // 0..127
  for (int idx = t; idx < GH * D; idx += kConsumerWarps * 32) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb_m[w * GH + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float f = exp2f(comb_m[w * GH + h] - M);  // 0 for a warp with no chunk
      L += f * comb_l[w * GH + h];
      O += f * comb_o[(w * GH + h) * D + d];
    }
    const int hq = h0 + h;
    if (nsplit == 1) {
      p.out[((int64_t)qs * p.Hq + hq) * D + d] = __float2bfloat16_rn(O / L * p.v_scale);
    } else {
      const int64_t row = ((int64_t)r * p.Hq + hq) * p.ws_splits + split;
      p.ws_o[row * D + d] = O * p.v_scale;
      if (d == 0) p.ws_ml[row] = make_float2(M, L);
    }
  }
}

// One CTA per (query head, request) with more than one split: combines the
// partials of the decode kernel by log-sum-exp.
template <int D>
__global__ void __launch_bounds__(D) merge_kernel(DecodeParams p) {
  const int h = blockIdx.x, r = blockIdx.y, d = threadIdx.x;
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return;
  const int seq = p.seq_lens[r];
  if (seq < 1 || seq > p.max_blocks * p.B) return;
  const int nsplit = (seq + p.split_tokens - 1) / p.split_tokens;
  if (nsplit <= 1 || nsplit > p.ws_splits) return;
  const int64_t row0 = ((int64_t)r * p.Hq + h) * p.ws_splits;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.ws_ml[row0 + s].x);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float2 ml = p.ws_ml[row0 + s];
    const float f = exp2f(ml.x - M);
    L += f * ml.y;
    O += f * p.ws_o[(row0 + s) * D + d];
  }
  p.out[((int64_t)qs * p.Hq + h) * D + d] = __float2bfloat16_rn(O / L);
}

template <int D, bool FP8, int GH>
constexpr int decode_smem_bytes() {
  return kStages * Geo<D, FP8>::kStageBytes + kConsumerWarps * GH * (D + 2) * 4 +
         (int)sizeof(SmemTail);
}

template <int D, bool FP8, int GH>
cudaError_t launch_decode_t(const DecodeParams& p, int R, int max_splits, cudaStream_t s) {
  constexpr int smem = decode_smem_bytes<D, FP8, GH>();
  auto k = decode_kernel<D, FP8, GH>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(max_splits, p.Hkv * (p.g / GH), R);
  k<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_decode_d(const DecodeParams& p, int GH, int R, int max_splits,
                            cudaStream_t s) {
  switch (GH) {
    case 1: return launch_decode_t<D, FP8, 1>(p, R, max_splits, s);
    case 2: return launch_decode_t<D, FP8, 2>(p, R, max_splits, s);
    default: return launch_decode_t<D, FP8, 4>(p, R, max_splits, s);
  }
}

}  // namespace

int decode_heads_per_cta(int g) { return g < 4 ? g : 4; }

cudaError_t launch_decode(const DecodeParams& p, int D, bool fp8, int R, int max_splits,
                          cudaStream_t s) {
  const int GH = decode_heads_per_cta(p.g);
  if (D == 128)
    return fp8 ? launch_decode_d<128, true>(p, GH, R, max_splits, s)
               : launch_decode_d<128, false>(p, GH, R, max_splits, s);
  return fp8 ? launch_decode_d<64, true>(p, GH, R, max_splits, s)
             : launch_decode_d<64, false>(p, GH, R, max_splits, s);
}

cudaError_t launch_merge(const DecodeParams& p, int D, int R, cudaStream_t s) {
  dim3 grid(p.Hq, R);
  if (D == 128)
    merge_kernel<128><<<grid, 128, 0, s>>>(p);
  else
    merge_kernel<64><<<grid, 64, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace pa
