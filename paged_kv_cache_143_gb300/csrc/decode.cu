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
//  - one CTA per (key split, kv head, request): all g query heads of the GQA
//    group that share the kv head are served from one read of the KV;
//  - warp 4 is a producer: per 16-key chunk, K and V are each one contiguous
//    run of the pool (a (block, kv head) is contiguous), moved by one bulk
//    async copy (cp.async.bulk, completing on the stage's mbarrier) into a
//    64 KB ring (8 bf16 / 16 E4M3 stages). The warp fetches the block ids of
//    32 chunks at a time and handles a group of chunks per step, lane i
//    waiting for and issuing chunk c0 + i, so waits and copy issue overlap;
//  - warps 0..3 compute, each owning every 4th chunk. g = 1 (decode_kernel):
//    lane (a, b) = (lane/8, lane%8) handles keys a, a+4, a+8, a+12 of the
//    chunk and a fixed 1/8 of the head dimension, so a quarter-warp reads 128
//    contiguous bytes of one key row (no bank conflicts); the dot products
//    use packed fp32 multiply-adds and finish with 3 xor-shuffles; P*V
//    accumulates in registers and is reduced across the key lanes once per
//    split. g >= 2 (decode_mma_kernel, described at its definition):
//    warp-level tensor-core products with the g query heads as rows;
//  - the warps merge through shared memory; one split writes bf16 output
//    directly, several write fp32 partials (o, m, l) for the merge kernel.
//    (Batches with shared-prefix groups run on cascade.cu's kernel, whose
//    partials the merge kernel below also combines.)
// FP8 E4M3 codes are widened in registers (exact); k_scale is folded into the
// query scale and v_scale into the output.
#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_kernels.h"
#include "tc_ptx.cuh"
#include "decode_rows.cuh"

namespace pa {
namespace {

constexpr int kThreads = (kConsumerWarps + 1) * 32;

// One piece of a key row as packed fp32 pairs (dims 2i, 2i+1).
template <int D, bool FP8>
__device__ __forceinline__ void load_piece2(const uint8_t* src, uint64_t* f2) {
  using G = Geo<D, FP8>;
  if constexpr (!FP8) {
    const uint4 v = *reinterpret_cast<const uint4*>(src);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f2[i] = f2_pack(bf16_lo(w[i]), bf16_hi(w[i]));
  } else {
    float f[G::kPieceElems];
    if constexpr (G::kPieceBytes == 16) {
      e4m3x16_to_f32(*reinterpret_cast<const uint4*>(src), f);
    } else {
      e4m3x8_to_f32(*reinterpret_cast<const uint2*>(src), f);
    }
#pragma unroll
    for (int i = 0; i < G::kPiecePairs; ++i) f2[i] = f2_pack(f[2 * i], f[2 * i + 1]);
  }
}

struct SmemTail {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  int abort;
};

// The producer warp of the decode kernels: it fetches the block ids of 32
// chunks at a time (lane i: chunk base + i, one coalesced load). Per 16-key
// chunk, K and V are each one contiguous run of the pool, moved by one bulk
// async copy each that completes on the stage's mbarrier by transaction
// bytes. The producer handles a group of chunks per step (lane i waits for
// the stage of chunk c0 + i and issues its copies), so that the waits and the
// copy issue of a group overlap; one chunk per step left only about two
// chunks in flight. kTma: the same runs move as TMA tensor boxes (16 rows of
// 128 codes, 128-byte swizzle) through the maps tk and tv, which view a pool
// as [block][kv head * B + offset][128].
// produce_run issues chunks [0, nch) of one key run (keys k_begin + 16 c of
// the block-table row `table`, kv head kvh) into ring positions q_base + c
// (stage = position mod kStages); it returns false if a wait gave up or the
// CTA aborted, and adds the positions it issued to *issued (the drain must
// wait for every one of them).
template <class G, bool kTma>
__device__ __forceinline__ bool produce_run(const DecodeParams& p, uint8_t* ring, SmemTail* tail,
                                            const int32_t* table, int kvh, int k_begin, int nch,
                                            int64_t q_base, int lane, const CUtensorMap* tk,
                                            const CUtensorMap* tv, int64_t* issued) {
  // chunks handled per step (half the ring, at most 8)
  constexpr int kGroup = G::kStages / 2 < 8 ? G::kStages / 2 : 8;
  static_assert(32 % kGroup == 0, "groups must tile the 32 chunks of a block-id fetch");
  const unsigned full = 0xffffffffu;
  const int64_t head_stride = (int64_t)p.B * G::kRowBytes;  // one (block, head)
  for (int base = 0; base < nch; base += 32) {
    const int c_lane = base + lane;
    const int key_lane = k_begin + c_lane * kChunk;
    int blk_lane = c_lane < nch ? __ldg(table + key_lane / p.B) : 0;
    const bool bad = c_lane < nch && (blk_lane < 0 || blk_lane >= p.num_blocks);
    if (__any_sync(full, bad) && lane == 0) raise_error(p.err, kErrBounds);
    if (bad) blk_lane = 0;  // read a valid block; the call's output is then unspecified
    // byte offset of each lane's chunk in the pool (one contiguous run of K, of
    // V), or its TMA coordinates (row within the block, block)
    const int64_t off_lane = ((int64_t)blk_lane * p.Hkv + kvh) * head_stride +
                             (int64_t)(key_lane % p.B) * G::kRowBytes;
    const int y_lane = kvh * p.B + key_lane % p.B;
    const int n = min(32, nch - base);
    for (int g0 = 0; g0 < n; g0 += kGroup) {
      const int gn = min(kGroup, n - g0);
      const int64_t q = q_base + base + g0 + lane;  // this lane's ring position
      const bool mine = lane < gn;
      const int stage = (int)(q % G::kStages);
      const int64_t round = q / G::kStages;
      bool free_ok = true;
      if (mine && round > 0) free_ok = mbar_wait(&tail->empty[stage], (round - 1) & 1, p.err);
      const bool ok = __all_sync(full, free_ok) && !*reinterpret_cast<volatile int*>(&tail->abort);
      if (!ok) {
        if (lane == 0) tail->abort = 1;
        *issued = q_base + base + g0;
        return false;
      }
      if constexpr (kTma) {
        const int y = __shfl_sync(full, y_lane, (g0 + lane) & 31);
        const int z = __shfl_sync(full, blk_lane, (g0 + lane) & 31);
        if (mine) {
          uint8_t* dst = ring + stage * G::kStageBytes;
          mbar_arrive_expect_tx(&tail->full[stage], G::kStageBytes);
          tc::tma_load_3d(dst, tk, 0, y, z, &tail->full[stage]);
          tc::tma_load_3d(dst + G::kChunkBytes, tv, 0, y, z, &tail->full[stage]);
        }
      } else {
        const int64_t off = __shfl_sync(full, off_lane, (g0 + lane) & 31);
        if (mine) {
          uint8_t* dst = ring + stage * G::kStageBytes;
          mbar_arrive_expect_tx(&tail->full[stage], G::kStageBytes);
          bulk_g2s(dst, p.k_pool + off, G::kChunkBytes, &tail->full[stage]);
          bulk_g2s(dst + G::kChunkBytes, p.v_pool + off, G::kChunkBytes, &tail->full[stage]);
        }
      }
    }
  }
  *issued = q_base + nch;
  return true;
}

// Waits until the copies of ring positions [0, issued) have landed (those
// still in flight are the last kStages), so that the CTA may exit.
template <class G>
__device__ __forceinline__ void drain(const DecodeParams& p, SmemTail* tail, int64_t issued,
                                      int lane) {
  if (lane == 0)
    for (int64_t q = issued - G::kStages > 0 ? issued - G::kStages : 0; q < issued; ++q)
      mbar_wait(&tail->full[q % G::kStages], (q / G::kStages) & 1, p.err);
}

// The whole producer of a one-run CTA: request r's key run, then the drain.
template <class G, bool kTma>
__device__ __forceinline__ void produce(const DecodeParams& p, uint8_t* ring, SmemTail* tail,
                                        int r, int kvh, int k_begin, int nch, int lane,
                                        const CUtensorMap* tk, const CUtensorMap* tv) {
  const int32_t* table = p.block_tables + (int64_t)r * p.max_blocks;
  int64_t issued = 0;
  produce_run<G, kTma>(p, ring, tail, table, kvh, k_begin, nch, 0, lane, tk, tv, &issued);
  drain<G>(p, tail, issued, lane);
}

// GH heads per warp, HG head groups per CTA (GH * HG = g).
template <int D, bool FP8, int GH, int HG>
__global__ void __launch_bounds__(kThreads, 2) decode_kernel(DecodeParams p) {
  launch_dependents();  // the merge that follows may be scheduled now
  using G = Geo<D, FP8>;
  constexpr int kStages = G::kStages;
  constexpr int CR = kConsumerWarps / HG;  // warps per head group (chunk residues)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;                                                      // kStages stages
  float* comb_o = reinterpret_cast<float*>(smem + kStages * G::kStageBytes);  // [4][GH][D]
  float* comb_m = comb_o + kConsumerWarps * GH * D;                          // [4][GH]
  float* comb_l = comb_m + kConsumerWarps * GH;                              // [4][GH]
  SmemTail* tail = reinterpret_cast<SmemTail*>(comb_l + kConsumerWarps * GH);

  const int r = blockIdx.z;
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return;  // not a decode request
  if (qs < 0 || qs >= p.T) {  // a device qsl that leaves q / out
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int seq = p.seq_lens[r];
  if (seq < 1 || seq > p.max_blocks * p.B) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int nsplit = (seq + p.split_tokens - 1) / p.split_tokens;
  if (nsplit > (int)gridDim.x || (nsplit > 1 && nsplit > p.ws_splits)) {
    // device seq_lens disagree with the host mirror
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int split = blockIdx.x;
  if (split >= nsplit) return;
  const int k_begin = split * p.split_tokens;
  const int k_end = min(seq, k_begin + p.split_tokens);
  const int nch = (k_end - k_begin + kChunk - 1) / kChunk;
  const int kvh = blockIdx.y;
  const int hq0 = kvh * p.g;  // first query head of the group

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&tail->full[i], 1);
      mbar_init(&tail->empty[i], HG);  // one arrival per head group
    }
    tail->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    produce<G, false>(p, ring, tail, r, kvh, k_begin, nch, lane, nullptr, nullptr);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int hg = warp % HG, cr = warp / HG;
  const int h0 = hq0 + hg * GH;  // first query head of this warp
  const int a = lane >> 3, b = lane & 7;
  uint64_t q2[GH][G::kPairsPerLane];
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
          for (int x = 0; x < 4; ++x)
            q2[h][(pc * G::kPieceElems + e) / 2 + x] =
                f2_pack(f[2 * x] * p.q_scale, f[2 * x + 1] * p.q_scale);
        }
  }
  uint64_t o2[GH][G::kPairsPerLane];
  float m[GH], l[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int d = 0; d < G::kPairsPerLane; ++d) o2[h][d] = 0ull;
  }

  bool ok = true;
  for (int c = cr; c < nch && ok; c += CR) {
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
      uint64_t acc[GH];
#pragma unroll
      for (int h = 0; h < GH; ++h) acc[h] = 0ull;
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc) {
        uint64_t k2[G::kPiecePairs];
        load_piece2<D, FP8>(krow + (pc * 8 + b) * G::kPieceBytes, k2);
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
          for (int e = 0; e < G::kPiecePairs; ++e)
            acc[h] = f2_fma(q2[h][pc * G::kPiecePairs + e], k2[e], acc[h]);
      }
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float lo, hi;
        f2_unpack(acc[h], lo, hi);
        s[i][h] = lo + hi;
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
      const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll
      for (int d = 0; d < G::kPairsPerLane; ++d) o2[h][d] = f2_mul(o2[h][d], a2);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (!valid[i]) continue;  // unwritten cells may hold NaN: never touch them
      const uint8_t* vrow = Vs + (a + 4 * i) * G::kRowBytes;
#pragma unroll
      for (int pc = 0; pc < G::kPieces; ++pc) {
        uint64_t v2[G::kPiecePairs];
        load_piece2<D, FP8>(vrow + (pc * 8 + b) * G::kPieceBytes, v2);
#pragma unroll
        for (int h = 0; h < GH; ++h) {
          const uint64_t p2 = f2_pack(s[i][h], s[i][h]);
#pragma unroll
          for (int e = 0; e < G::kPiecePairs; ++e)
            o2[h][pc * G::kPiecePairs + e] = f2_fma(p2, v2[e], o2[h][pc * G::kPiecePairs + e]);
        }
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
  }
  float o[GH][G::kDimsPerLane];
#pragma unroll
  for (int h = 0; h < GH; ++h)
#pragma unroll
    for (int d = 0; d < G::kPairsPerLane; ++d) {
      f2_unpack(o2[h][d], o[h][2 * d], o[h][2 * d + 1]);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        o[h][2 * d + x] += __shfl_xor_sync(0xffffffffu, o[h][2 * d + x], 8);
        o[h][2 * d + x] += __shfl_xor_sync(0xffffffffu, o[h][2 * d + x], 16);
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
  for (int idx = t; idx < HG * GH * D; idx += kConsumerWarps * 32) {
    const int hh = idx / D, d = idx % D;  // head within the group, dim
    const int grp = hh / GH, h = hh % GH;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < CR; ++k) M = fmaxf(M, comb_m[(grp + HG * k) * GH + h]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int k = 0; k < CR; ++k) {
      const int w = grp + HG * k;  // the warps of head group grp
      const float f = exp2f(comb_m[w * GH + h] - M);  // 0 for a warp with no chunk
      L += f * comb_l[w * GH + h];
      O += f * comb_o[(w * GH + h) * D + d];
    }
    const int hq = hq0 + hh;
    if (nsplit == 1) {
      p.out[((int64_t)qs * p.Hq + hq) * D + d] = __float2bfloat16_rn(O / L * p.v_scale);
    } else {
      const int64_t row = ((int64_t)r * p.Hq + hq) * p.ws_splits + split;
      p.ws_o[row * D + d] = O * p.v_scale;
      if (d == 0) p.ws_ml[row] = make_float2(M, L);
    }
  }
}

// Combines the four consumer warps' partial rows (comb buffers) of one key
// run and writes rows hq0 .. hq0 + nrows - 1 of request r: the bf16 output
// (direct), or the fp32 partial into split slot `slot`.
// All 128 consumer threads must call it (it holds a barrier).
template <int D>
__device__ __forceinline__ void combine_rows(const DecodeParams& p, const float* comb_o,
                                             float* comb_m, float* comb_l, int nrows, int r,
                                             int qs, int hq0, bool direct, int slot) {
  // each row's warp weights 2^(m_w - M) (0 for a warp with no chunk), its
  // max and its sum, once per row: thread t < nrows owns row t and replaces
  // the row's comb_m entries by the weights, its warp-0 and warp-1 comb_l
  // entries by the sum and the max
  if ((int)threadIdx.x < nrows) {
    const int row = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, comb_m[w * 16 + row]);
    float L = 0.f, f[kConsumerWarps];
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      f[w] = ex2_ftz(comb_m[w * 16 + row] - M);
      L += f[w] * comb_l[w * 16 + row];
    }
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) comb_m[w * 16 + row] = f[w];
    comb_l[row] = L;
    comb_l[16 + row] = M;
  }
  named_bar_sync(3, kConsumerWarps * 32);
  for (int idx = threadIdx.x; idx < nrows * D; idx += kConsumerWarps * 32) {
    const int row = idx / D, d = idx % D;
    const float L = comb_l[row], M = comb_l[16 + row];
    float O = 0.f;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w)
      O += comb_m[w * 16 + row] * comb_o[(w * 16 + row) * D + d];
    const int hq = hq0 + row;
    if (direct) {
      p.out[((int64_t)qs * p.Hq + hq) * D + d] = __float2bfloat16_rn(O / L * p.v_scale);
    } else {
      const int64_t orow = ((int64_t)r * p.Hq + hq) * p.ws_splits + slot;
      p.ws_o[orow * D + d] = O * p.v_scale;
      if (d == 0) p.ws_ml[orow] = make_float2(M, L);
    }
  }
}

// MR: the warp's MMA state, MmaRows (up to 16 query heads as the MMA rows)
// or MmaKeys (up to 8 heads as the columns, the keys as the rows).
template <int D, bool FP8, class MR>
__global__ void __launch_bounds__(kThreads, 2)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, DecodeParams p) {
  launch_dependents();  // the merge that follows may be scheduled now
  using G = Geo<D, FP8>;
  constexpr int kStages = G::kStages;
  constexpr int kRows = 16;        // MMA rows (query heads, zero padded)
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  if constexpr (MR::kSw) ring += (1024u - (smem_u32(smem) & 1023u)) & 1023u;  // 1024-byte aligned
  float* comb_o = reinterpret_cast<float*>(ring + kStages * G::kStageBytes);  // [4][16][D]
  float* comb_m = comb_o + kConsumerWarps * kRows * D;                       // [4][16]
  float* comb_l = comb_m + kConsumerWarps * kRows;                           // [4][16]
  SmemTail* tail = reinterpret_cast<SmemTail*>(comb_l + kConsumerWarps * kRows);

  const int r = blockIdx.z;
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return;  // not a decode request
  if (qs < 0 || qs >= p.T) {  // a device qsl that leaves q / out
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int seq = p.seq_lens[r];
  if (seq < 1 || seq > p.max_blocks * p.B) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int nsplit = (seq + p.split_tokens - 1) / p.split_tokens;
  if (nsplit > (int)gridDim.x || (nsplit > 1 && nsplit > p.ws_splits)) {
    // device seq_lens disagree with the host mirror
    if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int split = blockIdx.x;
  if (split >= nsplit) return;
  const int k_begin = split * p.split_tokens;
  const int k_end = min(seq, k_begin + p.split_tokens);
  const int nch = (k_end - k_begin + kChunk - 1) / kChunk;
  // CTA y serves query heads hq0 .. hq0 + g - 1 of kv head kvh (g <= 16)
  const int kvh = blockIdx.y / p.head_groups;
  const int part = blockIdx.y % p.head_groups;
  const int hq0 = kvh * p.g + 16 * part;
  const int g = min(16, p.g - 16 * part);

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
    if (MR::kSw && lane == 0) {
      tc::prefetch_tensormap(&tmap_k);
      tc::prefetch_tensormap(&tmap_v);
    }
    produce<G, MR::kSw>(p, ring, tail, r, kvh, k_begin, nch, lane, &tmap_k, &tmap_v);
    return;
  }

  const int grp = lane >> 2, tig = lane & 3;
  const unsigned full = 0xffffffffu;
  MR st;
  {
    const __nv_bfloat16* rows[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const int row = grp + 8 * ri;
      rows[ri] = row < g ? p.q + ((int64_t)qs * p.Hq + hq0 + row) * D : nullptr;
    }
    st.load_q(rows, p.q_scale, tig);
  }
  st.reset();
  for (int c = warp; c < nch; c += kConsumerWarps) {
    const int stage = c % kStages, round = c / kStages;
    if (!__all_sync(full, mbar_wait(&tail->full[stage], round & 1, p.err))) {
      tail->abort = 1;
      break;
    }
    const uint8_t* Ks = ring + stage * G::kStageBytes;
    st.chunk(Ks, Ks + G::kChunkBytes, k_begin + c * kChunk, k_end, grp, tig);
    __syncwarp();
    if (lane == 0) mbar_arrive(&tail->empty[stage]);
  }
  st.finish_sums();
  st.to_comb(comb_o, comb_m, comb_l, warp, g, grp, tig);
  // one decision for all consumer threads (combine_rows holds a barrier)
  if (named_bar_or(1, kConsumerWarps * 32, *reinterpret_cast<volatile int*>(&tail->abort)))
    return;
  combine_rows<D>(p, comb_o, comb_m, comb_l, g, r, qs, hq0, nsplit == 1, split);
}

// ---------------------------------------------------------------------------
// Persistent GQA decode (2 <= g <= 16), see PersistPlan: CTA b streams the
// chunks [b Q, b Q + Q) of the call's flat chunk space, unit after unit,
// without draining its ring between them: the producer warp runs ahead
// across unit boundaries (and stages each unit's query rows with one bulk
// copy), so the start of each unit overlaps the end of the previous one, and
// every CTA gets the same number of chunks whatever the request lengths.
// Within a unit the chunks go round-robin to the four consumer warps (by ring
// position), which combine through shared memory at the unit's end.
struct Seg {
  int r;           // the request
  int kvh;
  int c0, c1;      // chunks [c0, c1) of the unit
  int key_end;     // keys at or past it are masked (the sequence length)
  int piece, n_pieces;
  int64_t f_next;  // flat position after this piece
};

__device__ __forceinline__ Seg segment_at(const DecodeParams& p, const int32_t* pref,
                                          const int32_t* rseq, int64_t f, int64_t f_end,
                                          int64_t Q) {
  // the request r with Hkv pref[r] <= f < Hkv pref[r + 1] (requests of no
  // chunk are skipped: their pref does not grow)
  int lo = 0, hi = p.R - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if ((int64_t)p.Hkv * pref[mid] <= f) lo = mid; else hi = mid - 1;
  }
  const int64_t C = pref[lo + 1] - pref[lo];
  const int64_t off = f - (int64_t)p.Hkv * pref[lo];
  Seg sg;
  sg.r = lo;
  sg.kvh = (int)(off / C);
  sg.key_end = rseq[lo];
  const int64_t a = (int64_t)p.Hkv * pref[lo] + (int64_t)sg.kvh * C;
  const int64_t end = min(a + C, f_end);  // > f: f lies inside the unit
  sg.c0 = (int)(f - a);
  sg.c1 = (int)(end - a);
  sg.piece = (int)(f / Q - a / Q);
  sg.n_pieces = (int)flat_pieces(a, C, Q);
  sg.f_next = end;
  return sg;
}

// Chunks of request r's keys (0 if r is not a decode request; a bad device
// entry raises kErrBounds and counts 0).
__device__ __forceinline__ int tail_chunks(const DecodeParams& p, int r) {
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return 0;
  const int seq = p.seq_lens[r];
  if (qs < 0 || qs >= p.T || seq < 1 || seq > p.max_blocks * p.B) {
    raise_error(p.err, kErrBounds);
    return 0;
  }
  return (seq + kChunk - 1) / kChunk;
}

// Staged query rows of the persistent decode: up to kQSlots tail units ahead.
constexpr int kQSlots = 8;
constexpr int kQStageBytes = 8192;
struct PersistBars {
  uint64_t q_full[kQSlots];   // a unit's query rows landed (transaction bytes)
  uint64_t q_empty[kQSlots];  // the four consumer warps have read them
  SmemTail t;
};

template <int D, bool FP8, class MR>
__global__ void __launch_bounds__(kThreads, 2)
    decode_persist_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, DecodeParams p) {
  launch_dependents();  // the merge that follows may be scheduled now
  using G = Geo<D, FP8>;
  constexpr int kStages = G::kStages;
  constexpr int kRows = 16;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  if constexpr (MR::kSw) ring += (1024u - (smem_u32(smem) & 1023u)) & 1023u;
  float* comb_o = reinterpret_cast<float*>(ring + kStages * G::kStageBytes);  // [4][16][D]
  float* comb_m = comb_o + kConsumerWarps * kRows * D;                       // [4][16]
  float* comb_l = comb_m + kConsumerWarps * kRows;                           // [4][16]
  int32_t* pref = reinterpret_cast<int32_t*>(comb_l + kConsumerWarps * kRows);  // [R + 1]
  int32_t* rtok = pref + kMaxPersistR + 4;  // [R] each request's token (decodes)
  int32_t* rseq = rtok + kMaxPersistR;      // [R] and its sequence length
  // the query rows of the next tail units, staged by the producer: kQSlots
  // slots of g rows each (as many as fit kQStageBytes)
  __nv_bfloat16* qstage = reinterpret_cast<__nv_bfloat16*>(rseq + kMaxPersistR);
  PersistBars* pb = reinterpret_cast<PersistBars*>(reinterpret_cast<uint8_t*>(qstage) +
                                                   kQStageBytes);
  SmemTail* tail = &pb->t;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.R;
  const int q_slot_elems = p.g * D;  // one tail unit's g query rows
  const int n_qslots = min(kQSlots, kQStageBytes / (q_slot_elems * 2));
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&tail->full[i], 1);
      mbar_init(&tail->empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kQSlots; ++i) {
      mbar_init(&pb->q_full[i], 1);
      mbar_init(&pb->q_empty[i], kConsumerWarps);
    }
    tail->abort = 0;
    fence_mbar_init();
  }
  // the tails' chunk counts (then their exclusive running sum, warp 0), and
  // each request's token and length, kept for the units below
  for (int r = tid; r < R; r += kThreads) {
    pref[r] = tail_chunks(p, r);
    rtok[r] = pref[r] > 0 ? p.qsl[r] : -1;
    rseq[r] = pref[r] > 0 ? p.seq_lens[r] : 0;
  }
  __syncthreads();
  if (warp == 0) {
    int carry = 0;
    for (int base = 0; base < R; base += 32) {
      const int v = base + lane < R ? pref[base + lane] : 0;
      int x = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (base + lane < R) pref[base + lane] = carry + x - v;
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (lane == 0) pref[R] = carry;
  }
  __syncthreads();
  const int64_t W = (int64_t)p.Hkv * pref[R];
  const int64_t Q =
      max((W + (int64_t)gridDim.x - 1) / (int64_t)gridDim.x, (int64_t)max(p.pp.q_min, 1));
  if (blockIdx.x == 0) {  // the plan, for the merge kernel
    if (tid == 0) {
      p.pp.aux[0] = (int32_t)Q;
      p.pp.aux[1] = (int32_t)W;
      if (W > (int64_t)gridDim.x * Q) raise_error(p.err, kErrBounds);  // chunks no CTA takes
    }
    for (int r = tid; r <= R; r += kThreads) p.pp.aux[2 + r] = pref[r];
  }
  const int64_t f_begin = (int64_t)blockIdx.x * Q;
  const int64_t f_end = min(W, f_begin + Q);
  if (f_begin >= f_end) return;

  if (warp == kConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (MR::kSw && lane == 0) {
      tc::prefetch_tensormap(&tmap_k);
      tc::prefetch_tensormap(&tmap_v);
    }
    int64_t q = 0, issued = 0;
    int n_tail = 0;  // tail units whose query rows were staged
    bool ok = true;
    for (int64_t f = f_begin; f < f_end;) {
      const Seg sg = segment_at(p, pref, rseq, f, f_end, Q);
      if (sg.f_next <= f) break;  // cannot happen: f lies inside the unit
      f = sg.f_next;
      const int nch = sg.c1 - sg.c0;
      {
        // the unit's g query rows (contiguous in q) into the next staging slot,
        // once the consumers have read the unit that used it before
        const int slot = n_tail % n_qslots, use = n_tail / n_qslots;
        if (lane == 0) {
          if (use > 0) ok = mbar_wait(&pb->q_empty[slot], (use - 1) & 1, p.err);
          if (ok) {
            mbar_arrive_expect_tx(&pb->q_full[slot], (unsigned)(q_slot_elems * 2));
            bulk_g2s(qstage + slot * q_slot_elems,
                     p.q + ((int64_t)rtok[sg.r] * p.Hq + (int64_t)sg.kvh * p.g) * D,
                     (unsigned)(q_slot_elems * 2), &pb->q_full[slot]);
          }
        }
        if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
          if (lane == 0) tail->abort = 1;
          break;
        }
        ++n_tail;
      }
      const int32_t* table = p.block_tables + (int64_t)sg.r * p.max_blocks;
      if (!produce_run<G, MR::kSw>(p, ring, tail, table, sg.kvh, sg.c0 * kChunk, nch, q, lane,
                                   &tmap_k, &tmap_v, &issued))
        break;
      q += nch;
    }
    drain<G>(p, tail, issued, lane);
    // and the staged query rows still in flight (the last use of each slot)
    if (lane == 0)
      for (int u = n_tail - n_qslots > 0 ? n_tail - n_qslots : 0; u < n_tail; ++u)
        mbar_wait(&pb->q_full[u % n_qslots], (u / n_qslots) & 1, p.err);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int grp = lane >> 2, tig = lane & 3;
  const unsigned full = 0xffffffffu;
  const int g = p.g;
  int64_t q = 0;   // ring position of the unit's first chunk
  int n_tail = 0;  // units started (their query rows are staged)
  bool ok = true;
  MR st;
  for (int64_t f = f_begin; f < f_end;) {
    const Seg sg = segment_at(p, pref, rseq, f, f_end, Q);
    if (sg.f_next <= f) break;  // (as the producer)
    f = sg.f_next;
    const int nch = sg.c1 - sg.c0;
    const int k_begin = sg.c0 * kChunk;
    const int k_end = min(sg.key_end, sg.c1 * kChunk);
    // rows: the g heads of the request's token, staged by the producer
    const int qs = rtok[sg.r];
    const int hq0 = sg.kvh * g;
    {
      const int slot = n_tail % n_qslots;
      if (!__all_sync(full, mbar_wait(&pb->q_full[slot], (n_tail / n_qslots) & 1, p.err))) {
        tail->abort = 1;
        ok = false;
      }
      const __nv_bfloat16* rows[2];
#pragma unroll
      for (int ri = 0; ri < 2; ++ri) {
        const int row = grp + 8 * ri;
        rows[ri] = ok && row < g ? qstage + slot * q_slot_elems + row * D : nullptr;
      }
      st.load_q(rows, p.q_scale, tig);
      __syncwarp();
      if (lane == 0) mbar_arrive(&pb->q_empty[slot]);  // the rows are in registers
      ++n_tail;
    }
    st.reset();
    // chunk c sits at ring position q + c and belongs to warp (q + c) mod 4
    for (int c = (int)((warp - q % kConsumerWarps + kConsumerWarps) % kConsumerWarps);
         ok && c < nch; c += kConsumerWarps) {
      const int64_t pos = q + c;
      const int stage = (int)(pos % kStages);
      if (!__all_sync(full, mbar_wait(&tail->full[stage], (pos / kStages) & 1, p.err))) {
        tail->abort = 1;
        ok = false;
        break;
      }
      const uint8_t* Ks = ring + stage * G::kStageBytes;
      st.chunk(Ks, Ks + G::kChunkBytes, k_begin + c * kChunk, k_end, grp, tig);
      __syncwarp();
      if (lane == 0) mbar_arrive_cnt(&tail->empty[stage], kConsumerWarps);
    }
    st.finish_sums();
    st.to_comb(comb_o, comb_m, comb_l, warp, g, grp, tig);
    // one decision for all consumer threads (combine_rows holds a barrier)
    const bool failed = named_bar_or(1, kConsumerWarps * 32,
                                     !ok || *reinterpret_cast<volatile int*>(&tail->abort));
    // the output of a request read in one piece; else its piece's partial
    const bool direct = sg.n_pieces == 1;
    if (!direct && sg.piece >= p.ws_splits) {
      if (tid == 0) raise_error(p.err, kErrBounds);  // device lengths disagree with the plan
    } else if (!failed) {
      combine_rows<D>(p, comb_o, comb_m, comb_l, g, sg.r, qs, hq0, direct, sg.piece);
    }
    q += nch;
    // every consumer warp takes the same decision (and the comb buffer is
    // free again for the next unit)
    if (named_bar_or(2, kConsumerWarps * 32,
                     failed || *reinterpret_cast<volatile int*>(&tail->abort)))
      break;
  }
}

// One warp per (query head, request) with more than one split slot: combines
// the partials by log-sum-exp. Lane i holds the (max, sum) of slots i, i+32,
// ... and dims (D/32) i .. (D/32) i + D/32 - 1 of every slot's output, so the
// loads of all slots go out together.
constexpr int kMergeWarps = 8;
template <int D>
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(DecodeParams p) {
  constexpr int kV = D / 32;  // dims per lane
  grid_dependency_wait();  // the decode grid's partials are complete and visible
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x * kMergeWarps + (threadIdx.x >> 5), r = blockIdx.y;
  if (h >= p.Hq) return;
  const int qs = p.qsl[r], qe = p.qsl[r + 1], seq = p.seq_lens[r];
  if (qe - qs != 1 || qs < 0 || qs >= p.T) return;  // the decode kernel flagged a bad qsl
  if (seq < 1 || seq > p.max_blocks * p.B) return;
  const int grp_id = group_of(p.groups, r);
  const int k_lo = grp_id >= 0 ? p.groups.prefix_tokens[grp_id] : 0;
  if (k_lo >= seq) return;
  // slots: the shared-prefix pieces (group members) and the splits
  int nsplit;
  if (p.pp.on) {
    // the persistent kernel's partition, as it recorded it
    const int64_t Q = p.pp.aux[0];
    const int32_t* pref = p.pp.aux + 2;
    const int64_t C = pref[r + 1] - pref[r];
    if (C <= 0 || Q <= 0) return;
    const int64_t a = (int64_t)p.Hkv * pref[r] + (h / p.g) * C;
    nsplit = (int)flat_pieces(a, C, Q);  // 1: the decode kernel wrote the output
  } else {
    nsplit = prefix_slots(p.groups, grp_id) + (seq - k_lo + p.split_tokens - 1) / p.split_tokens;
  }
  if (nsplit <= 1 || nsplit > p.ws_splits) return;
  const int64_t row0 = ((int64_t)r * p.Hq + h) * p.ws_splits;
  const unsigned full = 0xffffffffu;
  float M = -INFINITY;
  for (int s = lane; s < nsplit; s += 32) M = fmaxf(M, p.ws_ml[row0 + s].x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(full, M, o));
  float L = 0.f, O[kV];
#pragma unroll
  for (int v = 0; v < kV; ++v) O[v] = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 32) {
    const int n = min(32, nsplit - s0);
    float f = 0.f;
    if (lane < n) {
      const float2 ml = p.ws_ml[row0 + s0 + lane];
      f = exp2f(ml.x - M);
      L += f * ml.y;
    }
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
      const float fi = __shfl_sync(full, f, i);
      const float* src = p.ws_o + (row0 + s0 + i) * D + kV * lane;
      if constexpr (kV == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        O[0] += fi * x.x; O[1] += fi * x.y; O[2] += fi * x.z; O[3] += fi * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        O[0] += fi * x.x; O[1] += fi * x.y;
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(full, L, o);
  __nv_bfloat16* dst = p.out + ((int64_t)qs * p.Hq + h) * D + kV * lane;
  if constexpr (kV == 4) {
    __nv_bfloat162 a = __floats2bfloat162_rn(O[0] / L, O[1] / L);
    __nv_bfloat162 b = __floats2bfloat162_rn(O[2] / L, O[3] / L);
    uint2 w;
    w.x = *reinterpret_cast<uint32_t*>(&a);
    w.y = *reinterpret_cast<uint32_t*>(&b);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(O[0] / L, O[1] / L);
  }
}

template <int D, bool FP8, int GH>
constexpr int decode_smem_bytes() {
  return Geo<D, FP8>::kStages * Geo<D, FP8>::kStageBytes + kConsumerWarps * GH * (D + 2) * 4 +
         (int)sizeof(SmemTail);
}

template <int D, bool FP8, int GH, int HG>
cudaError_t launch_decode_t(const DecodeParams& p, int R, int max_splits, cudaStream_t s) {
  constexpr int smem = decode_smem_bytes<D, FP8, GH>();
  auto k = decode_kernel<D, FP8, GH, HG>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(max_splits, p.Hkv, R);
  k<<<grid, kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_decode_mma_t(const DecodeParams& p, int R, int max_splits, cudaStream_t s) {
  constexpr bool kSw = FP8 && D == 128;
  constexpr int smem = (kSw ? 1024 : 0) + Geo<D, FP8>::kStages * Geo<D, FP8>::kStageBytes +
                       kConsumerWarps * 16 * (D + 2) * 4 + (int)sizeof(SmemTail);
  CUtensorMap tk, tv;
  cudaError_t e = decode_maps<D, FP8>(p, &tk, &tv);
  if (e != cudaSuccess) return e;
  // up to 8 heads: the keys as the MMA rows (half the MMAs of 16 padded rows)
  auto k = p.g <= 8 ? decode_mma_kernel<D, FP8, MmaKeys<D, FP8>>
                    : decode_mma_kernel<D, FP8, MmaRows<D, FP8>>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dim3 grid(max_splits, p.Hkv * p.head_groups, R);
  k<<<grid, kThreads, smem, s>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D, bool FP8>
cudaError_t launch_decode_persist_t(const DecodeParams& p, int n_cta, cudaStream_t s) {
  constexpr bool kSw = FP8 && D == 128;
  constexpr int smem = (kSw ? 1024 : 0) + Geo<D, FP8>::kStages * Geo<D, FP8>::kStageBytes +
                       kConsumerWarps * 16 * (D + 2) * 4 + (3 * kMaxPersistR + 4) * 4 +
                       kQStageBytes + (int)sizeof(PersistBars);
  static_assert(2 * (smem + 1024) <= 228 * 1024, "two CTAs per SM");
  if (p.g < 2 || p.g > 16 || p.head_groups != 1 || p.R > kMaxPersistR || p.R < 1 || !p.pp.on ||
      !p.pp.aux)
    return cudaErrorInvalidValue;
  CUtensorMap tk, tv;
  cudaError_t e = decode_maps<D, FP8>(p, &tk, &tv);
  if (e != cudaSuccess) return e;
  auto k = p.g <= 8 ? decode_persist_kernel<D, FP8, MmaKeys<D, FP8>>
                    : decode_persist_kernel<D, FP8, MmaRows<D, FP8>>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<n_cta, kThreads, smem, s>>>(tk, tv, p);
  return cudaGetLastError();
}

// g = 1: one head per kv head, CUDA-core dot products (a 16-row MMA would be
// 1/16 used); g >= 2: warp-level tensor-core MMAs for up to 16 heads at once
// (any g: rows past g are zero padding; g > 16 takes ceil(g / 16) CTAs per
// kv head, each reading the kv head's keys).
template <int D, bool FP8>
cudaError_t launch_decode_d(const DecodeParams& p, int R, int max_splits, cudaStream_t s) {
  if (p.g == 1) {
    if (p.head_groups != 1) return cudaErrorInvalidValue;
    return launch_decode_t<D, FP8, 1, 1>(p, R, max_splits, s);
  }
  if (p.g >= 2 && p.head_groups == (p.g + 15) / 16)
    return launch_decode_mma_t<D, FP8>(p, R, max_splits, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, int D, bool fp8, int R, int max_splits,
                          cudaStream_t s) {
  if (D == 128)
    return fp8 ? launch_decode_d<128, true>(p, R, max_splits, s)
               : launch_decode_d<128, false>(p, R, max_splits, s);
  return fp8 ? launch_decode_d<64, true>(p, R, max_splits, s)
             : launch_decode_d<64, false>(p, R, max_splits, s);
}

cudaError_t launch_decode_persist(const DecodeParams& p, int D, bool fp8, int n_cta,
                                  cudaStream_t s) {
  if (D == 128)
    return fp8 ? launch_decode_persist_t<128, true>(p, n_cta, s)
               : launch_decode_persist_t<128, false>(p, n_cta, s);
  return fp8 ? launch_decode_persist_t<64, true>(p, n_cta, s)
             : launch_decode_persist_t<64, false>(p, n_cta, s);
}

cudaError_t launch_merge(const DecodeParams& p, int D, int R, cudaStream_t s) {
  // a programmatic dependent launch: scheduled while the decode grid before
  // it drains, it waits for that grid's partials in grid_dependency_wait
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((p.Hq + kMergeWarps - 1) / kMergeWarps, R);
  cfg.blockDim = dim3(kMergeWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return D == 128 ? cudaLaunchKernelEx(&cfg, merge_kernel<128>, p)
                  : cudaLaunchKernelEx(&cfg, merge_kernel<64>, p);
}

}  // namespace pa
