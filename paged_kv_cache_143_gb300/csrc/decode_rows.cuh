// decode_rows.cuh — pieces shared by the decode kernels (decode.cu) and the
// shared-prefix decode (cascade.cu): the 16-key chunk geometry of a K/V
// stage, the warp-level tensor-core state of up to 16 query rows (MmaRows),
// and the TMA maps of the swizzled E4M3 stages.
#pragma once

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_kernels.h"
#include "tc_ptx.cuh"

namespace pa {
namespace {


constexpr int kChunk = 16;         // keys per pipeline stage
constexpr int kConsumerWarps = 4;  // compute warps of a decode CTA (warps 0..3)
constexpr int kMaxStages = 16;     // ring depth of the E4M3 kernels

template <int D, bool FP8>
struct Geo {
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElt;                  // one key row
  static constexpr int kPieceBytes = kRowBytes / 8 >= 16 ? 16 : kRowBytes / 8;
  static constexpr int kPieces = kRowBytes / (8 * kPieceBytes);
  static constexpr int kPieceElems = kPieceBytes / kElt;
  static constexpr int kPiecePairs = kPieceElems / 2;
  static constexpr int kDimsPerLane = kPieces * kPieceElems;  // = D / 8
  static constexpr int kPairsPerLane = kDimsPerLane / 2;
  static constexpr int kChunkBytes = kChunk * kRowBytes;
  static constexpr int kStageBytes = 2 * kChunkBytes;         // K then V
  // ring depth: 64 KB of K/V in flight per CTA whatever the element size
  // (8 stages of bf16 chunks, 16 of E4M3 chunks for D = 128); a multiple of
  // the consumer warp count
  static constexpr int kStages = 65536 / kStageBytes > kMaxStages ? kMaxStages
                                                                  : 65536 / kStageBytes;
  static_assert(kStages % kConsumerWarps == 0, "ring depth");
  static_assert(kDimsPerLane * 8 == D, "lane split must cover the head");
  // first dimension of piece p of lane b
  __device__ static constexpr int dim0(int p, int b) { return (p * 8 + b) * kPieceElems; }
};

// ---------------------------------------------------------------------------
// Decode for GQA groups g >= 2 on warp-level tensor-core MMAs.
//
// Per kv head the decode contraction is [g x D] . [D x keys] with g <= 16,
// below the smallest tcgen05 tile (M = 64), so each consumer warp issues
// mma.sync m16n8k16 (f32 accumulate) on register fragments: up to 16 query
// rows (padded with zero rows), a 16-key chunk is two n8 tiles. The operands
// come straight from the linear rows the bulk copies deliver:
//  - S = Q K^T: a fixed permutation of the head dimension, the same for Q and
//    K, maps k-steps 2j and 2j+1 of lane (grp, tig) onto the 8 contiguous
//    dims 32 j + 8 tig .. +7, so every K fragment is one 16-byte load of
//    key row grp (bf16), or one 8-byte load widened to f16 (E4M3);
//  - P is the S accumulator tile re-packed to 16 bits (no data movement);
//  - O += P V: output dim 16 grp + nt (D = 128; 8 grp + nt for D = 64) is
//    column grp of n-tile nt, so lane (grp, tig) reads rows 2tig, 2tig+1,
//    2tig+8, 2tig+9 over its 16 (8) contiguous dims and pairs them with prmt.
// E4M3 pools run f16 MMAs: the codes widen exactly to f16, and each query row
// is pre-scaled by a power of two into [2^14, 2^15) before its f16 rounding
// (undone in the score scale), so f16 range never limits the queries.
// E4M3 at D = 128: the stages arrive as TMA tensor boxes with the 128-byte
// swizzle (16-byte chunk c of row r stored at chunk c ^ (r & 7)). In linear
// rows the lanes that hold different keys of the same columns hit the same
// banks (rows are 128 B apart); swizzled, a lane reads the chunks 2 tig and
// 2 tig + 1 of its K row (the head-dimension permutation becomes: k-step
// pair j of lane tig = dims 32 tig + 8 j .. +7) and chunk grp of its V rows,
// and every 16-byte load of a quarter-warp falls on distinct banks.
//
// MmaRows holds one warp's state for up to 16 query rows: the Q fragments,
// the per-row score scale, and the running (O, max, sum) of the rows.
template <int D, bool FP8>
struct MmaRows {
  static constexpr int KJ = D / 32;  // pairs of k-steps
  static constexpr int DG = D / 8;   // output dims per lane group = n-tiles of O
  static constexpr bool kSw = FP8 && D == 128;  // swizzled stages (TMA tensor copies)
  using G = Geo<D, FP8>;
  uint32_t qa[KJ][2][4];  // qa[j][row][w] = the 16-bit pair of dims 32j + 8tig + 2w
  float sc[2];            // score scale of rows grp and grp + 8 (log2 units)
  float o[DG][4];
  float m[2], l[2];

  // The raw query rows of load_q (rows grp and grp + 8), fetched ahead of
  // their conversion so that the load latency overlaps other start-up work.
  struct QRaw {
    uint4 v[2][KJ];
  };
  static __device__ __forceinline__ void fetch_q(const __nv_bfloat16* const (&rows)[2], QRaw& r,
                                                 int tig) {
#pragma unroll
    for (int ri = 0; ri < 2; ++ri)
#pragma unroll
      for (int j = 0; j < KJ; ++j)
        r.v[ri][j] = rows[ri] ? *reinterpret_cast<const uint4*>(
                                    rows[ri] + (kSw ? 32 * tig + 8 * j : 32 * j + 8 * tig))
                              : make_uint4(0u, 0u, 0u, 0u);  // a zero padding row
  }

  // Loads rows grp and grp + 8 (rows[ri], nullptr: a zero padding row; a
  // row may sit in global or in shared memory).
  __device__ __forceinline__ void load_q(const __nv_bfloat16* const (&rows)[2], float q_scale,
                                         int tig) {
    QRaw r;
    fetch_q(rows, r, tig);
    load_q(r, q_scale, tig);
  }

  __device__ __forceinline__ void load_q(const QRaw& r, float q_scale, int tig) {
    const unsigned full = 0xffffffffu;
    float qf[2][KJ][8];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri)
#pragma unroll
      for (int j = 0; j < KJ; ++j) bf16x8_to_f32(r.v[ri][j], qf[ri][j]);
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      float up = 1.f;
      sc[ri] = q_scale;
      if (FP8) {
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < KJ; ++j)
#pragma unroll
          for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(qf[ri][j][e]));
        amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
        int e2 = 0;
        if (amax > 0.f) {
          const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
          e2 = min(100, max(-120, 14 - ex));
        }
        up = __uint_as_float((uint32_t)(e2 + 127) << 23);
        sc[ri] *= __uint_as_float((uint32_t)(127 - e2) << 23);
      }
#pragma unroll
      for (int j = 0; j < KJ; ++j)
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          if (FP8) {
            __half2 h = __floats2half2_rn(qf[ri][j][2 * w] * up, qf[ri][j][2 * w + 1] * up);
            qa[j][ri][w] = *reinterpret_cast<uint32_t*>(&h);
          } else {
            __nv_bfloat162 h = __floats2bfloat162_rn(qf[ri][j][2 * w], qf[ri][j][2 * w + 1]);
            qa[j][ri][w] = *reinterpret_cast<uint32_t*>(&h);
          }
        }
    }
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int nt = 0; nt < DG; ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  static __device__ __forceinline__ void mma(float (&c)[4], uint32_t a0, uint32_t a1,
                                             uint32_t a2, uint32_t a3, uint32_t b0,
                                             uint32_t b1) {
    if (FP8)
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
      asm volatile(
          "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
          "{%8,%9}, {%0,%1,%2,%3};"
          : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
          : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
  // 8 E4M3 codes -> four f16 pairs (exact)
  static __device__ __forceinline__ void widen8(uint32_t x, uint32_t y, uint32_t* w) {
    asm("{\n\t.reg .b16 a, b, c, d;\n\tmov.b32 {a, b}, %4;\n\tmov.b32 {c, d}, %5;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t"
        "cvt.rn.f16x2.e4m3x2 %2, c;\n\tcvt.rn.f16x2.e4m3x2 %3, d;\n\t}"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
        : "r"(x), "r"(y));
  }
  // 8 consecutive elements of a row -> four 16-bit pairs
  static __device__ __forceinline__ void load8(const uint8_t* src, uint32_t (&w)[4]) {
    if (FP8) {
      const uint2 v = *reinterpret_cast<const uint2*>(src);
      widen8(v.x, v.y, w);
    } else {
      const uint4 v = *reinterpret_cast<const uint4*>(src);
      w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    }
  }

  // The reference maximum of a row after a step whose largest score is mx
  // (log2 units): it moves to the new maximum only when that exceeds the
  // current reference by more than 2^8 (alpha = the factor that rescales
  // what was accumulated against the old reference; 1 when it stays). A stale
  // reference is exact algebra (every accumulated term and the sum share
  // it); it bounds the step's weights P by 2^8 and skips most rescales.
  static __device__ __forceinline__ float rebase(float m_cur, float mx, float& alpha) {
    const bool move = mx > m_cur + 8.f;  // (also the first step: m_cur = -inf)
    alpha = move ? ex2_ftz(m_cur - mx) : 1.f;
    return move ? mx : m_cur;
  }

  // NC consecutive 16-key chunks (K rows Ks[c], V rows Vs[c], keys key0 +
  // 16 c .. key0 + 16 c + 15, those at or past k_end masked): scores, one
  // online-softmax update over all NC * 16 keys, O += P V. Two chunks per call
  // give the warp twice the independent MMA chains and half the softmax
  // bookkeeping per key.
  template <int NC>
  __device__ __forceinline__ void chunks(const uint8_t* const (&Ks)[NC],
                                         const uint8_t* const (&Vs)[NC], int key0, int k_end,
                                         int grp, int tig) {
    const unsigned full = 0xffffffffu;
    constexpr int NT = 2 * NC;  // n-tiles of 8 keys
    // S for keys 8t + grp (B fragments), t = n-tile
    float s[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
      const uint8_t* krow = Ks[t >> 1] + (8 * (t & 1) + grp) * G::kRowBytes;
      if constexpr (kSw) {
        // k-step pairs 2h, 2h+1 of lane tig: dims 32 tig + 16 h .. +15, the
        // 16-byte chunk 2 tig + h of row grp, stored at chunk ^ grp
#pragma unroll
        for (int h = 0; h < KJ / 2; ++h) {
          const uint4 x =
              *reinterpret_cast<const uint4*>(krow + (((2 * tig + h) ^ grp) << 4));
          uint32_t kw[4];
          widen8(x.x, x.y, kw);
          mma(s[t], qa[2 * h][0][0], qa[2 * h][1][0], qa[2 * h][0][1], qa[2 * h][1][1], kw[0],
              kw[1]);
          mma(s[t], qa[2 * h][0][2], qa[2 * h][1][2], qa[2 * h][0][3], qa[2 * h][1][3], kw[2],
              kw[3]);
          widen8(x.z, x.w, kw);
          mma(s[t], qa[2 * h + 1][0][0], qa[2 * h + 1][1][0], qa[2 * h + 1][0][1],
              qa[2 * h + 1][1][1], kw[0], kw[1]);
          mma(s[t], qa[2 * h + 1][0][2], qa[2 * h + 1][1][2], qa[2 * h + 1][0][3],
              qa[2 * h + 1][1][3], kw[2], kw[3]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < KJ; ++j) {
          uint32_t kw[4];
          load8(krow + (32 * j + 8 * tig) * G::kElt, kw);
          mma(s[t], qa[j][0][0], qa[j][1][0], qa[j][0][1], qa[j][1][1], kw[0], kw[1]);
          mma(s[t], qa[j][0][2], qa[j][1][2], qa[j][0][3], qa[j][1][3], kw[2], kw[3]);
        }
      }
    }
    // scale, mask, online softmax of rows grp (c0, c1) and grp + 8 (c2, c3)
    const bool whole = key0 + 16 * NC <= k_end;  // no key of the step is masked
    float alpha[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      float mx = -INFINITY;
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& x = s[t][2 * ri + e];
          x = whole || key0 + 8 * t + 2 * tig + e < k_end ? x * sc[ri] : -INFINITY;
          mx = fmaxf(mx, x);
        }
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 2));
      const float m_ref = rebase(m[ri], mx, alpha[ri]);
      float ps = 0.f;
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float& x = s[t][2 * ri + e];
          x = ex2_ftz(x - m_ref);
          ps += x;
        }
      l[ri] = l[ri] * alpha[ri] + ps;
      m[ri] = m_ref;
    }
    if (__any_sync(full, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int nt = 0; nt < DG; ++nt) {
        o[nt][0] *= alpha[0];
        o[nt][1] *= alpha[0];
        o[nt][2] *= alpha[1];
        o[nt][3] *= alpha[1];
      }
    }
    auto pk = [](float x, float y) -> uint32_t {
      if (FP8) {
        __half2 h = __floats2half2_rn(x, y);
        return *reinterpret_cast<uint32_t*>(&h);
      }
      __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
      return *reinterpret_cast<uint32_t*>(&h);
    };
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      // P of chunk c as the A fragment of its 16-key step
      const uint32_t pa0 = pk(s[2 * c][0], s[2 * c][1]), pa1 = pk(s[2 * c][2], s[2 * c][3]);
      const uint32_t pa2 = pk(s[2 * c + 1][0], s[2 * c + 1][1]);
      const uint32_t pa3 = pk(s[2 * c + 1][2], s[2 * c + 1][3]);
      // V rows 2tig, 2tig+1, 2tig+8, 2tig+9 over dims DG grp .. DG grp + DG - 1
      uint32_t vw[4][DG / 2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kr = 2 * tig + (i & 1) + 8 * (i >> 1);
        if constexpr (kSw) {  // the 16-byte chunk grp of row kr, stored at grp ^ (kr & 7)
          const uint4 x = *reinterpret_cast<const uint4*>(Vs[c] + kr * G::kRowBytes +
                                                          ((grp ^ (kr & 7)) << 4));
          widen8(x.x, x.y, &vw[i][0]);
          widen8(x.z, x.w, &vw[i][4]);
        } else {
          const uint8_t* vrow = Vs[c] + kr * G::kRowBytes + DG * grp * G::kElt;
#pragma unroll
          for (int h = 0; h < DG / 8; ++h) {
            uint32_t w4[4];
            load8(vrow + 8 * h * G::kElt, w4);
#pragma unroll
            for (int w = 0; w < 4; ++w) vw[i][4 * h + w] = w4[w];
          }
        }
        if (!whole && key0 + 16 * c + kr >= k_end)  // unwritten cells may hold NaN; P = 0 must not meet them
#pragma unroll
          for (int w = 0; w < DG / 2; ++w) vw[i][w] = 0u;
      }
#pragma unroll
      for (int nt = 0; nt < DG; ++nt) {
        const uint32_t sel = (nt & 1) ? 0x7632u : 0x5410u;
        uint32_t b0, b1;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b0) : "r"(vw[0][nt >> 1]), "r"(vw[1][nt >> 1]), "r"(sel));
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(b1) : "r"(vw[2][nt >> 1]), "r"(vw[3][nt >> 1]), "r"(sel));
        mma(o[nt], pa0, pa1, pa2, pa3, b0, b1);
      }
    }
  }

  // One 16-key chunk (K rows Ks, V rows Vs, keys key0 .. key0 + 15).
  __device__ __forceinline__ void chunk(const uint8_t* Ks, const uint8_t* Vs, int key0, int k_end,
                                        int grp, int tig) {
    const uint8_t* const k[1] = {Ks};
    const uint8_t* const v[1] = {Vs};
    chunks<1>(k, v, key0, k_end, grp, tig);
  }

  // Per-row sums over the four lanes of a row (the maxima already agree).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      l[ri] += __shfl_xor_sync(0xffffffffu, l[ri], 1);
      l[ri] += __shfl_xor_sync(0xffffffffu, l[ri], 2);
    }
  }

  // This warp's rows into the combine buffer of warp `warp` (rows < nrows).
  __device__ __forceinline__ void to_comb(float* comb_o, float* comb_m, float* comb_l, int warp,
                                          int nrows, int grp, int tig) const {
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      const int row = grp + 8 * ri;
      if (row < nrows) {
#pragma unroll
        for (int nt = 0; nt < DG; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            comb_o[(warp * 16 + row) * D + DG * (2 * tig + e) + nt] = o[nt][2 * ri + e];
        if (tig == 0) {
          comb_m[warp * 16 + row] = m[ri];
          comb_l[warp * 16 + row] = l[ri];
        }
      }
    }
  }

  // After finish_sums: the unnormalised output this lane holds, as runs of
  // four consecutive dims, f(row, first dim, values, row max, row sum) for
  // rows grp and grp + 8; and each row's (max, sum) once, from one lane:
  // g(row, m, l).
  template <class F>
  __device__ __forceinline__ void for_each_run(int grp, int tig, F&& f) const {
#pragma unroll
    for (int ri = 0; ri < 2; ++ri)
#pragma unroll
      for (int e = 0; e < 2; ++e)
#pragma unroll
        for (int i = 0; i < DG / 4; ++i)
          f(grp + 8 * ri, DG * (2 * tig + e) + 4 * i,
            make_float4(o[4 * i][2 * ri + e], o[4 * i + 1][2 * ri + e], o[4 * i + 2][2 * ri + e],
                        o[4 * i + 3][2 * ri + e]),
            m[ri], l[ri]);
  }
  template <class F>
  __device__ __forceinline__ void for_each_stat(int grp, int tig, F&& f) const {
    if (tig == 0) {
      f(grp, m[0], l[0]);
      f(grp + 8, m[1], l[1]);
    }
  }
};

// ---------------------------------------------------------------------------
// The same warp-level decode with the roles of the MMA operands swapped, for
// GQA groups of at most 8 heads: the 16 keys of a chunk are the MMA rows and
// the heads the 8 columns,
//   S^T = K Q^T   (m16n8k16: A = K, 16 keys x 16 dims per k-step; B = Q^T),
//   O^T += V^T P^T (m16n8k16: A = V^T, 16 dims x 16 keys; B = P^T).
// A chunk then takes D/16 + D/16 MMAs instead of MmaRows' 2 D/16 + 2 D/16
// (whose 16 rows are mostly padding for g <= 8), and a lane holds four
// scores of a chunk instead of eight.
//  - S: a fixed permutation of the head dimension, the same for Q and K,
//    gives lane tig eight dims per pair of k-steps: k-steps 2q and 2q + 1
//    take dims b + {0,1}, b + {2,3} and b + {4,5}, b + {6,7} as their
//    k-columns (2 tig, 2 tig + 1) and (2 tig + 8, + 9), where b is
//    D/4 tig + 8 q for E4M3 pools (a lane's dims are one contiguous run: its
//    8-byte loads of the 128-byte-swizzled rows, or of the 64-byte rows at
//    D = 64, fall on distinct banks) and 32 q + 8 tig for bf16 pools (the four
//    lanes of a row read 64 contiguous bytes per load, as MmaRows does). The
//    K fragments are then loads of key rows grp and grp + 8, and Q^T's
//    fragments are head grp's dims, loaded once.
//  - softmax per head (column): lane (grp, tig) holds the scores of keys grp,
//    grp + 8 for heads 2 tig, 2 tig + 1; maxima reduce over the eight grp
//    lanes by xor-shuffles, sums stay per lane until finish_sums.
//  - P^T: the 16-bit P of keys 0..7 (and 8..15) is transposed in registers by
//    movmatrix.trans, which turns the accumulator layout (row key, columns
//    heads) into the B-operand layout (rows keys 2 tig, 2 tig + 1, column
//    head grp).
//  - O^T: m-tile mt holds output dims DG grp + 2 mt (row grp) and
//    DG grp + 2 mt + 1 (row grp + 8), DG = D / 8, so the A fragments come from
//    the same V rows 2 tig, 2 tig + 1, 2 tig + 8, 2 tig + 9 over dims
//    DG grp .. DG grp + DG - 1 that MmaRows reads, paired by prmt, and a lane
//    ends up holding DG contiguous output dims of heads 2 tig, 2 tig + 1.
// Same numerics as MmaRows: fp32 scores and accumulators, P rounded to 16
// bits, E4M3 codes widened exactly to f16, queries of E4M3 pools pre-scaled
// by a power of two per head.
template <int D, bool FP8>
struct MmaKeys {
  static constexpr int KS = D / 16;  // k-steps of S
  static constexpr int DG = D / 8;   // output dims per lane group
  static constexpr int MT = DG / 2;  // m-tiles of O^T
  static constexpr bool kSw = FP8 && D == 128;
  static constexpr int kLaneDims = D / 4;  // dims of Q and K per lane (tig)
  using G = Geo<D, FP8>;
  uint32_t qb[KS][2];  // B fragments of Q^T (head grp): k-step j, dims 4j + {0,1} / {2,3}
  float sc[2];         // score scale of heads 2 tig, 2 tig + 1 (log2 units)
  float o[MT][4];      // O^T: [mt] = (dim d0, head 2tig), (d0, 2tig+1), (d0+1, 2tig), (d0+1, 2tig+1)
  float m[2], l[2];    // heads 2 tig, 2 tig + 1 (l: this lane's keys until finish_sums)

  // Head grp's dims of lane tig (kdim8 below) as raw bf16 words.
  struct QRaw {
    uint4 v[kLaneDims / 8];
  };
  // First of the eight dims that lane tig takes for k-steps 2q, 2q + 1.
  static __device__ __forceinline__ int kdim8(int q, int tig) {
    return FP8 ? kLaneDims * tig + 8 * q : 32 * q + 8 * tig;
  }
  // rows[0]: the row of head grp (nullptr: a zero padding head); rows[1] is
  // not used (heads grp + 8 do not exist for g <= 8).
  static __device__ __forceinline__ void fetch_q(const __nv_bfloat16* const (&rows)[2], QRaw& r,
                                                 int tig) {
#pragma unroll
    for (int i = 0; i < kLaneDims / 8; ++i)
      r.v[i] = rows[0] ? *reinterpret_cast<const uint4*>(rows[0] + kdim8(i, tig))
                       : make_uint4(0u, 0u, 0u, 0u);
  }
  __device__ __forceinline__ void load_q(const __nv_bfloat16* const (&rows)[2], float q_scale,
                                         int tig) {
    QRaw r;
    fetch_q(rows, r, tig);
    load_q(r, q_scale, tig);
  }
  __device__ __forceinline__ void load_q(const QRaw& r, float q_scale, int tig) {
    const unsigned full = 0xffffffffu;
    float qf[kLaneDims];
#pragma unroll
    for (int i = 0; i < kLaneDims / 8; ++i) bf16x8_to_f32(r.v[i], qf + 8 * i);
    float up = 1.f, s_head = q_scale;
    if (FP8) {  // head grp's largest magnitude into [2^14, 2^15) before f16 rounding
      float amax = 0.f;
#pragma unroll
      for (int i = 0; i < kLaneDims; ++i) amax = fmaxf(amax, fabsf(qf[i]));
      amax = fmaxf(amax, __shfl_xor_sync(full, amax, 1));
      amax = fmaxf(amax, __shfl_xor_sync(full, amax, 2));
      int e2 = 0;
      if (amax > 0.f) {
        const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
        e2 = min(100, max(-120, 14 - ex));
      }
      up = __uint_as_float((uint32_t)(e2 + 127) << 23);
      s_head *= __uint_as_float((uint32_t)(127 - e2) << 23);
    }
#pragma unroll
    for (int j = 0; j < KS; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float a = qf[4 * j + 2 * h] * up, b = qf[4 * j + 2 * h + 1] * up;
        if (FP8) {
          __half2 x = __floats2half2_rn(a, b);
          qb[j][h] = *reinterpret_cast<uint32_t*>(&x);
        } else {
          __nv_bfloat162 x = __floats2bfloat162_rn(a, b);
          qb[j][h] = *reinterpret_cast<uint32_t*>(&x);
        }
      }
    // the scales of the two heads this lane's score columns belong to
    const int lane = threadIdx.x & 31;
    sc[0] = __shfl_sync(full, s_head, (2 * (lane & 3)) * 4);
    sc[1] = __shfl_sync(full, s_head, (2 * (lane & 3) + 1) * 4);
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }

  // The K fragments of k-steps 2q, 2q + 1 of key row `row` (lane tig's dims
  // kdim8(q, tig) .. + 7): w[0], w[1] = k-step 2q's (a0|a1, a2|a3 half),
  // w[2], w[3] = k-step 2q + 1's.
  static __device__ __forceinline__ void k_words(const uint8_t* krow, int row, int q, int tig,
                                                 uint32_t (&w)[4]) {
    if constexpr (FP8) {
      // 8 codes: dims kLaneDims tig + 8 q .. + 7, in a 16-byte chunk with the
      // next 8 (swizzled rows at D = 128)
      const int byte = kdim8(q, tig);
      const int chunk = byte >> 4;
      const uint8_t* src =
          krow + ((kSw ? (chunk ^ (row & 7)) : chunk) << 4) + (byte & 15);
      const uint2 x = *reinterpret_cast<const uint2*>(src);
      MmaRows<D, FP8>::widen8(x.x, x.y, w);
    } else {
      const uint4 x =
          *reinterpret_cast<const uint4*>(krow + kdim8(q, tig) * G::kElt);
      w[0] = x.x; w[1] = x.y; w[2] = x.z; w[3] = x.w;
    }
  }

  static __device__ __forceinline__ void movtrans(uint32_t& x) {
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %0;" : "+r"(x));
  }

  template <int NC>
  __device__ __forceinline__ void chunks(const uint8_t* const (&Ks)[NC],
                                         const uint8_t* const (&Vs)[NC], int key0, int k_end,
                                         int grp, int tig) {
    const unsigned full = 0xffffffffu;
    // S^T of chunk c: two accumulator chains (even / odd k-step pairs)
    float s[NC][4];
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      float acc[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h) acc[h][0] = acc[h][1] = acc[h][2] = acc[h][3] = 0.f;
      const uint8_t* r0 = Ks[c] + grp * G::kRowBytes;
      const uint8_t* r1 = Ks[c] + (grp + 8) * G::kRowBytes;
#pragma unroll
      for (int q = 0; q < KS / 2; ++q) {
        uint32_t w0[4], w1[4];
        k_words(r0, grp, q, tig, w0);
        k_words(r1, grp + 8, q, tig, w1);
        MmaRows<D, FP8>::mma(acc[q & 1], w0[0], w1[0], w0[1], w1[1], qb[2 * q][0], qb[2 * q][1]);
        MmaRows<D, FP8>::mma(acc[q & 1], w0[2], w1[2], w0[3], w1[3], qb[2 * q + 1][0],
                             qb[2 * q + 1][1]);
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) s[c][i] = acc[0][i] + acc[1][i];
    }
    // scale, mask, online softmax of heads 2 tig (c0, c2) and 2 tig + 1 (c1, c3)
    const bool whole = key0 + 16 * NC <= k_end;  // no key of the step is masked
    float alpha[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float& x = s[c][2 * h + e];
          x = whole || key0 + 16 * c + grp + 8 * h < k_end ? x * sc[e] : -INFINITY;
          mx = fmaxf(mx, x);
        }
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(full, mx, 16));
      const float m_ref = MmaRows<D, FP8>::rebase(m[e], mx, alpha[e]);
      float ps = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float& x = s[c][2 * h + e];
          x = ex2_ftz(x - m_ref);
          ps += x;
        }
      l[e] = l[e] * alpha[e] + ps;
      m[e] = m_ref;
    }
    if (__any_sync(full, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= alpha[0];
        o[mt][1] *= alpha[1];
        o[mt][2] *= alpha[0];
        o[mt][3] *= alpha[1];
      }
    }
    auto pk = [](float x, float y) -> uint32_t {
      if (FP8) {
        __half2 h = __floats2half2_rn(x, y);
        return *reinterpret_cast<uint32_t*>(&h);
      }
      __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
      return *reinterpret_cast<uint32_t*>(&h);
    };
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      // P^T of chunk c as the B fragments: keys 2 tig, 2 tig + 1 (and + 8) of head grp
      uint32_t b0 = pk(s[c][0], s[c][1]), b1 = pk(s[c][2], s[c][3]);
      movtrans(b0);
      movtrans(b1);
      // V rows 2tig, 2tig+1, 2tig+8, 2tig+9 over dims DG grp .. DG grp + DG - 1
      uint32_t vw[4][DG / 2];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int kr = 2 * tig + (i & 1) + 8 * (i >> 1);
        if constexpr (kSw) {  // the 16-byte chunk grp of row kr, stored at grp ^ (kr & 7)
          const uint4 x = *reinterpret_cast<const uint4*>(Vs[c] + kr * G::kRowBytes +
                                                          ((grp ^ (kr & 7)) << 4));
          MmaRows<D, FP8>::widen8(x.x, x.y, &vw[i][0]);
          MmaRows<D, FP8>::widen8(x.z, x.w, &vw[i][4]);
        } else {
          const uint8_t* vrow = Vs[c] + kr * G::kRowBytes + DG * grp * G::kElt;
#pragma unroll
          for (int h = 0; h < DG / 8; ++h) {
            uint32_t w4[4];
            MmaRows<D, FP8>::load8(vrow + 8 * h * G::kElt, w4);
#pragma unroll
            for (int w = 0; w < 4; ++w) vw[i][4 * h + w] = w4[w];
          }
        }
        if (!whole && key0 + 16 * c + kr >= k_end)  // unwritten cells may hold NaN; P = 0 must not meet them
#pragma unroll
          for (int w = 0; w < DG / 2; ++w) vw[i][w] = 0u;
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t a0, a1, a2, a3;
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a0) : "r"(vw[0][mt]), "r"(vw[1][mt]));
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a1) : "r"(vw[0][mt]), "r"(vw[1][mt]));
        asm("prmt.b32 %0, %1, %2, 0x5410;" : "=r"(a2) : "r"(vw[2][mt]), "r"(vw[3][mt]));
        asm("prmt.b32 %0, %1, %2, 0x7632;" : "=r"(a3) : "r"(vw[2][mt]), "r"(vw[3][mt]));
        MmaRows<D, FP8>::mma(o[mt], a0, a1, a2, a3, b0, b1);
      }
    }
  }

  __device__ __forceinline__ void chunk(const uint8_t* Ks, const uint8_t* Vs, int key0, int k_end,
                                        int grp, int tig) {
    const uint8_t* const k[1] = {Ks};
    const uint8_t* const v[1] = {Vs};
    chunks<1>(k, v, key0, k_end, grp, tig);
  }

  // Per-head sums over the eight key lanes of a head (the maxima already agree).
  __device__ __forceinline__ void finish_sums() {
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 4);
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 8);
      l[e] += __shfl_xor_sync(0xffffffffu, l[e], 16);
    }
  }

  template <class F>
  __device__ __forceinline__ void for_each_run(int grp, int tig, F&& f) const {
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int i = 0; i < DG / 4; ++i)
        f(2 * tig + e, DG * grp + 4 * i,
          make_float4(o[2 * i][e], o[2 * i][2 + e], o[2 * i + 1][e], o[2 * i + 1][2 + e]), m[e],
          l[e]);
  }
  template <class F>
  __device__ __forceinline__ void for_each_stat(int grp, int tig, F&& f) const {
    if (grp == 0) {
      f(2 * tig, m[0], l[0]);
      f(2 * tig + 1, m[1], l[1]);
    }
  }

  // This warp's rows (heads < nrows) into the combine buffer of warp `warp`.
  __device__ __forceinline__ void to_comb(float* comb_o, float* comb_m, float* comb_l, int warp,
                                          int nrows, int grp, int tig) const {
    for_each_run(grp, tig, [&](int row, int d0, float4 v, float, float) {
      if (row < nrows) *reinterpret_cast<float4*>(comb_o + (warp * 16 + row) * D + d0) = v;
    });
    for_each_stat(grp, tig, [&](int row, float mm, float ll) {
      if (row < nrows) {
        comb_m[warp * 16 + row] = mm;
        comb_l[warp * 16 + row] = ll;
      }
    });
  }
};

// TMA maps of the E4M3 pools at D = 128 (the swizzled stages): a pool as
// [block][kv head * B + offset][128 codes]; one box = one 16-key chunk of one
// kv head, 128-byte swizzled. Left empty for the other kernels.
template <int D, bool FP8>
cudaError_t decode_maps(const DecodeParams& p, CUtensorMap* tk, CUtensorMap* tv) {
  *tk = CUtensorMap{};
  *tv = CUtensorMap{};
  if constexpr (FP8 && D == 128) {
    auto encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    if (p.num_blocks < 1) return cudaErrorInvalidValue;
    cuuint64_t dims[3] = {128, (cuuint64_t)p.Hkv * p.B, (cuuint64_t)p.num_blocks};
    cuuint64_t strides[2] = {128, (cuuint64_t)p.Hkv * p.B * 128};
    cuuint32_t box[3] = {128, (cuuint32_t)kChunk, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(p.k_pool), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
        encode(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(p.v_pool), dims,
               strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

}  // namespace
}  // namespace pa
