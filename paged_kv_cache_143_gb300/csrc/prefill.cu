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
// One CTA = two consecutive tiles (A, B) of 128 query rows x one kv head; both
// tiles share every K/V tile that is loaded. A tile's rows are the (token,
// head) pairs of the GQA group that shares the kv head, packed token major
// (row = token * g + head), so K/V are read once per group: 128 / g tokens
// per tile (integer division; when g does not divide 128 the last
// 128 mod g rows of every tile stay unused, masked to P = 0), g <= 128.
// The CTAs go out longest first across all requests: the host plans a list
// of (request, tile pair) units sorted by the key tiles each walks, since the
// block scheduler hands out CTAs in grid order as SMs free up.
//   warpgroup 0  warp 0: TMA producer — the Q tiles once (a 4-D tensor map over
//                [T][Hkv][g][D]), then per 128-key tile one 2-D box per physical
//                block and 64-column chunk (coordinates from the block table),
//                all boxes of a tile issued by one warp instruction, into a
//                ring of stages (K of a stage released after its S MMAs, V
//                after its PV MMAs);
//                warp 1: allocates 512 TMEM columns; one thread issues the MMAs
//                in the order PV_A(j-1), S_A(j), PV_B(j-1), S_B(j), so that one
//                tile's MMAs run while the other tile's softmax works:
//                S_t = Q_t K_j^T (M 128, N 128, K = D, both operands K-major,
//                f32 in TMEM) and O_t += P_t V_j (P_t read from TMEM where it
//                overwrote S_t, V MN-major from shared memory).
//   warpgroups 1, 2  softmax of tiles A and B, one TMEM lane (= one query row)
//                per thread: read S, mask, online max/sum in log2 units, write
//                P as bf16 pairs over S; O is rescaled in TMEM only when the
//                running max grows by more than 2^8 (the stale max is otherwise
//                kept, which is exact algebra); epilogue O / l.
// E4M3 pools: S runs on E4M3 tensor-core operands at D = 128 (kind::f8f6f4:
// the K codes as stored, the query as the sum of three E4M3 terms after a
// power-of-two scale, ~2^-12 relative), while V is widened to f16 in place by
// two converter warps and P.V stays on f16 operands (P keeps f16 range).
// At D = 64 both K and V are widened and every MMA is f16.
// Every wait is bounded; a timeout sets the error word and the CTA unwinds
// (waits for its copies and MMAs, frees TMEM) without writing output.
#include <cudaTypedefs.h>

#include <mutex>

#include <cuda_fp8.h>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_kernels.h"
#include "tc_ptx.cuh"

namespace pa {
namespace {

constexpr int kM = 128;        // query rows per tile
constexpr int kN = 128;        // keys per KV tile
constexpr int kThreads = 384;  // 3 warpgroups
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.f;
// Register split: the block is launched with kLaunchRegs per thread (the
// __launch_bounds__ cap for 384 threads); warpgroup 0 lowers to
// kRegsProducer and the two softmax warpgroups raise to kRegsSoftmax. The
// raised total must not exceed the launched total, or the raise never
// completes.
constexpr uint32_t kLaunchRegs = 168;
constexpr uint32_t kRegsProducer = 64;
constexpr uint32_t kRegsSoftmax = 216;
static_assert(128 * kRegsProducer + 256 * kRegsSoftmax <= kThreads * kLaunchRegs,
              "register split exceeds the registers the block is launched with");
static_assert(kRegsProducer % 8 == 0 && kRegsSoftmax % 8 == 0, "setmaxnreg takes multiples of 8");

template <int D, bool F8>
struct Smem {
  static constexpr int kStages = D == 128 ? 2 : 4;     // KV tiles in flight
  static constexpr int kChunkBytes = kN * 128;         // 128 rows x 64 bf16 (one swizzle column)
  static constexpr int kChunks = D / 64;
  static constexpr int kQBytes = kM * D * 2;           // one Q tile (bf16, as loaded)
  static constexpr int kKVBytes = kN * D * 2;          // one K or V tile (16-bit)
  // E4M3 pools at D = 128: S runs on E4M3 operands. K tiles stay E4M3 codes
  // (128-byte rows, 128-byte swizzle, 16 KB); each Q tile becomes three E4M3
  // tiles (q ~ hi + mid + lo) written over and after its bf16 copy (48 KB).
  static constexpr bool kF8S = F8 && D == 128;
  static constexpr int kQPart = kM * 128;              // one E4M3 Q tile
  static constexpr int kQRegion = kF8S ? 3 * kQPart : kQBytes;
  static constexpr int kKBytes = kF8S ? kN * D : kKVBytes;
  static constexpr int kOffQ = 0;                      // Q_A, then Q_B
  static constexpr int kOffK = 2 * kQRegion;
  static constexpr int kOffV = kOffK + kStages * kKBytes;
  // E4M3 V (and K for D = 64): the tile of codes (rows of D bytes) of stage st
  // lands in the upper half of its own f16 stage for D = 128 and is widened in
  // place (row r of codes occupies exactly the bytes of row r of the upper
  // 64-column chunk, so a row's codes are read before its second half is
  // written); for D = 64 each stage has a staging tile of its own.
  static constexpr bool kInPlace = F8 && D == 128;
  static constexpr int kK8Bytes = F8 && !kInPlace ? kN * D : 0;  // per stage
  static constexpr int kOffK8 = kOffV + kStages * kKVBytes;
  static constexpr int kOffV8 = kOffK8 + kStages * kK8Bytes;
  static constexpr int kOffBar = kOffV8 + kStages * kK8Bytes;
  static constexpr int kBarBytes = 512;               // the mbarriers (struct Bars)
  static constexpr int kBytes = kOffBar + kBarBytes;
  static constexpr int kAlloc = kBytes + 1024;  // the base is rounded up to 1024 B
  static_assert(kAlloc <= 232448, "dynamic shared memory above the 227 KB per-block limit");
  static_assert(kOffK % 1024 == 0 && kOffV % 1024 == 0 && kKBytes % 1024 == 0,
                "128-byte-swizzled tiles start on 1024-byte boundaries");
  // where the E4M3 codes of stage st land (K only for D = 64)
  __host__ __device__ static constexpr int k8(int st) { return kOffK8 + st * kK8Bytes; }
  __host__ __device__ static constexpr int v8(int st) {
    return kInPlace ? kOffV + st * kKVBytes + kKVBytes / 2 : kOffV8 + st * kK8Bytes;
  }
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[4];
  uint64_t v_full[4];
  uint64_t k_empty[4];  // K of a stage is free once its S MMAs are done
  uint64_t v_empty[4];  // V of a stage is free once its PV MMAs are done
  uint64_t s_full[2];   // per Q tile
  uint64_t p_full[2];
  uint64_t pv_done[2];
  uint64_t final_mma;
  uint64_t k8_full[4], v8_full[4];  // E4M3 codes of a stage landed (k/v_full: widened)
  uint64_t q_conv;                  // Q tiles converted to f16 (E4M3 pools)
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

// Widens 16 E4M3 codes to f16 (exact: every E4M3 value is an f16 value).
__device__ __forceinline__ void e4m3x16_to_f16(const uint4& in, uint32_t (&out)[8]) {
  const uint32_t w[4] = {in.x, in.y, in.z, in.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(out[2 * i]), "=r"(out[2 * i + 1])
        : "r"(w[i]));
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmap_q,
                   const __grid_constant__ CUtensorMap tmap_k,
                   const __grid_constant__ CUtensorMap tmap_v, PrefillParams p) {
  using S = Smem<D, F8>;
  constexpr int kStages = S::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + S::kOffBar);
  static_assert(sizeof(Bars) <= S::kBarBytes, "the mbarriers overrun their shared-memory slot");

  // a tile pair of a prefill chunk of request r: from the unit list (grid
  // (Hkv, units), longest units first; unit = request << 16 | last << 15 |
  // pair, last marking the request's highest listed pair), else from the
  // grid (pairs, Hkv, requests), requests heaviest first and each request's
  // latest pairs first
  const bool listed = p.n_units > 0;
  const int unit = listed ? p.units[blockIdx.y] : 0;
  const int r = listed ? unit >> 16 : p.n_order ? p.order[blockIdx.z] : (int)blockIdx.z;
  const int q_begin = p.qsl[r];
  const int q_len = p.qsl[r + 1] - q_begin;
  // (one CTA per request reports a bad entry: the first kv head of a unit
  // on the list, else the request's first grid cell)
  const bool reporter = threadIdx.x == 0 && blockIdx.x == 0 && (listed || blockIdx.y == 0);
  if (q_len <= 1) {
    // decode requests and empty requests are not ours; a listed unit of one
    // means the device qsl disagrees with the host mirror the list came from
    if (listed && reporter) raise_error(p.err, kErrBounds);
    return;
  }
  const int seq = p.seq_lens[r];
  if (seq < q_len || seq > p.max_blocks * p.B || q_begin < 0 || q_begin + q_len > p.T) {
    if (reporter) raise_error(p.err, kErrBounds);
    return;
  }
  const int32_t* table = p.block_tables + (int64_t)r * p.max_blocks;
  const int g = p.g;
  const int tpt = kM / g;  // tokens per tile
  const int ntq = (q_len + tpt - 1) / tpt;
  const int npairs = (ntq + 1) / 2;
  int pair, kvh;
  if (listed) {
    pair = unit & 0x7FFF;
    kvh = blockIdx.x;
    // the device qsl disagrees with the host mirror the list was planned
    // from: a unit past the request's tiles, or tiles past the request's last
    // listed pair (those would be left unwritten)
    const bool last_listed = (unit & 0x8000) != 0;
    if (pair >= npairs || (last_listed && pair != npairs - 1)) {
      if (reporter) raise_error(p.err, kErrBounds);
      if (pair >= npairs) return;
    }
  } else {
    const int pair_x = blockIdx.x;
    if (npairs > (int)gridDim.x) {
      // more query tiles than the grid was planned for: device qsl disagrees
      // with the host mirror; the tiles past the grid would be left unwritten
      if (threadIdx.x == 0 && pair_x == 0 && blockIdx.y == 0) raise_error(p.err, kErrBounds);
    }
    if (pair_x >= npairs) return;
    pair = npairs - 1 - pair_x;  // heaviest (latest) pairs start first
    kvh = blockIdx.y;
  }
  const int P = seq - q_len;
  int q0[2], ntk[2], n_kv[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int tile = 2 * pair + t;
    q0[t] = tile * tpt;
    if (tile < ntq) {
      const int last = min(q_len, q0[t] + tpt) - 1;
      n_kv[t] = p.causal ? min(seq, P + last + 1) : seq;
      ntk[t] = (n_kv[t] + kN - 1) / kN;
    } else {
      n_kv[t] = 0;
      ntk[t] = 0;
    }
  }
  const int ntk_all = max(ntk[0], ntk[1]);
  const int n_kv_all = max(n_kv[0], n_kv[1]);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      // bf16: completed by the TMA bytes; E4M3: by the two converter warps
      mbar_init(&bars->k_full[s], F8 && !S::kF8S ? 2 : 1);
      mbar_init(&bars->v_full[s], F8 ? 2 : 1);
      mbar_init(&bars->k_empty[s], 1);
      mbar_init(&bars->v_empty[s], 1);
      mbar_init(&bars->k8_full[s], 1);
      mbar_init(&bars->v8_full[s], 1);
    }
    mbar_init(&bars->q_conv, 8);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 4);  // one arrival per softmax warp
      mbar_init(&bars->pv_done[t], 1);
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
  const uint32_t tmem = bars->tmem_base;  // S_t / P_t at column 128 t, O_t at 256 + 128 t

  // Warpgroup 0 (producer, MMA, two idle warps) gives registers to the two
  // softmax warpgroups (see kRegsProducer / kRegsSoftmax). The role branches never merge
  // (each ends with its own block-wide barrier), so each keeps its limit.
  if (warp < 4) {
    tc::regs_dec<kRegsProducer>();
    if (warp == 0) {
    // ----------------------------------------------------------- TMA producer
    const unsigned full = 0xffffffffu;
    if (lane == 0) {
      tc::prefetch_tensormap(&tmap_q);
      tc::prefetch_tensormap(&tmap_k);
      tc::prefetch_tensormap(&tmap_v);
      const int nq = ntk[1] > 0 ? 2 : 1;
      // each box holds the tile's (128 / g) * g rows of 64 dims
      mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(nq * tpt * g * D * 2));
      for (int t = 0; t < nq; ++t)
        for (int c = 0; c < S::kChunks; ++c)
          tc::tma_load_4d(smem + S::kOffQ + t * S::kQRegion + c * S::kChunkBytes, &tmap_q,
                          c * 64, 0, kvh, q_begin + q0[t], &bars->q_full);
    }
    const int nbt = kN / p.B;  // blocks per KV tile (<= 8)
    auto fetch = [&](int j) -> int {
      const int lb = j * nbt + lane;
      return (j < ntk_all && lane < nbt && lb * p.B < n_kv_all) ? __ldg(table + lb) : 0;
    };
    // lane -> one box of a K or V tile: block i, 64-column chunk c
    const int box_block = lane / S::kChunks;
    const int box_chunk = lane % S::kChunks;
    int ids = fetch(0);
    int issued_k = 0, issued_v = 0;
    for (int j = 0; j < ntk_all; ++j) {
      const int next = fetch(j + 1);
      const int st = j % kStages;
      int nload = 0;
      while (nload < nbt && (j * nbt + nload) * p.B < n_kv_all) ++nload;
      const bool bad = lane < nload && (ids < 0 || ids >= p.num_blocks);
      if (__any_sync(full, bad) && lane == 0) raise_error(p.err, kErrBounds);
      const int blk_lane = bad ? 0 : ids;  // a valid block; the output is then unspecified
      const int blk = __shfl_sync(full, blk_lane, box_block & 7);
      const uint32_t bytes = (uint32_t)(nload * p.B * D * (F8 ? 1 : 2));
      const bool issues = F8 ? lane < nload : box_block < nload;
      const int row = ((F8 ? blk_lane : blk) * p.Hkv + kvh) * p.B;
      // bf16: boxes of 64 columns into the swizzled stage; E4M3: one box of
      // D codes x B keys per block into the stage's tile of codes
      // K: bf16 — 64-column boxes into the swizzled stage; E4M3, D = 128 —
      // one box of 128 codes x B keys per block straight into the swizzled
      // stage (the MMA reads the codes); E4M3, D = 64 — into the code tile
      const int k_dst = S::kF8S ? S::kOffK + st * S::kKBytes + lane * p.B * 128
                        : F8    ? S::k8(st) + lane * p.B * D
                                : S::kOffK + st * S::kKBytes + box_chunk * S::kChunkBytes +
                                      box_block * p.B * 128;
      const int v_dst = F8 ? S::v8(st) + lane * p.B * D
                           : S::kOffV + st * S::kKVBytes + box_chunk * S::kChunkBytes +
                                 box_block * p.B * 128;
      uint64_t* kbar = F8 && !S::kF8S ? &bars->k8_full[st] : &bars->k_full[st];
      uint64_t* vbar = F8 ? &bars->v8_full[st] : &bars->v_full[st];
      // K of tile j: the stage is free once the S MMAs of tile j - kStages are
      // done (for E4M3 this implies its codes were widened, and read, before)
      bool ok = true;
      if (lane == 0 && j >= kStages)
        ok = mbar_wait(&bars->k_empty[st], ((j / kStages) - 1) & 1, p.err);
      if (!__shfl_sync(full, ok ? 1 : 0, 0) || aborted(bars)) {
        if (lane == 0) bars->abort = 1;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(kbar, bytes);
      __syncwarp();
      if (issues)
        tc::tma_load_2d(smem + k_dst, &tmap_k, F8 ? 0 : box_chunk * 64, row, kbar);
      issued_k = j + 1;
      // V of tile j: free once the PV MMAs of tile j - kStages are done
      if (lane == 0 && j >= kStages)
        ok = mbar_wait(&bars->v_empty[st], ((j / kStages) - 1) & 1, p.err);
      if (!__shfl_sync(full, ok ? 1 : 0, 0)) {
        if (lane == 0) bars->abort = 1;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(vbar, bytes);
      __syncwarp();
      if (issues)
        tc::tma_load_2d(smem + v_dst, &tmap_v, F8 ? 0 : box_chunk * 64, row, vbar);
      issued_v = j + 1;
      ids = next;
    }
    // every issued copy lands before the CTA may leave
    if (lane == 0) {
      mbar_wait(&bars->q_full, 0, p.err);
      for (int j = issued_k - kStages > 0 ? issued_k - kStages : 0; j < issued_k; ++j)
        mbar_wait(F8 && !S::kF8S ? &bars->k8_full[j % kStages] : &bars->k_full[j % kStages],
                  (j / kStages) & 1, p.err);
      for (int j = issued_v - kStages > 0 ? issued_v - kStages : 0; j < issued_v; ++j)
        mbar_wait(F8 ? &bars->v8_full[j % kStages] : &bars->v_full[j % kStages],
                  (j / kStages) & 1, p.err);
    }
    } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = tc::idesc_16bit_f32(kM, kN, false, false, F8);
      constexpr uint32_t idesc_o = tc::idesc_16bit_f32(kM, D, false, true, F8);
      bool ok = mbar_wait(F8 ? &bars->q_conv : &bars->q_full, 0, p.err);
      auto issue_s = [&](int t, int j) {
        const uint8_t* qs = smem + S::kOffQ + t * S::kQRegion;
        const uint8_t* ks = smem + S::kOffK + (j % kStages) * S::kKBytes;
        if constexpr (S::kF8S) {
          // S = (q_hi + q_mid + q_lo) . k on E4M3 operands: per Q part, four
          // K = 32 steps along a 128-byte row (32 bytes each)
          constexpr uint32_t idesc_s8 = tc::idesc_e4m3_f32(kM, kN);
#pragma unroll 1
          for (int part = 0; part < 3; ++part)
#pragma unroll
            for (int k = 0; k < D / 32; ++k) {
              const uint64_t a = tc::smem_desc_sw128(qs + part * S::kQPart + k * 32, 16, 1024);
              const uint64_t b = tc::smem_desc_sw128(ks + k * 32, 16, 1024);
              tc::mma_e4m3_ss(tmem + t * kN, a, b, idesc_s8, part > 0 || k > 0);
            }
        } else {
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint64_t a =
                tc::smem_desc_sw128(qs + (k >> 2) * S::kChunkBytes + (k & 3) * 32, 16, 1024);
            const uint64_t b =
                tc::smem_desc_sw128(ks + (k >> 2) * S::kChunkBytes + (k & 3) * 32, 16, 1024);
            tc::mma_bf16_ss(tmem + t * kN, a, b, idesc_s, k > 0);
          }
        }
        tc::mma_commit(&bars->s_full[t]);
      };
      auto issue_pv = [&](int t, int j) -> bool {
        if (!mbar_wait(&bars->p_full[t], j & 1, p.err)) return false;
        if (!mbar_wait(&bars->v_full[j % kStages], (j / kStages) & 1, p.err)) return false;
        if (aborted(bars)) return false;
        tc::fence_after_sync();
        const uint8_t* vs = smem + S::kOffV + (j % kStages) * S::kKVBytes;
#pragma unroll
        for (int k = 0; k < kN / 16; ++k) {
          const uint64_t b = tc::smem_desc_sw128(vs + k * 16 * 128, S::kChunkBytes, 1024);
          tc::mma_bf16_ts(tmem + 2 * kN + t * kN, tmem + t * kN + k * 8, b, idesc_o,
                          j > 0 || k > 0);
        }
        tc::mma_commit(&bars->pv_done[t]);
        return true;
      };
      for (int j = 0; ok && j < ntk_all; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(&bars->k_full[st], (j / kStages) & 1, p.err) || aborted(bars)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          // PV_t(j-1) reads P_t out of the S_t columns before S_t(j) overwrites them
          if (j >= 1 && j - 1 < ntk[t] && !issue_pv(t, j - 1)) ok = false;
          if (ok && j < ntk[t]) issue_s(t, j);
        }
        tc::mma_commit(&bars->k_empty[st]);
        if (j >= 1) tc::mma_commit(&bars->v_empty[(j - 1) % kStages]);
      }
      if (ok) {
        const int j = ntk_all - 1;
        for (int t = 0; t < 2 && ok; ++t)
          if (j < ntk[t] && !issue_pv(t, j)) ok = false;
        tc::mma_commit(&bars->v_empty[j % kStages]);
      }
      if (!ok) bars->abort = 1;
      tc::mma_commit(&bars->final_mma);
      mbar_wait(&bars->final_mma, 0, p.err);
    }
    } else if (F8) {
    // ------------------------------------------ E4M3 -> f16 converters (warps 2, 3)
    // Each 16-byte granule of codes (16 dims of one key) becomes two 16-byte
    // f16 granules at their 128-byte-swizzled places in the K/V tile; keys at
    // or past n_kv_all are written as zeros (so P = 0 never meets a NaN).
    // A warp covers whole key rows in each step (8 granules per row for
    // D = 128) and reads them all before it writes any, which makes the
    // in-place widening safe: only row r's own codes share bytes with row r's
    // upper half.
    const int tid = threadIdx.x - 64;  // 0..63
    constexpr int kGran = D / 16;       // granules of codes per key
    static_assert(32 % kGran == 0, "a warp step must cover whole key rows");
    auto convert = [&](const uint8_t* src, uint8_t* dst, int key0) {
#pragma unroll 4
      for (int G = tid; G < kN * kGran; G += 64) {
        const int row = G / kGran, gq = G % kGran;
        uint32_t h[8];
        const bool live = key0 + row < n_kv_all;
        uint4 in = make_uint4(0, 0, 0, 0);
        if (live) in = *reinterpret_cast<const uint4*>(src + row * D + gq * 16);
        __syncwarp();
        if (live) {
          e4m3x16_to_f16(in, h);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) h[i] = 0u;
        }
        const int c = gq >> 2, q = 2 * (gq & 3);
        uint8_t* line = dst + c * S::kChunkBytes + row * 128;
        *reinterpret_cast<uint4*>(line + ((q ^ (row & 7)) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(line + (((q + 1) ^ (row & 7)) << 4)) =
            make_uint4(h[4], h[5], h[6], h[7]);
      }
    };
    bool ok = true;
    for (int j = 0; j < ntk_all && ok; ++j) {
      const int st = j % kStages;
      // D = 128: only V is widened (S reads the K codes); D = 64: K and V
      for (int kv = S::kF8S ? 1 : 0; kv < 2 && ok; ++kv) {
        // the codes landed; the producer issued them only once the stage was
        // free (its MMAs of tile j - kStages done)
        uint64_t* landed = kv ? &bars->v8_full[st] : &bars->k8_full[st];
        ok = __all_sync(0xffffffffu, mbar_wait(landed, (j / kStages) & 1, p.err)) &&
             !aborted(bars);
        if (!ok) break;
        convert(smem + (kv ? S::v8(st) : S::k8(st)),
                smem + (kv ? S::kOffV : S::kOffK) + st * S::kKVBytes, j * kN);
        tc::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kv ? &bars->v_full[st] : &bars->k_full[st]);
      }
    }
    if (!ok) bars->abort = 1;
    }
    // teardown: after every thread of the block is done with TMEM
    tc::fence_before_sync();
    named_bar_sync(0, kThreads);
    if (warp == 1) {
      tc::fence_after_sync();
      tc::tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    tc::regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int t = warp >= 8 ? 1 : 0;  // Q tile of this warpgroup
    const int my_ntk = t ? ntk[1] : ntk[0];
    const int my_q0 = t ? q0[1] : q0[0];
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tmem_s = tmem + t * kN + lane_off;
    const uint32_t tmem_o = tmem + 2 * kN + t * kN + lane_off;
    const int tok = my_q0 + row / g;
    const int head = row % g;
    const bool valid_row = my_ntk > 0 && row < tpt * g && tok < q_len;
    const int limit = !valid_row ? 0 : (p.causal ? min(P + tok + 1, seq) : seq);
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    float score_scale = p.scale_log2;  // log2(e) * scale (* k_scale for E4M3)
    if (F8) {
      // E4M3 pools. D = 64: the MMAs run on f16 operands; this thread
      // converts its own Q row in place, pre-scaled by 2^e so that the row's
      // largest magnitude lands in [2^14, 2^15) (exact: a power of two), and
      // divides the scores by 2^e. D = 128: see the E4M3 split below.
      if (my_ntk > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->q_full, 0, p.err));
        if constexpr (S::kF8S) {
          if (ok) {
            // S runs on E4M3 operands: this thread's row becomes three E4M3
            // rows, q * 2^e ~ hi + mid + lo (each the E4M3 rounding of what the
            // earlier terms leave), after an exact power-of-two scale that puts
            // the row's largest magnitude in [2^7, 2^8); the scores are divided
            // by 2^e. The thread reads its whole bf16 row first: hi and mid
            // take the bytes of that row in the two bf16 chunks, lo the tile's
            // third 16 KB.
            uint8_t* tq = smem + S::kOffQ + t * S::kQRegion;
            const int sw = row & 7;
            uint4 bq[2][8];
            float amax = 0.f;
  #pragma unroll
            for (int c = 0; c < 2; ++c)
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                bq[c][q] = *reinterpret_cast<const uint4*>(tq + c * S::kChunkBytes + row * 128 +
                                                           ((q ^ sw) << 4));
                float f[8];
                bf16x8_to_f32(bq[c][q], f);
  #pragma unroll
                for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
              }
            int e2 = 0;
            if (amax > 0.f) {
              const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
              e2 = min(100, max(-120, 7 - ex));
            }
            const float up = __uint_as_float((uint32_t)(e2 + 127) << 23);
            score_scale *= __uint_as_float((uint32_t)(127 - e2) << 23);
            auto e4m3x2 = [](float a, float b) -> uint32_t {  // a in the low byte
              return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                        __NV_E4M3);
            };
            auto back = [](uint32_t codes, float& a, float& b) {  // exact
              uint32_t h;
              asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\t"
                  "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
                  : "=r"(h)
                  : "r"(codes));
              const __half2 x = *reinterpret_cast<const __half2*>(&h);
              a = __low2float(x);
              b = __high2float(x);
            };
  #pragma unroll
            for (int g = 0; g < 8; ++g) {  // 16 dims: 16g .. 16g + 15
              float f[16];
              bf16x8_to_f32(bq[g >> 2][2 * (g & 3)], *reinterpret_cast<float(*)[8]>(f));
              bf16x8_to_f32(bq[g >> 2][2 * (g & 3) + 1], *reinterpret_cast<float(*)[8]>(f + 8));
              uint32_t part[3][4];
  #pragma unroll
              for (int w = 0; w < 4; ++w) {
                uint32_t words[3] = {0u, 0u, 0u};
  #pragma unroll
                for (int hb = 0; hb < 2; ++hb) {  // two pairs of dims per 32-bit word
                  float x0 = f[4 * w + 2 * hb] * up, x1 = f[4 * w + 2 * hb + 1] * up;
  #pragma unroll
                  for (int pi = 0; pi < 3; ++pi) {
                    const uint32_t c2 = e4m3x2(x0, x1);
                    words[pi] |= c2 << (16 * hb);
                    float y0, y1;
                    back(c2, y0, y1);
                    x0 -= y0;
                    x1 -= y1;
                  }
                }
  #pragma unroll
                for (int pi = 0; pi < 3; ++pi) part[pi][w] = words[pi];
              }
  #pragma unroll
              for (int pi = 0; pi < 3; ++pi)
                *reinterpret_cast<uint4*>(tq + pi * S::kQPart + row * 128 + ((g ^ sw) << 4)) =
                    make_uint4(part[pi][0], part[pi][1], part[pi][2], part[pi][3]);
            }
            tc::fence_proxy_async_smem();
          }
        } else if (ok) {
          uint8_t* qrow = smem + S::kOffQ + t * S::kQRegion + row * 128;
          float amax = 0.f;
#pragma unroll
          for (int c = 0; c < S::kChunks; ++c)
#pragma unroll
            for (int gq = 0; gq < 8; ++gq) {
              const uint4 v = *reinterpret_cast<const uint4*>(qrow + c * S::kChunkBytes + gq * 16);
              float f[8];
              bf16x8_to_f32(v, f);
#pragma unroll
              for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(f[e]));
            }
          int e2 = 0;
          if (amax > 0.f) {
            const int ex = (int)((__float_as_uint(amax) >> 23) & 0xFF) - 127;
            e2 = min(100, max(-120, 14 - ex));
          }
          const float up = __uint_as_float((uint32_t)(e2 + 127) << 23);
          const float down = __uint_as_float((uint32_t)(127 - e2) << 23);
          score_scale *= down;
#pragma unroll
          for (int c = 0; c < S::kChunks; ++c)
#pragma unroll
            for (int gq = 0; gq < 8; ++gq) {
              uint4* ptr = reinterpret_cast<uint4*>(qrow + c * S::kChunkBytes + gq * 16);
              float f[8];
              bf16x8_to_f32(*ptr, f);
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                __half2 x = __floats2half2_rn(f[2 * e] * up, f[2 * e + 1] * up);
                h[e] = *reinterpret_cast<uint32_t*>(&x);
              }
              *ptr = make_uint4(h[0], h[1], h[2], h[3]);
            }
          tc::fence_proxy_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->q_conv);
    }
    for (int j = 0; ok && j < my_ntk; ++j) {
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->s_full[t], j & 1, p.err))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sr[kN];
#pragma unroll
      for (int c = 0; c < kN / 32; ++c)
        tc::tmem_ld32(tmem_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
      tc::tmem_wait_ld();
      float* s = reinterpret_cast<float*>(sr);
      const int key0 = j * kN;
      if (key0 + kN > limit) {
#pragma unroll
        for (int k = 0; k < kN; ++k)
          if (key0 + k >= limit) s[k] = -INFINITY;
      }
      // raw scores; the log2-domain max is max * scale_log2 (scale > 0);
      // eight independent partial maxima (chain u: columns u + 8 i) keep the
      // reduction off one dependency chain, three-input maxima halve the
      // instruction count
      float mx[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        mx[u] = fmax3(s[u], s[u + 8], s[u + 16]);
#pragma unroll
        for (int i = 3; i + 1 < kN / 8; i += 2) mx[u] = fmax3(mx[u], s[u + 8 * i], s[u + 8 * i + 8]);
        if constexpr ((kN / 8 - 3) % 2 == 1) mx[u] = fmaxf(mx[u], s[u + kN - 8]);
      }
      float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      mt *= score_scale;
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
      // p = 2^(s * scale - m) on column pairs: one packed fp32x2 multiply-add
      // per pair, the exponentials one by one, four packed partial sums
      const uint64_t sc2 = f2_pack(score_scale, score_scale);
      const uint64_t nm2 = f2_pack(-m_sub, -m_sub);
      uint64_t sum2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int k = 0; k < kN; k += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          float a, b;
          f2_unpack(f2_fma(f2_pack(s[k + 2 * u], s[k + 2 * u + 1]), sc2, nm2), a, b);
          s[k + 2 * u] = fast_exp2(a);
          s[k + 2 * u + 1] = fast_exp2(b);
          sum2[u] = f2_add(sum2[u], f2_pack(s[k + 2 * u], s[k + 2 * u + 1]));
        }
      float sum[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) f2_unpack(sum2[u], sum[2 * u], sum[2 * u + 1]);
      l_run = l_run * alpha + (((sum[0] + sum[1]) + (sum[2] + sum[3])) +
                               ((sum[4] + sum[5]) + (sum[6] + sum[7])));
      m_run = m_use;

      // rescale O_t (rare): PV_t(j-1) precedes S_t(j) in the MMA stream, so it
      // has completed; the wait only orders the TMEM accesses
      if (__any_sync(0xffffffffu, rescale)) {
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[t], (j - 1) & 1, p.err))) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const float a = rescale ? alpha : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tc::tmem_ld32(tmem_o + c * 32, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * a);
          tc::tmem_st32(tmem_o + c * 32, o);
        }
      }
      // P as 16-bit pairs (bf16, or f16 for E4M3 pools) over the first 64
      // columns of S_t (the A operand of PV)
#pragma unroll
      for (int c = 0; c < kN / 64; ++c) {
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          if (F8) {
            __half2 h = __floats2half2_rn(s[c * 64 + 2 * k], s[c * 64 + 2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
          } else {
            __nv_bfloat162 h = __floats2bfloat162_rn(s[c * 64 + 2 * k], s[c * 64 + 2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t*>(&h);
          }
        }
        tc::tmem_st32(tmem_s + c * 32, w);
      }
      tc::tmem_wait_st();
      // the CTA's last tile may hold keys past n_kv_all (unloaded blocks,
      // unwritten cells): zero those V rows so that P = 0 never meets a NaN
      if (!F8 && j == ntk_all - 1 && key0 + kN > n_kv_all) {
        const int st = j % kStages;
        if (!__all_sync(0xffffffffu, mbar_wait(&bars->v_full[st], (j / kStages) & 1, p.err))) {
          ok = false;
          break;
        }
        if (key0 + row >= n_kv_all) {
          uint8_t* vs = smem + S::kOffV + st * S::kKVBytes;
#pragma unroll
          for (int c = 0; c < S::kChunks; ++c)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<uint4*>(vs + c * S::kChunkBytes + row * 128 + q * 16) =
                  make_uint4(0, 0, 0, 0);
        }
        tc::fence_proxy_async_smem();
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->p_full[t]);
    }

    // epilogue: O_t / l once its last PV has landed
    if (ok && my_ntk > 0 &&
        !__all_sync(0xffffffffu, mbar_wait(&bars->pv_done[t], (my_ntk - 1) & 1, p.err)))
      ok = false;
    if (!ok) bars->abort = 1;
    if (ok && my_ntk > 0 && !aborted(bars)) {
      tc::fence_after_sync();
      const float inv_l = l_run > 0.f ? p.v_scale / l_run : 0.f;
      __nv_bfloat16* orow = p.out + ((int64_t)(q_begin + tok) * p.Hq + kvh * g + head) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tc::tmem_ld32(tmem_o + c * 32, o);
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
    tc::fence_before_sync();
    named_bar_sync(0, kThreads);
  }
}

// ----------------------------------------------------------- host launch

template <int D, bool F8>
cudaError_t launch_prefill_t(const PrefillLaunch& L, cudaStream_t s) {
  auto encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const PrefillParams& p = L.p;
  if (p.g < 1 || p.g > kM) return cudaErrorInvalidValue;  // a tile holds whole GQA groups
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
  // K and V as rows [(block * Hkv + head) * B + offset][D]. bf16: box = 64
  // dims x B rows, 128-byte swizzled (the MMA operand layout); E4M3: box =
  // D codes x B rows, unswizzled where the converter warps read it (V; K for
  // D = 64) and 128-byte swizzled where the MMA reads the codes (K, D = 128).
  {
    cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)p.num_blocks * p.Hkv * p.B};
    cuuint64_t strides[1] = {(cuuint64_t)D * (F8 ? 1 : 2)};
    cuuint32_t box[2] = {(cuuint32_t)(F8 ? D : 64), (cuuint32_t)p.B};
    cuuint32_t es[2] = {1, 1};
    const CUtensorMapDataType dt =
        F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const CUtensorMapSwizzle sw = F8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
    const CUtensorMapSwizzle sw_k = Smem<D, F8>::kF8S ? CU_TENSOR_MAP_SWIZZLE_128B : sw;
    if (encode(&tk, dt, 2, const_cast<void*>(L.k_pool), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw_k, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
    if (encode(&tv, dt, 2, const_cast<void*>(L.v_pool), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  constexpr int smem = Smem<D, F8>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<D, F8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // the register split inside the kernel assumes the block is launched with
  // kLaunchRegs per thread; refuse to launch a build that allocated fewer
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, prefill_kernel<D, F8>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs < (int)kLaunchRegs) return cudaErrorInvalidConfiguration;
  // kv heads x listed units, else tile pairs x kv heads x prefill requests
  const dim3 grid = p.n_units > 0 ? dim3(p.Hkv, p.n_units, 1)
                                  : dim3((L.max_q_tiles + 1) / 2, p.Hkv, p.n_order ? p.n_order : L.R);
  prefill_kernel<D, F8><<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s) {
  if (L.D == 128) return L.fp8 ? launch_prefill_t<128, true>(L, s) : launch_prefill_t<128, false>(L, s);
  return L.fp8 ? launch_prefill_t<64, true>(L, s) : launch_prefill_t<64, false>(L, s);
}

}  // namespace pa
