// cascade.cu — decode batches with shared prefixes (pa_forward_shared_prefix)
// in one launch: the prefix of each group read once for all its members, the
// private tails per request; the parts are merged by log-sum-exp afterwards
// (merge_kernel).
//
// [vLLM-wiki "블록 공유와 쓰기 시 복사"]: the members of a group (parallel samples
// of one prompt) reference the same physical blocks for the prompt. By the
// blockwise equation of [vLLM-wiki "블록 단위 어텐션 계산"] the softmax over a
// member's keys (prefix ∪ tail) splits exactly into per-part maxima, sums and
// unnormalised outputs merged by log-sum-exp, so the prefix part of every
// member's decode token can be computed against one read of the prefix.
//
// Both kinds of CTA are four warps; each warp owns up to 16 query rows and
// runs the warp-level tensor-core decode (decode_rows.cuh: mma.sync
// m16n8k16, S and P.V per 16-key chunk, two chunks per online-softmax
// update, everything in registers; tails of GQA groups of at most 8 heads
// with the keys as the MMA rows). Nothing is combined across
// warps: a warp writes its rows' partial (or final) output itself.
//  - prefix CTA (group k, piece, kv head, row block): rows = (member, head)
//    pairs of the group, 64 per CTA (16 per warp), against one piece of the
//    prefix read through the first member's table row. The four warps share
//    one ring of K/V stages: every warp consumes every chunk; the last warp
//    to finish a stage (a shared-memory counter) refills it with the chunk
//    one ring ahead, so the prefix bytes leave HBM once per row block.
//  - tail CTA (request r, task block x): warp w takes task 4x + w of r, a
//    (key split, kv head, 16-head part) of r's keys after its group's prefix
//    (all keys for an ungrouped decode), with a private quarter of the ring
//    that it fills itself, one quarter ahead. Short tails cost one warp, not a
//    CTA with a cross-warp combine.
// Many short CTAs (three per SM) rather than a persistent grid: a warp's
// start-up (block ids, query rows, first copies: a few microseconds of
// latency) then overlaps the other resident CTAs' work instead of stalling a
// stream of units (a persistent per-warp version of this kernel measured
// twice as slow on the prefix-shared sampling workload).
// Stages: per 16-key chunk, K then V, each one contiguous run of the pool
// moved by one bulk copy (E4M3 at D = 128: TMA tensor boxes with the
// 128-byte swizzle, the layout MmaRows reads without bank conflicts). Every
// wait is bounded; a wait that gives up sets the error word, and the CTA
// waits for its copies in flight before it exits.
#include "decode_rows.cuh"

namespace pa {
namespace {

constexpr int kCWarps = 4;  // warps per CTA, every one a consumer
constexpr int kCThreads = kCWarps * 32;
constexpr int kRowsPerCta = kCWarps * 16;

struct CascadeSmem {
  uint64_t full[kMaxStages];  // a stage's K and V landed (transaction bytes)
  int done[kMaxStages];       // prefix CTAs: warps that finished the stage (monotone)
  int issued;                 // prefix CTAs: chunks issued so far
  int abort;
};

template <int D, bool FP8>
struct CascadeGeo {
  using G = Geo<D, FP8>;
  static constexpr bool kSw = MmaRows<D, FP8>::kSw;
  static constexpr int kStages = G::kStages;
  static constexpr int kTailStages = kStages / kCWarps;  // per warp in a tail CTA
  static_assert(kTailStages >= 2, "a tail warp needs two stages");
  static constexpr int kSmem =
      (kSw ? 1024 : 0) + kStages * G::kStageBytes + (int)sizeof(CascadeSmem);
};

// One warp's source of block ids: lane i holds the id of chunk base + i of
// the key run starting at k_begin of `table` (ids outside the pool raise
// kErrBounds and read block 0; the call's output is then unspecified).
struct IdWindow {
  int base = -64;
  int id = 0;
  __device__ __forceinline__ int get(const DecodeParams& p, const int32_t* table, int k_begin,
                                     int nch, int c, int lane) {
    if (c < base || c >= base + 32) {
      base = c & ~31;
      const int cl = base + lane;
      int v = cl < nch ? __ldg(table + (k_begin + cl * kChunk) / p.B) : 0;
      const bool bad = cl < nch && (v < 0 || v >= p.num_blocks);
      if (__any_sync(0xffffffffu, bad) && lane == 0) raise_error(p.err, kErrBounds);
      id = bad ? 0 : v;
    }
    return __shfl_sync(0xffffffffu, id, c & 31);
  }
};

// Issues the chunk at key `key` of kv head kvh (physical block blk) into
// `stage` (one lane).
template <int D, bool FP8>
__device__ __forceinline__ void issue_chunk(const DecodeParams& p, uint8_t* ring, CascadeSmem* cs,
                                            const CUtensorMap* tk, const CUtensorMap* tv,
                                            int stage, int kvh, int key, int blk) {
  using G = Geo<D, FP8>;
  uint8_t* dst = ring + stage * G::kStageBytes;
  mbar_arrive_expect_tx(&cs->full[stage], G::kStageBytes);
  if constexpr (CascadeGeo<D, FP8>::kSw) {
    const int y = kvh * p.B + key % p.B;
    tc::tma_load_3d(dst, tk, 0, y, blk, &cs->full[stage]);
    tc::tma_load_3d(dst + G::kChunkBytes, tv, 0, y, blk, &cs->full[stage]);
  } else {
    const int64_t off = ((int64_t)blk * p.Hkv + kvh) * (int64_t)p.B * G::kRowBytes +
                        (int64_t)(key % p.B) * G::kRowBytes;
    bulk_g2s(dst, p.k_pool + off, G::kChunkBytes, &cs->full[stage]);
    bulk_g2s(dst + G::kChunkBytes, p.v_pool + off, G::kChunkBytes, &cs->full[stage]);
  }
}

// Where a warp's rows go: row i (< 16) of the warp is a (request, query
// token, query head), or padding.
struct WarpRows {
  int nrows;  // rows of the warp (0: none)
  // prefix CTA: (member, head) row r0 + i of the group of `first` (query
  // tokens from q_begin on), heads of kv head kvh; tail CTA: query head
  // hq0 + i of request `req` (query token qtok)
  bool prefix;
  int r0, first, q_begin, kvh;
  int req, qtok, hq0;
  __device__ __forceinline__ bool get(int g, int i, int& r, int& qt, int& hq) const {
    if (i >= nrows) return false;
    if (prefix) {
      const int gr = r0 + i, mem = gr / g;
      r = first + mem;
      qt = q_begin + mem;
      hq = kvh * g + gr % g;
    } else {
      r = req;
      qt = qtok;
      hq = hq0 + i;
    }
    return true;
  }
};

// One warp's key run and its rows: the chunks [0, nch) of keys k_begin + 16 c
// (masked at k_end) of kv head kvh through `table`, in the stages
// stage0 + (c mod sw) of the ring; a prefix CTA's warps share the ring (nact
// of them consume every chunk), a tail warp owns its sw stages.
struct WarpJob {
  const int32_t* table;
  int kvh, k_begin, k_end, nch, nact, sw, stage0, slot;
  bool prefix, direct, fills;
  WarpRows rows;
};

// The body of the kernel for one row-state type (MmaRows: up to 16 query
// rows; MmaKeys: up to 8 heads, keys as the MMA rows): start-up, streaming
// of the warp's key run, output.
template <int D, bool FP8, class RS>
__device__ __forceinline__ void cascade_warp(const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                             const DecodeParams& p, uint8_t* ring,
                                             CascadeSmem* cs, const WarpJob& jb) {
  using G = Geo<D, FP8>;
  constexpr int S = CascadeGeo<D, FP8>::kStages;
  const int lane = threadIdx.x & 31;
  const int grp = lane >> 2, tig = lane & 3;
  const unsigned full = 0xffffffffu;
  const int nch = jb.nch, sw = jb.sw, stage0 = jb.stage0;

  // start-up: the query rows and the first block ids are requested before
  // the barriers are set up, so that their latencies overlap
  IdWindow win;
  typename RS::QRaw qraw;
  if (nch > 0) {
    const __nv_bfloat16* rows[2];
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
      int r, qt, hq;
      rows[ri] = jb.rows.get(p.g, grp + 8 * ri, r, qt, hq)
                     ? p.q + ((int64_t)qt * p.Hq + hq) * D
                     : nullptr;
    }
    RS::fetch_q(rows, qraw, tig);
  }
  if (jb.fills && nch > 0) win.get(p, jb.table, jb.k_begin, nch, 0, lane);  // lane i: chunk i
  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&cs->full[i], 1);
      cs->done[i] = 0;
    }
    cs->issued = 0;
    cs->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ---- the first stages: a prefix CTA's ring filled by warp 0, a tail
  // warp's quarter by the warp itself (lane i: chunk i)
  if (jb.fills && nch > 0) {
    if (CascadeGeo<D, FP8>::kSw && lane == 0) {
      tc::prefetch_tensormap(tmap_k);
      tc::prefetch_tensormap(tmap_v);
    }
    const int n0 = min(sw, nch);
    if (lane < n0)
      issue_chunk<D, FP8>(p, ring, cs, tmap_k, tmap_v, stage0 + lane, jb.kvh,
                          jb.k_begin + lane * kChunk, win.id);
    if (jb.prefix && lane == 0) cs->issued = n0;
  }

  RS st;
  bool ok = true;
  int consumed = 0, issued_w = jb.fills ? min(sw, nch) : 0;  // tail warps: own accounting
  if (nch > 0) {
    st.load_q(qraw, p.q_scale, tig);
    st.reset();
    // two chunks per step where the ring holds at least two steps of them
    const bool pairs = sw >= 4;
    for (int c = 0; c < nch;) {
      const int n = pairs && c + 1 < nch ? 2 : 1;
      const int st0 = stage0 + c % sw, st1 = stage0 + (c + 1) % sw;
      bool ready = mbar_wait(&cs->full[st0], (c / sw) & 1, p.err);
      if (n == 2) ready = ready && mbar_wait(&cs->full[st1], ((c + 1) / sw) & 1, p.err);
      if (!__all_sync(full, ready) || *reinterpret_cast<volatile int*>(&cs->abort)) {
        cs->abort = 1;
        ok = false;
        break;
      }
      const uint8_t* K0 = ring + st0 * G::kStageBytes;
      if (n == 2) {
        const uint8_t* K1 = ring + st1 * G::kStageBytes;
        const uint8_t* const ks[2] = {K0, K1};
        const uint8_t* const vs[2] = {K0 + G::kChunkBytes, K1 + G::kChunkBytes};
        st.template chunks<2>(ks, vs, jb.k_begin + c * kChunk, jb.k_end, grp, tig);
      } else {
        st.chunk(K0, K0 + G::kChunkBytes, jb.k_begin + c * kChunk, jb.k_end, grp, tig);
      }
      consumed = c + n;
      // each stage takes the chunk one ring ahead next, issued by the last
      // warp done with it (the warps' reads of the stage have completed:
      // their values are in registers, consumed by MMAs already issued)
      for (int i = 0; i < n; ++i) {
        const int cc = c + i, stage = stage0 + cc % sw, cn = cc + sw;
        const int id = cn < nch ? win.get(p, jb.table, jb.k_begin, nch, cn, lane) : 0;
        __syncwarp();
        bool last = true;
        if (jb.prefix && cn < nch) {
          int old = 0;
          if (lane == 0) {
            __threadfence_block();
            old = atomicAdd(&cs->done[stage], 1);
          }
          last = (__shfl_sync(full, old, 0) + 1) % jb.nact == 0;
        }
        if (last && cn < nch) {
          if (lane == 0) {
            __threadfence_block();
            issue_chunk<D, FP8>(p, ring, cs, tmap_k, tmap_v, stage, jb.kvh,
                                jb.k_begin + cn * kChunk, id);
            if (jb.prefix) atomicMax(&cs->issued, cn + 1);
          }
          issued_w = cn + 1;
        }
      }
      c += n;
    }
    if (ok) {
      // the rows: the final bf16 output (direct) or the fp32 partial
      // (o * v_scale, max, sum) into split slot jb.slot
      st.finish_sums();
      st.for_each_run(grp, tig, [&](int row, int d0, float4 v, float, float l) {
        int r, qt, hq;
        if (!jb.rows.get(p.g, row, r, qt, hq)) return;
        if (jb.direct) {
          const float f = p.v_scale / l;
          const __nv_bfloat162 a = __floats2bfloat162_rn(v.x * f, v.y * f);
          const __nv_bfloat162 b = __floats2bfloat162_rn(v.z * f, v.w * f);
          *reinterpret_cast<uint2*>(p.out + ((int64_t)qt * p.Hq + hq) * D + d0) =
              make_uint2(*reinterpret_cast<const uint32_t*>(&a),
                         *reinterpret_cast<const uint32_t*>(&b));
        } else {
          const int64_t orow = ((int64_t)r * p.Hq + hq) * p.ws_splits + jb.slot;
          const float s = p.v_scale;
          *reinterpret_cast<float4*>(p.ws_o + orow * D + d0) =
              make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
        }
      });
      if (!jb.direct)
        st.for_each_stat(grp, tig, [&](int row, float m, float l) {
          int r, qt, hq;
          if (jb.rows.get(p.g, row, r, qt, hq))
            p.ws_ml[((int64_t)r * p.Hq + hq) * p.ws_splits + jb.slot] = make_float2(m, l);
        });
    }
  }
  // copies still in flight after a wait gave up land before the CTA exits
  if (!jb.prefix) {
    if (!ok && lane == 0)
      for (int c = consumed; c < issued_w; ++c)
        mbar_wait(&cs->full[stage0 + c % sw], (c / sw) & 1, p.err);
    return;
  }
  __syncthreads();
  if (threadIdx.x == 0 && cs->abort) {
    const int n = cs->issued;
    for (int c = n - S > 0 ? n - S : 0; c < n; ++c) mbar_wait(&cs->full[c % S], (c / S) & 1, p.err);
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kCThreads, 3)
    cascade_decode_kernel(const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v, DecodeParams p,
                          CascadePlan cp) {
  launch_dependents();  // the merge that follows may be scheduled now
  using G = Geo<D, FP8>;
  using CG = CascadeGeo<D, FP8>;
  constexpr int S = CG::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* ring = smem;
  if constexpr (CG::kSw) ring += (1024u - (smem_u32(smem) & 1023u)) & 1023u;  // 1024-byte aligned
  CascadeSmem* cs = reinterpret_cast<CascadeSmem*>(ring + S * G::kStageBytes);
  const int warp = threadIdx.x >> 5;

  // ---- this warp's key run, rows and destination
  WarpJob jb{};
  jb.prefix = (int)blockIdx.x < cp.n_prefix_ctas;
  jb.rows.prefix = jb.prefix;
  if (jb.prefix) {
    int b = blockIdx.x;
    const int rb = b % cp.row_blocks;
    b /= cp.row_blocks;
    jb.kvh = b % p.Hkv;
    b /= p.Hkv;
    const int piece = b % cp.pieces;
    const int k = b / cp.pieces;
    if (k >= p.groups.n) return;
    const int first = p.groups.first[k], n = p.groups.size[k];
    const int q_begin = p.qsl[first];
    if (p.qsl[first + n] - q_begin != n || q_begin < 0 || q_begin + n > p.T) {
      // members are not all decodes, or a device qsl leaves q / out
      if (threadIdx.x == 0 && rb == 0 && jb.kvh == 0 && piece == 0)
        raise_error(p.err, kErrBounds);
      return;
    }
    jb.k_begin = piece * p.groups.prefix_split_tokens;
    if (jb.k_begin >= p.groups.prefix_tokens[k]) return;
    jb.k_end = min(p.groups.prefix_tokens[k], jb.k_begin + p.groups.prefix_split_tokens);
    const int rows = n * p.g;  // (member, head) rows of the group
    const int row0 = rb * kRowsPerCta;
    if (row0 >= rows) return;
    jb.nact = min(kCWarps, (rows - row0 + 15) / 16);
    jb.table = p.block_tables + (int64_t)first * p.max_blocks;
    jb.sw = S;
    jb.stage0 = 0;
    jb.slot = piece;
    jb.fills = warp == 0;
    jb.rows.r0 = row0 + warp * 16;
    jb.rows.nrows = warp < jb.nact ? min(16, rows - jb.rows.r0) : 0;
    jb.rows.first = first;
    jb.rows.q_begin = q_begin;
    jb.rows.kvh = jb.kvh;
    // a warp without rows only takes part in the barriers
    jb.nch = jb.rows.nrows > 0 ? (jb.k_end - jb.k_begin + kChunk - 1) / kChunk : 0;
    cascade_warp<D, FP8, MmaRows<D, FP8>>(&tmap_k, &tmap_v, p, ring, cs, jb);
    return;
  }
  const int b = (int)blockIdx.x - cp.n_prefix_ctas;
  const int r = b / cp.tail_ctas, x = b % cp.tail_ctas;
  if (r >= p.R) return;
  const int qs = p.qsl[r];
  if (p.qsl[r + 1] - qs != 1) return;  // not a decode request
  const int seq = p.seq_lens[r];
  if (qs < 0 || qs >= p.T || seq < 1 || seq > p.max_blocks * p.B) {
    if (threadIdx.x == 0 && x == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int grp_id = group_of(p.groups, r);
  const int k_lo = grp_id >= 0 ? p.groups.prefix_tokens[grp_id] : 0;
  const int slot0 = prefix_slots(p.groups, grp_id);
  if (k_lo >= seq) {
    if (threadIdx.x == 0 && x == 0) raise_error(p.err, kErrBounds);
    return;
  }
  const int nsplit = (seq - k_lo + p.split_tokens - 1) / p.split_tokens;
  const int units = p.Hkv * p.head_groups;  // (kv head, 16-head part) of a split
  if ((int64_t)nsplit * units > (int64_t)cp.tail_ctas * kCWarps ||
      (slot0 + nsplit > 1 && slot0 + nsplit > p.ws_splits)) {
    // device seq_lens disagree with the host mirror the grid was planned from
    if (threadIdx.x == 0 && x == 0) raise_error(p.err, kErrBounds);
    return;
  }
  if (x * kCWarps >= nsplit * units) return;
  const int t = x * kCWarps + warp;
  const int split = t / units, u = t % units;
  jb.kvh = u / p.head_groups;
  const int part = u % p.head_groups;
  jb.rows.nrows = t < nsplit * units ? min(16, p.g - 16 * part) : 0;
  jb.rows.req = r;
  jb.rows.qtok = qs;
  jb.rows.hq0 = jb.kvh * p.g + 16 * part;
  jb.k_begin = k_lo + split * p.split_tokens;
  jb.k_end = min(seq, jb.k_begin + p.split_tokens);
  jb.nch = jb.rows.nrows > 0 ? (jb.k_end - jb.k_begin + kChunk - 1) / kChunk : 0;
  jb.table = p.block_tables + (int64_t)r * p.max_blocks;
  jb.nact = 1;
  jb.sw = CG::kTailStages;
  jb.stage0 = warp * CG::kTailStages;
  jb.direct = slot0 + nsplit == 1;
  jb.slot = slot0 + split;
  jb.fills = jb.nch > 0;
  if (p.g <= 8)
    cascade_warp<D, FP8, MmaKeys<D, FP8>>(&tmap_k, &tmap_v, p, ring, cs, jb);
  else
    cascade_warp<D, FP8, MmaRows<D, FP8>>(&tmap_k, &tmap_v, p, ring, cs, jb);
}

template <int D, bool FP8>
cudaError_t launch_cascade_t(const DecodeParams& p, const CascadePlan& cp, cudaStream_t s) {
  constexpr int smem = CascadeGeo<D, FP8>::kSmem;
  static_assert(3 * (smem + 1024) <= 228 * 1024, "three CTAs per SM");
  CUtensorMap tk, tv;
  cudaError_t e = decode_maps<D, FP8>(p, &tk, &tv);
  if (e != cudaSuccess) return e;
  auto k = cascade_decode_kernel<D, FP8>;
  e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int64_t n = (int64_t)cp.n_prefix_ctas + (int64_t)p.R * cp.tail_ctas;
  if (n < 1 || n > INT32_MAX) return cudaErrorInvalidValue;
  k<<<(unsigned)n, kCThreads, smem, s>>>(tk, tv, p, cp);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_cascade(const DecodeParams& p, const CascadePlan& cp, int D, bool fp8,
                           cudaStream_t s) {
  if (D == 128)
    return fp8 ? launch_cascade_t<128, true>(p, cp, s) : launch_cascade_t<128, false>(p, cp, s);
  return fp8 ? launch_cascade_t<64, true>(p, cp, s) : launch_cascade_t<64, false>(p, cp, s);
}

}  // namespace pa
