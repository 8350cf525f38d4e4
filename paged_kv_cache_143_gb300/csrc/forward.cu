// forward.cu — pa_forward: checks, planning from the host mirrors, dispatch of
// the decode (split-KV + merge) and prefill kernels on the caller's stream.
//
// [vLLM-wiki "엔진 구조와 주요 기능"] (one token budget per step shared by decodes
// and prefill chunks) and [V1-blog "고정 예산 기반 청크 분할 알고리즘"]: a step packs
// one token per running decode next to prefill chunks; requests with q_len = 1
// go to the decode kernels, requests with q_len > 1 to the prefill kernel.
// [MRV2 "재설계 4"]: query_start_loc and seq_lens describe the batch; their host
// mirrors let the planner size grids without a device synchronisation.
#include <algorithm>
#include <cmath>

#include "pa_internal.h"
#include "pa_kernels.h"
#include "prefill_plan.h"

namespace {

size_t split_row_bytes(int64_t R, int64_t Hq, int64_t D) {
  return (size_t)(R * Hq) * (size_t)(D * 4 + 8);
}

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// The workspace starts with the persistent decode's plan area (see
// pa::PersistPlan), then the split partials: fp32 o [R][Hq][S][D], then
// (max, sum) [R][Hq][S].
size_t plan_area_bytes(int64_t R) {
  return (size_t)((pa::persist_aux_words(R) * 4 + 255) / 256 * 256);
}

}  // namespace

extern "C" size_t pa_forward_workspace_size(int32_t num_reqs, int32_t num_q_heads,
                                            int32_t head_dim, int32_t max_splits) {
  if (num_reqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_splits <= 0) return 0;
  return plan_area_bytes(num_reqs) +
         split_row_bytes(num_reqs, num_q_heads, head_dim) * (size_t)max_splits;
}

namespace {

// Optional groups of decode requests that share their first blocks.
struct Cascade {
  int32_t n;
  const int32_t* first_host;          // [n]
  const int32_t* size_host;           // [n]
  const int32_t* prefix_blocks_host;  // [n]
};

pa_status forward_impl(const void* q, void* out, const int32_t* query_start_loc,
                       const int32_t* seq_lens, const int32_t* qsl_host,
                       const int32_t* seq_lens_host, const int32_t* block_tables,
                       int32_t max_blocks, int32_t num_reqs, int32_t num_tokens,
                       int32_t num_q_heads, const pa_kv_pool* pool, float scale, int32_t causal,
                       const Cascade* cas, void* workspace, size_t workspace_bytes,
                       pa_stream_t stream) {
  pa_status st = pa::check_pool(pool);
  if (st != PA_OK) return st;
  const int R = num_reqs, T = num_tokens, Hq = num_q_heads;
  const int Hkv = pool->num_kv_heads, D = pool->head_dim, B = pool->block_size;
  if (R < 0 || T < 0 || Hq <= 0 || max_blocks < 0) return PA_ERR_INVALID;
  if (Hq % Hkv != 0) return PA_ERR_UNSUPPORTED;
  const int g = Hq / Hkv;
  if (!(scale > 0.f) || !std::isfinite(scale)) return PA_ERR_INVALID;
  if (causal != 0 && causal != 1) return PA_ERR_INVALID;
  if (cas && cas->n < 0) return PA_ERR_INVALID;
  if (cas && cas->n > pa::kMaxGroups) return PA_ERR_UNSUPPORTED;
  if (cas && cas->n > 0 && (!cas->first_host || !cas->size_host || !cas->prefix_blocks_host))
    return PA_ERR_INVALID;
  if (R == 0) return T == 0 && (!cas || cas->n == 0) ? PA_OK : PA_ERR_INVALID;
  if (T > 0 && pool->num_blocks == 0) return PA_ERR_INVALID;  // no block a table could name
  if (!qsl_host || !seq_lens_host || !query_start_loc || !seq_lens || !block_tables)
    return PA_ERR_INVALID;
  if (T > 0 && (!q || !out || !pa::aligned16(q) || !pa::aligned16(out))) return PA_ERR_INVALID;
  if (workspace_bytes > 0 && (!workspace || !pa::aligned16(workspace))) return PA_ERR_INVALID;

  // ---- plan from the host mirrors
  if (qsl_host[0] != 0 || qsl_host[R] != T) return PA_ERR_INVALID;
  int n_pre = 0, max_q_tiles = 0;
  for (int r = 0; r < R; ++r) {
    const int ql = qsl_host[r + 1] - qsl_host[r];
    if (ql < 0) return PA_ERR_INVALID;
    if (ql == 0) continue;
    const int seq = seq_lens_host[r];
    if (seq < ql || (int64_t)seq > (int64_t)max_blocks * B) return PA_ERR_INVALID;
    if (ql > 1) {
      // a prefill tile (128 rows of token x head) must hold a whole GQA group
      if (g > 128) return PA_ERR_UNSUPPORTED;
      ++n_pre;
      const int tiles = (ql + 128 / g - 1) / (128 / g);
      if (tiles > max_q_tiles) max_q_tiles = tiles;
    }
  }
  if (R > 65535) return PA_ERR_UNSUPPORTED;

  // ---- shared-prefix groups: consecutive decode requests, each with keys
  // past the prefix
  pa::GroupDesc gd{};
  int max_prefix = 0, max_members = 0;
  if (cas && cas->n > 0) {
    gd.n = cas->n;
    int prev_end = 0;
    for (int k = 0; k < cas->n; ++k) {
      const int a = cas->first_host[k], n = cas->size_host[k];
      const int pb = cas->prefix_blocks_host[k];
      if (a < prev_end || n < 1 || (int64_t)a + n > R || pb < 1 || pb > max_blocks)
        return PA_ERR_INVALID;
      prev_end = a + n;
      const int pt = pb * B;
      for (int r = a; r < a + n; ++r)
        if (qsl_host[r + 1] - qsl_host[r] != 1 || seq_lens_host[r] <= pt) return PA_ERR_INVALID;
      gd.first[k] = a;
      gd.size[k] = n;
      gd.prefix_tokens[k] = pt;
      max_prefix = std::max(max_prefix, pt);
      max_members = std::max(max_members, n);
    }
  }
  const size_t row_bytes = split_row_bytes(R, Hq, D);
  const size_t plan_bytes = plan_area_bytes(R);
  const size_t part_bytes = workspace_bytes > plan_bytes ? workspace_bytes - plan_bytes : 0;
  const int64_t ws_splits = row_bytes ? (int64_t)(part_bytes / row_bytes) : 0;
  // the pieces of a prefix and at least one tail split each need a slot
  if (gd.n > 0 && ws_splits < 2) return PA_ERR_INVALID;
  int pieces = 0;
  if (gd.n > 0) {
    // prefix pieces of 512 keys (32 chunks: a ring and a half of stages per
    // CTA), fewer and longer when the workspace's slots run out: a member
    // needs one slot per piece and at least one for its tail
    const int64_t want = (max_prefix + ws_splits - 2) / (ws_splits - 1);
    gd.prefix_split_tokens = round_up((int)std::max<int64_t>(512, want), 16);
    pieces = (max_prefix + gd.prefix_split_tokens - 1) / gd.prefix_split_tokens;
  }
  // decode key range of request r: [k_lo, seq)
  auto group_slots = [&](int r, int* k_lo) {
    const int k = pa::group_of(gd, r);
    *k_lo = k >= 0 ? gd.prefix_tokens[k] : 0;
    return pa::prefix_slots(gd, k);
  };
  int n_dec = 0, max_dec_len = 0;
  int64_t dec_keys = 0;
  for (int r = 0; r < R; ++r) {
    if (qsl_host[r + 1] - qsl_host[r] != 1) continue;
    int k_lo;
    group_slots(r, &k_lo);
    const int len = seq_lens_host[r] - k_lo;
    ++n_dec;
    dec_keys += len;
    max_dec_len = std::max(max_dec_len, len);
  }

  unsigned* err = pa::error_word();
  if (!err) return PA_ERR_CUDA;
  cudaStream_t s = pa::as_stream(stream);
  const bool fp8 = pool->dtype == PA_KV_FP8_E4M3;
  const float kLog2e = 1.4426950408889634f;
  float* ws_o = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + plan_bytes);
  float2* ws_ml = reinterpret_cast<float2*>(reinterpret_cast<uint8_t*>(ws_o) +
                                            (size_t)R * Hq * ws_splits * D * 4);

  auto prefill_launch = [&]() {
    pa::PrefillLaunch L{};
    L.p.out = static_cast<__nv_bfloat16*>(out);
    L.p.T = T;
    L.p.qsl = query_start_loc;
    L.p.seq_lens = seq_lens;
    L.p.block_tables = block_tables;
    L.p.max_blocks = max_blocks;
    L.p.Hq = Hq;
    L.p.Hkv = Hkv;
    L.p.g = g;
    L.p.num_blocks = pool->num_blocks;
    L.p.B = B;
    L.p.causal = causal;
    L.p.scale_log2 = scale * kLog2e * (fp8 ? pool->k_scale : 1.f);
    L.p.v_scale = fp8 ? pool->v_scale : 1.f;
    L.fp8 = fp8;
    L.p.err = err;
    L.q = q;
    L.k_pool = pool->k_pool;
    L.v_pool = pool->v_pool;
    L.T = T;
    L.R = R;
    L.D = D;
    return L;
  };

  // ---- persistent GQA decode: the decode work as one flat chunk space cut
  // into equal per-CTA ranges (pa::PersistPlan); batches with shared-prefix
  // groups take the grid kernels (and the prefix pieces on tensor cores)
  pa::PersistPlan pp{};
  int persist_ctas = 0;
  if (n_dec > 0 && g >= 2 && g <= 16 && R <= pa::kMaxPersistR && ws_splits >= 2 && gd.n == 0) {
    int64_t W = 0;
    for (int r = 0; r < R; ++r)
      if (qsl_host[r + 1] - qsl_host[r] == 1) W += (int64_t)Hkv * ((seq_lens_host[r] + 15) / 16);
    // slots a request may need with Q chunks per CTA: a unit of C chunks
    // falls into at most ceil((C - 1) / Q) + 1 CTA ranges (1 if Q >= W)
    auto fits = [&](int64_t Q) {
      for (int r = 0; r < R; ++r) {
        if (qsl_host[r + 1] - qsl_host[r] != 1) continue;
        const int64_t C = (seq_lens_host[r] + 15) / 16;
        if ((Q >= W ? 1 : (C + Q - 2) / Q + 1) > ws_splits) return false;
      }
      return true;
    };
    int64_t lo = 1, hi = std::max<int64_t>(W, 1);  // fits(W) holds: one range
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (fits(mid)) hi = mid; else lo = mid + 1;
    }
    const int64_t q_min = lo;
    const int64_t n_max = (int64_t)pa::num_sms() * 2;  // two CTAs per SM
    const int64_t Q = std::max(q_min, (W + n_max - 1) / n_max);
    if (W > 0 && W < INT32_MAX && Q < INT32_MAX) {
      pp.on = 1;
      pp.q_min = (int32_t)q_min;
      pp.aux = static_cast<int32_t*>(workspace);
      persist_ctas = (int)((W + Q - 1) / Q);
    }
  }

  if (n_dec > 0) {
    pa::DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.out = static_cast<__nv_bfloat16*>(out);
    p.T = T;
    p.qsl = query_start_loc;
    p.seq_lens = seq_lens;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.g = g;
    p.head_groups = g > 16 ? (g + 15) / 16 : 1;
    if ((int64_t)Hkv * p.head_groups > 65535) return PA_ERR_UNSUPPORTED;
    p.k_pool = static_cast<const uint8_t*>(pool->k_pool);
    p.v_pool = static_cast<const uint8_t*>(pool->v_pool);
    p.num_blocks = pool->num_blocks;
    p.B = B;
    p.q_scale = scale * kLog2e * (fp8 ? pool->k_scale : 1.f);
    p.v_scale = fp8 ? pool->v_scale : 1.f;
    p.err = err;
    p.groups = gd;
    p.R = R;
    p.pp = pp;

    if (gd.n > 0) {
      // shared-prefix batch: the groups' prefix pieces and every decode's keys
      // after its prefix in one launch (cascade.cu), then the merge. Tail
      // splits of at least 256 keys, few enough for the slots left after a
      // member's prefix pieces.
      int64_t sp = 256;
      for (int r = 0; r < R; ++r) {
        if (qsl_host[r + 1] - qsl_host[r] != 1) continue;
        int k_lo;
        const int free_slots = (int)ws_splits - group_slots(r, &k_lo);
        sp = std::max<int64_t>(sp, (seq_lens_host[r] - k_lo + free_slots - 1) / free_slots);
      }
      sp = round_up((int)sp, 16);
      const int units = Hkv * p.head_groups;
      int64_t tail_ctas = 1;
      for (int r = 0; r < R; ++r) {
        if (qsl_host[r + 1] - qsl_host[r] != 1) continue;
        int k_lo;
        group_slots(r, &k_lo);
        const int64_t ns = (seq_lens_host[r] - k_lo + sp - 1) / sp;
        tail_ctas = std::max<int64_t>(tail_ctas, (ns * units + 3) / 4);
      }
      pa::CascadePlan cp{};
      cp.pieces = pieces;
      cp.row_blocks = (int)(((int64_t)max_members * g + 63) / 64);
      const int64_t n_pref = (int64_t)gd.n * pieces * Hkv * cp.row_blocks;
      if (n_pref + (int64_t)R * tail_ctas > INT32_MAX) return PA_ERR_UNSUPPORTED;
      cp.n_prefix_ctas = (int32_t)n_pref;
      cp.tail_ctas = (int32_t)tail_ctas;
      p.split_tokens = (int)sp;
      p.ws_splits = (int)ws_splits;
      p.ws_o = ws_o;
      p.ws_ml = ws_ml;
      if (pa::launch_cascade(p, cp, D, fp8, s) != cudaSuccess) return PA_ERR_CUDA;
      pa::count_launches(1);
      // every group member has a prefix partial and a tail partial
      if (pa::launch_merge(p, D, R, s) != cudaSuccess) return PA_ERR_CUDA;
      pa::count_launches(1);
    } else if (pp.on) {
      // every decode in one persistent launch, then the merge of the pieces
      p.ws_splits = (int)ws_splits;
      p.ws_o = ws_o;
      p.ws_ml = ws_ml;
      if (pa::launch_decode_persist(p, D, fp8, persist_ctas, s) != cudaSuccess) return PA_ERR_CUDA;
      pa::count_launches(1);
      if (pa::launch_merge(p, D, R, s) != cudaSuccess) return PA_ERR_CUDA;
      pa::count_launches(1);
    } else {
      // Split size: enough CTAs for ~4 waves of 2 CTAs per SM, each split at
      // least 256 keys, a multiple of the 16-key chunk; bounded by the slots
      // the workspace holds. Depends only on seq_lens, never on placement.
      const int64_t target_ctas = (int64_t)pa::num_sms() * 2 * 4;
      int64_t split = (dec_keys * Hkv * p.head_groups + target_ctas - 1) / target_ctas;
      split = std::max<int64_t>(split, 256);
      split = std::min<int64_t>(split, max_dec_len);
      split = round_up((int)split, 16);
      auto plan = [&](int64_t sp, int* grid_x) {
        int gx = 0;
        for (int r = 0; r < R; ++r)
          if (qsl_host[r + 1] - qsl_host[r] == 1)
            gx = std::max(gx, (int)((seq_lens_host[r] + sp - 1) / sp));
        *grid_x = gx;
        return gx;  // split slots a request needs
      };
      int grid_x;
      int need = plan(split, &grid_x);
      if (need > 1 && need > ws_splits) {
        if (ws_splits <= 1) {  // no groups here: one split per request, no workspace
          split = round_up(max_dec_len, 16);
        } else {
          split = round_up((int)((max_dec_len + ws_splits - 1) / ws_splits), 16);
        }
        need = plan(split, &grid_x);
      }
      if (grid_x > 65535) return PA_ERR_UNSUPPORTED;
      p.split_tokens = (int)split;
      p.ws_splits = need > 1 ? (int)ws_splits : 1;
      if (need > 1) {
        p.ws_o = ws_o;
        p.ws_ml = ws_ml;
      }
      if (pa::launch_decode(p, D, fp8, R, grid_x, s) != cudaSuccess) return PA_ERR_CUDA;
      pa::count_launches(1);
      if (need > 1) {
        if (pa::launch_merge(p, D, R, s) != cudaSuccess) return PA_ERR_CUDA;
        pa::count_launches(1);
      }
    }
  }

  if (n_pre > 0) {
    pa::PrefillLaunch L = prefill_launch();
    L.max_q_tiles = max_q_tiles;
    // Launch order (prefill_plan.h): the (request, tile pair) units longest
    // first across all requests, each unit's kv heads side by side. Units
    // past the list's capacity fall back to a (pairs, Hkv, requests) grid
    // with the requests ordered by their causal pairs.
    const int n_units =
        pa::plan_prefill_units<pa::kMaxPrefillUnits>(qsl_host, seq_lens_host, R, g, causal != 0,
                                                     L.p.units);
    if (n_units >= 0) {
      L.p.n_units = n_units;
    } else if (n_pre <= pa::kMaxOrderedPrefill) {
      int n = 0;
      for (int r = 0; r < R; ++r)
        if (qsl_host[r + 1] - qsl_host[r] > 1) L.p.order[n++] = r;
      auto work = [&](int r) {
        const int64_t ql = qsl_host[r + 1] - qsl_host[r];
        const int64_t P = seq_lens_host[r] - ql;
        return causal ? ql * P + ql * (ql + 1) / 2 : ql * (int64_t)seq_lens_host[r];
      };
      std::stable_sort(L.p.order, L.p.order + n,
                       [&](int a, int b) { return work(a) > work(b); });
      L.p.n_order = n;
    }
    if (pa::launch_prefill(L, s) != cudaSuccess) return PA_ERR_CUDA;
    pa::count_launches(1);
  }
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_forward(const void* q, void* out, const int32_t* query_start_loc,
                                const int32_t* seq_lens, const int32_t* qsl_host,
                                const int32_t* seq_lens_host, const int32_t* block_tables,
                                int32_t max_blocks, int32_t num_reqs, int32_t num_tokens,
                                int32_t num_q_heads, const pa_kv_pool* pool, float scale,
                                int32_t causal, void* workspace, size_t workspace_bytes,
                                pa_stream_t stream) {
  return forward_impl(q, out, query_start_loc, seq_lens, qsl_host, seq_lens_host, block_tables,
                      max_blocks, num_reqs, num_tokens, num_q_heads, pool, scale, causal,
                      nullptr, workspace, workspace_bytes, stream);
}

extern "C" pa_status pa_forward_shared_prefix(
    const void* q, void* out, const int32_t* query_start_loc, const int32_t* seq_lens,
    const int32_t* qsl_host, const int32_t* seq_lens_host, const int32_t* block_tables,
    int32_t max_blocks, int32_t num_reqs, int32_t num_tokens, int32_t num_q_heads,
    const pa_kv_pool* pool, float scale, int32_t causal, int32_t num_groups,
    const int32_t* group_first_host, const int32_t* group_size_host,
    const int32_t* prefix_blocks_host, void* workspace, size_t workspace_bytes,
    pa_stream_t stream) {
  const Cascade c{num_groups, group_first_host, group_size_host, prefix_blocks_host};
  return forward_impl(q, out, query_start_loc, seq_lens, qsl_host, seq_lens_host, block_tables,
                      max_blocks, num_reqs, num_tokens, num_q_heads, pool, scale, causal, &c,
                      workspace, workspace_bytes, stream);
}
