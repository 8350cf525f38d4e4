// pa_kernels.h — launch interfaces between the pa_forward planner and the
// attention kernels (internal to libpa).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Groups of consecutive decode requests whose first blocks are shared.
constexpr int kMaxGroups = 64;
struct GroupDesc {
  int32_t n;                          // number of groups (0: none)
  int32_t first[kMaxGroups];          // group k = requests [first[k], first[k] + size[k]),
  int32_t size[kMaxGroups];           //   increasing and disjoint
  int32_t prefix_tokens[kMaxGroups];  // shared prefix length (whole blocks)
  // the prefix is cut into pieces of this many keys (a multiple of 16);
  // piece i of a member's prefix lands in split slot i, its tail after them
  int32_t prefix_split_tokens;
};

// Group of request r (-1 if none), by binary search over the group starts.
__host__ __device__ inline int group_of(const GroupDesc& gd, int r) {
  if (gd.n == 0 || r < gd.first[0]) return -1;
  int lo = 0, hi = gd.n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (gd.first[mid] <= r) lo = mid; else hi = mid - 1;
  }
  return r < gd.first[lo] + gd.size[lo] ? lo : -1;
}

// Split slots that a group member's prefix pieces take (0 if ungrouped).
__host__ __device__ inline int prefix_slots(const GroupDesc& gd, int grp) {
  return grp < 0 ? 0
                 : (gd.prefix_tokens[grp] + gd.prefix_split_tokens - 1) / gd.prefix_split_tokens;
}

// ---------------------------------------------------------------------------
// Persistent GQA decode (2 <= g <= 16; batches without shared-prefix groups).
// The decode work of one call is laid out as one sequence of 16-key chunks,
// the "flat space": unit (request r, kv head h) holds the chunks of r's keys
// [0, seq_len) for the g heads of r's token, at Hkv * pref[r] + h * C_r, pref
// the exclusive running sum of C_r over the requests (0 for non-decodes).
// CTA b of the grid takes the chunks [b Q, b Q + Q), with
// Q = max(ceil(W / grid), q_min); the CTA ranges cut each unit [a, a + C)
// into pieces, piece i being the part in CTA floor(a / Q) + i. A request read
// in one piece writes its output directly; otherwise every piece writes a
// partial into split slot i, merged by log-sum-exp.
constexpr int kMaxPersistR = 512;   // requests the persistent path handles

struct PersistPlan {
  int32_t on;                          // 1: decodes run on the persistent kernel
  int32_t q_min;                       // minimum chunks per CTA (bounds the slots)
  int32_t* aux;                        // workspace: [0] Q, [1] W, [2 + r] pref[r], r <= R
};

// Pieces of a unit of C chunks starting at a, for ranges of Q chunks.
__host__ __device__ inline int64_t flat_pieces(int64_t a, int64_t C, int64_t Q) {
  return C <= 0 ? 0 : (a + C - 1) / Q - a / Q + 1;
}

// Words of the persistent plan's area at the start of the workspace.
__host__ __device__ inline int64_t persist_aux_words(int64_t R) { return R + 3; }

struct DecodeParams {
  const __nv_bfloat16* q;      // [T][Hq][D]
  __nv_bfloat16* out;          // [T][Hq][D]
  int32_t T;                   // rows of q and out: every device qsl entry must be <= T
  const int32_t* qsl;          // [R+1]
  const int32_t* seq_lens;     // [R]
  const int32_t* block_tables; // [R][max_blocks]
  int32_t max_blocks;
  int32_t Hq, Hkv, g;
  // CTAs per kv head along grid y: 1, or ceil(g / 16) for g > 16 (the MMA
  // decode serves at most 16 query heads per CTA; CTA y = kv head *
  // head_groups + part serves heads part * 16 .. of the group)
  int32_t head_groups;
  const uint8_t* k_pool;       // [num_blocks][Hkv][B][D] elements of 1 or 2 bytes
  const uint8_t* v_pool;
  int32_t num_blocks, B;
  float q_scale;               // softmax scale * log2(e) * k_scale (FP8) or * 1
  float v_scale;               // v_scale (FP8) or 1
  int32_t split_tokens;        // keys per split (multiple of 16)
  int32_t ws_splits;           // split stride of the workspace arrays
  float* ws_o;                 // [R][Hq][ws_splits][D] unnormalised partial outputs
  float2* ws_ml;               // [R][Hq][ws_splits] (max in log2 units, sum)
  unsigned* err;
  // requests in a group attend only to their keys after the shared prefix
  // (key range [prefix_tokens, seq_len)) and always write partials into
  // split slots 1.. (slot 0 holds the prefix partial)
  GroupDesc groups;
  int32_t R;                   // requests
  PersistPlan pp;              // the persistent kernel's plan (pp.on == 0: grid kernels)
};

constexpr int kMaxOrderedPrefill = 256;
constexpr int kMaxPrefillUnits = 1024;

struct PrefillParams {
  __nv_bfloat16* out;          // [T][Hq][D]
  int32_t T;                   // rows of q and out: every device qsl entry must be <= T
  const int32_t* qsl;          // [R+1]
  const int32_t* seq_lens;     // [R]
  const int32_t* block_tables; // [R][max_blocks]
  int32_t max_blocks;
  int32_t Hq, Hkv, g;
  int32_t num_blocks, B;
  int32_t causal;
  float scale_log2;            // softmax scale * log2(e) (* k_scale for E4M3 pools)
  float v_scale;               // v_scale for E4M3 pools, else 1
  unsigned* err;
  // prefill requests in launch order (most work first); n_order == 0 means
  // grid.z walks every request in batch order
  int32_t n_order;
  int32_t order[kMaxOrderedPrefill];
  // (request, tile pair) units in launch order, the most key tiles first
  // across all requests: unit = request << 16 | last << 15 | pair, last set
  // on the request's highest pair. With n_units > 0 the grid is
  // (Hkv, n_units) and order/n_order are unused.
  int32_t n_units;
  int32_t units[kMaxPrefillUnits];
};

struct PrefillLaunch {
  PrefillParams p;
  const void* q;               // bf16 [T][Hq][D]
  const void* k_pool;          // [num_blocks][Hkv][B][D]
  const void* v_pool;
  int32_t T, R, D;
  bool fp8;                    // E4M3 pools
  int32_t max_q_tiles;         // max over prefill requests of ceil(q_len / (128 / g))
};

cudaError_t launch_prefill(const PrefillLaunch& L, cudaStream_t s);

// Grid of the shared-prefix decode (cascade.cu): n_prefix_ctas CTAs for the
// groups' prefixes, laid out as [group][piece][kv head][row block] (a row
// block = 64 of the group's (member, head) rows, member-major), then
// tail_ctas CTAs per request, each taking four (key split, kv head, 16-head
// part) tasks of the request.
struct CascadePlan {
  int32_t n_prefix_ctas;
  int32_t pieces;       // prefix pieces per group (of groups.prefix_split_tokens keys)
  int32_t row_blocks;   // row blocks per (group, piece, kv head)
  int32_t tail_ctas;    // CTAs per request
};
// Prefix pieces and private tails of a batch with shared-prefix groups, into
// the split slots of the workspace (p.ws_o, p.ws_ml): a member's prefix
// piece i in slot i, its tail splits after them; an ungrouped request read
// in one split writes its bf16 output directly.
cudaError_t launch_cascade(const DecodeParams& p, const CascadePlan& cp, int D, bool fp8,
                           cudaStream_t s);

cudaError_t launch_decode(const DecodeParams& p, int D, bool fp8, int R, int max_splits,
                          cudaStream_t s);
// The persistent decode on n_cta CTAs (p.pp.on == 1).
cudaError_t launch_decode_persist(const DecodeParams& p, int D, bool fp8, int n_cta,
                                  cudaStream_t s);
cudaError_t launch_merge(const DecodeParams& p, int D, int R, cudaStream_t s);

}  // namespace pa
