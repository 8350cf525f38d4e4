// prefill_plan.h — launch order of the prefill kernel's CTAs, planned on the
// host from the query-start and sequence-length mirrors (plain C++: no CUDA
// types, so host tests compile it alone).
//
// [V1-blog "고정 예산 기반 청크 분할 알고리즘"]: a prefill chunk of q_len tokens
// follows P = seq_len - q_len cached tokens; under causal masking query j of
// the chunk sees keys 0 .. P + j. The prefill kernel gives one CTA to a pair
// of consecutive query tiles (tpt = 128 / g tokens each) of one kv head and
// walks the key tiles (128 keys) of the pair's later tile, so a CTA's time
// grows with that count. The block scheduler hands out CTAs in grid order as
// SMs free up; listing the (request, tile pair) units longest first across
// all requests keeps the long ones from forming the grid's tail.
#pragma once

#include <algorithm>
#include <cstdint>

namespace pa {

// Key tiles walked by tile pair `pair` of a chunk of q_len tokens with
// seq_len keys in all (the later tile's last token bounds the causal keys).
inline int prefill_pair_key_tiles(int q_len, int seq_len, int pair, int tpt, bool causal) {
  const int last = std::min(q_len, (2 * pair + 2) * tpt);
  const int n_kv = causal ? seq_len - q_len + last : seq_len;
  return (n_kv + 127) / 128;
}

// Writes the prefill units of requests r = 0 .. R-1 with q_len > 1 into
// units[0 .. n-1] and returns n, or -1 if there are more than MaxUnits. A
// unit is request << 16 | last << 15 | pair, last set on the request's
// highest pair. Order: key tiles walked, descending; ties keep request
// order, and within a request the later pairs first. Requires R <= 65535,
// 1 <= g <= 128 and pairs < 2^15 (which MaxUnits <= 2^15 guarantees).
template <int MaxUnits>
int plan_prefill_units(const int32_t* qsl_host, const int32_t* seq_lens_host, int R, int g,
                       bool causal, int32_t* units) {
  static_assert(MaxUnits <= (1 << 15), "pair index must fit in 15 bits");
  const int tpt = 128 / g;
  int64_t total = 0;
  for (int r = 0; r < R; ++r) {
    const int ql = qsl_host[r + 1] - qsl_host[r];
    if (ql > 1) total += ((ql + tpt - 1) / tpt + 1) / 2;
  }
  if (total > MaxUnits) return -1;
  struct Unit {
    int32_t steps, id;
  };
  Unit list[MaxUnits];
  int n = 0;
  for (int r = 0; r < R; ++r) {
    const int ql = qsl_host[r + 1] - qsl_host[r];
    if (ql <= 1) continue;
    const int npairs = ((ql + tpt - 1) / tpt + 1) / 2;
    for (int pair = npairs - 1; pair >= 0; --pair) {
      const int last = pair == npairs - 1 ? 0x8000 : 0;
      list[n++] = Unit{prefill_pair_key_tiles(ql, seq_lens_host[r], pair, tpt, causal),
                       (r << 16) | last | pair};
    }
  }
  std::stable_sort(list, list + n, [](const Unit& a, const Unit& b) { return a.steps > b.steps; });
  for (int i = 0; i < n; ++i) units[i] = list[i].id;
  return n;
}

}  // namespace pa
