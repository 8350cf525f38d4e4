// Host-test driver for prefill_plan.h: reads "R g causal cap" then the R + 1
// query starts and the R sequence lengths from stdin, prints the number of
// units (-1: over capacity) and the units, one per line.
#include <cstdio>
#include <vector>

#include "../paged_kv_cache_143_gb300/csrc/prefill_plan.h"

int main() {
  int R, g, causal, cap;
  if (std::scanf("%d %d %d %d", &R, &g, &causal, &cap) != 4) return 2;
  std::vector<int32_t> qsl(R + 1), seq(R), units(1024);
  for (auto& x : qsl)
    if (std::scanf("%d", &x) != 1) return 2;
  for (auto& x : seq)
    if (std::scanf("%d", &x) != 1) return 2;
  int n;
  if (cap == 1024)
    n = pa::plan_prefill_units<1024>(qsl.data(), seq.data(), R, g, causal != 0, units.data());
  else if (cap == 16)
    n = pa::plan_prefill_units<16>(qsl.data(), seq.data(), R, g, causal != 0, units.data());
  else
    return 2;
  std::printf("%d\n", n);
  for (int i = 0; i < n; ++i) std::printf("%d\n", units[i]);
  return 0;
}
