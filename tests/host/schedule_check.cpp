// Host check of the CTA-pair GEMM's tile sequence (compiled and run by tests/test_host_logic.py):
// the static waves of every pair plus the claimed tail, claimed in a scrambled order of pairs,
// cover every tile exactly once, and every pair ends on the -1 it is given past the last tile.
// Usage: schedule_check num_tiles pairs seed   -> prints "ok <n_static>" or an error.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "internal.h"

int main(int argc, char** argv) {
  if (argc != 4) return 2;
  const int num_tiles = atoi(argv[1]);
  const int pairs = atoi(argv[2]);
  unsigned seed = static_cast<unsigned>(atoi(argv[3]));
  std::vector<int> seen(num_tiles, 0);
  std::vector<qkvcte::PairSchedule> s;
  for (int p = 0; p < pairs; ++p) s.emplace_back(num_tiles, p, pairs);
  for (int p = 0; p < pairs; ++p)
    for (int q = 0; q < s[p].n_static; ++q) {
      const int t = s[p].static_tile(q);
      if (t < 0 || t >= num_tiles) { printf("static tile %d out of range\n", t); return 1; }
      seen[t]++;
    }
  // the claimed tail: pairs claim in a pseudo-random order; a claim past the end gives -1
  unsigned counter = 0;
  std::vector<int> done(pairs, 0);
  int left = pairs;
  while (left > 0) {
    seed = seed * 1103515245u + 12345u;
    const int p = static_cast<int>((seed >> 8) % static_cast<unsigned>(pairs));
    if (done[p]) continue;
    const long long t = static_cast<long long>(s[p].dyn_base) + counter++;
    if (t >= num_tiles) { done[p] = 1; --left; continue; }
    seen[t]++;
  }
  for (int t = 0; t < num_tiles; ++t)
    if (seen[t] != 1) { printf("tile %d taken %d times\n", t, seen[t]); return 1; }
  printf("ok %d\n", s[0].n_static);
  return 0;
}
