// Host check of the GEMM's banded tile order (compiled and run by tests/test_host_logic.py).
// Usage: bands_check T H I tile_n k_end band_tiles [m_chunks]   -> prints "ok <n_bands>" or an error.
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "internal.h"

int main(int argc, char** argv) {
  if (argc != 7 && argc != 8) return 2;
  qkvcte::GemmShape g{};
  g.T = atoi(argv[1]);
  g.H = atoi(argv[2]);
  g.I = atoi(argv[3]);
  g.tile_n = atoi(argv[4]);
  const int k_end = atoi(argv[5]);
  const int band_tiles = atoi(argv[6]);
  g.m_tiles = (g.T + 127) / 128;
  g.n_tiles = (g.I + g.tile_n - 1) / g.tile_n;
  g.n_qk_tiles = (k_end + g.tile_n - 1) / g.tile_n;
  if (g.n_qk_tiles > g.n_tiles) g.n_qk_tiles = g.n_tiles;
  const int m_chunks = argc == 8 ? atoi(argv[7]) : 1;
  qkvcte::make_bands(g, band_tiles, m_chunks);
  const int total = g.m_tiles * g.n_tiles;
  if (g.band_tile0[g.n_bands] != total) { printf("bad total %d vs %d\n", g.band_tile0[g.n_bands], total); return 1; }
  if (g.n_bands > qkvcte::kMaxBands) { printf("too many bands\n"); return 1; }
  std::vector<int> seen(total, 0);
  bool in_v = false;
  for (int t = 0; t < total; ++t) {
    int m, n;
    qkvcte::tile_coords(g, t, m, n);
    if (m < 0 || m >= g.m_tiles || n < 0 || n >= g.n_tiles) { printf("out of range at %d\n", t); return 1; }
    seen[m * g.n_tiles + n]++;
    const bool qk = n < g.n_qk_tiles;
    if (in_v && qk) { printf("Q/K tile after a V tile at %d\n", t); return 1; }
    in_v = in_v || !qk;
  }
  for (int i = 0; i < total; ++i)
    if (seen[i] != 1) { printf("tile %d visited %d times\n", i, seen[i]); return 1; }
  const int v_tiles = g.n_tiles - g.n_qk_tiles;
  const int need = (v_tiles + band_tiles - 1) / band_tiles + (g.n_qk_tiles + band_tiles - 1) / band_tiles;
  // With row-panel chunks, every chunk's Q/K tiles come before the next chunk's.
  if (m_chunks > 1) {
    int last_m0 = -1;
    for (int s = 0; s < g.n_bands && g.band_n0[s] < g.n_qk_tiles; ++s) {
      if (g.band_m0[s] < last_m0) { printf("chunk order broken at segment %d\n", s); return 1; }
      last_m0 = g.band_m0[s];
    }
  }
  if (need <= qkvcte::kMaxBands && m_chunks == 1) {  // otherwise bands are widened to fit the cap
    for (int b = 0; b < g.n_bands; ++b)
      if (g.band_nc[b] > band_tiles) { printf("band %d too wide\n", b); return 1; }
  }
  printf("ok %d\n", g.n_bands);
  return 0;
}
