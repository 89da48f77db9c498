// Brute-force check of the library's host-side tiling arithmetic (fa_common.cuh):
// the key / query tile ranges a tile of rows (keys) can see, the interior-tile test
// that lets the kernels skip the per-element mask, the key-range count of short query
// sequences, and the range set the dQ range sum adds up. Built and run by
// tests/test_host_tiling.py; prints "ok <checks>" or the first failure (exit 1).
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "fa_common.cuh"

using namespace fa;

// key j is visible to query row i: the mask rule of the source pages as restated
// here, independently of the library (top-left causal, window counting self)
static bool visible(int i, int j, int Sk, int causal, int window) {
  if (j < 0 || j >= Sk) return false;
  if (causal && j > i) return false;
  if (window > 0 && j < i - window + 1) return false;
  return true;
}

static long long checks = 0;
static void fail(const char* what, int a, int b, int c, int d, int e, int f) {
  std::printf("FAIL %s: %d %d %d %d %d %d\n", what, a, b, c, d, e, f);
  std::exit(1);
}

// the key tiles [lo, hi) must be exactly the tiles holding a visible key of some row
static void check_kv(int r0, int r1, int Sk, int causal, int window) {
  int lo, hi;
  kv_tile_range(r0, r1, Sk, causal, window, &lo, &hi);
  const int n_kt = (Sk + BLOCK_N - 1) / BLOCK_N;
  for (int t = 0; t < n_kt; ++t) {
    bool any = false;
    for (int i = r0; i <= r1 && !any; ++i)
      for (int j = t * BLOCK_N; j < (t + 1) * BLOCK_N && !any; ++j) any = visible(i, j, Sk, causal, window);
    if (any != (t >= lo && t < hi)) fail("kv_tile_range", r0, r1, Sk, causal, window, t);
  }
  ++checks;
}

// the query tiles [lo, hi) must be exactly the tiles holding a row that sees some key
static void check_q(int c0, int c1, int Sq, int Sk, int causal, int window) {
  int lo, hi;
  q_tile_range(c0, c1, Sq, causal, window, &lo, &hi);
  const int n_qt = (Sq + BLOCK_M - 1) / BLOCK_M;
  for (int t = 0; t < n_qt; ++t) {
    bool any = false;
    for (int i = t * BLOCK_M; i < (t + 1) * BLOCK_M && i < Sq && !any; ++i)
      for (int j = c0; j <= c1 && !any; ++j) any = visible(i, j, Sk, causal, window);
    if (any != (t >= lo && t < hi)) fail("q_tile_range", c0, c1, Sq, causal, window, t);
  }
  ++checks;
}

// a tile pair said to need no mask must have every pair visible
static void check_mask(int r0, int r1, int c0, int Sk, int causal, int window) {
  const int c1 = c0 + BLOCK_N - 1;
  if (tile_needs_mask(r0, r1, c0, c1, Sk, causal, window)) return;
  for (int i = r0; i <= r1; ++i)
    for (int j = c0; j <= c1; ++j)
      if (!visible(i, j, Sk, causal, window)) fail("tile_needs_mask", r0, r1, c0, Sk, causal, window);
  ++checks;
}

int main() {
  const int windows[] = {0, 1, 2, 100, 127, 128, 129, 300, 1000};
  const int sizes[] = {1, 2, 127, 128, 129, 255, 256, 300, 513};
  for (int causal = 0; causal < 2; ++causal)
    for (int window : windows)
      for (int Sq : sizes)
        for (int Sk : sizes) {
          // rows of one tile and of a two-tile item (the forward's row pairs)
          for (int r0 = 0; r0 < Sq; r0 += BLOCK_M) {
            check_kv(r0, std::min(r0 + BLOCK_M - 1, Sq - 1), Sk, causal, window);
            check_kv(r0, std::min(r0 + 2 * BLOCK_M - 1, Sq - 1), Sk, causal, window);
            for (int c0 = 0; c0 < Sk + BLOCK_N; c0 += BLOCK_N)
              check_mask(r0, r0 + BLOCK_M - 1, c0, Sk, causal, window);
          }
          for (int c0 = 0; c0 < Sk; c0 += BLOCK_N)
            check_q(c0, std::min(c0 + BLOCK_N - 1, Sk - 1), Sq, Sk, causal, window);
        }
  // key-range count: no split unless the items are fewer than the SMs and there are
  // at least 8 key tiles; otherwise ranges of >= 4 tiles, at most MAX_KEY_RANGES of
  // them, and no range count with a lower estimated cost
  const int sms = 152;
  auto cost = [&](int base, int n_kt, int s) {
    const int t = (n_kt + s - 1) / s, ns = (n_kt + t - 1) / t;
    return ((long long)base * ns + sms - 1) / sms * (t + 2);
  };
  for (int base = 1; base <= 200; ++base)
    for (int n_kt = 1; n_kt <= 260; ++n_kt) {
      const int t = key_range_tiles(base, n_kt, sms);
      const int ns = (n_kt + t - 1) / t;
      if (base >= sms || n_kt < 8) {
        if (t != n_kt) fail("key_range_tiles (no split)", base, n_kt, t, 0, 0, 0);
      } else {
        if (ns > MAX_KEY_RANGES || (ns > 1 && t < 4)) fail("key_range_tiles (limits)", base, n_kt, t, ns, 0, 0);
        const long long got = (long long)((base * (long long)ns + sms - 1) / sms) * (t + 2);
        for (int s = 1; s <= MAX_KEY_RANGES && s <= n_kt / 4; ++s)
          if (cost(base, n_kt, s) < got) fail("key_range_tiles (not minimal)", base, n_kt, t, s, 0, 0);
      }
      ++checks;
    }
  // the ranges the dQ range sum adds up, [lo / tps, (hi - 1) / tps], are exactly the
  // ranges s whose key tiles [s tps, (s + 1) tps) meet the query tile's [lo, hi)
  for (int tps = 1; tps <= 12; ++tps)
    for (int lo = 0; lo < 60; ++lo)
      for (int hi = lo; hi <= 60; ++hi) {
        const int s_lo = lo / tps, s_hi = hi > lo ? (hi - 1) / tps + 1 : 0;
        for (int s = 0; s * tps < 60; ++s) {
          const bool meets = std::max(lo, s * tps) < std::min(hi, (s + 1) * tps);
          const bool summed = hi > lo && s >= s_lo && s < s_hi;
          if (meets != summed) fail("range sum", tps, lo, hi, s, 0, 0);
        }
        ++checks;
      }
  std::printf("ok %lld\n", checks);
  return 0;
}
