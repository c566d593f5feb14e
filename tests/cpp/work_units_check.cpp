// Host check of the attention launch's work units (paged_decode_attention_02_gb300/csrc/
// work_units.h): for many tile counts W, warp counts NW and chunk limits, the units tile
// [0, W) exactly and in order, every tile's owner holds it, the claim order names each pool
// chunk once, and an all-static split is exactly the equal split floor(w W / NW).
// Prints "ok" and exits 0, or prints the first failing case and exits 1.
#include <cstdio>
#include <cstdint>
#include <set>

#include "../../paged_decode_attention_02_gb300/csrc/work_units.h"

using pda::Units;

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;
static uint64_t next_u64() {  // xorshift64*
  rng_state ^= rng_state >> 12;
  rng_state ^= rng_state << 25;
  rng_state ^= rng_state >> 27;
  return rng_state * 0x2545f4914f6cdd1dull;
}
static int rand_in(int lo, int hi) {  // inclusive
  return lo + static_cast<int>(next_u64() % static_cast<uint64_t>(hi - lo + 1));
}

static bool check(int W, int NW, int k_max) {
  const Units un = pda::make_units(W, NW, k_max);
  const int n = un.units();
#define FAIL(msg)                                                                        \
  do {                                                                                   \
    std::printf("FAIL W=%d NW=%d k_max=%d k=%d: %s\n", W, NW, k_max, un.k, msg);         \
    return false;                                                                        \
  } while (0)
  if (un.k < 0 || un.k > k_max || un.k > PDA_POOL_CHUNKS_PER_WARP) FAIL("chunk count");
  if (un.start(0) != 0 || un.start(n) != W) FAIL("units do not span [0, W)");
  const int stride = n <= 20000 ? 1 : n / 20000 + 1;
  for (int u = 0; u < n; u += stride) {
    const int a = un.start(u), b = un.start(u + 1);
    if (a > b) FAIL("units out of order");
    if (un.k == 0 && a != static_cast<int>((static_cast<long long>(u) * W) / NW))
      FAIL("all-static split is not floor(w W / NW)");
    if (a < b && (un.owner(a) != u || un.owner(b - 1) != u)) FAIL("owner does not invert start");
    if (un.live(u) != (a < b)) FAIL("live");
  }
  for (int i = 0; i < 200 && W > 0; ++i) {
    const int t = rand_in(0, W - 1);
    const int u = un.owner(t);
    if (u < 0 || u >= n || un.start(u) > t || t >= un.start(u + 1)) FAIL("tile owner");
  }
  if (un.k > 0) {
    std::set<int> seen;
    for (int g = 0; g < NW * un.k; ++g) {
      const int u = un.chunk_unit(g);
      if (u < 0 || u >= n || u % (un.k + 1) == 0 || !seen.insert(u).second)
        FAIL("claim order does not name each chunk once");
    }
  }
  return true;
#undef FAIL
}

int main() {
  const int nws[] = {1, 2, 3, 8, 12, 96, 152, 192, 372, 1104, 1216, 1824, 4096, 16383};
  for (int NW : nws) {
    const int Ws[] = {1, 7, NW - 1 > 0 ? NW - 1 : 1, NW, NW + 1, 9 * NW, 24 * NW, 80 * NW - 1,
                      80 * NW, 361 * NW + 17, 658992, 2000000, 2147483647 / 2};
    for (int W : Ws) {
      if (W <= 0) continue;
      for (int k_max = 0; k_max <= PDA_POOL_CHUNKS_PER_WARP; ++k_max)
        if (!check(W, NW, k_max)) return 1;
    }
    for (int i = 0; i < 300; ++i)
      if (!check(rand_in(1, 5000000), NW, rand_in(0, PDA_POOL_CHUNKS_PER_WARP))) return 1;
  }
  std::printf("ok\n");
  return 0;
}
