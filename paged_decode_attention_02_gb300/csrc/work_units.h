// work_units.h -- how one attention launch cuts its tile list into units of work: each
// warp's static share, and the pool chunks that warps claim at run time. Host and device
// code both use it (the launch plan sizes the workspace's piece slots from it; a host test
// checks its arithmetic).
#pragma once

#if defined(__CUDACC__)
#define PDA_HD __host__ __device__ __forceinline__
#else
#define PDA_HD inline
#endif

namespace pda {

#ifndef PDA_POOL_PCT
#define PDA_POOL_PCT 10          // share of each warp's range left to claimed chunks
#endif
#ifndef PDA_POOL_CHUNKS_PER_WARP
#define PDA_POOL_CHUNKS_PER_WARP 2  // chunks each warp's pooled share is cut into (at most)
#endif
#ifndef PDA_POOL_FIRST_CHUNK_PCT
#define PDA_POOL_FIRST_CHUNK_PCT 50  // share of a warp's pooled tiles in its first chunk (k = 2)
#endif
constexpr int kMinChunkTiles = 4;  // a pool chunk is at least about this many tiles

// Work units over the tile list. Warp w's range [a_w, a_{w+1}) (an equal split of the W
// tiles over the NW warps) is cut into its static share [a_w, m_w), which warp w runs
// itself, and k chunks of the remaining PDA_POOL_PCT percent, which any warp may claim once
// its own static share is done. SMs stream at different rates (whole groups of them
// consistently slower than the rest), and an equal static split ends with the slowest; the
// claimed chunks move the last tenth of the work to the SMs that are ahead. Keeping each
// chunk beside its warp's static share cuts a long (request, kv-head) segment into a few
// pieces more, not into hundreds as a pool at the end of the list would. Units are numbered
// in tile order (u = w (k + 1) + j: j = 0 the static share, j = 1..k the chunks), so the
// pieces of a segment are merged in the same order whichever warp ran each chunk, and
// results do not depend on timing. With k = 0 the units are the plain equal split.
struct Units {
  int W, NW, k;
  int q, r;       // W = q NW + r
  float per_inv;  // NW / W, for a first guess of a tile's warp
  // a(w): first tile of warp w's range, floor(w W / NW) (w r < NW^2 < 2^32)
  PDA_HD int a(int w) const {
    return w * q + static_cast<int>((static_cast<unsigned>(w) * static_cast<unsigned>(r)) /
                                    static_cast<unsigned>(NW));
  }
  // m_w: end of warp w's static share
  PDA_HD static int m_of(int aw, int aw1) {
    return aw + static_cast<int>((static_cast<long long>(aw1 - aw) * (100 - PDA_POOL_PCT)) / 100);
  }
  PDA_HD int units() const { return NW * (k + 1); }
  PDA_HD int start(int u) const {
    if (k == 0) return a(u);
    const int w = k == 1 ? (u >> 1) : u / 3, j = u - w * (k + 1);
    const int aw = a(w);
    if (j == 0) return aw;
    const int aw1 = a(w + 1), mw = m_of(aw, aw1);
    return j == 1 ? mw : mid(mw, aw1);
  }
  // end of the first chunk of a warp whose pooled tiles are [mw, aw1) (k = 2)
  PDA_HD static int mid(int mw, int aw1) {
    return mw + static_cast<int>((static_cast<long long>(aw1 - mw) * PDA_POOL_FIRST_CHUNK_PCT) /
                                 100);
  }
  // the warp whose range holds tile t: the largest w with a(w) <= t
  PDA_HD int warp_of(int t) const {
    int w = static_cast<int>(static_cast<float>(t) * per_inv);
    w = w < 0 ? 0 : (w >= NW ? NW - 1 : w);
    while (w + 1 < NW && a(w + 1) <= t) ++w;
    while (w > 0 && a(w) > t) --w;
    return w;
  }
  // the unit whose range holds tile t
  PDA_HD int owner(int t) const {
    const int w = warp_of(t);
    if (k == 0) return w;
    const int aw1 = a(w + 1), mw = m_of(a(w), aw1);
    if (t < mw) return w * (k + 1);
    if (k == 1) return 2 * w + 1;
    return 3 * w + (t < mid(mw, aw1) ? 1 : 2);
  }
  PDA_HD bool live(int u) const { return start(u) != start(u + 1); }
  // Pool chunk g (claim order) -> its unit: first chunk 1 of every warp, then chunk 2, ...
  PDA_HD int chunk_unit(int g) const {
    return (g % NW) * (k + 1) + 1 + g / NW;
  }
};
static_assert(PDA_POOL_CHUNKS_PER_WARP >= 0 && PDA_POOL_CHUNKS_PER_WARP <= 2,
              "Units cuts a warp's pooled share into at most two chunks");

// The units of W tiles over NW warps, with at most k_max chunks per warp (0: all static).
// Chunks stay at least kMinChunkTiles tiles, so short launches keep the plain split.
PDA_HD Units make_units(int W, int NW, int k_max) {
  int k = 0;  // stays a compile-time 0 where k_max is one (the tensor-core steps)
  if (k_max > 0) {
    const long long kc = (static_cast<long long>(W) * PDA_POOL_PCT) /
                         (100ll * NW * kMinChunkTiles);
    k = kc < k_max ? static_cast<int>(kc) : k_max;
  }
  return Units{W, NW, k, W / NW, W % NW,
               W > 0 ? static_cast<float>(NW) / static_cast<float>(W) : 0.f};
}

}  // namespace pda
