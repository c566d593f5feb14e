// decode_attention.cu -- batched single-query attention over a paged KV cache, sm_103a.
//
// What it computes: for each request b and query head h (kv-head k = h / G, G = H / H_kv),
//   out[b,h] = sum_t softmax_t(scale * q[b,h] . K_t[k]) V_t[k],  t < context_lens[b],
// with token t in physical block block_tables[b][t / 16], row t % 16. Decode reads the
// whole cached history each step (page "Disaggregated LLM Serving: from PD disaggregation
// to attention offload", sec. 1 and sec. 6.1); the history is paged (page "From
// PagedAttention to Prefill-Decode disaggregation", sec. 2.2).
//
// How (GB300 design):
//  * Unit of work = one tile = one physical block (16 tokens) of one kv-head: 16 rows of
//    D elements for K and for V. Tiles are numbered request-major, then kv-head, then
//    block, so the tiles of one (request, kv-head) "segment" are consecutive.
//  * The total tile count is split evenly over all warps of a persistent grid (one block
//    per SM, at most sm_cap SMs). Each warp is an independent worker: it streams its tile
//    range through its own ring of shared-memory stages filled by TMA (3-D tiled
//    cp.async.bulk.tensor for the K and V rows, a 1-D bulk copy for the segment's q rows),
//    each stage guarded by an mbarrier. There is no block-wide synchronisation in the loop.
//  * The G query heads that share a kv-head are processed together, so each K/V byte is
//    read from HBM once (GQA).
//  * Scores use fp32 FMAs; the partial dot products of a lane group are summed with a
//    shuffle reduce-scatter, which leaves each lane owning a few complete (head, token)
//    scores. Softmax is online, in base 2 (q is pre-scaled by scale * log2 e).
//  * A segment that lies wholly inside one worker's range is normalised and written
//    directly. A segment cut by a range boundary leaves (m, l, o) pieces in the workspace
//    (at most two per worker); the warp that registers a segment's last piece merges them
//    with a log-sum-exp combine, so no second kernel is needed. This is the split and merge
//    of Orca's iteration-level batching (page "Disaggregated LLM Serving", sec. 2.1),
//    applied along the sequence.
//  * bf16 and fp32 caches run on the CUDA cores: per kv-head and token this is G dot
//    products of length D against 2 * D * sizeof(elem) bytes, and the bf16 path already
//    streams at the HBM rate. Quantised caches (FP8, NVFP4) at D = 128 carry two to four
//    times as many tokens per byte, so their dot products go to the tensor cores
//    (warp_attn_tc.cuh), mostly on units of two adjacent kv-heads (one TMA box for both);
//    the pipeline, scheduling and merge below are shared and see a pair as one unit with
//    2 G query heads.
#include <math.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <cmath>
#include <mutex>
#include <utility>
#include <vector>

#include "pda_device.cuh"
#include "pda_internal.h"
#include "warp_attn_tc.cuh"
#include "work_units.h"

namespace pda {

#ifndef PDA_ATTN_WARPS
#define PDA_ATTN_WARPS 12     // preferred warps (workers) per block
#endif
#ifndef PDA_ATTN_MAX_STAGES
#define PDA_ATTN_MAX_STAGES 4  // most pipeline stages per warp
#endif

// A launch uses no more warps than give each at least this many tiles. With fewer, a small
// batch spreads over thousands of warps and every (request, kv-head) segment is cut into
// dozens of pieces for its merge to read back: one 13B-shape request ran 51 us over 1824
// warps and 31 us at 8 tiles per warp (4 and 16 measured slower).
#ifndef PDA_MIN_TILES_PER_WARP
#define PDA_MIN_TILES_PER_WARP 8
#endif

#ifndef PDA_TC_WARPS
#define PDA_TC_WARPS 12        // warps (workers) per block of the tensor-core tile step
#endif

constexpr int kBS = 16;             // tokens per physical block (box height of the TMA)
constexpr int kMaxWarps = PDA_ATTN_WARPS > PDA_TC_WARPS ? PDA_ATTN_WARPS : PDA_TC_WARPS;
// Warps per block for a GQA group of G: on the CUDA cores the group of 8 keeps 8 warps so
// its 8 heads of q and o stay in registers (up to 255 per thread); the tensor-core tile
// step holds q and o in mma fragments and keeps all warps.
__host__ __device__ constexpr int warps_for_group(int G, bool tc) {
  return tc ? PDA_TC_WARPS : (G >= 8 ? 8 : PDA_ATTN_WARPS);
}
// The two-head tensor-core step holds both heads' q fragments and running state (about 230
// registers). A scheduler's register file (16K) holds three warps only below 171 registers
// each. FP8 runs it with 8 warps (two per scheduler, no spills); NVFP4, whose longer
// dequantisation chains need more warps to hide, with 12 and a few spilled registers
// (measured 9-10 % faster for NVFP4 and 2 % slower for FP8 than the other choice).
#ifndef PDA_TC_PAIR_WARPS_FP8
#define PDA_TC_PAIR_WARPS_FP8 8
#endif
#ifndef PDA_TC_PAIR_WARPS_NVFP4
#define PDA_TC_PAIR_WARPS_NVFP4 12
#endif
static_assert(PDA_TC_PAIR_WARPS_FP8 <= kMaxWarps && PDA_TC_PAIR_WARPS_NVFP4 <= kMaxWarps,
              "per-warp shared arrays are sized for kMaxWarps");
__host__ __device__ constexpr int warps_for_mode(int G, int mode, bool fp4) {
  return mode == 2 ? (fp4 ? PDA_TC_PAIR_WARPS_NVFP4 : PDA_TC_PAIR_WARPS_FP8)
                   : warps_for_group(G, mode != 0);
}
// Stage alignment: the tensor-core step reads TMA tiles written with the 128-byte (FP8) or
// 64-byte (NVFP4) swizzle, whose pattern repeats every 1024 (512) bytes.
__host__ __device__ constexpr int stage_align(bool tc) { return tc ? 1024 : 128; }

// Tile steps (see attn_partial_kernel).
constexpr int kModeCuda = 0;
constexpr int kModeTc = 1;
constexpr int kModeTcPair = 2;
constexpr int kMetaBytesPerWarp = 2 * 32 * 8;  // two groups of 32 (block id, length) pairs
constexpr int kMaxBatch = 8192;     // prefix table size bound (shared memory)
constexpr int kSmemBudget = 226 * 1024;  // dynamic bytes; static shared memory sits on top
constexpr int kMinResidentSmem = 116 * 1024;  // > half an SM: never two blocks per SM

struct AttnParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_o;                    // [2 * units][G][D]   piece outputs (two slots per unit)
  float* ws_ml;                   // [2 * units][G][2]   piece (max, sum)
  unsigned long long* ws_arrive;  // [B * H_kv] piece arrivals (tagged counters, see arrive)
  unsigned long long* ws_claim;   // pool chunks claimed so far (tagged counter)
  unsigned long long call;        // this call's number (48 bits)
  int pool_k;                     // most pool chunks per warp the workspace holds pieces for
  int32_t* error_word;
  float v_scale;                  // value of a stored V element = code * v_scale (1 if plain)
  const uint8_t* k_bscales;       // NVFP4: [blocks, H_kv, 16, D/16] E4M3 block scales
  const uint8_t* v_bscales;
  int B, H, H_kv, num_blocks, max_blocks, max_context_len;
  int block_size;                 // tokens per physical block: 16 << bs_shift
  int bs_shift;                   // log2 of the 16-row tiles per physical block
  int out_kind;                   // output type: 0 fp32, 1 bf16, 2 fp16
  float scale_log2;
  int num_workers;
  int stages;
  uint32_t stage_bytes;   // one stage: K tile, V tile, q slot
  uint32_t prefix_bytes;  // shared bytes reserved for the prefix table
};

// Reduce-scatter over the lanes of one row group: n values per lane, xor masks from
// `mask` down to 1. While n > 1 every lane keeps the lower half of its values and adds the
// partner's upper half; once one value is left the remaining steps are plain butterflies.
// This leaves each lane with complete sums only because every lane stores its values in a
// lane-dependent order (see WarpAttn::init): local index u holds real index u ^ idx0, so a
// lane's lower half is exactly the half its partner sends it.
template <int n, int mask>
struct ReduceScatter {
  static __device__ __forceinline__ void run(float* v) {
    if constexpr (mask == 0) {
      return;
    } else if constexpr (n > 1) {
#pragma unroll
      for (int i = 0; i < n / 2; ++i) v[i] += __shfl_xor_sync(kFullMask, v[i + n / 2], mask);
      ReduceScatter<n / 2, mask / 2>::run(v);
    } else {
      v[0] += __shfl_xor_sync(kFullMask, v[0], mask);
      ReduceScatter<1, mask / 2>::run(v);
    }
  }
};

template <typename KV, typename QT, int D, int G>
struct Geometry {
  using E = Elem<KV>;
  static constexpr int VEC = E::kVec;               // elements per lane per row (16 bytes)
  static constexpr int LPR = D / VEC;               // lanes covering one row
  static constexpr int RPW = 32 / LPR;              // rows a warp covers per step
  static constexpr int TPL = kBS / RPW;             // token slots per lane per tile
  static constexpr int N = G * TPL;                 // partial dots per lane per tile
  static constexpr int C = N >= LPR ? N / LPR : 1;  // complete scores per lane
  static constexpr int DUP = N >= LPR ? 1 : LPR / N;  // lanes holding the same score
  static constexpr int LPH = N >= LPR ? LPR / G : LPR;  // lanes of a row group per head
  // Scores of two token slots share one packed fp32x2 FMA when q fits twice in registers.
  static constexpr bool PAIR_QK = G * VEC <= 32 && TPL % 2 == 0;
  // NVFP4: every row of a tile comes with one E4M3 scale per 16 elements
  static constexpr bool SCALED = std::is_same<KV, nvfp4>::value;
  static constexpr int ROW_SCALES = D / 16;  // scale bytes per row (NVFP4)
  static constexpr uint32_t TILE_BYTES = kBS * D * E::kBits / 8;
  static constexpr uint32_t SCALE_BYTES = SCALED ? kBS * ROW_SCALES : 0;  // per K or V tile
  static constexpr uint32_t Q_BYTES = G * D * sizeof(QT);
  static_assert(32 % LPR == 0 && kBS % RPW == 0, "row geometry");
  static_assert(LPR >= G, "one head per lane after the reduce-scatter");
  static_assert(VEC % 2 == 0, "packed fp32x2 accumulation");
  static_assert(TILE_BYTES % 128 == 0 && Q_BYTES % 16 == 0, "smem alignment");
  static_assert(!SCALED || (VEC <= 16 && 16 % VEC == 0), "a lane's dims share one scale");
};

// Per-warp online-softmax state and tile arithmetic.
//
// Lane layout: lane = rw * LPR + cl; the lane covers dims [cl*VEC, cl*VEC + VEC) of the
// rows rw, rw + RPW, ... (token slot i is row rw + RPW * i of the 16-row tile). Each lane
// forms N = G * TPL partial dot products (head j, slot i; real index j * TPL + i), sums
// them with the other lanes of its row group by a reduce-scatter, and is left with C
// complete scores of one head: real indices idx0 .. idx0 + C - 1.
template <typename KV, typename QT, int D, int G>
struct WarpAttn {
  using Geo = Geometry<KV, QT, D, G>;
  using E = typename Geo::E;
  static constexpr int VEC = Geo::VEC, LPR = Geo::LPR, RPW = Geo::RPW, TPL = Geo::TPL;
  static constexpr int N = Geo::N, C = Geo::C, DUP = Geo::DUP, LPH = Geo::LPH;
  static constexpr bool PAIR_QK = Geo::PAIR_QK;
  static constexpr bool SCALED = Geo::SCALED;
  static constexpr int ROW_SCALES = Geo::ROW_SCALES;

  int lane, rw, cl, idx0;
  int sblk;                      // NVFP4: index of this lane's 16-element block in a row
  int srow[SCALED ? TPL : 1];    // NVFP4: scale offset of the K row behind local slot il
  int hp;             // local head jl holds real head jl ^ hp
  int krow[TPL];      // element offset of the K row behind local slot il (real slot il ^ tp)
  float2 q2[PAIR_QK ? G : 1][PAIR_QK ? VEC : 1];  // q (scaled), duplicated, local head order
  float qs[PAIR_QK ? 1 : G][PAIR_QK ? 1 : VEC];   // q (scaled), local head order
  float2 o2[G][VEC / 2];  // unnormalised output, real head order, dims pairs
  float m_own;  // running max of this lane's head (log2 domain)
  float l_own;  // this lane's share of the running sum of its head

  __device__ __forceinline__ void init(int lane_) {
    lane = lane_;
    rw = lane / LPR;
    cl = lane % LPR;
    idx0 = (cl / DUP) * C;
    hp = idx0 / TPL;
    const int tp = idx0 % TPL;
#pragma unroll
    for (int il = 0; il < TPL; ++il) krow[il] = (rw + RPW * (il ^ tp)) * D + cl * VEC;
    sblk = (cl * VEC) / 16;
    if constexpr (SCALED) {
#pragma unroll
      for (int il = 0; il < TPL; ++il) srow[il] = (rw + RPW * (il ^ tp)) * ROW_SCALES + sblk;
    }
  }

  __device__ __forceinline__ void reset(const QT* q_smem, float scale_log2) {
#pragma unroll
    for (int jl = 0; jl < G; ++jl) {
      float t[VEC];
      load_elems<QT, VEC>(q_smem + (jl ^ hp) * D + cl * VEC, t);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        const float qv = t[e] * scale_log2;
        if constexpr (PAIR_QK)
          q2[jl][e] = make_float2(qv, qv);
        else
          qs[jl][e] = qv;
      }
    }
#pragma unroll
    for (int j = 0; j < G; ++j)
#pragma unroll
      for (int e = 0; e < VEC / 2; ++e) o2[j][e] = make_float2(0.f, 0.f);
    m_own = -INFINITY;
    l_own = 0.f;
  }

  // ksc/vsc: the tile's NVFP4 block scales ([16 rows][D/16] E4M3 bytes), unused otherwise.
  template <bool kPartial>
  __device__ __forceinline__ void tile(const KV* ks, const KV* vs, const uint8_t* ksc,
                                       const uint8_t* vsc, int n_valid) {
    // ---- scores: part[jl * TPL + il] = q(real head jl ^ hp) . K(real slot il ^ tp)
    float part[N];
    if constexpr (PAIR_QK) {
#pragma unroll
      for (int m = 0; m < TPL / 2; ++m) {
        float k0[VEC], k1[VEC];
        E::load(elem_ptr<KV>(ks, krow[2 * m]), k0);
        E::load(elem_ptr<KV>(ks, krow[2 * m + 1]), k1);
        float2 sk = make_float2(1.f, 1.f);
        if constexpr (SCALED)
          sk = make_float2(e4m3_to_f32(ksc[srow[2 * m]]), e4m3_to_f32(ksc[srow[2 * m + 1]]));
#pragma unroll
        for (int jl = 0; jl < G; ++jl) {
          float2 acc = __fmul2_rn(q2[jl][0], make_float2(k0[0], k1[0]));
#pragma unroll
          for (int e = 1; e < VEC; ++e)
            acc = __ffma2_rn(q2[jl][e], make_float2(k0[e], k1[e]), acc);
          if constexpr (SCALED) acc = __fmul2_rn(acc, sk);
          part[jl * TPL + 2 * m] = acc.x;
          part[jl * TPL + 2 * m + 1] = acc.y;
        }
      }
    } else {
#pragma unroll
      for (int il = 0; il < TPL; ++il) {
        float k[VEC];
        E::load(elem_ptr<KV>(ks, krow[il]), k);
        float sk = 1.f;
        if constexpr (SCALED) sk = e4m3_to_f32(ksc[srow[il]]);
#pragma unroll
        for (int jl = 0; jl < G; ++jl) {
          float acc = qs[jl][0] * k[0];
#pragma unroll
          for (int e = 1; e < VEC; ++e) acc = fmaf(qs[jl][e], k[e], acc);
          part[jl * TPL + il] = SCALED ? acc * sk : acc;
        }
      }
    }
    ReduceScatter<N, LPR / 2>::run(part);

    // part[0..C) are now complete scores of real index idx0 + r: head (idx0 + r) / TPL,
    // slot (idx0 + r) % TPL.
    float tmax = -INFINITY;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      if (kPartial) {
        const int t = rw + RPW * ((idx0 + r) % TPL);
        if (t >= n_valid) part[r] = -INFINITY;
      }
      tmax = fmaxf(tmax, part[r]);
    }
    // lanes cl and cl ^ m for m < DUP hold the same scores, so the max skips those masks
#pragma unroll
    for (int mask = LPH / 2; mask >= DUP; mask >>= 1)
      tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, mask));
#pragma unroll
    for (int mask = LPR; mask < 32; mask <<= 1)
      tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, mask));

    const float m_new = fmaxf(m_own, tmax);
    const float alpha = ex2(m_own - m_new);
    m_own = m_new;
    float psum = 0.f;
#pragma unroll
    for (int r = 0; r < C; ++r) {
      part[r] = ex2(part[r] - m_new);
      psum += part[r];
    }
    l_own = l_own * alpha + ((cl % DUP) == 0 ? psum : 0.f);
#pragma unroll
    for (int j = 0; j < G; ++j) {
      const float a = (G == 1) ? alpha : __shfl_sync(kFullMask, alpha, j * LPH);
      const float2 a2 = make_float2(a, a);
#pragma unroll
      for (int e = 0; e < VEC / 2; ++e) o2[j][e] = __fmul2_rn(o2[j][e], a2);
    }

    // ---- o[j] += p(j, slot i) * V(row of slot i), real order
#pragma unroll
    for (int i = 0; i < TPL; ++i) {
      const int t = rw + RPW * i;
      float v[VEC];
      E::load(elem_ptr<KV>(vs, t * D + cl * VEC), v);
      float sv = 1.f;  // NVFP4: this lane's block scale of row t, folded into p
      if constexpr (SCALED) sv = e4m3_to_f32(vsc[t * ROW_SCALES + sblk]);
      if (kPartial && t >= n_valid) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = 0.f;
        sv = 0.f;
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int idx = j * TPL + i;
        const int src = rw * LPR + (idx / C) * DUP;
        float p = __shfl_sync(kFullMask, part[idx % C], src);
        if constexpr (SCALED) p *= sv;
        const float2 p2 = make_float2(p, p);
#pragma unroll
        for (int e = 0; e < VEC / 2; ++e)
          o2[j][e] = __ffma2_rn(p2, make_float2(v[2 * e], v[2 * e + 1]), o2[j][e]);
      }
    }
  }

  // Sums the state over lanes; afterwards lanes of row group 0 hold, for every head j,
  // o[j] over their dims, and lj[j], mj[j] on every lane.
  __device__ __forceinline__ void reduce(float* lj, float* mj) {
    float l = l_own;
#pragma unroll
    for (int mask = LPH / 2; mask >= 1; mask >>= 1) l += __shfl_xor_sync(kFullMask, l, mask);
#pragma unroll
    for (int mask = LPR; mask < 32; mask <<= 1) l += __shfl_xor_sync(kFullMask, l, mask);
#pragma unroll
    for (int j = 0; j < G; ++j) {
#pragma unroll
      for (int e = 0; e < VEC / 2; ++e)
#pragma unroll
        for (int mask = LPR; mask < 32; mask <<= 1) {
          o2[j][e].x += __shfl_xor_sync(kFullMask, o2[j][e].x, mask);
          o2[j][e].y += __shfl_xor_sync(kFullMask, o2[j][e].y, mask);
        }
      lj[j] = __shfl_sync(kFullMask, l, j * LPH);
      mj[j] = __shfl_sync(kFullMask, m_own, j * LPH);
    }
  }

  __device__ __forceinline__ float o(int j, int e) const {
    return (e & 1) ? o2[j][e >> 1].y : o2[j][e >> 1].x;
  }

  // Calls f(head, d, values, VEC, l of the head) for each run of output elements this lane
  // writes (lanes of row group 0 hold the reduced state); lj as filled by reduce().
  template <typename F>
  __device__ __forceinline__ void for_each_out(const float* lj, F&& f) const {
    if (rw != 0) return;
#pragma unroll
    for (int j = 0; j < G; ++j) {
      float v[VEC];
#pragma unroll
      for (int e = 0; e < VEC; ++e) v[e] = o(j, e);
      f(j, cl * VEC, v, VEC, lj[j]);
    }
  }
  __device__ __forceinline__ bool writes_ml(int lane_) const { return lane_ == 0; }
};

// n fp32 values (n = 2 or a multiple of 4, p aligned to n * 4 bytes up to 16).
__device__ __forceinline__ void store_f32(float* p, const float* v, int n) {
  if (n == 2) {
    *reinterpret_cast<float2*>(p) = make_float2(v[0], v[1]);
    return;
  }
  for (int e = 0; e < n; e += 4)
    *reinterpret_cast<float4*>(p + e) = make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]);
}

// Output kinds (AttnParams::out_kind).
constexpr int kOutF32 = 0;
constexpr int kOutBF16 = 1;
constexpr int kOutF16 = 2;

__device__ __forceinline__ void store_one(void* out, size_t off, float v, int kind) {
  if (kind == kOutBF16)
    reinterpret_cast<__nv_bfloat16*>(out)[off] = __float2bfloat16_rn(v);
  else if (kind == kOutF16)
    reinterpret_cast<__half*>(out)[off] = __float2half_rn(v);
  else
    reinterpret_cast<float*>(out)[off] = v;
}

__device__ __forceinline__ void store_out(void* out, size_t off, const float* v, int n,
                                          int kind) {
  if (kind == kOutF16) {
    __half* p = reinterpret_cast<__half*>(out) + off;
    if (n % 2 == 0) {
      for (int e = 0; e < n; e += 2)
        *reinterpret_cast<__half2*>(p + e) = __floats2half2_rn(v[e], v[e + 1]);
    } else {
      for (int e = 0; e < n; ++e) p[e] = __float2half_rn(v[e]);
    }
  } else if (kind == kOutBF16) {
    __nv_bfloat16* p = reinterpret_cast<__nv_bfloat16*>(out) + off;
    if (n == 2) {
      *reinterpret_cast<__nv_bfloat162*>(p) = __floats2bfloat162_rn(v[0], v[1]);
    } else if (n == 8) {
      uint4 w;
      __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]);
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2], v[3]);
      __nv_bfloat162 c = __floats2bfloat162_rn(v[4], v[5]);
      __nv_bfloat162 d = __floats2bfloat162_rn(v[6], v[7]);
      w.x = *reinterpret_cast<uint32_t*>(&a);
      w.y = *reinterpret_cast<uint32_t*>(&b);
      w.z = *reinterpret_cast<uint32_t*>(&c);
      w.w = *reinterpret_cast<uint32_t*>(&d);
      *reinterpret_cast<uint4*>(p) = w;
    } else {
      for (int e = 0; e < n; ++e) p[e] = __float2bfloat16_rn(v[e]);
    }
  } else {
    store_f32(reinterpret_cast<float*>(out) + off, v, n);
  }
}

// Arrival counters hold ((call number << 16) | count) ^ kTagMix. A counter written by an
// earlier call (or one that was aborted) carries another call number and counts as 0. The
// mix keeps other data from passing for a live counter: a workspace reused for calls of
// other shapes holds fp32 partial results where this call's counters lie, and zeros or
// small values there would otherwise read as the tag of one of the first calls.
constexpr unsigned long long kTagMix = 0xa5c396e17b2d0000ull;

__device__ __forceinline__ unsigned long long arrival_reset(unsigned long long call) {
  return (call << 16) ^ kTagMix;
}

// Registers one more piece of a segment and returns how many pieces of it this call has
// registered so far.
__device__ __forceinline__ unsigned arrive(unsigned long long* counter,
                                           unsigned long long call) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(counter);
  while (true) {
    const unsigned long long cur = old ^ kTagMix;
    const unsigned long long next = ((cur >> 16) == call) ? cur + 1 : ((call << 16) | 1ull);
    const unsigned long long seen = atomicCAS(counter, old, next ^ kTagMix);
    if (seen == old) return static_cast<unsigned>(next & 0xffffull);
    old = seen;
  }
}

// Makes the pool's claim counter this call's, with nothing claimed yet, unless it already is
// (a counter of another call, or one never written, is replaced). Each warp does this once,
// before its first claim.
__device__ __forceinline__ void register_claims(unsigned long long* c, unsigned long long call) {
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(c);
  while (((old ^ kTagMix) >> 16) != call) {
    const unsigned long long seen = atomicCAS(c, old, arrival_reset(call));
    if (seen == old) return;
    old = seen;
  }
}

// Claims the next pool chunk and returns its index (NW k or more once the pool is used up).
// The tag mix leaves the low 16 bits alone, so the count adds without unmixing; a call makes
// at most NW k + NW claims, below 2^16.
__device__ __forceinline__ unsigned claim_chunk(unsigned long long* c) {
  return static_cast<unsigned>(atomicAdd(c, 1ull) & 0xffffull);
}

// Log-sum-exp merge of the pieces of one segment (request b, kv-head h) into out, done by
// the warp that registered the segment's last piece. Pieces come from units w0..w1 (the
// first may hold it as its tail piece); empty units hold none. For each head j:
//   M = max m_i,  L = sum l_i 2^(m_i - M),  out = sum o_i 2^(m_i - M) / L.
// All heads are merged together so the loads of one pass are in flight at once: lane i
// reads piece i's (m, l) of every head, then lanes stream the pieces' o rows. Pieces are
// read from L2 (ld.cg): other SMs wrote them during this launch.
template <int D, int G, int HP>
__device__ __forceinline__ void merge_heads(const AttnParams& p, int b, int h, int j0, int w0,
                                            int w1, bool w0_tail, const Units un, int lane) {
  constexpr int PER = D / 32;
  auto slot_of = [&](int w) { return 2 * w + ((w == w0 && w0_tail) ? 1 : 0); };
  const float* ml = p.ws_ml;
  // pass 1: M[j] over all pieces (lane i looks at unit w0 + i, w0 + i + 32, ...)
  float M[HP];
#pragma unroll
  for (int j = 0; j < HP; ++j) M[j] = -INFINITY;
  for (int w = w0 + lane; w <= w1; w += 32) {
    if (!un.live(w)) continue;
    const float2* mlw =
        reinterpret_cast<const float2*>(ml) + static_cast<size_t>(slot_of(w)) * G + j0;
#pragma unroll
    for (int j = 0; j < HP; ++j) M[j] = fmaxf(M[j], __ldcg(mlw + j).x);
  }
#pragma unroll
  for (int j = 0; j < HP; ++j)
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) M[j] = fmaxf(M[j], __shfl_xor_sync(kFullMask, M[j], m));

  // pass 2: weights, L[j], and the weighted o rows
  float acc[HP][PER], Lsum[HP];
#pragma unroll
  for (int j = 0; j < HP; ++j) {
    Lsum[j] = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[j][e] = 0.f;
  }
  for (int base = w0; base <= w1; base += 32) {
    const int w = base + lane;
    float f[HP];
#pragma unroll
    for (int j = 0; j < HP; ++j) f[j] = 0.f;
    const bool mine = w <= w1 && un.live(w);
    const unsigned live_mask = __ballot_sync(kFullMask, mine);  // bit i: unit base + i
    if (mine) {
      const float2* mlw =
          reinterpret_cast<const float2*>(ml) + static_cast<size_t>(slot_of(w)) * G + j0;
#pragma unroll
      for (int j = 0; j < HP; ++j) {
        const float2 v = __ldcg(mlw + j);
        f[j] = ex2(v.x - M[j]);
        Lsum[j] += v.y * f[j];
      }
    }
    // The live pieces of this group of 32 units, U rows in flight at once (each load is an L2
    // round trip), in increasing unit order. Empty units are skipped outright: a launch with
    // fewer tiles than warps leaves most units empty, and a segment's range of units can
    // hold hundreds of them. A missing slot of the last batch reads piece w0's row (always
    // written: w0 holds the segment's first tile) and is left out of the sum by its flag, not
    // by a zero weight (its row may hold NaN).
    constexpr int U = HP * PER <= 4 ? 4 : 1;  // wider would spill in the kernels with G >= 2
    unsigned rest = live_mask;  // the same on every lane
    while (rest != 0u) {
      float v[U][HP][PER];
      float fu[U][HP];
      bool use[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        use[u] = rest != 0u;
        const int i = use[u] ? __ffs(rest) - 1 : 0;
        rest &= rest - 1u;  // no-op once empty
        const float* row =
            p.ws_o + (static_cast<size_t>(slot_of(use[u] ? base + i : w0)) * G + j0) * D;
#pragma unroll
        for (int j = 0; j < HP; ++j) {
          fu[u][j] = __shfl_sync(kFullMask, f[j], i);
#pragma unroll
          for (int e = 0; e < PER; ++e) v[u][j][e] = __ldcg(row + j * D + lane + 32 * e);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (!use[u]) continue;
#pragma unroll
        for (int j = 0; j < HP; ++j)
#pragma unroll
          for (int e = 0; e < PER; ++e) acc[j][e] = fmaf(v[u][j][e], fu[u][j], acc[j][e]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < HP; ++j) {
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) Lsum[j] += __shfl_xor_sync(kFullMask, Lsum[j], m);
    const size_t row = (static_cast<size_t>(b) * p.H + static_cast<size_t>(h) * G + j0 + j) * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      const float v = acc[j][e] * (p.v_scale / Lsum[j]);
      store_one(p.out, row + lane + 32 * e, v, p.out_kind);
    }
  }
}

// Merges all G heads of a segment, at most four heads per pass (register budget).
template <int D, int G>
__device__ void merge_segment(const AttnParams& p, int b, int h, int w0, int w1, bool w0_tail,
                              const Units un, int lane) {
  constexpr int HP = G < 4 ? G : 4;
#pragma unroll 1
  for (int j0 = 0; j0 < G; j0 += HP)
    merge_heads<D, G, HP>(p, b, h, j0, w0, w1, w0_tail, un, lane);
}

// MODE selects the tile step: kModeCuda (CUDA cores), kModeTc (tensor cores, one kv-head
// per tile) or kModeTcPair (tensor cores, two adjacent kv-heads per tile, loaded by one
// 4-D TMA box). G is the unit's query heads: the kv-head's G, or 2 G for a pair; p.H_kv
// counts units (kv-heads, or pairs).
template <typename KV, typename QT, int D, int G, int MODE>
__global__ void __launch_bounds__(warps_for_mode(G, MODE, std::is_same<KV, nvfp4>::value) * 32,
                                  1)
    attn_partial_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  constexpr bool TC = MODE != kModeCuda;
  using Geo = Geometry<KV, QT, D, G>;
  using W = std::conditional_t<
      MODE == kModeCuda, WarpAttn<KV, QT, D, G>,
      std::conditional_t<MODE == kModeTc, WarpAttnTC<KV, D, G>, WarpAttnTCPair<KV, D, G / 2>>>;
  // a unit's tile: one head tile, or a pair's two head tiles back to back
  constexpr int kHeads = MODE == kModeTcPair ? 2 : 1;
  constexpr uint32_t kTile = kHeads * Geo::TILE_BYTES;
  constexpr uint32_t kScales = kHeads * Geo::SCALE_BYTES;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  // The host reserves stage_align(TC) - 128 spare bytes; the layout starts at the first
  // aligned address (swizzled TMA tiles need the swizzle period's alignment).
  constexpr uint32_t kAlign = stage_align(TC);
  unsigned char* smem =
      smem_raw + ((kAlign - (smem_addr(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  if ((smem_addr(smem_raw) & 127u) != 0) {  // TMA destinations assume 128-byte alignment
    if (threadIdx.x == 0) atomic_or_error(p.error_word, PDA_DEVERR_TIMEOUT);
    return;
  }

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int B = p.B;

  // ---- shared layout: prefix table | stage buffers | barriers | stage info words
  int32_t* s_pre = reinterpret_cast<int32_t*>(smem);
  unsigned char* s_stage = smem + p.prefix_bytes;
  const size_t stage_region = static_cast<size_t>(nwarps) * p.stages * p.stage_bytes;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(s_stage + stage_region);
  int32_t* s_info = reinterpret_cast<int32_t*>(s_bar + nwarps * p.stages);
  int2* s_meta = reinterpret_cast<int2*>(
      (reinterpret_cast<uintptr_t>(s_info + nwarps * p.stages) + 7) & ~uintptr_t(7));

  // The tensor maps' descriptors are fetched while the prologue below reads the lengths.
  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }

  // ---- 1. block prefix sums of per-request tile counts (every block computes its own)
  const int cap_tokens = min(p.max_blocks * p.block_size, p.max_context_len);
  {
    const int per = (B + blockDim.x - 1) / blockDim.x;
    const int lo = min(B, tid * per), hi = min(B, lo + per);
    int local = 0;
    for (int b = lo; b < hi; ++b) {
      const int L = p.context_lens[b];
      const bool ok = L >= 0 && L <= cap_tokens;
      local += ok ? (L + kBS - 1) / kBS : 0;
    }
    // block-wide exclusive scan of `local`
    int incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(kFullMask, incl, d);
      if (lane >= d) incl += y;
    }
    __shared__ int warp_tot[kMaxWarps];
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += warp_tot[w];
    int run = base + incl - local;
    for (int b = lo; b < hi; ++b) {
      s_pre[b] = run;
      const int L = p.context_lens[b];
      const bool ok = L >= 0 && L <= cap_tokens;
      run += ok ? (L + kBS - 1) / kBS : 0;
    }
    if (tid == blockDim.x - 1) s_pre[B] = run;
  }
  // barrier init (one lane per warp, its own stages)
  if (lane == 0) {
    // one arrive carries the byte count of the stage's copies
    for (int s = 0; s < p.stages; ++s) mbar_init(&s_bar[warp * p.stages + s], 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- 2. rows that get no tiles: empty histories (zeros) and invalid lengths (NaN)
  for (int b = blockIdx.x; b < B; b += gridDim.x) {
    if (s_pre[b + 1] != s_pre[b]) continue;
    const int L = p.context_lens[b];
    const bool bad = !(L >= 0 && L <= cap_tokens);
    if (bad && tid == 0) atomic_or_error(p.error_word, PDA_DEVERR_CONTEXT_LEN);
    const float val = bad ? __int_as_float(0x7fc00000) : 0.f;
    for (int i = tid; i < p.H * D; i += blockDim.x) {
      const size_t off = static_cast<size_t>(b) * p.H * D + i;
      store_one(p.out, off, val, p.out_kind);
    }
  }

  // ---- 3. this warp's work: its static unit, then pool chunks while any are left
  const int H_kv = p.H_kv;
  const int W_tiles = s_pre[B] * H_kv;
  // Workers: the grid's warps, but no more than give each PDA_MIN_TILES_PER_WARP tiles of
  // this launch (the host sized the grid by its bound on the lengths; the lengths on the
  // device may be shorter). The others leave here. Only the CUDA-core step leaves a pool
  // (see make_plan); the tensor-core steps compile without it.
  const int nw = max(1, min(p.num_workers,
                            (W_tiles + PDA_MIN_TILES_PER_WARP - 1) / PDA_MIN_TILES_PER_WARP));
  const int wi = blockIdx.x * nwarps + warp;
  if (wi >= nw) return;
  const Units un = make_units(W_tiles, nw, MODE == kModeCuda ? p.pool_k : 0);
  const int w = wi * (un.k + 1);  // this warp's static unit
  if (un.k == 0 && !un.live(w)) return;

  unsigned char* my_stage = s_stage + static_cast<size_t>(warp) * p.stages * p.stage_bytes;
  uint64_t* my_bar = s_bar + warp * p.stages;
  int32_t* my_info = s_info + warp * p.stages;
  auto k_buf = [&](int s) { return reinterpret_cast<KV*>(my_stage + s * p.stage_bytes); };
  auto v_buf = [&](int s) {
    return reinterpret_cast<KV*>(my_stage + s * p.stage_bytes + kTile);
  };
  auto ks_buf = [&](int s) {  // NVFP4 block scales of the K tile, [kHeads][16][D/16]
    return reinterpret_cast<uint8_t*>(my_stage + s * p.stage_bytes + 2 * kTile);
  };
  auto vs_buf = [&](int s) {
    return reinterpret_cast<uint8_t*>(my_stage + s * p.stage_bytes + 2 * kTile + kScales);
  };
  auto q_buf = [&](int s) {
    return reinterpret_cast<QT*>(my_stage + s * p.stage_bytes + 2 * kTile + 2 * kScales);
  };

  // (request, kv-head, block) of tile y
  auto locate = [&](int y, int& b, int& h, int& blk, int& nb) {
    int lo = 0, hi = B;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_pre[mid] * H_kv <= y) lo = mid; else hi = mid;
    }
    b = lo;
    nb = s_pre[b + 1] - s_pre[b];
    const int rem = y - s_pre[b] * H_kv;
    h = rem / nb;
    blk = rem - h * nb;
  };

  const uint64_t policy = l2_policy_evict_first();
  int2* my_meta = s_meta + warp * 64;
  const int S = p.stages;
  // The stage ring persists across units: every tile a unit loads is consumed within it, so
  // the next unit starts on the stage (and phase) after the last one used.
  int stage = 0;
  uint32_t phase = 0;
  W st;
  st.init(lane);
  bool registered = false;

  // Runs tiles [t_begin, t_end) as unit `unit`. When claim_next is set, lane 0 claims the
  // next pool chunk as soon as the range has no more tiles to load (the atomic's latency
  // hides behind the range's last tiles); the claimed index is returned through `claimed`.
  // Returns false after a wait that timed out (the error bit is set).
  auto run = [&](int t_begin, int t_end, int unit, bool claim_next, unsigned& claimed) -> bool {
    // Issue-side metadata, one group of 32 tiles at a time: lane i describes tile
    // g_base + i. The block id and context length of the next group are fetched with
    // cp.async a whole group ahead into this warp's two-slot ring, so the lane that issues a
    // tile never waits on a global load. Each lane reads only the slot it filled itself.
    int g_base = t_begin, g_buf = 0;
    int cur_b = 0, cur_h = 0, cur_blk = 0, cur_pid = 0, cur_len = 0;
    int nxt_b = 0, nxt_h = 0, nxt_blk = 0;
    auto prefetch = [&](int base, int buf) {
      const int y = base + lane;
      if (y < t_end) {
        int nb;
        locate(y, nxt_b, nxt_h, nxt_blk, nb);
        cp_async4(&my_meta[buf * 32 + lane].x, p.block_tables +
                                                       static_cast<size_t>(nxt_b) * p.max_blocks +
                                                       (nxt_blk >> p.bs_shift));
        cp_async4(&my_meta[buf * 32 + lane].y, p.context_lens + nxt_b);
      }
      cp_async_commit();
    };
    auto enter = [&](int base, int buf) {  // the group starting at `base` becomes current
      cp_async_wait_all();
      g_base = base;
      g_buf = buf;
      cur_b = nxt_b;
      cur_h = nxt_h;
      cur_blk = nxt_blk;
      const int2 m = my_meta[buf * 32 + lane];
      cur_pid = m.x;
      cur_len = m.y;
      if (base + 32 < t_end) prefetch(base + 32, buf ^ 1);
    };
    prefetch(t_begin, 0);
    enter(t_begin, 0);
    auto issue = [&](int x, int s) {
      if (x >= g_base + 32) enter(g_base + 32, g_buf ^ 1);
      if (lane == x - g_base) {
        const bool bad = cur_pid < 0 || cur_pid >= p.num_blocks;
        const bool need_q = (cur_blk == 0) || (x == t_begin);
        const int n_valid = min(kBS, cur_len - cur_blk * kBS);
        my_info[s] = n_valid | (bad ? 0x100 : 0);
        if (bad) atomic_or_error(p.error_word, PDA_DEVERR_BLOCK_ID);
        const uint32_t bytes = 2 * kTile + 2 * kScales + (need_q ? Geo::Q_BYTES : 0);
        mbar_arrive_expect_tx(&my_bar[s], bytes);
        // the tile is rows sub * 16 .. + 15 of its physical block
        const int sub = cur_blk & ((1 << p.bs_shift) - 1);
        const int row = (bad ? 0 : cur_pid) * p.block_size + sub * kBS;
        if constexpr (Geo::SCALED) {
          // scales [blocks][heads][block_size][D/16]: each head's 16 rows are one run; with
          // 16-token blocks a pair's two runs are adjacent (one copy)
          constexpr uint32_t kRun = Geo::SCALE_BYTES;  // one head's 16 rows
          const size_t head0 = static_cast<size_t>(bad ? 0 : cur_pid) * H_kv * kHeads +
                               static_cast<size_t>(cur_h) * kHeads;
          const size_t off = (head0 * p.block_size + static_cast<size_t>(sub) * kBS) *
                             Geo::ROW_SCALES;
          if (kHeads == 1 || p.bs_shift == 0) {
            bulk_load(ks_buf(s), p.k_bscales + off, kScales, &my_bar[s]);
            bulk_load(vs_buf(s), p.v_bscales + off, kScales, &my_bar[s]);
          } else {
            const size_t step = static_cast<size_t>(p.block_size) * Geo::ROW_SCALES;
#pragma unroll
            for (int u = 0; u < kHeads; ++u) {
              bulk_load(ks_buf(s) + u * kRun, p.k_bscales + off + u * step, kRun, &my_bar[s]);
              bulk_load(vs_buf(s) + u * kRun, p.v_bscales + off + u * step, kRun, &my_bar[s]);
            }
          }
        }
        if constexpr (MODE == kModeTcPair) {  // both heads of pair cur_h in one box
          tma_load_4d(k_buf(s), &tmK, 0, row, 0, cur_h, &my_bar[s], policy);
          tma_load_4d(v_buf(s), &tmV, 0, row, 0, cur_h, &my_bar[s], policy);
        } else {
          tma_load_3d(k_buf(s), &tmK, 0, cur_h, row, &my_bar[s], policy);
          tma_load_3d(v_buf(s), &tmV, 0, cur_h, row, &my_bar[s], policy);
        }
        if (need_q) {
          const QT* src = reinterpret_cast<const QT*>(p.q) +
                          (static_cast<size_t>(cur_b) * p.H + static_cast<size_t>(cur_h) * G) * D;
          bulk_load(q_buf(s), src, Geo::Q_BYTES, &my_bar[s]);
        }
      }
    };

    const int n_tiles = t_end - t_begin;
    for (int i = 0; i < S && i < n_tiles; ++i) issue(t_begin + i, (stage + i) % S);
    if (claim_next && !registered) {  // overlaps the first loads
      if (lane == 0) register_claims(p.ws_claim, p.call);
      registered = true;
    }
    unsigned next_claim = 0;
    if (claim_next && n_tiles < S && lane == 0) next_claim = claim_chunk(p.ws_claim);

    // Consumer-side sequential position.
    int cb, ch, cblk, cnb;
    locate(t_begin, cb, ch, cblk, cnb);
    bool seg_bad = false;

    for (int x = t_begin; x < t_end; ++x) {
      const bool ready = __all_sync(kFullMask, mbar_wait_bounded(&my_bar[stage], phase));
      if (!ready) {
        atomic_or_error(p.error_word, PDA_DEVERR_TIMEOUT);
        cp_async_wait_all();
        // Give copies still in flight a bounded chance to land before leaving.
        for (int y = x; y < min(t_end, x + S); ++y) {
          const int s2 = (stage + (y - x)) % S;
          const uint32_t ph2 = phase ^ (((stage + (y - x)) / S) & 1);
          mbar_wait_bounded(&my_bar[s2], ph2);
        }
        return false;
      }
      const int info = my_info[stage];
      const int n_valid = info & 0xff;
      if (cblk == 0 || x == t_begin) {
        st.reset(q_buf(stage), p.scale_log2);
        seg_bad = false;
      }
      seg_bad |= (info & 0x100) != 0;
      if (n_valid == kBS)
        st.template tile<false>(k_buf(stage), v_buf(stage), ks_buf(stage), vs_buf(stage),
                                n_valid);
      else
        st.template tile<true>(k_buf(stage), v_buf(stage), ks_buf(stage), vs_buf(stage),
                               n_valid);

      // hand the stage back to the TMA engine
      __syncwarp();
      fence_proxy_async_smem();
      if (x + S < t_end)
        issue(x + S, stage);
      else if (claim_next && x + S == t_end && lane == 0)  // nothing left to load
        next_claim = claim_chunk(p.ws_claim);
      if (++stage == S) {
        stage = 0;
        phase ^= 1;
      }

      // segment end?
      const bool last_of_seg = (cblk + 1 == cnb);
      if (last_of_seg || x + 1 == t_end) {
        float lj[G], mj[G];
        st.reduce(lj, mj);
        const int seg_start = s_pre[cb] * H_kv + ch * cnb;
        const int seg_end = seg_start + cnb;
        const bool complete = seg_start >= t_begin && seg_end <= t_end;
        if (complete) {
          st.for_each_out(lj, [&](int j, int d, const float* o, int n, float l) {
            float v[8];
            const float inv = seg_bad ? __int_as_float(0x7fc00000) : p.v_scale / l;
#pragma unroll
            for (int e = 0; e < 8; ++e)
              if (e < n) v[e] = o[e] * inv;
            const size_t off =
                (static_cast<size_t>(cb) * p.H + static_cast<size_t>(ch) * G + j) * D + d;
            store_out(p.out, off, v, n, p.out_kind);
          });
        } else {
          // A piece of a segment cut by a unit boundary: store (m, l, o), register it, and
          // merge the segment if this was its last piece.
          const int slot = 2 * unit + (seg_start <= t_begin ? 0 : 1);
          st.for_each_out(lj, [&](int j, int d, const float* o, int n, float) {
            store_f32(p.ws_o + (static_cast<size_t>(slot) * G + j) * D + d, o, n);
          });
          if (st.writes_ml(lane)) {
#pragma unroll
            for (int j = 0; j < G; ++j) {
              p.ws_ml[(static_cast<size_t>(slot) * G + j) * 2 + 0] = mj[j];
              p.ws_ml[(static_cast<size_t>(slot) * G + j) * 2 + 1] =
                  seg_bad ? __int_as_float(0x7fc00000) : lj[j];
            }
          }
          __threadfence();  // this lane's piece stores before the arrival below
          __syncwarp();
          const int seg = cb * H_kv + ch;
          unsigned arrived = 0;
          if (lane == 0) arrived = arrive(p.ws_arrive + seg, p.call);
          arrived = __shfl_sync(kFullMask, arrived, 0);
          const int w0 = un.owner(seg_start);
          const int w1 = un.owner(seg_end - 1);
          unsigned pieces = 0;
          for (int wb = w0; wb <= w1; wb += 32) {
            const int ww = wb + lane;
            pieces += __popc(__ballot_sync(kFullMask, ww <= w1 && un.live(ww)));
          }
          if (arrived == pieces) {
            __threadfence();  // see the other pieces' stores
            merge_segment<D, G>(p, cb, ch, w0, w1, seg_start != un.start(w0), un, lane);
            if (lane == 0) atomicExch(p.ws_arrive + seg, arrival_reset(p.call));
          }
        }
      }
      // advance the consumer position
      if (++cblk == cnb) {
        cblk = 0;
        if (++ch == H_kv) {
          ch = 0;
          do {
            ++cb;
          } while (cb < B && s_pre[cb + 1] == s_pre[cb]);
        }
        if (cb < B) cnb = s_pre[cb + 1] - s_pre[cb];
      }
    }
    claimed = __shfl_sync(kFullMask, next_claim, 0);
    return true;
  };

  const bool pool = un.k > 0;
  const unsigned n_chunks = static_cast<unsigned>(un.NW) * un.k;
  unsigned c = 0;
  if (un.live(w)) {
    if (!run(un.start(w), un.start(w + 1), w, pool, c)) return;
  } else if (pool) {
    if (lane == 0) {
      register_claims(p.ws_claim, p.call);
      c = claim_chunk(p.ws_claim);
    }
    registered = true;
    c = __shfl_sync(kFullMask, c, 0);
  }
  // pool chunks, each the next one nobody has taken yet
  while (pool && c < n_chunks) {
    const int u = un.chunk_unit(static_cast<int>(c));
    if (un.live(u)) {
      if (!run(un.start(u), un.start(u + 1), u, true, c)) return;
    } else {
      if (lane == 0) c = claim_chunk(p.ws_claim);
      c = __shfl_sync(kFullMask, c, 0);
    }
  }
}

// ------------------------------------------------------------------ host side
namespace {

struct LaunchPlan {
  int nwarps, stages, grid;
  int pool_k;  // pool chunks per warp the workspace has piece slots for (0: all static)
  uint32_t stage_bytes, prefix_bytes;
  size_t smem_bytes;
  size_t ws_arrive, ws_claim, ws_ml, ws_o, ws_total;  // byte offsets / total
};

// q is bf16 beside a quantised cache, otherwise of the cache's own type.
size_t q_bytes_for(pda_dtype kv) {
  return (kv == PDA_FP8_E4M3 || kv == PDA_NVFP4) ? 2u : dtype_bytes(kv);
}

// How a launch tiles the work: the tile step and the unit (one kv-head, or a pair).
struct Tiling {
  int mode;   // kModeCuda, kModeTc or kModeTcPair
  int H_u;    // units per request (kv-heads, or pairs)
  int G_u;    // query heads per unit
};

// Quantised caches at D = 128 run on the tensor cores. Where H_kv is even and G <= 4, two
// adjacent kv-heads share a tile (one TMA box and one pipeline step for both): per byte
// that halves the TMA operations, which bound small quantised tiles (about one per 120 SM
// cycles, whatever their size), and the per-tile pipeline work. Otherwise a quantised tile
// is one kv-head on the tensor cores for G >= 2, and on the CUDA cores for G = 1 (a plain
// GEMV, where they keep up: measured equal to the single-head tensor-core step).
Tiling tiling_for(pda_dtype kv, int D, int H_kv, int G) {
  const bool quantised = kv == PDA_FP8_E4M3 || kv == PDA_NVFP4;
  if (quantised && D == 128 && G <= 4 && H_kv % 2 == 0) return {kModeTcPair, H_kv / 2, 2 * G};
  if (quantised && D == 128 && G >= 2) return {kModeTc, H_kv, G};
  return {kModeCuda, H_kv, G};
}

// One pipeline stage: the K and V tiles, (NVFP4) their block scales, the q rows, for a unit.
uint32_t stage_bytes_for(pda_dtype kv, int D, const Tiling& t) {
  const size_t heads = t.mode == kModeTcPair ? 2 : 1;
  const size_t tile = heads * (kv == PDA_NVFP4 ? kBS * D / 2 : kBS * D * dtype_bytes(kv));
  const size_t scales = heads * (kv == PDA_NVFP4 ? 2 * kBS * D / 16 : 0);
  const size_t q = static_cast<size_t>(t.G_u) * D * q_bytes_for(kv);
  return static_cast<uint32_t>(
      round_up(2 * tile + scales + q, stage_align(t.mode != kModeCuda)));
}

// pool: leave a share of the tiles to chunks claimed at run time (see Units); the
// workspace then holds piece slots for them as well.
bool make_plan(int B, int H_kv, int G, int D, pda_dtype kv, int sm_cap, int num_sms, bool pool,
               LaunchPlan* pl) {
  const Tiling t = tiling_for(kv, D, H_kv, G);
  const bool tc = t.mode != kModeCuda;
  const size_t align = stage_align(tc);
  pl->stage_bytes = stage_bytes_for(kv, D, t);
  pl->prefix_bytes = static_cast<uint32_t>(round_up(static_cast<size_t>(B + 1) * 4, align));
  // + alignment of the metadata ring, + room to align the layout's start
  const size_t fixed = pl->prefix_bytes + 8 + (align - 128);
  if (fixed >= static_cast<size_t>(kSmemBudget)) return false;
  pl->nwarps = 0;
  // The most warps that still get two stages each; then as many stages as fit.
  for (int nw = warps_for_mode(t.G_u, t.mode, kv == PDA_NVFP4); nw >= 2; --nw) {
    const size_t per_stage = static_cast<size_t>(nw) * (pl->stage_bytes + 8 + 4);
    const size_t meta = static_cast<size_t>(nw) * kMetaBytesPerWarp;
    if (fixed + meta >= static_cast<size_t>(kSmemBudget)) continue;
    const int stages = static_cast<int>((kSmemBudget - fixed - meta) / per_stage);
    if (stages >= 2) {
      pl->nwarps = nw;
      pl->stages = stages > PDA_ATTN_MAX_STAGES ? PDA_ATTN_MAX_STAGES : stages;
      break;
    }
  }
  if (pl->nwarps == 0) return false;
  size_t smem = fixed + static_cast<size_t>(pl->nwarps) * kMetaBytesPerWarp +
                static_cast<size_t>(pl->nwarps) * pl->stages * (pl->stage_bytes + 8 + 4);
  smem = round_up(smem, 128);
  if (smem < static_cast<size_t>(kMinResidentSmem)) smem = kMinResidentSmem;
  pl->smem_bytes = smem;
  int grid = num_sms;
  if (sm_cap > 0 && sm_cap < grid) grid = sm_cap;
  pl->grid = grid;
  const size_t nw_total = static_cast<size_t>(grid) * pl->nwarps;
  // Pool chunks pay off where the grid covers the whole chip: there SMs stream at unequal
  // rates (measured: whole runs of SMs about 10 % slower than the rest, at every workload),
  // while a capped grid leaves room around its SMs and runs evenly, so the chunks' extra
  // pieces and pipeline refills would cost more than they balance. The tensor-core steps
  // (quantised caches) process a tile in a fraction of the time and pay relatively more for
  // both; they keep the static split. A call claims at most NW k chunks plus one failed claim
  // per warp, within 16 bits.
  pl->pool_k = pool && t.mode == kModeCuda && grid == num_sms &&
                       nw_total * (PDA_POOL_CHUNKS_PER_WARP + 1) < 65536
                   ? PDA_POOL_CHUNKS_PER_WARP
                   : 0;
  const size_t units = nw_total * (1 + pl->pool_k);
  pl->ws_arrive = 0;
  pl->ws_claim = static_cast<size_t>(B) * t.H_u * 8;
  pl->ws_ml = round_up(pl->ws_claim + 8, 256);
  pl->ws_o = pl->ws_ml + round_up(2 * units * t.G_u * 2 * 4, 256);
  pl->ws_total = pl->ws_o + round_up(2 * units * t.G_u * static_cast<size_t>(D) * 4, 256);
  return true;
}

using KernelFn = void (*)(const CUtensorMap, const CUtensorMap, const AttnParams);

// The kernel for a unit of G_u query heads in the given mode.
template <typename KV, typename QT, int D>
KernelFn pick_g(int G_u, int mode) {
  if constexpr (std::is_same<KV, fp8e4m3>::value || std::is_same<KV, nvfp4>::value) {
    if constexpr (D == 128) {
      if (mode == kModeTcPair) {
        switch (G_u) {
          case 2: return attn_partial_kernel<KV, QT, D, 2, kModeTcPair>;
          case 4: return attn_partial_kernel<KV, QT, D, 4, kModeTcPair>;
          case 8: return attn_partial_kernel<KV, QT, D, 8, kModeTcPair>;
          default: return nullptr;
        }
      }
      if (mode == kModeTc) {
        switch (G_u) {
          case 2: return attn_partial_kernel<KV, QT, D, 2, kModeTc>;
          case 4: return attn_partial_kernel<KV, QT, D, 4, kModeTc>;
          case 8: return attn_partial_kernel<KV, QT, D, 8, kModeTc>;
          default: return nullptr;
        }
      }
    }
  }
  if (mode != kModeCuda) return nullptr;
  switch (G_u) {
    case 1: return attn_partial_kernel<KV, QT, D, 1, kModeCuda>;
    case 2: return attn_partial_kernel<KV, QT, D, 2, kModeCuda>;
    case 4: return attn_partial_kernel<KV, QT, D, 4, kModeCuda>;
    case 8: return attn_partial_kernel<KV, QT, D, 8, kModeCuda>;
    default: return nullptr;
  }
}

KernelFn pick_kernel(pda_dtype kv, int D, const Tiling& t) {
  if (kv == PDA_F16) {
    if (D == 128) return pick_g<__half, __half, 128>(t.G_u, t.mode);
    if (D == 64) return pick_g<__half, __half, 64>(t.G_u, t.mode);
  } else if (kv == PDA_BF16) {
    if (D == 128) return pick_g<__nv_bfloat16, __nv_bfloat16, 128>(t.G_u, t.mode);
    if (D == 64) return pick_g<__nv_bfloat16, __nv_bfloat16, 64>(t.G_u, t.mode);
  } else if (kv == PDA_FP8_E4M3) {
    if (D == 128) return pick_g<fp8e4m3, __nv_bfloat16, 128>(t.G_u, t.mode);
    if (D == 64) return pick_g<fp8e4m3, __nv_bfloat16, 64>(t.G_u, t.mode);
  } else if (kv == PDA_NVFP4) {
    if (D == 128) return pick_g<nvfp4, __nv_bfloat16, 128>(t.G_u, t.mode);
    if (D == 64) return pick_g<nvfp4, __nv_bfloat16, 64>(t.G_u, t.mode);
  } else {
    if (D == 128) return pick_g<float, float, 128>(t.G_u, t.mode);
    if (D == 64) return pick_g<float, float, 64>(t.G_u, t.mode);
  }
  return nullptr;
}

bool supported_g(int G) { return G == 1 || G == 2 || G == 4 || G == 8; }
// Physical blocks of 16, 32, ..., 256 tokens (a tile is 16 rows of one block).
bool supported_block_size(int bs) {
  return bs >= kBS && bs <= 16 * kBS && (bs & (bs - 1)) == 0;
}

// Numbers the calls, so a call recognises arrival counters left by earlier ones.
std::atomic<unsigned long long> g_call{1};

// Raises a kernel's dynamic shared-memory limit to the full budget once per device, so
// later calls (and calls made while a stream is being captured) skip the runtime call.
std::mutex g_attr_mu;
std::vector<std::pair<const void*, int>> g_attr_done;

pda_status allow_max_smem(const void* fn, int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const auto& e : g_attr_done)
    if (e.first == fn && e.second == dev) return PDA_OK;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget) !=
      cudaSuccess)
    return PDA_ERR_CUDA;
  g_attr_done.emplace_back(fn, dev);
  return PDA_OK;
}

// The last few encoded KV tensor maps, keyed by everything the encoding depends on.
struct MapKey {
  const void* base;
  int num_blocks, block_size, H_kv, D, dtype, swizzle;
  bool pair;
  bool operator==(const MapKey& o) const {
    return base == o.base && num_blocks == o.num_blocks && block_size == o.block_size &&
           H_kv == o.H_kv && D == o.D && dtype == o.dtype && swizzle == o.swizzle &&
           pair == o.pair;
  }
};
constexpr int kMapCache = 8;
std::mutex g_map_mu;
MapKey g_map_key[kMapCache];
CUtensorMap g_map_val[kMapCache];
int g_map_used = 0, g_map_next = 0;

// pair: the two-head map of encode_kv_pair_tensor_map (byte caches; D = row bytes).
pda_status cached_kv_tensor_map(CUtensorMap* tm, const void* base, int num_blocks,
                                int block_size, int H_kv, int D, pda_dtype dtype,
                                int swizzle_bytes, bool pair) {
  const MapKey key{base, num_blocks, block_size, H_kv, D, static_cast<int>(dtype),
                   swizzle_bytes, pair};
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < g_map_used; ++i)
      if (g_map_key[i] == key) {
        *tm = g_map_val[i];
        return PDA_OK;
      }
  }
  // boxes are one tile: kBS rows of one physical block (block_size is a multiple of kBS)
  const pda_status st =
      pair ? encode_kv_pair_tensor_map(tm, base, num_blocks, block_size, H_kv, D, swizzle_bytes,
                                       kBS)
           : encode_kv_tensor_map(tm, base, num_blocks, block_size, H_kv, D, dtype,
                                  swizzle_bytes, kBS);
  if (st != PDA_OK) return st;
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_map_key[g_map_next] = key;
  g_map_val[g_map_next] = *tm;
  g_map_next = (g_map_next + 1) % kMapCache;
  if (g_map_used < kMapCache) ++g_map_used;
  return PDA_OK;
}

}  // namespace
}  // namespace pda

using namespace pda;

extern "C" pda_status pda_attention_workspace_size(int B, int H, int H_kv, int D, int block_size,
                                                   pda_dtype kv_dtype, int sm_cap,
                                                   size_t* bytes) {
  if (bytes == nullptr || B < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || D <= 0 ||
      block_size <= 0 || sm_cap < 0 || !(dtype_ok(kv_dtype) || kv_dtype == PDA_NVFP4))
    return PDA_ERR_INVALID_ARG;
  if (!supported_block_size(block_size) || (D != 64 && D != 128) || !supported_g(H / H_kv) ||
      B > kMaxBatch)
    return PDA_ERR_UNSUPPORTED;
  int dev, sms;
  const pda_status st = current_device_sms(&dev, &sms);
  if (st != PDA_OK) return st;
  LaunchPlan pl;
  if (!make_plan(B, H_kv, H / H_kv, D, kv_dtype, sm_cap, sms, true, &pl))
    return PDA_ERR_UNSUPPORTED;
  *bytes = pl.ws_total;
  return PDA_OK;
}

namespace pda {
namespace {

// The attention launch behind every public entry point. kv_dtype selects the cache format;
// k_scale and v_scale are the values of one stored unit of K and V (1 for plain caches).
pda_status launch_attention(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const void* k_bscales, const void* v_bscales,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int max_context_len, int B, int H,
                            int H_kv, int D, int block_size, int num_blocks, float scale,
                            float k_scale, float v_scale, pda_dtype q_dtype,
                            pda_dtype kv_dtype, pda_dtype out_dtype, int sm_cap,
                            void* workspace, size_t workspace_bytes, int32_t* error_word,
                            cudaStream_t stream, bool pool = true, bool clear_arrivals = false) {
  // ---- host-side validation, before any CUDA call
  if (B < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || D <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks_per_seq < 0 || max_context_len < 0 || sm_cap < 0 ||
      !float_dtype_ok(q_dtype) || !(dtype_ok(kv_dtype) || kv_dtype == PDA_NVFP4) ||
      !float_dtype_ok(out_dtype) ||
      !isfinite(scale) || !isfinite(k_scale) || !isfinite(v_scale))
    return PDA_ERR_INVALID_ARG;
  if (B == 0) return PDA_OK;
  if (out == nullptr || q == nullptr || k_cache == nullptr || v_cache == nullptr ||
      block_tables == nullptr || context_lens == nullptr)
    return PDA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache))
    return PDA_ERR_INVALID_ARG;
  if (kv_dtype == PDA_NVFP4 && (k_bscales == nullptr || v_bscales == nullptr ||
                                !aligned16(k_bscales) || !aligned16(v_bscales)))
    return PDA_ERR_INVALID_ARG;
  const int G = H / H_kv;
  const bool quantised = kv_dtype == PDA_FP8_E4M3 || kv_dtype == PDA_NVFP4;
  const bool q_ok = quantised ? q_dtype == PDA_BF16 : q_dtype == kv_dtype;
  if (!supported_block_size(block_size) || (D != 64 && D != 128) || !supported_g(G) || !q_ok ||
      B > kMaxBatch)
    return PDA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= (1ll << 31) ||
      static_cast<long long>(B) * max_blocks_per_seq * H_kv >= (1ll << 31))
    return PDA_ERR_UNSUPPORTED;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return PDA_ERR_WORKSPACE;

  int dev, sms;
  pda_status st = current_device_sms(&dev, &sms);
  if (st != PDA_OK) return st;
  LaunchPlan pl;
  if (!make_plan(B, H_kv, G, D, kv_dtype, sm_cap, sms, pool, &pl)) return PDA_ERR_UNSUPPORTED;
  if (workspace_bytes < pl.ws_total) return PDA_ERR_WORKSPACE;

  const Tiling tiling = tiling_for(kv_dtype, D, H_kv, G);
  // No more blocks than give every warp PDA_MIN_TILES_PER_WARP tiles at the host's bound on
  // the lengths (every request at max_context_len); the kernel applies the same rule to the
  // lengths it reads. The workspace, sized for the full grid, is large enough for fewer
  // workers.
  {
    const long long max_len =
        std::min<long long>(max_context_len, static_cast<long long>(max_blocks_per_seq) * block_size);
    const long long tiles = static_cast<long long>(B) * tiling.H_u * ((max_len + kBS - 1) / kBS);
    const long long per_block = static_cast<long long>(pl.nwarps) * PDA_MIN_TILES_PER_WARP;
    const long long blocks = (tiles + per_block - 1) / per_block;
    if (blocks < pl.grid) {
      pl.grid = static_cast<int>(std::max<long long>(1, blocks));
      pl.pool_k = 0;  // the pool is for the whole chip's grid
    }
  }
  KernelFn fn = pick_kernel(kv_dtype, D, tiling);
  if (fn == nullptr) return PDA_ERR_UNSUPPORTED;
  st = allow_max_smem(reinterpret_cast<const void*>(fn), dev);
  if (st != PDA_OK) return st;

  // the TMA sees an NVFP4 row as D/2 bytes; the tensor-core step reads swizzled tiles whose
  // swizzle span is one whole row (128 bytes FP8, 64 bytes NVFP4)
  const int row_elems = kv_dtype == PDA_NVFP4 ? D / 2 : D;
  const pda_dtype map_type = kv_dtype == PDA_NVFP4 ? PDA_FP8_E4M3 : kv_dtype;
  const int swizzle = tiling.mode != kModeCuda ? row_elems : 0;
  const bool pair = tiling.mode == kModeTcPair;
  CUtensorMap tmK, tmV;
  st = cached_kv_tensor_map(&tmK, k_cache, num_blocks, block_size, H_kv, row_elems, map_type,
                            swizzle, pair);
  if (st != PDA_OK) return st;
  st = cached_kv_tensor_map(&tmV, v_cache, num_blocks, block_size, H_kv, row_elems, map_type,
                            swizzle, pair);
  if (st != PDA_OK) return st;

  unsigned char* ws = static_cast<unsigned char*>(workspace);
  AttnParams ap;
  ap.out = out;
  ap.q = q;
  ap.block_tables = block_tables;
  ap.context_lens = context_lens;
  ap.ws_arrive = reinterpret_cast<unsigned long long*>(ws + pl.ws_arrive);
  ap.ws_claim = reinterpret_cast<unsigned long long*>(ws + pl.ws_claim);
  ap.pool_k = pl.pool_k;
  ap.call = g_call.fetch_add(1, std::memory_order_relaxed) & ((1ull << 48) - 1);
  ap.ws_ml = reinterpret_cast<float*>(ws + pl.ws_ml);
  ap.ws_o = reinterpret_cast<float*>(ws + pl.ws_o);
  ap.error_word = error_word;
  ap.v_scale = v_scale;
  ap.k_bscales = static_cast<const uint8_t*>(k_bscales);
  ap.v_bscales = static_cast<const uint8_t*>(v_bscales);
  ap.B = B;
  ap.H = H;
  ap.H_kv = tiling.H_u;  // units: kv-heads, or pairs of them
  ap.num_blocks = num_blocks;
  ap.max_blocks = max_blocks_per_seq;
  ap.max_context_len = max_context_len;
  ap.block_size = block_size;
  ap.bs_shift = 0;
  while ((kBS << ap.bs_shift) < block_size) ++ap.bs_shift;
  ap.out_kind = out_dtype == PDA_BF16 ? kOutBF16 : out_dtype == PDA_F16 ? kOutF16 : kOutF32;
  // the K scale folds into q's pre-scale: s = scale * (k_scale * code) . q
  ap.scale_log2 = scale * k_scale * 1.4426950408889634f;
  ap.num_workers = pl.grid * pl.nwarps;
  ap.stages = pl.stages;
  ap.stage_bytes = pl.stage_bytes;
  ap.prefix_bytes = pl.prefix_bytes;

  // clear_arrivals: zero the arrival counters first (a memset on the same stream), so no
  // counter left in the workspace by an earlier call can pass for one of this call's
  if (clear_arrivals && cudaMemsetAsync(ap.ws_arrive, 0, pl.ws_claim + 8, stream) != cudaSuccess)
    return PDA_ERR_CUDA;
  fn<<<pl.grid, pl.nwarps * 32, pl.smem_bytes, stream>>>(tmK, tmV, ap);
  if (cudaGetLastError() != cudaSuccess) return PDA_ERR_CUDA;
  return PDA_OK;
}

}  // namespace
}  // namespace pda

extern "C" pda_status pda_paged_decode_attention(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int B, int H, int H_kv, int D, int block_size, int num_blocks,
    float scale, pda_dtype q_dtype, pda_dtype kv_dtype, pda_dtype out_dtype, int sm_cap,
    void* workspace, size_t workspace_bytes, int32_t* error_word, cudaStream_t stream) {
  if (kv_dtype == PDA_FP8_E4M3) return PDA_ERR_UNSUPPORTED;  // needs its scales: _fp8 entry
  return launch_attention(out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, B, H, H_kv, D,
                          block_size, num_blocks, scale, 1.f, 1.f, q_dtype, kv_dtype, out_dtype,
                          sm_cap, workspace, workspace_bytes, error_word, stream);
}

extern "C" pda_status pda_paged_decode_attention_fp8(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int B, int H, int H_kv, int D, int block_size, int num_blocks,
    float scale, float k_scale, float v_scale, pda_dtype q_dtype, pda_dtype out_dtype,
    int sm_cap, void* workspace, size_t workspace_bytes, int32_t* error_word,
    cudaStream_t stream) {
  return launch_attention(out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, B, H, H_kv, D,
                          block_size, num_blocks, scale, k_scale, v_scale, q_dtype,
                          PDA_FP8_E4M3, out_dtype, sm_cap, workspace, workspace_bytes,
                          error_word, stream);
}

extern "C" pda_status pda_paged_decode_attention_nvfp4(
    void* out, const void* q, const void* k_data, const void* v_data,
    const void* k_block_scales, const void* v_block_scales, const int32_t* block_tables,
    int max_blocks_per_seq, const int32_t* context_lens, int max_context_len, int B, int H,
    int H_kv, int D, int block_size, int num_blocks, float scale, float k_scale, float v_scale,
    pda_dtype q_dtype, pda_dtype out_dtype, int sm_cap, void* workspace,
    size_t workspace_bytes, int32_t* error_word, cudaStream_t stream) {
  return launch_attention(out, q, k_data, v_data, k_block_scales, v_block_scales,
                          block_tables, max_blocks_per_seq, context_lens, max_context_len, B, H,
                          H_kv, D, block_size, num_blocks, scale, k_scale, v_scale, q_dtype,
                          PDA_NVFP4, out_dtype, sm_cap, workspace, workspace_bytes, error_word,
                          stream);
}

// ------------------------------------------------------------------ no-allocation variant
// Scratch for pda_paged_decode_attention_noalloc: a fixed device array in this module, for
// callers that may not allocate device memory while they run: a plugin whose host
// framework owns all device memory and hands it only inputs and outputs, or a serving loop
// that forbids allocation once it has started. Host code must not pass `g_noalloc_scratch`
// itself to a kernel (on the host it names a host-side shadow, not device memory); it
// passes the address cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PDA_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int kNoallocMaxDevices = 64;
std::atomic<void*> g_noalloc_ptr[kNoallocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the scratch array on `dev` (the current device), looked up once.
pda_status noalloc_scratch(int dev, void** ptr) {
  if (dev < 0 || dev >= kNoallocMaxDevices) return PDA_ERR_UNSUPPORTED;
  void* p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    p = g_noalloc_ptr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return PDA_ERR_CUDA;
      g_noalloc_ptr[dev].store(p, std::memory_order_release);
    }
  }
  *ptr = p;
  return PDA_OK;
}
}  // namespace

extern "C" pda_status pda_paged_decode_attention_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int B, int H, int H_kv, int D, int block_size, int num_blocks,
    float scale, pda_dtype q_dtype, pda_dtype kv_dtype, pda_dtype out_dtype, int sm_cap,
    int32_t* error_word, cudaStream_t stream) {
  if (kv_dtype == PDA_FP8_E4M3) return PDA_ERR_UNSUPPORTED;  // as pda_paged_decode_attention
  // The same checks as pda_attention_workspace_size, for the all-static split (no pool of
  // claimed chunks, whose piece slots would not fit the fixed array).
  if (B < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || D <= 0 || block_size <= 0 ||
      sm_cap < 0 || !(dtype_ok(kv_dtype) || kv_dtype == PDA_NVFP4))
    return PDA_ERR_INVALID_ARG;
  if (!supported_block_size(block_size) || (D != 64 && D != 128) || !supported_g(H / H_kv) ||
      B > kMaxBatch)
    return PDA_ERR_UNSUPPORTED;
  int dev = 0, sms = 0;
  pda_status st = current_device_sms(&dev, &sms);
  if (st != PDA_OK) return st;
  LaunchPlan pl;
  if (!make_plan(B, H_kv, H / H_kv, D, kv_dtype, sm_cap, sms, false, &pl))
    return PDA_ERR_UNSUPPORTED;
  if (pl.ws_total > PDA_NOALLOC_SCRATCH_BYTES) return PDA_ERR_TOO_LARGE;
  void* scratch = nullptr;
  st = noalloc_scratch(dev, &scratch);
  if (st != PDA_OK) return st;
  // The shared array keeps whatever the previous call left, which may be a call of another
  // shape or one that timed out: its counters are cleared before the kernel runs.
  return launch_attention(out, q, k_cache, v_cache, nullptr, nullptr, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, B, H, H_kv, D,
                          block_size, num_blocks, scale, 1.f, 1.f, q_dtype, kv_dtype, out_dtype,
                          sm_cap, scratch, PDA_NOALLOC_SCRATCH_BYTES, error_word, stream,
                          /*pool=*/false, /*clear_arrivals=*/true);
}
