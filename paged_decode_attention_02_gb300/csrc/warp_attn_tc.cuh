// warp_attn_tc.cuh -- one warp's tile step on the tensor cores, for quantised caches
// (FP8 E4M3, and NVFP4: E2M1 codes with one E4M3 scale per 16 elements) at D = 128.
//
// A head tile is one physical block (16 tokens) of one kv-head. Per head tile the warp
// computes, with mma.sync m16n8k16 (fp16 operands, fp32 accumulators):
//   S  = Q K^T    M = query heads (rows g of the fragment), N = 16 tokens (two n-tiles),
//                 K = d in eight k-steps;
//   O^T += V^T P^T  M = d (eight m-tiles of 16), N = 8 heads, K = 16 tokens.
// The accumulator of S (row = head g, columns = token pairs 2t, 2t+1) has exactly the layout
// of the P^T operand (column = head g, k pairs = tokens 2t, 2t+1), so the probabilities go
// from the softmax into the second product without any exchange between lanes.
//
// Two steps use these products:
//  * WarpAttnTC: one kv-head per tile, its G (2 to 8) query heads in rows and columns 0..G-1.
//  * WarpAttnTCPair: two adjacent kv-heads A, B per tile (one TMA box carries both head
//    tiles), G <= 4 query heads each: A's heads in output columns 0..G-1, B's in 4..4+G-1,
//    so both share one set of accumulators; each head's scores have their own accumulator.
//    Half the TMA operations and half the per-tile pipeline work per byte.
//
// Why mma.sync and not tcgen05: K and V reach the tensor cores only after a dequantisation
// that runs in registers, and with at most 8 query rows per kv-head the reduction runs over
// tokens; tcgen05 wants its operands in shared memory (or TMEM) and 64 or 128 rows of M.
//
// Exactness: E4M3 codes, E2M1 codes and their products with E4M3 block scales are all
// exact in fp16, so the K and V operands are the cached values themselves; q is exact in
// fp16 after a power-of-two rescale that keeps it in range (folded back into the score
// scale). The probabilities enter P^T V as the sum of two fp16 parts, hi = fp16(p) and
// lo = fp16(p - hi), both multiplied into the same accumulator: one fp16 part alone
// (relative error 2^-12) moves an output by up to 2^-12 of the largest |V|, which is too
// much where the weighted V values cancel; the pair leaves about 2^-22.
//
// Shared-memory layout: the TMA writes each 16-row head tile with the 128-byte swizzle (FP8,
// 128-byte rows: 16-byte chunk c of row r lands at chunk c ^ (r & 7)) or the 64-byte
// swizzle (NVFP4, 64-byte rows: chunk c ^ ((r >> 1) & 3)), which makes every load below
// free of bank conflicts. The element order along d inside a k-step is permuted (the same
// permutation for q and K), which leaves the dot products unchanged.
#pragma once

#include <math.h>
#include <type_traits>

#include "pda_device.cuh"

namespace pda {

// The per-head products, shared by the single- and two-head steps. Lane = 4 g + t4.
template <typename KV, int D>
struct TCOps {
  static_assert(D == 128, "tensor-core tile step is laid out for D = 128");
  static constexpr bool FP4 = std::is_same<KV, nvfp4>::value;
  static_assert(FP4 || std::is_same<KV, fp8e4m3>::value, "quantised caches only");
  static constexpr int ROW_BYTES = FP4 ? D / 2 : D;  // bytes of one K or V row
  static constexpr int TILE_BYTES = 16 * ROW_BYTES;  // one head tile

  // ldmatrix row addresses of this lane inside a V head tile (bytes), one per pair of
  // 16-byte chunks.
  static __device__ __forceinline__ void v_offsets(int lane, int* v_off) {
    const int j = lane & 7;                   // row inside the 8x8 matrix this lane addresses
    const int r = j + 8 * ((lane >> 3) & 1);  // token row of the tile
    const int ch = lane >> 4;                 // second chunk of the pair
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int chunk = 2 * q + ch;  // NVFP4 uses q < 2 only: four 16-byte chunks per row
      v_off[q] = FP4 ? r * ROW_BYTES + (((chunk ^ ((r >> 1) & 3)) & 3) << 4)
                     : r * ROW_BYTES + ((chunk ^ (r & 7)) << 4);
    }
  }

  // q of one head (32 consecutive d from 32 t4, in fp32) as A fragments: k-step s holds
  // d = 32 t4 + 4 s + {0, 1} (first pair) and + {2, 3} (second pair).
  static __device__ __forceinline__ void q_fragments(const float* qv, float down,
                                                     uint32_t (&qa)[8][2]) {
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      qa[s][0] = f16x2_bits(__floats2half2_rn(qv[4 * s] * down, qv[4 * s + 1] * down));
      qa[s][1] = f16x2_bits(__floats2half2_rn(qv[4 * s + 2] * down, qv[4 * s + 3] * down));
    }
  }

  // S[nt] += Q K^T over one head tile: n-tile nt covers tokens 8 nt .. 8 nt + 7 (token g of
  // it on this lane). ksc: the tile's block scales, row r at ksc + r * ksc_stride (NVFP4).
  static __device__ __forceinline__ void qk(float (&sc)[2][4], const uint32_t (&qa)[8][2],
                                            const unsigned char* ks, const uint8_t* ksc,
                                            int ksc_stride, int g, int t4) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      const int r = g + 8 * nt;
      if constexpr (FP4) {
        // 16 bytes = d 32 t4 .. 32 t4 + 31; byte 2s (+1) holds k-step s's first (second) pair
        const uint4 w = *reinterpret_cast<const uint4*>(
            ks + r * ROW_BYTES + ((t4 ^ ((r >> 1) & 3)) << 4));
        const uint32_t sp =
            e4m3x2_to_f16x2(*reinterpret_cast<const uint16_t*>(ksc + r * ksc_stride + 2 * t4));
        const __half2 s_lo = __low2half2(as_half2(sp));   // block 2 t4: k-steps 0-3
        const __half2 s_hi = __high2half2(as_half2(sp));  // block 2 t4 + 1: k-steps 4-7
        const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t h[4];
          e2m1x8_to_f16x2(words[u], h);
          const __half2 sb = u < 2 ? s_lo : s_hi;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int s = 2 * u + k;
            const uint32_t b0 = f16x2_bits(__hmul2(as_half2(h[2 * k]), sb));
            const uint32_t b1 = f16x2_bits(__hmul2(as_half2(h[2 * k + 1]), sb));
            mma_f16_16816(sc[nt], qa[s][0], 0u, qa[s][1], 0u, b0, b1);
          }
        }
      } else {
        // chunk 2 t4 + hh = d 32 t4 + 16 hh .. + 15; word u of it is k-step 4 hh + u
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint4 w = *reinterpret_cast<const uint4*>(
              ks + r * ROW_BYTES + (((2 * t4 + hh) ^ (r & 7)) << 4));
          const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t b0, b1;
            e4m3x4_to_f16x2(words[u], b0, b1);
            mma_f16_16816(sc[nt], qa[4 * hh + u][0], 0u, qa[4 * hh + u][1], 0u, b0, b1);
          }
        }
      }
    }
  }

  // Per token half of this lane's V pairs: which of (token 2t4 [+8], token 2t4+1 [+8]) are
  // valid; the masks clear the invalid token's bytes (FP8) or fp16 halves (NVFP4).
  static __device__ __forceinline__ void keep_masks(int t4, int n_valid, uint32_t& keep_lo,
                                                    uint32_t& keep_hi) {
    const bool a = 2 * t4 < n_valid, b = 2 * t4 + 1 < n_valid;
    const bool c = 8 + 2 * t4 < n_valid, d = 9 + 2 * t4 < n_valid;
    if constexpr (FP4) {
      keep_lo = (a ? 0x0000ffffu : 0u) | (b ? 0xffff0000u : 0u);
      keep_hi = (c ? 0x0000ffffu : 0u) | (d ? 0xffff0000u : 0u);
    } else {
      keep_lo = (a ? 0x00ff00ffu : 0u) | (b ? 0xff00ff00u : 0u);
      keep_hi = (c ? 0x00ff00ffu : 0u) | (d ? 0xff00ff00u : 0u);
    }
  }

  // O^T += V^T P^T over one head tile, P^T given as this lane's B fragments (hi and lo
  // fp16 parts). ldmatrix.trans hands this lane, per 16-byte chunk of the rows 0-7 (and
  // 8-15), two bytes of token 2t4 and the same two bytes of token 2t4 + 1. vsc: the tile's
  // block scales, row t at vsc + t * vsc_stride (NVFP4).
  static __device__ __forceinline__ void pv(float (&o)[8][4], const unsigned char* vs,
                                            const uint8_t* vsc, int vsc_stride,
                                            const int (&v_off)[4], int g, int t4,
                                            uint32_t pb0, uint32_t pb1, uint32_t pl0,
                                            uint32_t pl1, uint32_t keep_lo, uint32_t keep_hi) {
    if constexpr (FP4) {
      // scale pairs (token t0, token t0 + 1) of this lane's block in chunk c: rows 2t4(+1)
      // and 8 + 2t4 (+1); the block is 2c + g / 4
      const uint2 w0 = *reinterpret_cast<const uint2*>(vsc + (2 * t4) * vsc_stride);
      const uint2 w1 = *reinterpret_cast<const uint2*>(vsc + (2 * t4 + 1) * vsc_stride);
      const uint2 w2 = *reinterpret_cast<const uint2*>(vsc + (8 + 2 * t4) * vsc_stride);
      const uint2 w3 = *reinterpret_cast<const uint2*>(vsc + (9 + 2 * t4) * vsc_stride);
      const uint32_t bsel = g >> 2;
#pragma unroll
      for (int qq = 0; qq < 2; ++qq) {
        uint32_t r[4];
        ldmatrix_x4_trans(r, vs + v_off[qq]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int chunk = 2 * qq + cc;
          const uint32_t k = 2 * (chunk & 1) + bsel;
          const uint32_t sel = k | ((k + 4) << 4);
          const __half2 sv_lo = as_half2(e4m3x2_to_f16x2(
              prmt(chunk < 2 ? w0.x : w0.y, chunk < 2 ? w1.x : w1.y, sel)));
          const __half2 sv_hi = as_half2(e4m3x2_to_f16x2(
              prmt(chunk < 2 ? w2.x : w2.y, chunk < 2 ? w3.x : w3.y, sel)));
          // A words (token pair) for d0 + u, d0 = 32 chunk + 4 g
          uint32_t alo[4], ahi[4];
          {
            uint32_t h[4];
            e2m1x8_to_f16x2(r[2 * cc], h);  // t0: (d0,d0+1) (d0+2,d0+3); t1: same
            alo[0] = prmt(h[0], h[2], 0x5410u);
            alo[1] = prmt(h[0], h[2], 0x7632u);
            alo[2] = prmt(h[1], h[3], 0x5410u);
            alo[3] = prmt(h[1], h[3], 0x7632u);
            e2m1x8_to_f16x2(r[2 * cc + 1], h);
            ahi[0] = prmt(h[0], h[2], 0x5410u);
            ahi[1] = prmt(h[0], h[2], 0x7632u);
            ahi[2] = prmt(h[1], h[3], 0x5410u);
            ahi[3] = prmt(h[1], h[3], 0x7632u);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            alo[u] = f16x2_bits(__hmul2(as_half2(alo[u]), sv_lo)) & keep_lo;
            ahi[u] = f16x2_bits(__hmul2(as_half2(ahi[u]), sv_hi)) & keep_hi;
          }
          // m-tile 2 chunk + v: row g = d0 + 2v, row g + 8 = d0 + 2v + 1
          mma_f16_16816(o[2 * chunk], alo[0], alo[1], ahi[0], ahi[1], pb0, pb1);
          mma_f16_16816(o[2 * chunk], alo[0], alo[1], ahi[0], ahi[1], pl0, pl1);
          mma_f16_16816(o[2 * chunk + 1], alo[2], alo[3], ahi[2], ahi[3], pb0, pb1);
          mma_f16_16816(o[2 * chunk + 1], alo[2], alo[3], ahi[2], ahi[3], pl0, pl1);
        }
      }
    } else {
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        uint32_t r[4];
        ldmatrix_x4_trans(r, vs + v_off[qq]);
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          // bytes (t0 d0, t0 d0+1, t1 d0, t1 d0+1) -> (t0 d0, t1 d0, t0 d0+1, t1 d0+1)
          const uint32_t lo = prmt(r[2 * cc], 0u, 0x3120u) & keep_lo;
          const uint32_t hi = prmt(r[2 * cc + 1], 0u, 0x3120u) & keep_hi;
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2(lo, a0, a1);  // d0 = 16 chunk + 2 g (row g), d0 + 1 (row g + 8)
          e4m3x4_to_f16x2(hi, a2, a3);
          mma_f16_16816(o[2 * qq + cc], a0, a1, a2, a3, pb0, pb1);
          mma_f16_16816(o[2 * qq + cc], a0, a1, a2, a3, pl0, pl1);
        }
      }
    }
  }

  // d of row g of m-tile i (row g + 8 is d + 1).
  static __device__ __forceinline__ int d_of(int i, int g) {
    return FP4 ? 32 * (i >> 1) + 4 * g + 2 * (i & 1) : 16 * i + 2 * g;
  }

  // Power-of-two factor that brings max |q| (over the warp) below 2^15: returns `down`, the
  // factor q is multiplied by, and sets `up` = 1 / down for the score scale.
  static __device__ __forceinline__ float q_shift(float amax_lane, float& up) {
    float amax = amax_lane;
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
    const int shift = e > 14 ? (e - 14 < 126 ? e - 14 : 126) : 0;
    up = __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
    return __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
  }

  // The 32 q values of row `row` this lane holds (d 32 t4 ..), zeros if `real` is false;
  // returns their max |q|.
  static __device__ __forceinline__ float load_q(const __nv_bfloat16* q_smem, int row,
                                                 bool real, int t4, float* qv) {
    float amax = 0.f;
    if (real) {
      const uint4* src = reinterpret_cast<const uint4*>(q_smem + row * D + 32 * t4);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 w = src[i];
        qv[8 * i + 0] = bf16_lo(w.x);
        qv[8 * i + 1] = bf16_hi(w.x);
        qv[8 * i + 2] = bf16_lo(w.y);
        qv[8 * i + 3] = bf16_hi(w.y);
        qv[8 * i + 4] = bf16_lo(w.z);
        qv[8 * i + 5] = bf16_hi(w.z);
        qv[8 * i + 6] = bf16_lo(w.w);
        qv[8 * i + 7] = bf16_hi(w.w);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[i]));
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] = 0.f;
    }
    return amax;
  }

  // fp16 hi and lo parts of two probabilities as f16x2 words.
  static __device__ __forceinline__ void split_p(float p0, float p1, uint32_t& hi,
                                                 uint32_t& lo) {
    const __half2 h = __floats2half2_rn(p0, p1);
    const float2 r = __half22float2(h);
    hi = f16x2_bits(h);
    lo = f16x2_bits(__floats2half2_rn(p0 - r.x, p1 - r.y));
  }

  // One head's softmax step over this lane's four scores x (tokens 2t4, 2t4+1, 8+2t4,
  // 9+2t4; already scaled): the tile max over the lane's row group, whether the running max
  // must move (by more than kLag), and the probabilities against the running max after it.
  // Returns the rescale factor (1 where the max stays, 0 on the first tile).
  static __device__ __forceinline__ float softmax(float (&x)[4], float& m_run, float& l_run,
                                                  bool& grow) {
    float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 2));
    grow = tmax > m_run + kLag;
    const float m_new = grow ? tmax : m_run;
    const float alpha = ex2(m_run - m_new);  // 0 on the first tile, 1 where m is kept
    m_run = m_new;
    l_run *= alpha;
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = ex2(x[e] - m_run);
    l_run += (x[0] + x[1]) + (x[2] + x[3]);
    return alpha;
  }

  // The max a head's running maximum may lag the true one by (log2 units): probabilities
  // then stay below 2^8, well inside fp16, and the output is rescaled only when a new
  // maximum exceeds the old by more than this.
  static constexpr float kLag = 8.f;
};

// One kv-head per tile; its G query heads in fragment rows / output columns 0..G-1.
template <typename KV, int D, int G>
struct WarpAttnTC {
  static_assert(G == 2 || G == 4 || G == 8, "2 to 8 heads per kv-head (G = 1 is a GEMV)");
  using Ops = TCOps<KV, D>;
  static constexpr int ROW_SCALES = D / 16;  // NVFP4 scale bytes per row and head

  int g, t4;
  uint32_t qa[8][2];  // q of head g as A fragments
  float o[8][4];      // O^T accumulators: m-tile i, (d row g | g + 8) x heads (2t4, 2t4+1)
  float m_run;        // running max of head g (log2 units, scaled)
  float l_run;        // this lane's share of head g's running sum
  float c;            // score scale: scale * log2(e) * k_scale * 2^qshift
  int v_off[4];
  float l_cols[2];    // after reduce(): full sums of heads 2 t4 and 2 t4 + 1

  __device__ __forceinline__ void init(int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    Ops::v_offsets(lane, v_off);
  }

  // q of this warp's segment (G rows of D bf16 in shared memory), pre-scale scale_log2.
  __device__ __forceinline__ void reset(const __nv_bfloat16* q_smem, float scale_log2) {
    float qv[32];
    const float amax = Ops::load_q(q_smem, g, g < G, t4, qv);
    float up;
    const float down = Ops::q_shift(amax, up);
    c = scale_log2 * up;
    Ops::q_fragments(qv, down, qa);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
    m_run = -INFINITY;
    l_run = 0.f;
  }

  // ks/vs: the tile's K and V rows (swizzled); ksc/vsc: NVFP4 block scales, [16][D/16].
  template <bool kPartial>
  __device__ __forceinline__ void tile(const KV* ks, const KV* vs, const uint8_t* ksc,
                                       const uint8_t* vsc, int n_valid) {
    float sc[2][4] = {};
    Ops::qk(sc, qa, reinterpret_cast<const unsigned char*>(ks), ksc, ROW_SCALES, g, t4);
    float x[4] = {sc[0][0] * c, sc[0][1] * c, sc[1][0] * c, sc[1][1] * c};
    if (kPartial) {
      const int tok[4] = {2 * t4, 2 * t4 + 1, 8 + 2 * t4, 9 + 2 * t4};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (tok[e] >= n_valid) x[e] = -INFINITY;
    }
    bool grow;
    const float alpha = Ops::softmax(x, m_run, l_run, grow);
    if (__any_sync(kFullMask, grow)) {
      // the O^T columns of this lane are heads 2 t4 and 2 t4 + 1 (lanes 8 t4, 8 t4 + 4)
      const float2 a2 = make_float2(__shfl_sync(kFullMask, alpha, 8 * t4),
                                    __shfl_sync(kFullMask, alpha, 8 * t4 + 4));
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 lo = __fmul2_rn(make_float2(o[i][0], o[i][1]), a2);
        const float2 hi = __fmul2_rn(make_float2(o[i][2], o[i][3]), a2);
        o[i][0] = lo.x;
        o[i][1] = lo.y;
        o[i][2] = hi.x;
        o[i][3] = hi.y;
      }
    }
    uint32_t pb0, pb1, pl0, pl1;  // tokens (2t4, 2t4+1) and (8+2t4, 9+2t4)
    Ops::split_p(x[0], x[1], pb0, pl0);
    Ops::split_p(x[2], x[3], pb1, pl1);
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (kPartial) Ops::keep_masks(t4, n_valid, keep_lo, keep_hi);
    Ops::pv(o, reinterpret_cast<const unsigned char*>(vs), vsc, ROW_SCALES, v_off, g, t4, pb0,
            pb1, pl0, pl1, keep_lo, keep_hi);
  }

  // After the last tile: lj[j], mj[j] of every head j < G on every lane.
  __device__ __forceinline__ void reduce(float* lj, float* mj) {
    float l = l_run;
    l += __shfl_xor_sync(kFullMask, l, 1);
    l += __shfl_xor_sync(kFullMask, l, 2);
#pragma unroll
    for (int j = 0; j < G; ++j) {
      lj[j] = __shfl_sync(kFullMask, l, 4 * j);
      mj[j] = __shfl_sync(kFullMask, m_run, 4 * j);
    }
    l_cols[0] = __shfl_sync(kFullMask, l, 8 * t4);
    l_cols[1] = __shfl_sync(kFullMask, l, 8 * t4 + 4);
  }

  // Calls f(head, d, values, 2, l of the head) for each pair of output elements this lane
  // holds (the head's sum comes from reduce(), so lj is not indexed here).
  template <typename F>
  __device__ __forceinline__ void for_each_out(const float*, F&& f) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int j = 2 * t4 + jj;
        if (j < G) {
          const float v[2] = {o[i][jj], o[i][2 + jj]};
          f(j, Ops::d_of(i, g), v, 2, l_cols[jj]);
        }
      }
    }
  }
  __device__ __forceinline__ bool writes_ml(int lane) const { return lane == 0; }
};

// Two adjacent kv-heads A (tile bytes [0, TILE_BYTES)) and B ([TILE_BYTES, 2 TILE_BYTES)) per
// tile, GH <= 4 query heads each; NVFP4 scales likewise, A's [16][D/16] then B's. Unit head j: A's local j for j < GH, B's local j - GH
// otherwise (the q rows and output rows of the unit are in that order). Lane g holds head
// A_g's and B_g's scores (separate accumulators) and running state; the shared O^T holds
// A's heads in columns 0..GH-1 and B's in 4..4+GH-1: the PV products of head A get P^T
// columns 0-3 (lanes g < 4 supply P_A[g], lanes g >= 4 zero), those of head B columns 4-7
// (lanes g >= 4 supply P_B[g - 4], fetched from lane - 16, lanes g < 4 zero).
template <typename KV, int D, int GH>
struct WarpAttnTCPair {
  static_assert(GH == 1 || GH == 2 || GH == 4, "1 to 4 heads per kv-head of a pair");
  using Ops = TCOps<KV, D>;
  static constexpr int G = 2 * GH;                 // query heads of the unit
  static constexpr int ROW_SCALES = D / 16;        // NVFP4 scale bytes per row and head
  static constexpr int HEAD_SCALES = 16 * ROW_SCALES;  // a head's tile of scales: A's, B's

  int g, t4;
  uint32_t qa[2][8][2];  // q of heads A_g, B_g as A fragments
  float o[8][4];
  float m_run[2], l_run[2];  // heads A_g, B_g
  float c;
  int v_off[4];
  float l_cols[2];

  __device__ __forceinline__ void init(int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    Ops::v_offsets(lane, v_off);
  }

  __device__ __forceinline__ void reset(const __nv_bfloat16* q_smem, float scale_log2) {
    float qa_v[32], qb_v[32];
    const float amax = fmaxf(Ops::load_q(q_smem, g, g < GH, t4, qa_v),
                             Ops::load_q(q_smem, GH + g, g < GH, t4, qb_v));
    float up;
    const float down = Ops::q_shift(amax, up);
    c = scale_log2 * up;
    Ops::q_fragments(qa_v, down, qa[0]);
    Ops::q_fragments(qb_v, down, qa[1]);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[i][e] = 0.f;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      m_run[u] = -INFINITY;
      l_run[u] = 0.f;
    }
  }

  template <bool kPartial>
  __device__ __forceinline__ void tile(const KV* ks_, const KV* vs_, const uint8_t* ksc,
                                       const uint8_t* vsc, int n_valid) {
    const unsigned char* ks = reinterpret_cast<const unsigned char*>(ks_);
    const unsigned char* vs = reinterpret_cast<const unsigned char*>(vs_);
    float sc[2][2][4] = {};  // head, n-tile
#pragma unroll
    for (int u = 0; u < 2; ++u)
      Ops::qk(sc[u], qa[u], ks + u * Ops::TILE_BYTES, ksc + u * HEAD_SCALES, ROW_SCALES, g,
              t4);
    float x[2][4];
    float alpha[2];
    bool grow[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      x[u][0] = sc[u][0][0] * c;
      x[u][1] = sc[u][0][1] * c;
      x[u][2] = sc[u][1][0] * c;
      x[u][3] = sc[u][1][1] * c;
      if (kPartial) {
        const int tok[4] = {2 * t4, 2 * t4 + 1, 8 + 2 * t4, 9 + 2 * t4};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (tok[e] >= n_valid) x[u][e] = -INFINITY;
      }
      alpha[u] = Ops::softmax(x[u], m_run[u], l_run[u], grow[u]);
    }
    if (__any_sync(kFullMask, grow[0] || grow[1])) {
      // columns 2t4, 2t4+1 of this lane: A heads (t4 < 2) or B heads 2t4-4, 2t4-3 (t4 >= 2),
      // owned by lanes 8 (t4 & 1) and 8 (t4 & 1) + 4
      const int src = 8 * (t4 & 1);
      const float aA0 = __shfl_sync(kFullMask, alpha[0], src);
      const float aA1 = __shfl_sync(kFullMask, alpha[0], src + 4);
      const float aB0 = __shfl_sync(kFullMask, alpha[1], src);
      const float aB1 = __shfl_sync(kFullMask, alpha[1], src + 4);
      const float2 a2 = t4 < 2 ? make_float2(aA0, aA1) : make_float2(aB0, aB1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 lo = __fmul2_rn(make_float2(o[i][0], o[i][1]), a2);
        const float2 hi = __fmul2_rn(make_float2(o[i][2], o[i][3]), a2);
        o[i][0] = lo.x;
        o[i][1] = lo.y;
        o[i][2] = hi.x;
        o[i][3] = hi.y;
      }
    }
    // P^T fragments: column g of head A's product is P_A[g] on lanes g < 4; column g of head
    // B's product is P_B[g - 4], owned by lane - 16, on lanes g >= 4
    uint32_t pA[4], pB[4];  // hi0, hi1, lo0, lo1
    Ops::split_p(x[0][0], x[0][1], pA[0], pA[2]);
    Ops::split_p(x[0][2], x[0][3], pA[1], pA[3]);
    Ops::split_p(x[1][0], x[1][1], pB[0], pB[2]);
    Ops::split_p(x[1][2], x[1][3], pB[1], pB[3]);
    const bool low = g < 4;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t from = __shfl_xor_sync(kFullMask, pB[k], 16);
      pA[k] = low ? pA[k] : 0u;
      pB[k] = low ? 0u : from;
    }
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;
    if (kPartial) Ops::keep_masks(t4, n_valid, keep_lo, keep_hi);
    Ops::pv(o, vs, vsc, ROW_SCALES, v_off, g, t4, pA[0], pA[1], pA[2], pA[3], keep_lo,
            keep_hi);
    Ops::pv(o, vs + Ops::TILE_BYTES, vsc + HEAD_SCALES, ROW_SCALES, v_off, g, t4, pB[0],
            pB[1], pB[2], pB[3], keep_lo, keep_hi);
  }

  // lj[j], mj[j] of every unit head j < 2 GH on every lane.
  __device__ __forceinline__ void reduce(float* lj, float* mj) {
    float l[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      l[u] = l_run[u];
      l[u] += __shfl_xor_sync(kFullMask, l[u], 1);
      l[u] += __shfl_xor_sync(kFullMask, l[u], 2);
    }
#pragma unroll
    for (int j = 0; j < GH; ++j) {
      lj[j] = __shfl_sync(kFullMask, l[0], 4 * j);
      mj[j] = __shfl_sync(kFullMask, m_run[0], 4 * j);
      lj[GH + j] = __shfl_sync(kFullMask, l[1], 4 * j);
      mj[GH + j] = __shfl_sync(kFullMask, m_run[1], 4 * j);
    }
    const int src = 8 * (t4 & 1);
    const float lA0 = __shfl_sync(kFullMask, l[0], src);
    const float lA1 = __shfl_sync(kFullMask, l[0], src + 4);
    const float lB0 = __shfl_sync(kFullMask, l[1], src);
    const float lB1 = __shfl_sync(kFullMask, l[1], src + 4);
    l_cols[0] = t4 < 2 ? lA0 : lB0;
    l_cols[1] = t4 < 2 ? lA1 : lB1;
  }

  // Calls f(unit head, d, values, 2, l of the head) for this lane's output pairs.
  template <typename F>
  __device__ __forceinline__ void for_each_out(const float*, F&& f) const {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        const int n = 2 * t4 + jj;               // output column
        const int local = n & 3;                 // head within its kv-head
        const int j = n < 4 ? local : GH + local;  // unit head
        if (local < GH) {
          const float v[2] = {o[i][jj], o[i][2 + jj]};
          f(j, Ops::d_of(i, g), v, 2, l_cols[jj]);
        }
      }
    }
  }
  __device__ __forceinline__ bool writes_ml(int lane) const { return lane == 0; }
};

}  // namespace pda
