// warp_attn_tc.cuh -- one warp's tile step on the tensor cores, for quantised caches
// (FP8 E4M3, and NVFP4: E2M1 codes with one E4M3 scale per 16 elements) at D = 128.
//
// A tile is one physical block (16 tokens) of one kv-head; the G (2 to 8) query heads of
// that kv-head go through it together. Per tile the warp computes, with mma.sync m16n8k16
// (fp16 operands, fp32 accumulators):
//   S  = Q K^T    M = heads (G real, padded to 16), N = 16 tokens (two n-tiles), K = d;
//   O^T += V^T P^T  M = d (eight m-tiles of 16), N = heads (8), K = 16 tokens.
// The accumulator of S (row = head g, columns = token pairs 2t, 2t+1) has exactly the layout
// of the P^T operand (column = head g, k pairs = tokens 2t, 2t+1), so the probabilities go
// from the softmax into the second product without any exchange between lanes.
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
// Shared-memory layout: the TMA writes each 16-row tile with the 128-byte swizzle (FP8,
// 128-byte rows: 16-byte chunk c of row r lands at chunk c ^ (r & 7)) or the 64-byte
// swizzle (NVFP4, 64-byte rows: chunk c ^ ((r >> 1) & 3)), which makes every load below
// free of bank conflicts. The element order along d inside a k-step is permuted (the same
// permutation for q and K), which leaves the dot products unchanged.
#pragma once

#include <math.h>
#include <type_traits>

#include "pda_device.cuh"

#ifndef PDA_TC_QK_SPLIT
#define PDA_TC_QK_SPLIT 0  // 1: even and odd k-steps of S = Q K^T accumulate separately
#endif

namespace pda {

template <typename KV, int D, int G>
struct WarpAttnTC {
  static_assert(D == 128, "tensor-core tile step is laid out for D = 128");
  static_assert(G == 2 || G == 4 || G == 8, "2 to 8 heads per kv-head (G = 1 is a GEMV)");
  static constexpr bool FP4 = std::is_same<KV, nvfp4>::value;
  static_assert(FP4 || std::is_same<KV, fp8e4m3>::value, "quantised caches only");
  static constexpr int ROW_BYTES = FP4 ? D / 2 : D;  // bytes of one K or V row
  static constexpr int ROW_SCALES = D / 16;           // NVFP4 scale bytes per row
  // The max a head's running maximum may lag the true one by (log2 units): probabilities
  // then stay below 2^8, well inside fp16, and the output is rescaled only when a new
  // maximum exceeds the old by more than this.
  static constexpr float kLag = 8.f;

  int g, t4;
  uint32_t qa[8][2];  // q of head g as A fragments: k-step s, k pairs (2t4, 2t4 + 8)
  float o[8][4];      // O^T accumulators: m-tile i, (d row g | g + 8) x heads (2t4, 2t4+1)
  float m_run;        // running max of head g (log2 units, scaled)
  float l_run;        // this lane's share of head g's running sum
  float c;            // score scale: scale * log2(e) * k_scale * 2^qshift
  int v_off[4];       // ldmatrix row addresses of this lane inside a V tile (bytes)
  float l_cols[2];    // after reduce(): full sums of heads 2 t4 and 2 t4 + 1

  __device__ __forceinline__ void init(int lane) {
    g = lane >> 2;
    t4 = lane & 3;
    const int j = lane & 7;              // row inside the 8x8 matrix this lane addresses
    const int r = j + 8 * ((lane >> 3) & 1);  // token row of the tile
    const int ch = lane >> 4;            // second chunk of the pair
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (FP4) {
        const int chunk = 2 * q + ch;  // only q < 2 is used: four 16-byte chunks per row
        v_off[q] = r * ROW_BYTES + (((chunk ^ ((r >> 1) & 3)) & 3) << 4);
      } else {
        const int chunk = 2 * q + ch;
        v_off[q] = r * ROW_BYTES + ((chunk ^ (r & 7)) << 4);
      }
    }
  }

  // q of this warp's segment (G rows of D bf16 in shared memory), pre-scale scale_log2.
  __device__ __forceinline__ void reset(const __nv_bfloat16* q_smem, float scale_log2) {
    float qv[32];
    if (g < G) {
      const uint4* src = reinterpret_cast<const uint4*>(q_smem + g * D + 32 * t4);
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
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) qv[i] = 0.f;
    }
    // power-of-two shift that brings max |q| below 2^15 (fp16 range)
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(qv[i]));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, m));
    const int e = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127;
    const int shift = e > 14 ? (e - 14 < 126 ? e - 14 : 126) : 0;
    const float down = __uint_as_float(static_cast<uint32_t>(127 - shift) << 23);
    c = scale_log2 * __uint_as_float(static_cast<uint32_t>(127 + shift) << 23);
    // k-step s holds d = 32 t4 + 4 s + {0, 1} (first pair) and + {2, 3} (second pair)
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      qa[s][0] = f16x2_bits(__floats2half2_rn(qv[4 * s] * down, qv[4 * s + 1] * down));
      qa[s][1] = f16x2_bits(__floats2half2_rn(qv[4 * s + 2] * down, qv[4 * s + 3] * down));
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) o[i][e2] = 0.f;
    m_run = -INFINITY;
    l_run = 0.f;
  }

  // ks/vs: the tile's K and V rows (swizzled); ksc/vsc: NVFP4 block scales, [16][D/16].
  template <bool kPartial>
  __device__ __forceinline__ void tile(const KV* ks_, const KV* vs_, const uint8_t* ksc,
                                       const uint8_t* vsc, int n_valid) {
    const unsigned char* ks = reinterpret_cast<const unsigned char*>(ks_);
    const unsigned char* vs = reinterpret_cast<const unsigned char*>(vs_);

    // ---- S = Q K^T: n-tile nt covers tokens 8 nt .. 8 nt + 7 (token g of it on this lane)
    // with PDA_TC_QK_SPLIT the odd k-steps go to a second accumulator (two shorter chains)
    float sc[2][4], sc_odd[2][4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[nt][e] = sc_odd[nt][e] = 0.f;
      const int r = g + 8 * nt;
      if constexpr (FP4) {
        // 16 bytes = d 32 t4 .. 32 t4 + 31; byte 2s (+1) holds k-step s's first (second) pair
        const uint4 w = *reinterpret_cast<const uint4*>(
            ks + r * ROW_BYTES + ((t4 ^ ((r >> 1) & 3)) << 4));
        const uint32_t sp = e4m3x2_to_f16x2(
            *reinterpret_cast<const uint16_t*>(ksc + r * ROW_SCALES + 2 * t4));
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
            mma_f16_16816((PDA_TC_QK_SPLIT && (s & 1)) ? sc_odd[nt] : sc[nt], qa[s][0], 0u,
                          qa[s][1], 0u, b0, b1);
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
            mma_f16_16816((PDA_TC_QK_SPLIT && (u & 1)) ? sc_odd[nt] : sc[nt],
                          qa[4 * hh + u][0], 0u, qa[4 * hh + u][1], 0u, b0, b1);
          }
        }
      }
      if (PDA_TC_QK_SPLIT) {
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] += sc_odd[nt][e];
      }
    }

    // ---- online softmax of head g over tokens (2t4, 2t4+1, 8+2t4, 9+2t4)
    float x[4] = {sc[0][0] * c, sc[0][1] * c, sc[1][0] * c, sc[1][1] * c};
    if (kPartial) {
      const int tok[4] = {2 * t4, 2 * t4 + 1, 8 + 2 * t4, 9 + 2 * t4};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (tok[e] >= n_valid) x[e] = -INFINITY;
    }
    float tmax = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 1));
    tmax = fmaxf(tmax, __shfl_xor_sync(kFullMask, tmax, 2));
    const bool grow = tmax > m_run + kLag;
    if (__any_sync(kFullMask, grow)) {
      const float m_new = grow ? tmax : m_run;
      const float alpha = ex2(m_run - m_new);  // 0 on the first tile, 1 where m is kept
      m_run = m_new;
      l_run *= alpha;
      // the O^T columns of this lane are heads 2 t4 and 2 t4 + 1 (lanes 8 t4, 8 t4 + 4)
      const float a0 = __shfl_sync(kFullMask, alpha, 8 * t4);
      const float a1 = __shfl_sync(kFullMask, alpha, 8 * t4 + 4);
      const float2 a2 = make_float2(a0, a1);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float2 lo = __fmul2_rn(make_float2(o[i][0], o[i][1]), a2);
        float2 hi = __fmul2_rn(make_float2(o[i][2], o[i][3]), a2);
        o[i][0] = lo.x;
        o[i][1] = lo.y;
        o[i][2] = hi.x;
        o[i][3] = hi.y;
      }
    }
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) p[e] = ex2(x[e] - m_run);
    l_run += (p[0] + p[1]) + (p[2] + p[3]);
    // tokens (2t4, 2t4+1) and (8+2t4, 9+2t4): high fp16 parts, then the remainders
    const __half2 h0 = __floats2half2_rn(p[0], p[1]);
    const __half2 h1 = __floats2half2_rn(p[2], p[3]);
    const float2 r0 = __half22float2(h0), r1 = __half22float2(h1);
    const uint32_t pb0 = f16x2_bits(h0), pb1 = f16x2_bits(h1);
    const uint32_t pl0 = f16x2_bits(__floats2half2_rn(p[0] - r0.x, p[1] - r0.y));
    const uint32_t pl1 = f16x2_bits(__floats2half2_rn(p[2] - r1.x, p[3] - r1.y));

    // ---- O^T += V^T P^T. ldmatrix.trans hands this lane, per 16-byte chunk of the rows
    // 0-7 (and 8-15), two bytes of token 2t4 and the same two bytes of token 2t4 + 1.
    uint32_t keep_lo = 0xffffffffu, keep_hi = 0xffffffffu;  // per token half (partial)
    if (kPartial) {
      const bool a = 2 * t4 < n_valid, b = 2 * t4 + 1 < n_valid;
      const bool cc = 8 + 2 * t4 < n_valid, d = 9 + 2 * t4 < n_valid;
      if constexpr (FP4) {
        keep_lo = (a ? 0x0000ffffu : 0u) | (b ? 0xffff0000u : 0u);
        keep_hi = (cc ? 0x0000ffffu : 0u) | (d ? 0xffff0000u : 0u);
      } else {
        keep_lo = (a ? 0x00ff00ffu : 0u) | (b ? 0xff00ff00u : 0u);
        keep_hi = (cc ? 0x00ff00ffu : 0u) | (d ? 0xff00ff00u : 0u);
      }
    }
    if constexpr (FP4) {
      // scale pairs (token t0, token t0 + 1) of this lane's block in chunk c: rows 2t4(+1)
      // and 8 + 2t4 (+1); the block is 2c + g / 4
      const uint2 w0 = *reinterpret_cast<const uint2*>(vsc + (2 * t4) * ROW_SCALES);
      const uint2 w1 = *reinterpret_cast<const uint2*>(vsc + (2 * t4 + 1) * ROW_SCALES);
      const uint2 w2 = *reinterpret_cast<const uint2*>(vsc + (8 + 2 * t4) * ROW_SCALES);
      const uint2 w3 = *reinterpret_cast<const uint2*>(vsc + (9 + 2 * t4) * ROW_SCALES);
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

  // d of row g of m-tile i (row g + 8 is d + 1).
  __device__ __forceinline__ int d_of(int i) const {
    return FP4 ? 32 * (i >> 1) + 4 * g + 2 * (i & 1) : 16 * i + 2 * g;
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
          f(j, d_of(i), v, 2, l_cols[jj]);
        }
      }
    }
  }
  __device__ __forceinline__ bool writes_ml(int lane) const { return lane == 0; }
};

}  // namespace pda
