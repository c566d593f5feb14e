// pda_device.cuh -- device primitives for the sm_103a kernels: mbarriers, TMA loads,
// bounded waits, bf16 unpacking and warp helpers. Inline PTX only; no library code.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pda.h"

namespace pda {

constexpr unsigned kFullMask = 0xffffffffu;

// A pipeline wait gives up after this many nanoseconds of %globaltimer and reports
// PDA_DEVERR_TIMEOUT instead of spinning forever.
constexpr unsigned long long kWaitLimitNs = 1000000000ull;

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later async-proxy
// (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete; false after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) return false;
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* tm) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tm)) : "memory");
}

// 3-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_addr(bar)),
      "l"(policy)
      : "memory");
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* tm, int c0, int c1,
                                            int c2, int c3, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
      "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// 4-byte asynchronous copy global -> shared (generic proxy; visible to the issuing thread
// after cp_async_wait_all).
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------- math helpers
// 2^x with the hardware approximation (ex2.approx, relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The two bf16 values packed in a 32-bit word, widened exactly to fp32.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void atomic_or_error(int32_t* error_word, int32_t bits) {
  if (error_word != nullptr) atomicOr(error_word, bits);
}

// ---------------------------------------------------------------- element access
// FP8 E4M3 code (the OCP format with no infinities), one byte.
struct fp8e4m3 {
  uint8_t bits;
};
// Two FP4 E2M1 codes per byte (even element in the low nibble); the values of a row come
// with one E4M3 scale per 16 elements, held in a separate tensor.
struct nvfp4 {
  uint8_t bits;
};

template <typename T>
struct Elem;

// Each lane moves kVec elements per access; load() widens them exactly to fp32.
template <>
struct Elem<float> {
  static constexpr int kBits = 32;
  static constexpr int kBytes = 4;
  static constexpr int kVec = 4;  // one 16-byte access
  static __device__ __forceinline__ void load(const void* p, float* out) {
    const float4 v = *reinterpret_cast<const float4*>(p);
    out[0] = v.x;
    out[1] = v.y;
    out[2] = v.z;
    out[3] = v.w;
  }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kBits = 16;
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;  // one 16-byte access
  static __device__ __forceinline__ void load(const void* p, float* out) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    out[0] = bf16_lo(v.x);
    out[1] = bf16_hi(v.x);
    out[2] = bf16_lo(v.y);
    out[3] = bf16_hi(v.y);
    out[4] = bf16_lo(v.z);
    out[5] = bf16_hi(v.z);
    out[6] = bf16_lo(v.w);
    out[7] = bf16_hi(v.w);
  }
};

template <>
struct Elem<__half> {
  static constexpr int kBits = 16;
  static constexpr int kBytes = 2;
  static constexpr int kVec = 8;  // one 16-byte access
  static __device__ __forceinline__ void load(const void* p, float* out) {
    const uint4 v = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[i]));
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
};

// Four E4M3 codes in a 32-bit word, widened exactly (E4M3 values are all exact in fp16).
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float* out) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  out[0] = a.x;
  out[1] = a.y;
  out[2] = b.x;
  out[3] = b.y;
}

template <>
struct Elem<fp8e4m3> {
  static constexpr int kBits = 8;
  static constexpr int kBytes = 1;
  static constexpr int kVec = 8;  // one 8-byte access (keeps the bf16 lane geometry)
  static __device__ __forceinline__ void load(const void* p, float* out) {
    const uint2 v = *reinterpret_cast<const uint2*>(p);
    e4m3x4_to_f32(v.x, out);
    e4m3x4_to_f32(v.y, out + 4);
  }
};

// One E4M3 code (in the low byte of w) widened exactly to fp32.
__device__ __forceinline__ float e4m3_to_f32(uint32_t w) {
  uint32_t h;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t}"
      : "=r"(h)
      : "r"(w & 0xffu));
  return __half2float(__ushort_as_half(static_cast<unsigned short>(h & 0xffffu)));
}

template <>
struct Elem<nvfp4> {
  static constexpr int kBits = 4;
  static constexpr int kVec = 8;  // one 4-byte access: 8 codes of one 16-element block
  // The raw E2M1 values (without the block scale), widened exactly to fp32.
  static __device__ __forceinline__ void load(const void* p, float* out) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    uint32_t h[4];
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
        : "r"(w));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[i]));
      out[2 * i] = f.x;
      out[2 * i + 1] = f.y;
    }
  }
};

// ---------------------------------------------------------------- tensor-core helpers
// D += A * B for one 16x8x16 tile, fp16 operands, fp32 accumulators (register fragments).
// a: rows (g, g+8) x k pairs (2t, 2t+8) as four f16x2 words; b: k pairs (2t, 2t+8) of
// column g; d/c: (row g, cols 2t, 2t+1), (row g+8, cols 2t, 2t+1), with g = lane / 4 and
// t = lane % 4.
__device__ __forceinline__ void mma_f16_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, "
      "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four 8x8 matrices of 16-bit elements from shared memory, transposed: lane 8i + j gives
// the address of row j of matrix i; afterwards word i of lane (g, t) holds elements
// (row 2t, col g) in its low half and (row 2t + 1, col g) in its high half.
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t* r, const void* row_addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_addr(row_addr))
               : "memory");
}

// Byte permute: byte i of the result is byte sel_i (0-7) of the pair {a, b}.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Four E4M3 codes -> two f16x2 words (codes 0,1 -> lo; codes 2,3 -> hi), exact.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// Two E4M3 codes in the low 16 bits of w -> one f16x2 word (low byte -> low half), exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
  uint32_t h;
  asm("{\n\t.reg .b16 l, u;\n\t"
      "mov.b32 {l, u}, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t}"
      : "=r"(h)
      : "r"(w));
  return h;
}

// Eight E2M1 codes (four bytes, even element in each low nibble) -> four f16x2 words,
// word i holding the two codes of byte i (low nibble -> low half), exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t* h) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t f16x2_bits(__half2 v) {
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ __half2 as_half2(uint32_t w) {
  return *reinterpret_cast<__half2*>(&w);
}

// Address of element `off` of a row of T that starts at `base`.
template <typename T>
__device__ __forceinline__ const void* elem_ptr(const void* base, int off) {
  return reinterpret_cast<const unsigned char*>(base) + (off * Elem<T>::kBits) / 8;
}

// Loads n elements of type T (n a multiple of Elem<T>::kVec) widened to fp32.
template <typename T, int n>
__device__ __forceinline__ void load_elems(const T* p, float* out) {
  static_assert(n % Elem<T>::kVec == 0, "whole accesses");
#pragma unroll
  for (int i = 0; i < n; i += Elem<T>::kVec) Elem<T>::load(p + i, out + i);
}

}  // namespace pda
