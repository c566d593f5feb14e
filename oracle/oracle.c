/*
 * oracle.c -- plain fp64 CPU reference for decode attention over a paged KV cache,
 * for the per-step KV append, and for the gather of one request's blocks into a
 * contiguous transfer buffer.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's CPU
 * baseline load this file. It shares no code, header, table or helper with the CUDA
 * library; it is written from the problem statement alone:
 *
 *  - Decode step (page "Disaggregated LLM Serving: from PD disaggregation to attention
 *    offload", sec. 1 "starting from autoregressive generation", item 2 of the second
 *    list): each decode step reads the whole cached K/V history of the request and
 *    appends the new token's K/V to it.
 *  - Paged layout (page "From PagedAttention to Prefill-Decode disaggregation", sec. 2.2
 *    steps 1-2): the cache is split into fixed-size physical blocks, each holding the K
 *    and V of a fixed number of tokens; a per-request table maps logical block i of the
 *    request to a physical block, and the physical blocks need not be contiguous.
 *  - Shared prefixes (same page, sec. 2.3): several requests may map to the same
 *    physical blocks; attention only reads them.
 *  - Request-level transfer of the KV (page on goodput and PD disaggregation,
 *    0539edu.com, sec. 5.4 "request-level granularity"): after prefill the whole KV of
 *    a request is sent in one piece, which needs it gathered into one buffer (pack) and,
 *    on the receiving instance, scattered into the blocks allocated there (unpack).
 *
 * Attention is the plain definition, with no online or split softmax:
 *      s_t = scale * sum_d q[d] * K_t[d]            for t < L
 *      p_t = exp(s_t - max_u s_u) / sum_u exp(s_u - max_u s_u)
 *      out = sum_t p_t * V_t
 * Everything is computed in double; stored bf16/fp16/fp32 inputs are upcast exactly, and FP8
 * E4M3 codes are decoded exactly and multiplied by their tensor's scale. Quantised KV
 * caches (page "From PagedAttention to Prefill-Decode disaggregation", sec. 6.2: a 4-bit KV
 * cache dequantised to FP8 before attention) are read through that decode.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - Cache tensors are dense row-major [num_blocks, block_size, H_kv, D].
 *  - Query head h reads kv-head h / (H / H_kv) (contiguous grouping for GQA).
 *  - Token t of request b lives in physical block block_tables[b][t / block_size] at
 *    row t % block_size.
 *  - context_lens counts the tokens after this step's append.
 *  - A request with context length 0 yields a zero row; a negative length, a length
 *    beyond the table's capacity or a block id outside [0, num_blocks) yields NaN rows
 *    for that request and the status ORC_ERR_DATA.
 *
 * The functions oracle_attention_partial and oracle_lse_combine exist only so that a
 * test can show that the split-and-merge arithmetic gives back the plain definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8_E4M3 = 2, ORC_NVFP4 = 3, ORC_F16 = 4 };
enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_DATA = 4 };

static size_t orc_elem_size(int dtype) {
  return (dtype == ORC_BF16 || dtype == ORC_F16) ? 2u : (dtype == ORC_FP8_E4M3 ? 1u : 4u);
}

static int orc_dtype_ok(int dtype) {
  return dtype == ORC_F32 || dtype == ORC_BF16 || dtype == ORC_FP8_E4M3 || dtype == ORC_F16;
}

/*
 * IEEE 754 binary16: sign bit, 5 exponent bits with bias 15, 10 mantissa bits. Exponent 0
 * encodes the subnormals m * 2^-24; exponent 31 is infinity (m = 0) or NaN; every other
 * code is (1 + m/1024) * 2^(e - 15) = (1024 + m) * 2^(e - 25).
 */
static double orc_f16(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double mag;
  if (e == 31)
    mag = m ? NAN : INFINITY;
  else if (e == 0)
    mag = ldexp((double)m, -24);
  else
    mag = ldexp((double)(1024 + m), e - 25);
  return sign ? -mag : mag;
}

double oracle_decode_f16(int bits) { return orc_f16((uint16_t)(bits & 0xffff)); }

/*
 * FP8 E4M3 (the OCP 8-bit format with no infinities): sign bit, 4 exponent bits with bias
 * 7, 3 mantissa bits. Exponent 0 encodes subnormals m/8 * 2^-6; exponent 15 with mantissa 7
 * is NaN; every other code is (1 + m/8) * 2^(e - 7). Largest finite magnitude 448.
 */
static double orc_e4m3(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  if (e == 15 && m == 7) return NAN;
  const double mag = (e == 0) ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

double oracle_decode_e4m3(int code) { return orc_e4m3((uint8_t)(code & 255)); }

/*
 * FP4 E2M1: sign bit, 2 exponent bits with bias 1, 1 mantissa bit. Exponent 0 encodes the
 * subnormals 0 and 0.5; otherwise (1 + m/2) * 2^(e - 1). Magnitudes 0, 0.5, 1, 1.5, 2, 3,
 * 4, 6; no infinities or NaN.
 */
static double orc_e2m1(unsigned code) {
  const int sign = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
  const double mag = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
  return sign ? -mag : mag;
}

double oracle_decode_e2m1(int code) { return orc_e2m1((unsigned)(code & 15)); }

/* Exact upcast of stored element idx. A bf16 value is the upper 16 bits of a binary32. */
static double orc_load(const void* base, size_t idx, int dtype) {
  if (dtype == ORC_FP8_E4M3) return orc_e4m3(((const uint8_t*)base)[idx]);
  if (dtype == ORC_F16) {
    uint16_t h;
    memcpy(&h, (const char*)base + idx * 2u, 2u);
    return orc_f16(h);
  }
  if (dtype == ORC_BF16) {
    uint16_t h;
    memcpy(&h, (const char*)base + idx * 2u, 2u);
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, 4u);
    return (double)f;
  }
  float f;
  memcpy(&f, (const char*)base + idx * 4u, 4u);
  return (double)f;
}

int oracle_version(void) { return 1; }

/*
 * KV append: for each request b whose slot s = slot_mapping[b] is >= 0, write the
 * new token's K and V (H_kv x D elements each) to block s / block_size, row
 * s % block_size. Bitwise copy. A slot >= num_blocks * block_size is an error and is
 * skipped; a negative slot means "no token" (padding) and is skipped silently.
 */
int oracle_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                     const int32_t* slot_mapping, int B, int H_kv, int D, int block_size,
                     int num_blocks, int dtype) {
  if (B < 0 || H_kv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 || !orc_dtype_ok(dtype))
    return ORC_ERR_ARG;
  const size_t e = orc_elem_size(dtype);
  const size_t row_bytes = (size_t)H_kv * (size_t)D * e;
  int status = ORC_OK;
  for (int b = 0; b < B; ++b) {
    const int32_t s = slot_mapping[b];
    if (s < 0) continue;
    if ((int64_t)s >= (int64_t)num_blocks * block_size) {
      status = ORC_ERR_DATA;
      continue;
    }
    const int64_t block = s / block_size;
    const int64_t offset = s % block_size;
    const size_t dst = ((size_t)block * (size_t)block_size + (size_t)offset) * row_bytes;
    memcpy((char*)k_cache + dst, (const char*)k_new + (size_t)b * row_bytes, row_bytes);
    memcpy((char*)v_cache + dst, (const char*)v_new + (size_t)b * row_bytes, row_bytes);
  }
  return status;
}

/*
 * KV pack: out[t, 0, h, :] = K of logical token t, out[t, 1, h, :] = V of token t, for
 * t < context_len, with token t found through block_table_row as for attention.
 * Bitwise copy into a dense [context_len, 2, H_kv, D] buffer.
 */
int oracle_kv_pack_blocks(void* out, const void* k_cache, const void* v_cache,
                          const int32_t* block_table_row, int context_len, int H_kv, int D,
                          int block_size, int num_blocks, int dtype) {
  if (context_len < 0 || H_kv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 ||
      !orc_dtype_ok(dtype))
    return ORC_ERR_ARG;
  const size_t e = orc_elem_size(dtype);
  const size_t row_bytes = (size_t)H_kv * (size_t)D * e;
  for (int t = 0; t < context_len; ++t) {
    const int32_t block = block_table_row[t / block_size];
    if (block < 0 || block >= num_blocks) return ORC_ERR_DATA;
    const size_t src = ((size_t)block * (size_t)block_size + (size_t)(t % block_size)) * row_bytes;
    char* dst = (char*)out + (size_t)t * 2u * row_bytes;
    memcpy(dst, (const char*)k_cache + src, row_bytes);
    memcpy(dst + row_bytes, (const char*)v_cache + src, row_bytes);
  }
  return ORC_OK;
}

/*
 * KV unpack, the receiving side of a request-level transfer: for t < context_len, write
 * in[t, 0, h, :] to the K row and in[t, 1, h, :] to the V row of logical token t, token t
 * being row t % block_size of physical block block_table_row[t / block_size]. Bitwise.
 * A block id out of range is an error; that token is skipped.
 */
int oracle_kv_unpack_blocks(const void* in, void* k_cache, void* v_cache,
                            const int32_t* block_table_row, int context_len, int H_kv, int D,
                            int block_size, int num_blocks, int dtype) {
  if (context_len < 0 || H_kv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 ||
      !orc_dtype_ok(dtype))
    return ORC_ERR_ARG;
  const size_t e = orc_elem_size(dtype);
  const size_t row_bytes = (size_t)H_kv * (size_t)D * e;
  int status = ORC_OK;
  for (int t = 0; t < context_len; ++t) {
    const int32_t block = block_table_row[t / block_size];
    if (block < 0 || block >= num_blocks) {
      status = ORC_ERR_DATA;
      continue;
    }
    const size_t dst = ((size_t)block * (size_t)block_size + (size_t)(t % block_size)) * row_bytes;
    const char* src = (const char*)in + (size_t)t * 2u * row_bytes;
    memcpy((char*)k_cache + dst, src, row_bytes);
    memcpy((char*)v_cache + dst, src + row_bytes, row_bytes);
  }
  return status;
}

/*
 * The same three copies for an NVFP4 block-scale cache, laid out per block and kv-head:
 * [num_blocks, H_kv, block_size, row_bytes] (row_bytes = D/16 scale bytes). The new rows
 * and the transfer buffer keep the token-major order of the data: new [B, H_kv, row_bytes],
 * buffer [context_len, 2, H_kv, row_bytes]. Scale row of (token slot s, kv-head h): block
 * s / block_size, offset s % block_size, at ((block * H_kv + h) * block_size + offset).
 */
static size_t orc_scale_row(int64_t block, int64_t offset, int h, int H_kv, int block_size) {
  return ((size_t)block * (size_t)H_kv + (size_t)h) * (size_t)block_size + (size_t)offset;
}

int oracle_kv_append_block_scales(const void* k_new, const void* v_new, void* k_scales,
                                  void* v_scales, const int32_t* slot_mapping, int B, int H_kv,
                                  int row_bytes, int block_size, int num_blocks) {
  if (B < 0 || H_kv <= 0 || row_bytes <= 0 || block_size <= 0 || num_blocks <= 0)
    return ORC_ERR_ARG;
  int status = ORC_OK;
  for (int b = 0; b < B; ++b) {
    const int32_t s = slot_mapping[b];
    if (s < 0) continue;
    if ((int64_t)s >= (int64_t)num_blocks * block_size) {
      status = ORC_ERR_DATA;
      continue;
    }
    for (int h = 0; h < H_kv; ++h) {
      const size_t dst = orc_scale_row(s / block_size, s % block_size, h, H_kv, block_size) *
                         (size_t)row_bytes;
      const size_t src = ((size_t)b * (size_t)H_kv + (size_t)h) * (size_t)row_bytes;
      memcpy((char*)k_scales + dst, (const char*)k_new + src, (size_t)row_bytes);
      memcpy((char*)v_scales + dst, (const char*)v_new + src, (size_t)row_bytes);
    }
  }
  return status;
}

int oracle_kv_pack_block_scales(void* out, const void* k_scales, const void* v_scales,
                                const int32_t* block_table_row, int context_len, int H_kv,
                                int row_bytes, int block_size, int num_blocks) {
  if (context_len < 0 || H_kv <= 0 || row_bytes <= 0 || block_size <= 0 || num_blocks <= 0)
    return ORC_ERR_ARG;
  for (int t = 0; t < context_len; ++t) {
    const int32_t block = block_table_row[t / block_size];
    if (block < 0 || block >= num_blocks) return ORC_ERR_DATA;
    for (int h = 0; h < H_kv; ++h) {
      const size_t src =
          orc_scale_row(block, t % block_size, h, H_kv, block_size) * (size_t)row_bytes;
      char* dst = (char*)out + (((size_t)t * 2u) * (size_t)H_kv + (size_t)h) * (size_t)row_bytes;
      memcpy(dst, (const char*)k_scales + src, (size_t)row_bytes);
      memcpy(dst + (size_t)H_kv * (size_t)row_bytes, (const char*)v_scales + src,
             (size_t)row_bytes);
    }
  }
  return ORC_OK;
}

int oracle_kv_unpack_block_scales(const void* in, void* k_scales, void* v_scales,
                                  const int32_t* block_table_row, int context_len, int H_kv,
                                  int row_bytes, int block_size, int num_blocks) {
  if (context_len < 0 || H_kv <= 0 || row_bytes <= 0 || block_size <= 0 || num_blocks <= 0)
    return ORC_ERR_ARG;
  int status = ORC_OK;
  for (int t = 0; t < context_len; ++t) {
    const int32_t block = block_table_row[t / block_size];
    if (block < 0 || block >= num_blocks) {
      status = ORC_ERR_DATA;
      continue;
    }
    for (int h = 0; h < H_kv; ++h) {
      const size_t dst =
          orc_scale_row(block, t % block_size, h, H_kv, block_size) * (size_t)row_bytes;
      const char* src =
          (const char*)in + (((size_t)t * 2u) * (size_t)H_kv + (size_t)h) * (size_t)row_bytes;
      memcpy((char*)k_scales + dst, src, (size_t)row_bytes);
      memcpy((char*)v_scales + dst, src + (size_t)H_kv * (size_t)row_bytes, (size_t)row_bytes);
    }
  }
  return status;
}

/*
 * Element d of kv-head hk in row `offset` of physical block `block`, before the per-tensor
 * scale. NVFP4 (the 4-bit KV format with fine-grained E4M3 block scales, page "From
 * PagedAttention to Prefill-Decode disaggregation", sec. 6.2): the data tensor is
 * [num_blocks, block_size, H_kv, D/2] bytes holding two E2M1 codes each, element d in the low
 * nibble of byte d/2 when d is even and in the high nibble when d is odd; the scale tensor
 * holds one E4M3 byte per 16 consecutive elements, laid out per block and kv-head,
 * [num_blocks, H_kv, block_size, D/16]. The element's value is
 * e2m1(code) * e4m3(scale of its 16-element block).
 */
static double orc_kv(const void* cache, const void* block_scales, size_t block, size_t offset,
                     int block_size, int hk, int d, int H_kv, int D, int dtype) {
  const size_t r = (block * (size_t)block_size + offset) * (size_t)H_kv + (size_t)hk;
  if (dtype == ORC_NVFP4) {
    const uint8_t byte = ((const uint8_t*)cache)[r * (size_t)(D / 2) + (size_t)(d / 2)];
    const unsigned code = (d & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15);
    const size_t srow = (block * (size_t)H_kv + (size_t)hk) * (size_t)block_size + offset;
    const uint8_t sc = ((const uint8_t*)block_scales)[srow * (size_t)(D / 16) + (size_t)(d / 16)];
    return orc_e2m1(code) * orc_e4m3(sc);
  }
  return orc_load(cache, r * (size_t)D + (size_t)d, dtype);
}

/*
 * Gather the K and V of kv-head hk of request b into contiguous [L, D] arrays of
 * doubles, each element times its tensor's scale. Returns 0, or -1 when a block id is out
 * of range.
 */
static int orc_gather(double* Kc, double* Vc, const void* k_cache, const void* v_cache,
                      const void* k_bs, const void* v_bs, const int32_t* table_row, int L,
                      int hk, int H_kv, int D, int block_size, int num_blocks, int kv_dtype,
                      double k_scale, double v_scale) {
  for (int t = 0; t < L; ++t) {
    const int32_t block = table_row[t / block_size];
    if (block < 0 || block >= num_blocks) return -1;
    const size_t off = (size_t)(t % block_size);
    for (int d = 0; d < D; ++d) {
      Kc[(size_t)t * D + d] =
          orc_kv(k_cache, k_bs, (size_t)block, off, block_size, hk, d, H_kv, D, kv_dtype) * k_scale;
      Vc[(size_t)t * D + d] =
          orc_kv(v_cache, v_bs, (size_t)block, off, block_size, hk, d, H_kv, D, kv_dtype) * v_scale;
    }
  }
  return 0;
}

static void orc_fill_rows(double* out, int b, int H, int D, double value) {
  for (size_t i = 0; i < (size_t)H * D; ++i) out[(size_t)b * H * D + i] = value;
}

/*
 * Decode attention over the paged cache. out is [B, H, D] doubles. q is [B, H, D] in
 * q_dtype; caches are [num_blocks, block_size, H_kv, D] in kv_dtype; block_tables is
 * [B, max_blocks]; context_lens is [B]. scale is the binary32 value a caller passes to
 * the kernel, used upcast to double. A stored K element means its decoded value times
 * k_scale, a V element its value times v_scale (1 for unquantised caches; for FP8 caches
 * the per-tensor scales of the quantisation). num_threads <= 0 uses the OpenMP default.
 */
static int orc_attention(double* out, const void* q, const void* k_cache, const void* v_cache,
                         const void* k_bs, const void* v_bs, const int32_t* block_tables,
                         int max_blocks, const int32_t* context_lens, int B, int H, int H_kv,
                         int D, int block_size, int num_blocks, float scale, int q_dtype,
                         int kv_dtype, float k_scale, float v_scale, int num_threads) {
  if (B < 0 || H <= 0 || H_kv <= 0 || H % H_kv != 0 || D <= 0 || block_size <= 0 ||
      num_blocks <= 0 || max_blocks < 0 || !orc_dtype_ok(q_dtype) ||
      !(orc_dtype_ok(kv_dtype) || (kv_dtype == ORC_NVFP4 && D % 16 == 0 && k_bs && v_bs)))
    return ORC_ERR_ARG;
  const int group = H / H_kv;
  const double sc = (double)scale;
  int status = ORC_OK;
  const int64_t n_pairs = (int64_t)B * H_kv;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1) reduction(max : status)
  for (int64_t pair = 0; pair < n_pairs; ++pair) {
    const int b = (int)(pair / H_kv);
    const int hk = (int)(pair % H_kv);
    const int L = context_lens[b];
    if (L < 0 || (int64_t)L > (int64_t)max_blocks * block_size) {
      if (hk == 0) orc_fill_rows(out, b, H, D, NAN);
      status = ORC_ERR_DATA;
      continue;
    }
    if (L == 0) {
      for (int j = 0; j < group; ++j)
        for (int d = 0; d < D; ++d) out[((size_t)b * H + (size_t)hk * group + j) * D + d] = 0.0;
      continue;
    }
    double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)L);
    const int32_t* row = block_tables + (size_t)b * max_blocks;
    if (orc_gather(Kc, Vc, k_cache, v_cache, k_bs, v_bs, row, L, hk, H_kv, D, block_size,
                   num_blocks, kv_dtype, (double)k_scale, (double)v_scale) != 0) {
      for (int j = 0; j < group; ++j)
        for (int d = 0; d < D; ++d)
          out[((size_t)b * H + (size_t)hk * group + j) * D + d] = NAN;
      status = ORC_ERR_DATA;
      free(Kc);
      free(Vc);
      free(s);
      continue;
    }
    for (int j = 0; j < group; ++j) {
      const int h = hk * group + j; /* query head h reads kv-head h / group == hk */
      const size_t qoff = ((size_t)b * H + h) * (size_t)D;
      double mx = -INFINITY;
      for (int t = 0; t < L; ++t) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += orc_load(q, qoff + d, q_dtype) * Kc[(size_t)t * D + d];
        s[t] = sc * dot;
        if (s[t] > mx) mx = s[t];
      }
      double den = 0.0;
      for (int t = 0; t < L; ++t) den += exp(s[t] - mx);
      double* o = out + qoff;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (int t = 0; t < L; ++t) {
        const double p = exp(s[t] - mx) / den;
        for (int d = 0; d < D; ++d) o[d] += p * Vc[(size_t)t * D + d];
      }
    }
    free(Kc);
    free(Vc);
    free(s);
  }
  return status;
}

int oracle_paged_decode_attention(double* out, const void* q, const void* k_cache,
                                  const void* v_cache, const int32_t* block_tables,
                                  int max_blocks, const int32_t* context_lens, int B, int H,
                                  int H_kv, int D, int block_size, int num_blocks, float scale,
                                  int q_dtype, int kv_dtype, float k_scale, float v_scale,
                                  int num_threads) {
  return orc_attention(out, q, k_cache, v_cache, NULL, NULL, block_tables, max_blocks,
                       context_lens, B, H, H_kv, D, block_size, num_blocks, scale, q_dtype,
                       kv_dtype, k_scale, v_scale, num_threads);
}

/*
 * The same attention over an NVFP4 cache: k_data/v_data are [num_blocks, block_size, H_kv,
 * D/2] bytes, k_block_scales/v_block_scales [num_blocks, H_kv, block_size, D/16] E4M3 bytes;
 * a K element means e2m1(code) * e4m3(block scale) * k_scale (see orc_kv).
 */
int oracle_paged_decode_attention_nvfp4(double* out, const void* q, const void* k_data,
                                        const void* v_data, const void* k_block_scales,
                                        const void* v_block_scales, const int32_t* block_tables,
                                        int max_blocks, const int32_t* context_lens, int B,
                                        int H, int H_kv, int D, int block_size, int num_blocks,
                                        float scale, int q_dtype, float k_scale, float v_scale,
                                        int num_threads) {
  return orc_attention(out, q, k_data, v_data, k_block_scales, v_block_scales, block_tables,
                       max_blocks, context_lens, B, H, H_kv, D, block_size, num_blocks, scale,
                       q_dtype, ORC_NVFP4, k_scale, v_scale, num_threads);
}

/*
 * Unnormalised attention of query head h of request b over tokens [t0, t1):
 *   m = max_t s_t,  l = sum_t exp(s_t - m),  o = sum_t exp(s_t - m) V_t.
 * This is the per-piece state of a sequence split; it is here only to show, in a test,
 * that merging pieces gives back the plain definition above.
 */
int oracle_attention_partial(double* m_out, double* l_out, double* o_out, const void* q,
                             const void* k_cache, const void* v_cache,
                             const int32_t* block_tables, int max_blocks, int b, int h, int t0,
                             int t1, int H, int H_kv, int D, int block_size, int num_blocks,
                             float scale, int q_dtype, int kv_dtype) {
  if (t0 < 0 || t1 <= t0 || H % H_kv != 0 || !orc_dtype_ok(q_dtype) || !orc_dtype_ok(kv_dtype))
    return ORC_ERR_ARG;
  const int hk = h / (H / H_kv);
  const int L = t1;
  double* Kc = (double*)malloc(sizeof(double) * (size_t)L * D);
  double* Vc = (double*)malloc(sizeof(double) * (size_t)L * D);
  const int32_t* row = block_tables + (size_t)b * max_blocks;
  if (orc_gather(Kc, Vc, k_cache, v_cache, NULL, NULL, row, L, hk, H_kv, D, block_size,
                 num_blocks, kv_dtype, 1.0, 1.0) != 0) {
    free(Kc);
    free(Vc);
    return ORC_ERR_DATA;
  }
  const size_t qoff = ((size_t)b * H + h) * (size_t)D;
  double mx = -INFINITY;
  double* s = (double*)malloc(sizeof(double) * (size_t)L);
  for (int t = t0; t < t1; ++t) {
    double dot = 0.0;
    for (int d = 0; d < D; ++d) dot += orc_load(q, qoff + d, q_dtype) * Kc[(size_t)t * D + d];
    s[t] = (double)scale * dot;
    if (s[t] > mx) mx = s[t];
  }
  double l = 0.0;
  for (int d = 0; d < D; ++d) o_out[d] = 0.0;
  for (int t = t0; t < t1; ++t) {
    const double w = exp(s[t] - mx);
    l += w;
    for (int d = 0; d < D; ++d) o_out[d] += w * Vc[(size_t)t * D + d];
  }
  *m_out = mx;
  *l_out = l;
  free(Kc);
  free(Vc);
  free(s);
  return ORC_OK;
}

/*
 * Log-sum-exp merge of n pieces (m_j, l_j, o_j[D]):
 *   M = max_j m_j,  L = sum_j l_j exp(m_j - M),  out = sum_j o_j exp(m_j - M) / L.
 */
int oracle_lse_combine(int n, const double* m, const double* l, const double* o, int D,
                       double* out) {
  if (n <= 0 || D <= 0) return ORC_ERR_ARG;
  double M = -INFINITY;
  for (int j = 0; j < n; ++j)
    if (m[j] > M) M = m[j];
  double Lsum = 0.0;
  for (int j = 0; j < n; ++j) Lsum += l[j] * exp(m[j] - M);
  for (int d = 0; d < D; ++d) {
    double acc = 0.0;
    for (int j = 0; j < n; ++j) acc += o[(size_t)j * D + d] * exp(m[j] - M);
    out[d] = acc / Lsum;
  }
  return ORC_OK;
}
