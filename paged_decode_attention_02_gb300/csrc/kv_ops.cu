// kv_ops.cu -- KV append (scatter of each request's new token into its slot), KV pack
// (gather of one request's scattered blocks into a contiguous transfer buffer) and KV
// unpack (the receiving side: scatter of such a buffer into freshly allocated blocks).
//
// All three are pure copies of rows of H_kv * D elements, done as 16-byte vectors with
// streaming (evict-first) loads and stores so a large pack does not flush L2.
//  * append: each decode step writes the new token's K/V (page "Disaggregated LLM
//    Serving: from PD disaggregation to attention offload", sec. 1, second list item 2)
//    into slot s = block * block_size + row, i.e. block s / block_size, row s % block_size.
//  * pack: request-level KV transfer needs the request's KV in one buffer (page on goodput
//    and PD disaggregation, 0539edu.com, sec. 5.4); out[t] = (K row, V row) of token t,
//    token t being row t % block_size of block table[t / block_size].
//  * unpack: the decode instance receives that buffer and writes it into the blocks it
//    allocated for the request (same page, sec. 3: the KV is migrated to the decode worker;
//    page "From PagedAttention to Prefill-Decode disaggregation", sec. 2.2 step 3).
//  * pack / unpack over layers: one request's blocks in every layer's cache (all layers
//    share the request's block table) in one launch -- the request-level transfer of a whole
//    model; layer-by-layer streaming (page on goodput and PD disaggregation, sec. 5.4, layer
//    granularity; page "Disaggregated LLM Serving", sec. 5.6) issues one layer at a time.
//  * the same three moves for the E4M3 block scales of an NVFP4 cache (page "From
//    PagedAttention to Prefill-Decode disaggregation", sec. 6.2), whose per-block head-major
//    layout differs from the token-major K/V rows.
#include "pda_device.cuh"
#include "pda_internal.h"

namespace pda {

__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k_new,
                                                        const uint4* __restrict__ v_new,
                                                        uint4* __restrict__ k_cache,
                                                        uint4* __restrict__ v_cache,
                                                        const int32_t* __restrict__ slots, int B,
                                                        int row_vecs, int block_size,
                                                        int num_blocks, int32_t* error_word) {
  const long long total = static_cast<long long>(B) * 2 * row_vecs;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / (2 * row_vecs));
    const int rem = static_cast<int>(i % (2 * row_vecs));
    const int which = rem / row_vecs;  // 0: K, 1: V
    const int c = rem % row_vecs;
    const int s = slots[b];
    if (s < 0) continue;  // padding
    const long long block = s / block_size;
    const long long row = s % block_size;
    if (block >= num_blocks) {
      if (rem == 0) atomic_or_error(error_word, PDA_DEVERR_SLOT);
      continue;
    }
    const size_t dst = static_cast<size_t>(block * block_size + row) * row_vecs + c;
    const size_t src = static_cast<size_t>(b) * row_vecs + c;
    if (which == 0)
      k_cache[dst] = k_new[src];
    else
      v_cache[dst] = v_new[src];
  }
}

struct PackJob {
  uint4* buf;  // the request's dense [len, 2, H_kv, D] buffer (pack: written, unpack: read)
  const int32_t* table;
  uint4* k_cache;  // the cache this job reads (pack) or writes (unpack)
  uint4* v_cache;
  int len;
};

// N: most jobs one launch carries (kernel parameter space: N * 40 bytes).
template <int N>
struct PackParams {
  int32_t* error_word;
  int n, row_vecs, block_size, num_blocks;
  PackJob jobs[N];
};

// Tokens per thread per iteration (loads in flight). Measured on the 8 longest requests of
// the GQA 32/8 workload (2.0 GB moved): pack 296 us with 8 (or 2) against 323 us with 4;
// unpack 308 us with 4 against 315 (2) and 329 (8).
#ifndef PDA_PACK_TOKENS
#define PDA_PACK_TOKENS 8
#endif
#ifndef PDA_UNPACK_TOKENS
#define PDA_UNPACK_TOKENS 4
#endif
template <bool kUnpack>
__host__ __device__ constexpr int tokens_per_iter() {
  return kUnpack ? PDA_UNPACK_TOKENS : PDA_PACK_TOKENS;
}

// Pack (cache rows -> dense buffer) or unpack (dense buffer -> cache rows).
// blockIdx.y selects the request. A token's copy is its K row then its V row, 2 * row_vecs
// 16-byte vectors; thread i of the block always moves vectors i, i + blockDim.x, ... of a
// token (so no per-vector division), for tokens_per_iter<kUnpack>() tokens at a time.
// Pack: a token in a block out of range reads as 0xFF bytes. Unpack: it is not written.
// Both set PDA_DEVERR_BLOCK_ID.
template <bool kUnpack, int N>
__global__ void __launch_bounds__(256) kv_blocks_kernel(const __grid_constant__ PackParams<N> p) {
  const PackJob job = p.jobs[blockIdx.y];
  const int rv = p.row_vecs;
  const int row2 = 2 * rv;
  const int bs = p.block_size;
  constexpr int kPackTokens = tokens_per_iter<kUnpack>();
  for (int t0 = blockIdx.x * kPackTokens; t0 < job.len; t0 += gridDim.x * kPackTokens) {
    int blk[kPackTokens];
#pragma unroll
    for (int k = 0; k < kPackTokens; ++k) {
      const int t = t0 + k;
      blk[k] = t < job.len ? job.table[t / bs] : 0;
      if (t < job.len && (blk[k] < 0 || blk[k] >= p.num_blocks)) {
        if (threadIdx.x == 0) atomic_or_error(p.error_word, PDA_DEVERR_BLOCK_ID);
        blk[k] = -1;
      }
    }
    for (int c = threadIdx.x; c < row2; c += blockDim.x) {
      const bool is_v = c >= rv;
      const int cv = is_v ? c - rv : c;
      uint4* cache = is_v ? job.v_cache : job.k_cache;
      uint4 v[kPackTokens];
#pragma unroll
      for (int k = 0; k < kPackTokens; ++k) {
        const int t = t0 + k;
        if (t >= job.len) continue;
        const size_t buf_at = static_cast<size_t>(t) * row2 + c;
        const size_t row_at =
            (static_cast<size_t>(blk[k] < 0 ? 0 : blk[k]) * bs + t % bs) * rv + cv;
        if (kUnpack)
          v[k] = __ldcs(job.buf + buf_at);
        else
          v[k] = blk[k] < 0 ? make_uint4(0xffffffffu, 0xffffffffu, 0xffffffffu, 0xffffffffu)
                            : __ldcs(cache + row_at);
      }
#pragma unroll
      for (int k = 0; k < kPackTokens; ++k) {
        const int t = t0 + k;
        if (t >= job.len) continue;
        const size_t buf_at = static_cast<size_t>(t) * row2 + c;
        const size_t row_at =
            (static_cast<size_t>(blk[k] < 0 ? 0 : blk[k]) * bs + t % bs) * rv + cv;
        if (!kUnpack)
          __stcs(job.buf + buf_at, v[k]);
        else if (blk[k] >= 0)
          __stcs(cache + row_at, v[k]);
      }
    }
  }
}

// ---- NVFP4 block scales: [num_blocks, H_kv, block_size, D/16] E4M3 bytes, per block and
// head-major, so a (block, kv-head) tile's scales are one contiguous run (what the attention
// kernel fetches in one bulk copy). The row of (block, offset, head) is
// (block * H_kv + head) * block_size + offset; these calls move rows of D/16 bytes as
// 4-byte words (rw words a row).
struct ScaleJob {
  uint32_t* buf;  // [len, 2, H_kv, D/16] (pack: written, unpack: read)
  const int32_t* table;
  int len;
};

template <int N>
struct ScaleParams {
  int32_t* error_word;
  uint32_t* k_scales;
  uint32_t* v_scales;
  int n, H_kv, rw, block_size, num_blocks;
  ScaleJob jobs[N];
};

__device__ __forceinline__ size_t scale_word(long long block, int offset, int h, int H_kv,
                                             int block_size, int rw, int w) {
  return (static_cast<size_t>(block * H_kv + h) * block_size + offset) * rw + w;
}

// Append: k_new/v_new [B, H_kv, D/16]; thread i copies word i of the flattened
// (b, K|V, head, word) space into the row of slot slot_mapping[b].
__global__ void __launch_bounds__(256) kv_append_scales_kernel(
    const uint32_t* __restrict__ k_new, const uint32_t* __restrict__ v_new,
    uint32_t* __restrict__ k_scales, uint32_t* __restrict__ v_scales,
    const int32_t* __restrict__ slots, int B, int H_kv, int rw, int block_size, int num_blocks,
    int32_t* error_word) {
  const int per = H_kv * rw;
  const long long total = static_cast<long long>(B) * 2 * per;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int b = static_cast<int>(i / (2 * per));
    const int rem = static_cast<int>(i % (2 * per));
    const int which = rem / per;
    const int hw = rem % per;
    const int s = slots[b];
    if (s < 0) continue;  // padding
    const long long block = s / block_size;
    if (block >= num_blocks) {
      if (rem == 0) atomic_or_error(error_word, PDA_DEVERR_SLOT);
      continue;
    }
    const size_t dst = scale_word(block, s % block_size, hw / rw, H_kv, block_size, rw, hw % rw);
    const size_t src = static_cast<size_t>(b) * per + hw;
    if (which == 0)
      k_scales[dst] = k_new[src];
    else
      v_scales[dst] = v_new[src];
  }
}

// Pack (scale rows -> [len, 2, H_kv, D/16]) or unpack (the reverse); blockIdx.y selects the
// request, threads stride over the buffer's words in order. A block id out of range sets
// PDA_DEVERR_BLOCK_ID; pack writes 0xFF bytes for its tokens, unpack skips them.
template <bool kUnpack, int N>
__global__ void __launch_bounds__(256) kv_scales_kernel(const __grid_constant__ ScaleParams<N> p) {
  const ScaleJob job = p.jobs[blockIdx.y];
  const int per = p.H_kv * p.rw;
  const long long total = static_cast<long long>(job.len) * 2 * per;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(i / (2 * per));
    const int rem = static_cast<int>(i % (2 * per));
    const int which = rem / per;
    const int hw = rem % per;
    const int block = job.table[t / p.block_size];
    const bool bad = block < 0 || block >= p.num_blocks;
    if (bad && rem == 0) atomic_or_error(p.error_word, PDA_DEVERR_BLOCK_ID);
    uint32_t* cache = which == 0 ? p.k_scales : p.v_scales;
    const size_t at =
        scale_word(bad ? 0 : block, t % p.block_size, hw / p.rw, p.H_kv, p.block_size, p.rw,
                   hw % p.rw);
    if (kUnpack) {
      if (!bad) cache[at] = job.buf[i];
    } else {
      job.buf[i] = bad ? 0xffffffffu : cache[at];
    }
  }
}

namespace {

pda_status check_kv_rows(int H_kv, int D, int block_size, int num_blocks, pda_dtype dt,
                         int* row_vecs) {
  if (H_kv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0 || !dtype_ok(dt))
    return PDA_ERR_INVALID_ARG;
  const size_t row_bytes = static_cast<size_t>(H_kv) * D * dtype_bytes(dt);
  if (row_bytes % 16 != 0 || row_bytes / 16 > (1u << 28)) return PDA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= (1ll << 31)) return PDA_ERR_UNSUPPORTED;
  *row_vecs = static_cast<int>(row_bytes / 16);
  return PDA_OK;
}

template <int N>
pda_status launch_blocks(const PackParams<N>& p, int max_len, bool unpack, cudaStream_t stream) {
  const int tok = unpack ? tokens_per_iter<true>() : tokens_per_iter<false>();
  int gx = (max_len + tok - 1) / tok;
  if (gx > 8192) gx = 8192;
  if (gx < 1) gx = 1;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(p.n));
  // one thread per 16-byte vector of a token's K|V row, at most 256
  const int threads = 2 * p.row_vecs >= 256 ? 256 : (2 * p.row_vecs + 31) / 32 * 32;
  if (unpack)
    kv_blocks_kernel<true, N><<<grid, threads, 0, stream>>>(p);
  else
    kv_blocks_kernel<false, N><<<grid, threads, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

// Shared front end of the batched pack and unpack calls: validates, fills the jobs, launches.
pda_status blocks_batched(void* const* bufs, const int32_t* const* block_table_rows,
                          const int32_t* context_lens, int n, const void* k_cache,
                          const void* v_cache, int H_kv, int D, int block_size, int num_blocks,
                          pda_dtype kv_dtype, int32_t* error_word, bool unpack,
                          cudaStream_t stream) {
  if (n < 0 || n > PDA_PACK_MAX_BATCH) return n < 0 ? PDA_ERR_INVALID_ARG : PDA_ERR_UNSUPPORTED;
  int rv = 0;
  const pda_status st = check_kv_rows(H_kv, D, block_size, num_blocks, kv_dtype, &rv);
  if (st != PDA_OK) return st;
  if (n == 0) return PDA_OK;
  if (bufs == nullptr || block_table_rows == nullptr || context_lens == nullptr ||
      k_cache == nullptr || v_cache == nullptr)
    return PDA_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PDA_ERR_INVALID_ARG;
  PackParams<PDA_PACK_MAX_BATCH> p;
  p.error_word = error_word;
  p.row_vecs = rv;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  int m = 0;
  int max_len = 0;
  for (int i = 0; i < n; ++i) {
    const int len = context_lens[i];
    if (len < 0) return PDA_ERR_INVALID_ARG;
    if (len == 0) continue;
    if (bufs[i] == nullptr || block_table_rows[i] == nullptr || !aligned16(bufs[i]))
      return PDA_ERR_INVALID_ARG;
    p.jobs[m].buf = static_cast<uint4*>(bufs[i]);
    p.jobs[m].table = block_table_rows[i];
    p.jobs[m].k_cache = static_cast<uint4*>(const_cast<void*>(k_cache));
    p.jobs[m].v_cache = static_cast<uint4*>(const_cast<void*>(v_cache));
    p.jobs[m].len = len;
    if (len > max_len) max_len = len;
    ++m;
  }
  if (m == 0) return PDA_OK;
  p.n = m;
  return launch_blocks(p, max_len, unpack, stream);
}

// Shared front end of the layer calls: one request, one job per layer.
pda_status blocks_layers(void* const* bufs, void* const* k_caches, void* const* v_caches,
                         int n_layers, const int32_t* block_table_row, int context_len, int H_kv,
                         int D, int block_size, int num_blocks, pda_dtype kv_dtype,
                         int32_t* error_word, bool unpack, cudaStream_t stream) {
  if (n_layers < 0 || context_len < 0) return PDA_ERR_INVALID_ARG;
  if (n_layers > PDA_PACK_MAX_LAYERS) return PDA_ERR_UNSUPPORTED;
  int rv = 0;
  const pda_status st = check_kv_rows(H_kv, D, block_size, num_blocks, kv_dtype, &rv);
  if (st != PDA_OK) return st;
  if (n_layers == 0 || context_len == 0) return PDA_OK;
  if (bufs == nullptr || k_caches == nullptr || v_caches == nullptr ||
      block_table_row == nullptr)
    return PDA_ERR_INVALID_ARG;
  PackParams<PDA_PACK_MAX_LAYERS> p;
  p.error_word = error_word;
  p.row_vecs = rv;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.n = n_layers;
  for (int i = 0; i < n_layers; ++i) {
    if (bufs[i] == nullptr || k_caches[i] == nullptr || v_caches[i] == nullptr ||
        !aligned16(bufs[i]) || !aligned16(k_caches[i]) || !aligned16(v_caches[i]))
      return PDA_ERR_INVALID_ARG;
    p.jobs[i].buf = static_cast<uint4*>(bufs[i]);
    p.jobs[i].table = block_table_row;
    p.jobs[i].k_cache = static_cast<uint4*>(k_caches[i]);
    p.jobs[i].v_cache = static_cast<uint4*>(v_caches[i]);
    p.jobs[i].len = context_len;
  }
  return launch_blocks(p, context_len, unpack, stream);
}


// Scale rows: D/16 bytes, moved as 4-byte words.
pda_status check_scale_rows(int H_kv, int D, int block_size, int num_blocks, int* rw) {
  if (H_kv <= 0 || D <= 0 || block_size <= 0 || num_blocks <= 0) return PDA_ERR_INVALID_ARG;
  if (D % 64 != 0) return PDA_ERR_UNSUPPORTED;
  if (static_cast<long long>(num_blocks) * block_size >= (1ll << 31)) return PDA_ERR_UNSUPPORTED;
  *rw = D / 64;
  return PDA_OK;
}

pda_status scales_batched(void* const* bufs, const int32_t* const* block_table_rows,
                          const int32_t* context_lens, int n, const void* k_scales,
                          const void* v_scales, int H_kv, int D, int block_size, int num_blocks,
                          int32_t* error_word, bool unpack, cudaStream_t stream) {
  if (n < 0 || n > PDA_PACK_MAX_BATCH) return n < 0 ? PDA_ERR_INVALID_ARG : PDA_ERR_UNSUPPORTED;
  int rw = 0;
  const pda_status st = check_scale_rows(H_kv, D, block_size, num_blocks, &rw);
  if (st != PDA_OK) return st;
  if (n == 0) return PDA_OK;
  if (bufs == nullptr || block_table_rows == nullptr || context_lens == nullptr ||
      k_scales == nullptr || v_scales == nullptr)
    return PDA_ERR_INVALID_ARG;
  if (!aligned4(k_scales) || !aligned4(v_scales)) return PDA_ERR_INVALID_ARG;
  ScaleParams<PDA_PACK_MAX_BATCH> p;
  p.error_word = error_word;
  p.k_scales = static_cast<uint32_t*>(const_cast<void*>(k_scales));
  p.v_scales = static_cast<uint32_t*>(const_cast<void*>(v_scales));
  p.H_kv = H_kv;
  p.rw = rw;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  int m = 0, max_len = 0;
  for (int i = 0; i < n; ++i) {
    const int len = context_lens[i];
    if (len < 0) return PDA_ERR_INVALID_ARG;
    if (len == 0) continue;
    if (bufs[i] == nullptr || block_table_rows[i] == nullptr || !aligned4(bufs[i]))
      return PDA_ERR_INVALID_ARG;
    p.jobs[m].buf = static_cast<uint32_t*>(bufs[i]);
    p.jobs[m].table = block_table_rows[i];
    p.jobs[m].len = len;
    if (len > max_len) max_len = len;
    ++m;
  }
  if (m == 0) return PDA_OK;
  p.n = m;
  const long long words = static_cast<long long>(max_len) * 2 * H_kv * rw;
  long long gx = (words + 255) / 256;
  if (gx > 4096) gx = 4096;
  const dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(m));
  if (unpack)
    kv_scales_kernel<true, PDA_PACK_MAX_BATCH><<<grid, 256, 0, stream>>>(p);
  else
    kv_scales_kernel<false, PDA_PACK_MAX_BATCH><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

}  // namespace
}  // namespace pda

using namespace pda;

extern "C" pda_status pda_kv_pack_layers(void* const* outs, const void* const* k_caches,
                                         const void* const* v_caches, int n_layers,
                                         const int32_t* block_table_row, int context_len,
                                         int H_kv, int D, int block_size, int num_blocks,
                                         pda_dtype kv_dtype, int32_t* error_word,
                                         cudaStream_t stream) {
  return blocks_layers(outs, const_cast<void* const*>(k_caches),
                       const_cast<void* const*>(v_caches), n_layers, block_table_row,
                       context_len, H_kv, D, block_size, num_blocks, kv_dtype, error_word, false,
                       stream);
}

extern "C" pda_status pda_kv_unpack_layers(const void* const* ins, void* const* k_caches,
                                           void* const* v_caches, int n_layers,
                                           const int32_t* block_table_row, int context_len,
                                           int H_kv, int D, int block_size, int num_blocks,
                                           pda_dtype kv_dtype, int32_t* error_word,
                                           cudaStream_t stream) {
  return blocks_layers(const_cast<void* const*>(ins), k_caches, v_caches, n_layers,
                       block_table_row, context_len, H_kv, D, block_size, num_blocks, kv_dtype,
                       error_word, true, stream);
}

extern "C" pda_status pda_kv_append(const void* k_new, const void* v_new, void* k_cache,
                                    void* v_cache, const int32_t* slot_mapping, int B, int H_kv,
                                    int D, int block_size, int num_blocks, pda_dtype kv_dtype,
                                    int32_t* error_word, cudaStream_t stream) {
  if (B < 0) return PDA_ERR_INVALID_ARG;
  int rv = 0;
  const pda_status st = check_kv_rows(H_kv, D, block_size, num_blocks, kv_dtype, &rv);
  if (st != PDA_OK) return st;
  if (B == 0) return PDA_OK;
  if (k_new == nullptr || v_new == nullptr || k_cache == nullptr || v_cache == nullptr ||
      slot_mapping == nullptr)
    return PDA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
    return PDA_ERR_INVALID_ARG;
  const long long total = static_cast<long long>(B) * 2 * rv;
  long long grid = (total + 255) / 256;
  if (grid > 65535) grid = 65535;
  kv_append_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new),
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), slot_mapping, B, rv,
      block_size, num_blocks, error_word);
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

extern "C" pda_status pda_kv_pack_blocks_batched(void* const* outs,
                                                 const int32_t* const* block_table_rows,
                                                 const int32_t* context_lens, int n,
                                                 const void* k_cache, const void* v_cache,
                                                 int H_kv, int D, int block_size, int num_blocks,
                                                 pda_dtype kv_dtype, int32_t* error_word,
                                                 cudaStream_t stream) {
  return blocks_batched(outs, block_table_rows, context_lens, n, k_cache, v_cache, H_kv, D,
                        block_size, num_blocks, kv_dtype, error_word, false, stream);
}

extern "C" pda_status pda_kv_pack_blocks(void* out, const void* k_cache, const void* v_cache,
                                         const int32_t* block_table_row, int context_len,
                                         int H_kv, int D, int block_size, int num_blocks,
                                         pda_dtype kv_dtype, int32_t* error_word,
                                         cudaStream_t stream) {
  void* outs[1] = {out};
  const int32_t* rows[1] = {block_table_row};
  const int32_t lens[1] = {context_len};
  return pda_kv_pack_blocks_batched(outs, rows, lens, 1, k_cache, v_cache, H_kv, D, block_size,
                                    num_blocks, kv_dtype, error_word, stream);
}

extern "C" pda_status pda_kv_unpack_blocks_batched(const void* const* ins,
                                                   const int32_t* const* block_table_rows,
                                                   const int32_t* context_lens, int n,
                                                   void* k_cache, void* v_cache, int H_kv, int D,
                                                   int block_size, int num_blocks,
                                                   pda_dtype kv_dtype, int32_t* error_word,
                                                   cudaStream_t stream) {
  return blocks_batched(const_cast<void* const*>(ins), block_table_rows, context_lens, n,
                        k_cache, v_cache, H_kv, D, block_size, num_blocks, kv_dtype, error_word,
                        true, stream);
}

extern "C" pda_status pda_kv_unpack_blocks(const void* in, void* k_cache, void* v_cache,
                                           const int32_t* block_table_row, int context_len,
                                           int H_kv, int D, int block_size, int num_blocks,
                                           pda_dtype kv_dtype, int32_t* error_word,
                                           cudaStream_t stream) {
  const void* ins[1] = {in};
  const int32_t* rows[1] = {block_table_row};
  const int32_t lens[1] = {context_len};
  return pda_kv_unpack_blocks_batched(ins, rows, lens, 1, k_cache, v_cache, H_kv, D,
                                      block_size, num_blocks, kv_dtype, error_word, stream);
}

extern "C" pda_status pda_kv_append_block_scales(const void* k_new, const void* v_new,
                                                 void* k_scales, void* v_scales,
                                                 const int32_t* slot_mapping, int B, int H_kv,
                                                 int D, int block_size, int num_blocks,
                                                 int32_t* error_word, cudaStream_t stream) {
  if (B < 0) return PDA_ERR_INVALID_ARG;
  int rw = 0;
  const pda_status st = check_scale_rows(H_kv, D, block_size, num_blocks, &rw);
  if (st != PDA_OK) return st;
  if (B == 0) return PDA_OK;
  if (k_new == nullptr || v_new == nullptr || k_scales == nullptr || v_scales == nullptr ||
      slot_mapping == nullptr)
    return PDA_ERR_INVALID_ARG;
  if (!aligned4(k_new) || !aligned4(v_new) || !aligned4(k_scales) || !aligned4(v_scales))
    return PDA_ERR_INVALID_ARG;
  const long long total = static_cast<long long>(B) * 2 * H_kv * rw;
  long long grid = (total + 255) / 256;
  if (grid > 65535) grid = 65535;
  kv_append_scales_kernel<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
      static_cast<const uint32_t*>(k_new), static_cast<const uint32_t*>(v_new),
      static_cast<uint32_t*>(k_scales), static_cast<uint32_t*>(v_scales), slot_mapping, B, H_kv,
      rw, block_size, num_blocks, error_word);
  return cudaGetLastError() == cudaSuccess ? PDA_OK : PDA_ERR_CUDA;
}

extern "C" pda_status pda_kv_pack_block_scales_batched(
    void* const* outs, const int32_t* const* block_table_rows, const int32_t* context_lens,
    int n, const void* k_scales, const void* v_scales, int H_kv, int D, int block_size,
    int num_blocks, int32_t* error_word, cudaStream_t stream) {
  return scales_batched(outs, block_table_rows, context_lens, n, k_scales, v_scales, H_kv, D,
                        block_size, num_blocks, error_word, false, stream);
}

extern "C" pda_status pda_kv_unpack_block_scales_batched(
    const void* const* ins, const int32_t* const* block_table_rows, const int32_t* context_lens,
    int n, void* k_scales, void* v_scales, int H_kv, int D, int block_size, int num_blocks,
    int32_t* error_word, cudaStream_t stream) {
  return scales_batched(const_cast<void* const*>(ins), block_table_rows, context_lens, n,
                        k_scales, v_scales, H_kv, D, block_size, num_blocks, error_word, true,
                        stream);
}
