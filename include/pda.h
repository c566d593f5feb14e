/*
 * pda.h -- C ABI of the paged decode-attention library for GB300 (sm_103a).
 *
 * The library implements the data-parallel hot path of one decode step over a paged KV
 * cache: the append of each request's new K/V, the attention of each request's single
 * query token over its whole cached history, and the gather of one request's scattered
 * KV blocks into a contiguous buffer for transfer.
 *
 * Conventions shared by every entry point:
 *  - Every pointer argument is a DEVICE pointer unless its comment says "host". The caller
 *    owns all memory; the library allocates nothing. Apart from the fixed scratch array of
 *    pda_paged_decode_attention_noalloc it keeps no state between calls.
 *  - Tensors are dense and row-major with exactly the shapes given; no strides.
 *  - KV caches are [num_blocks, block_size, H_kv, D]: physical block p holds block_size
 *    consecutive tokens, token row r of block p is at ((p * block_size + r) * H_kv) * D.
 *    (Page "From PagedAttention to Prefill-Decode disaggregation", sec. 2.2 step 1: the
 *    cache is cut into fixed-size physical blocks, each holding the K and V of a fixed
 *    number of tokens.)
 *  - block_tables is [B, max_blocks_per_seq] int32: logical block i of request b is
 *    physical block block_tables[b * max_blocks_per_seq + i]; blocks need not be
 *    contiguous or ordered, and several requests may share blocks (same page, sec. 2.2
 *    step 2 and sec. 2.3). Entries past a request's last block are never read.
 *  - Query head h reads kv-head h / (H / H_kv) (grouped-query attention, contiguous groups).
 *  - Every call is asynchronous on `stream`, never synchronises the host and allocates no
 *    device memory. A sequence of the calls other than pda_paged_decode_attention_noalloc
 *    can be captured in a CUDA graph once each kernel has been launched outside capture.
 *  - Host-checkable errors (null pointers, bad sizes, unsupported dtypes or shapes,
 *    misaligned pointers) return a status before anything is launched. Errors in device
 *    data (a block id or slot out of range, a context length beyond capacity) cannot be
 *    seen on the host without a sync; kernels OR a PDA_DEVERR_* bit into *error_word
 *    (when error_word is not NULL) and never trap. The caller zeroes the error word and
 *    reads it back whenever it chooses to synchronise.
 */
#ifndef PDA_H
#define PDA_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PDA_OK = 0,
  PDA_ERR_INVALID_ARG = 1, /* null pointer, negative or inconsistent size, misalignment */
  PDA_ERR_UNSUPPORTED = 2, /* a valid request the library does not implement */
  PDA_ERR_CUDA = 3,        /* a CUDA runtime call failed; see cudaGetLastError */
  PDA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required */
  PDA_ERR_TOO_LARGE = 5    /* needs more scratch than pda_paged_decode_attention_noalloc has */
} pda_status;

/* Element types. PDA_F32, PDA_BF16 and PDA_F16 (IEEE binary16, the precision the pages'
 * decode kernels were measured in) are q, output and KV-cache types. PDA_FP8_E4M3 (the OCP
 * 8-bit format without infinities) is a KV-cache type only: append, pack and unpack copy
 * its bytes, and pda_paged_decode_attention_fp8 reads it with per-tensor scales. PDA_NVFP4
 * names the 4-bit cache read by pda_paged_decode_attention_nvfp4 (and sizes its workspace);
 * its data tensors are moved as 1-byte rows by append, pack and unpack, its block scales by
 * the *_block_scales calls. */
typedef enum {
  PDA_F32 = 0,
  PDA_BF16 = 1,
  PDA_FP8_E4M3 = 2,
  PDA_NVFP4 = 3,
  PDA_F16 = 4
} pda_dtype;

/* Bits OR-ed into *error_word by the kernels. */
#define PDA_DEVERR_CONTEXT_LEN 0x1 /* context_lens[b] < 0, > max_context_len or > table capacity */
#define PDA_DEVERR_BLOCK_ID 0x2    /* a block id needed by a request is outside [0, num_blocks) */
#define PDA_DEVERR_SLOT 0x4        /* slot_mapping[b] >= num_blocks * block_size */
#define PDA_DEVERR_TIMEOUT 0x8     /* a pipeline wait passed its time limit; results invalid */

/* Bytes of the fixed device scratch behind pda_paged_decode_attention_noalloc. */
#define PDA_NOALLOC_SCRATCH_BYTES (8u << 20)

/* Most requests one batched pack or unpack call takes. */
#define PDA_PACK_MAX_BATCH 64

/* Most layers one pda_kv_pack_layers / pda_kv_unpack_layers call takes. */
#define PDA_PACK_MAX_LAYERS 256

/* Human-readable name of a status. Never NULL. */
const char* pda_status_string(pda_status status);

/* ABI version of this library (incremented on incompatible change). */
int pda_version(void);

/* Number of SMs of the current device, written to *num_sms (host). */
pda_status pda_device_sm_count(int* num_sms);

/*
 * pda_kv_append -- write each request's new token into the paged cache.
 *
 * Defined by the decode step of page "Disaggregated LLM Serving: from PD disaggregation to
 * attention offload", sec. 1 (second list, item 2): every decode step reads the cached
 * history and appends the new token's K/V; the slot comes from the block table (page "From
 * PagedAttention to Prefill-Decode disaggregation", sec. 2.2 step 3: blocks are handed out
 * as tokens arrive).
 *
 *  k_new, v_new   [B, H_kv, D] in kv_dtype: this step's K and V of each request.
 *  k_cache,v_cache [num_blocks, block_size, H_kv, D] in kv_dtype, updated in place.
 *  slot_mapping   [B] int32: flat slot s = block * block_size + row for request b. s < 0
 *                 means "no token" (padding) and is skipped; s >= num_blocks * block_size
 *                 sets PDA_DEVERR_SLOT and is skipped.
 *  The copy is bitwise. Two requests given the same slot race; the caller must not do so.
 *  Requires H_kv * D * sizeof(kv_dtype) to be a multiple of 16 bytes and 16-byte aligned
 *  pointers. B == 0 is a no-op.
 */
pda_status pda_kv_append(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const int32_t* slot_mapping, int B, int H_kv, int D, int block_size,
                         int num_blocks, pda_dtype kv_dtype, int32_t* error_word,
                         cudaStream_t stream);

/*
 * pda_attention_workspace_size -- bytes of device workspace pda_paged_decode_attention
 * needs on the current device for these sizes. The bound does not depend on the context
 * lengths. Written to *bytes (host).
 */
pda_status pda_attention_workspace_size(int B, int H, int H_kv, int D, int block_size,
                                        pda_dtype kv_dtype, int sm_cap, size_t* bytes);

/*
 * pda_paged_decode_attention -- one query token per head attends over its request's whole
 * cached history, read through the block table.
 *
 * Defined by: decode reads the request's whole KV history each step (page "Disaggregated
 * LLM Serving", sec. 1, and sec. 6.1 on why this is memory-bound); the history lives in
 * fixed-size blocks reached through a per-request table (page "From PagedAttention to
 * Prefill-Decode disaggregation", sec. 2.2). For each request b and query head h with
 * kv-head k = h / (H / H_kv) and L = context_lens[b]:
 *      s_t = scale * q[b,h,:] . K_t[k,:],   t < L
 *      out[b,h,:] = sum_t softmax(s)_t * V_t[k,:]
 * The work is split per request and kv-head and, for long histories, along the sequence;
 * the pieces are merged with a log-sum-exp combine (the per-request split and merge of
 * Orca's iteration-level batching, page "Disaggregated LLM Serving", sec. 2.1, applied
 * also along the sequence). Accumulation is fp32.
 *
 *  out            [B, H, D] in out_dtype (PDA_F32, PDA_BF16 or PDA_F16).
 *  q              [B, H, D] in q_dtype; q_dtype must equal kv_dtype.
 *  k_cache,v_cache [num_blocks, block_size, H_kv, D] in kv_dtype (PDA_F32, PDA_BF16 or
 *                 PDA_F16; an FP8 cache goes through pda_paged_decode_attention_fp8); read
 *                 only.
 *  block_tables   [B, max_blocks_per_seq] int32.
 *  context_lens   [B] int32 (device): tokens of history including this step's token.
 *                 L == 0 gives a zero row. L < 0, L > max_context_len or
 *                 L > max_blocks_per_seq * block_size gives NaN rows and
 *                 PDA_DEVERR_CONTEXT_LEN. A block id out of range gives NaN rows for
 *                 that (request, kv-head group) and PDA_DEVERR_BLOCK_ID.
 *  max_context_len host upper bound of context_lens (validation only).
 *  scale          softmax scale, usually 1/sqrt(D).
 *  sm_cap         0 runs on every SM; n > 0 confines the kernel to at most n SMs (one
 *                 resident block per SM, a persistent grid walks the work). This models
 *                 attention sharing the GPU with other work on a fraction of its SMs
 *                 (review of "Injecting Adrenaline into LLM Serving", sec. 3.3).
 *  workspace      device scratch of at least pda_attention_workspace_size(...) bytes,
 *                 256-byte aligned; not shared by calls that may run concurrently. No
 *                 initialisation is needed: its arrival counters are tagged with a number
 *                 the library gives each call, mixed with a fixed 48-bit pattern so that
 *                 what another call left there (zeros, or the fp32 partial results of a call
 *                 of another shape) is not taken for a live counter. (A call captured in a
 *                 CUDA graph keeps its number on every replay; if a replay ever reports
 *                 PDA_DEVERR_TIMEOUT, zero the workspace before the next replay.)
 *  Supported: D in {64, 128}; block_size in {16, 32, 64, 128, 256} (the kernel works in
 *  tiles of 16 rows of one physical block); H / H_kv in {1, 2, 4, 8}; B <= 8192;
 *  kv_dtype in {PDA_F32, PDA_BF16, PDA_F16}. Pointers 16-byte aligned. Other sizes return
 *  PDA_ERR_UNSUPPORTED.
 */
pda_status pda_paged_decode_attention(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      int max_blocks_per_seq, const int32_t* context_lens,
                                      int max_context_len, int B, int H, int H_kv, int D,
                                      int block_size, int num_blocks, float scale,
                                      pda_dtype q_dtype, pda_dtype kv_dtype, pda_dtype out_dtype,
                                      int sm_cap, void* workspace, size_t workspace_bytes,
                                      int32_t* error_word, cudaStream_t stream);

/*
 * pda_paged_decode_attention_fp8 -- pda_paged_decode_attention over an FP8 E4M3 KV cache.
 *
 * A quantised KV cache cuts the bytes each decode step must read (page "From
 * PagedAttention to Prefill-Decode disaggregation", sec. 6.2: a low-precision KV cache,
 * dequantised to FP8 before attention, raises memory bandwidth and throughput). Each
 * stored K code means decode(code) * k_scale and each V code decode(code) * v_scale
 * (per-tensor scales); the result is softmax(scale * q K^T) V over those values, exactly as
 * pda_paged_decode_attention computes it. Codes are widened exactly in registers. At D = 128
 * the products run on the tensor cores: K, V (exact in fp16) and q (exact in fp16 after a
 * power-of-two rescale) as fp16 operands, fp32 accumulation, probabilities entering P V as
 * two fp16 parts (relative error about 2^-22); softmax in fp32. At D = 64 all arithmetic is
 * fp32.
 *
 *  k_cache, v_cache [num_blocks, block_size, H_kv, D] bytes (E4M3 codes).
 *  q               [B, H, D] in q_dtype, which must be PDA_BF16.
 *  k_scale, v_scale finite per-tensor scales.
 *  Every other argument, the workspace (pda_attention_workspace_size with PDA_FP8_E4M3),
 *  the supported sizes and the errors are those of pda_paged_decode_attention.
 */
pda_status pda_paged_decode_attention_fp8(void* out, const void* q, const void* k_cache,
                                          const void* v_cache, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int max_context_len, int B, int H, int H_kv, int D,
                                          int block_size, int num_blocks, float scale,
                                          float k_scale, float v_scale, pda_dtype q_dtype,
                                          pda_dtype out_dtype, int sm_cap, void* workspace,
                                          size_t workspace_bytes, int32_t* error_word,
                                          cudaStream_t stream);

/*
 * pda_paged_decode_attention_nvfp4 -- pda_paged_decode_attention over an NVFP4 KV cache.
 *
 * The 4-bit KV format with fine-grained block scaling in E4M3 (page "From PagedAttention to
 * Prefill-Decode disaggregation", sec. 6.2: NVFP4 KV stores 4-bit values with fine-grained
 * block scales and E4M3 scale factors). Element d of the K row of (token row r, kv-head h)
 * means  e2m1(code) * e4m3(block scale) * k_scale,  with
 *   code        = nibble d % 2 (0: low, 1: high) of k_data[r][h][d / 2],
 *   block scale = k_block_scales[r / block_size][h][r % block_size][d / 16]
 *                 (one per 16 consecutive elements),
 * and the same for V. E2M1 is the 4-bit float with 2 exponent bits (bias 1) and 1 mantissa
 * bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6. Values are dequantised exactly in registers
 * (the pages describe a dequantisation to FP8 before attention; fp16 and fp32 hold every
 * product e2m1 * e4m3 exactly, so nothing is rounded before the attention arithmetic),
 * which at D = 128 runs on the tensor cores as for pda_paged_decode_attention_fp8.
 *
 *  k_data, v_data   [num_blocks, block_size, H_kv, D / 2] bytes.
 *  k_block_scales, v_block_scales [num_blocks, H_kv, block_size, D / 16] E4M3 bytes,
 *                   16-byte aligned: per block and head-major, so the scales of the 16
 *                   rows of one kv-head that a tile covers are one contiguous run of D
 *                   bytes (the pages give no layout; this is the one the kernel reads in
 *                   one bulk copy per tile and head).
 *  q                [B, H, D] in q_dtype, which must be PDA_BF16.
 *  k_scale, v_scale finite per-tensor scales.
 *  Every other argument, the workspace (pda_attention_workspace_size with PDA_NVFP4), the
 *  supported sizes and the errors are those of pda_paged_decode_attention.
 *  Append, pack and unpack: the data tensors are token-major byte caches, moved by
 *  pda_kv_append, pda_kv_pack_blocks[_batched] and pda_kv_unpack_blocks[_batched] with
 *  kv_dtype PDA_FP8_E4M3 (any 1-byte type) and D / 2 as the row length (H_kv * D / 2 a
 *  multiple of 16 bytes); the block scales by pda_kv_append_block_scales,
 *  pda_kv_pack_block_scales_batched and pda_kv_unpack_block_scales_batched.
 */
pda_status pda_paged_decode_attention_nvfp4(void* out, const void* q, const void* k_data,
                                            const void* v_data, const void* k_block_scales,
                                            const void* v_block_scales,
                                            const int32_t* block_tables, int max_blocks_per_seq,
                                            const int32_t* context_lens, int max_context_len,
                                            int B, int H, int H_kv, int D, int block_size,
                                            int num_blocks, float scale, float k_scale,
                                            float v_scale, pda_dtype q_dtype,
                                            pda_dtype out_dtype, int sm_cap, void* workspace,
                                            size_t workspace_bytes, int32_t* error_word,
                                            cudaStream_t stream);

/*
 * pda_paged_decode_attention_noalloc -- pda_paged_decode_attention without a workspace
 * argument, for callers that cannot allocate device memory.
 *
 * The pages describe no such call; it exists for code that may not call cudaMalloc or any
 * allocator when it runs: a plugin inside a host framework that owns all device memory and
 * hands out only inputs and outputs, or a serving loop that forbids allocation once it has
 * started. Such a caller still provides q, the caches, the tables, the lengths and out
 * exactly as for pda_paged_decode_attention (same meaning, layout and errors); the scratch
 * the kernels need comes from one fixed array of PDA_NOALLOC_SCRATCH_BYTES bytes compiled
 * into the library as a device global. Every GPU that loads the library holds that array
 * until the process exits. The call itself never calls cudaMalloc, cudaFree or any
 * allocating routine.
 *
 *  - Sizes whose scratch need exceeds PDA_NOALLOC_SCRATCH_BYTES (see
 *    pda_attention_workspace_size) are rejected with PDA_ERR_TOO_LARGE before any launch.
 *    On a 152-SM GB300 this admits every supported shape with H / H_kv <= 4 at D = 128
 *    (about 5 MB) and rejects H / H_kv = 8 at D = 128 (about 10 MB).
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 *    with that device current) and caches it for later calls.
 *  - Every call shares the one array, which keeps the previous call's contents: those of a
 *    call of another shape, or of one that stopped early with PDA_DEVERR_TIMEOUT. Partial
 *    results are written before they are read. The per-segment arrival counters at the
 *    head of the array must not carry counts from an earlier call, so every call first
 *    clears them (B * H_kv * 8 bytes or less, one cudaMemsetAsync on `stream`, which
 *    allocates nothing) and then launches the kernel.
 *    Calls that overlap on the GPU (on different streams, or from different host threads)
 *    race on the array and produce wrong results; serialise them.
 */
pda_status pda_paged_decode_attention_noalloc(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int max_context_len, int B, int H, int H_kv, int D, int block_size, int num_blocks,
    float scale, pda_dtype q_dtype, pda_dtype kv_dtype, pda_dtype out_dtype, int sm_cap,
    int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_pack_blocks -- gather one request's KV into one contiguous buffer.
 *
 * Defined by the request-level KV transfer of PD disaggregation (page on goodput and PD
 * disaggregation, 0539edu.com, sec. 5.4: after prefill, a request's whole KV is sent in
 * one transfer) over the paged layout above: for t < context_len,
 *      out[t, 0, :, :] = K of token t,   out[t, 1, :, :] = V of token t,
 * token t being row t % block_size of physical block block_table_row[t / block_size].
 *
 *  out            [context_len, 2, H_kv, D] in kv_dtype, dense.
 *  block_table_row device pointer to the request's table row (int32).
 *  context_len    host int, tokens to pack; 0 is a no-op.
 *  A block id out of range sets PDA_DEVERR_BLOCK_ID and fills that token's output with
 *  0xFF bytes (a NaN pattern). The copy is bitwise. Needs H_kv * D * sizeof(kv_dtype) to be
 *  a multiple of 16 bytes and 16-byte aligned pointers.
 */
pda_status pda_kv_pack_blocks(void* out, const void* k_cache, const void* v_cache,
                              const int32_t* block_table_row, int context_len, int H_kv, int D,
                              int block_size, int num_blocks, pda_dtype kv_dtype,
                              int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_pack_blocks_batched -- pda_kv_pack_blocks for n requests in one launch.
 *
 *  outs, block_table_rows, context_lens: HOST arrays of n entries; outs[i] and
 *  block_table_rows[i] are device pointers, context_lens[i] a host count. The arrays are
 *  copied into the launch, so the caller may reuse them when the call returns.
 *  n <= PDA_PACK_MAX_BATCH. Same semantics per request as pda_kv_pack_blocks.
 */
pda_status pda_kv_pack_blocks_batched(void* const* outs, const int32_t* const* block_table_rows,
                                      const int32_t* context_lens, int n, const void* k_cache,
                                      const void* v_cache, int H_kv, int D, int block_size,
                                      int num_blocks, pda_dtype kv_dtype, int32_t* error_word,
                                      cudaStream_t stream);

/*
 * pda_kv_unpack_blocks -- the receiving side of a request-level KV transfer: scatter one
 * request's contiguous KV buffer into the blocks allocated for it.
 *
 * Defined by the KV migration of PD disaggregation (page on goodput and PD disaggregation,
 * 0539edu.com, sec. 3: after prefill the request's KV moves to a decode worker; sec. 5.4:
 * request-level transfer sends it in one piece) into the paged layout, whose blocks are
 * allocated on demand (page "From PagedAttention to Prefill-Decode disaggregation", sec. 2.2
 * step 3). The inverse of pda_kv_pack_blocks: for t < context_len, the K row of token t
 * (row t % block_size of block block_table_row[t / block_size]) = in[t, 0, :, :] and the V
 * row = in[t, 1, :, :].
 *
 *  in             [context_len, 2, H_kv, D] in kv_dtype, dense; read only.
 *  k_cache,v_cache [num_blocks, block_size, H_kv, D], updated in place; rows of other
 *                 tokens are not touched.
 *  A block id out of range sets PDA_DEVERR_BLOCK_ID and that token is not written. Tokens
 *  that map to the same row race (the caller must not do that). Bitwise copy; 16-byte rows
 *  and alignment as for pack.
 */
pda_status pda_kv_unpack_blocks(const void* in, void* k_cache, void* v_cache,
                                const int32_t* block_table_row, int context_len, int H_kv,
                                int D, int block_size, int num_blocks, pda_dtype kv_dtype,
                                int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_unpack_blocks_batched -- pda_kv_unpack_blocks for n requests in one launch.
 *  ins, block_table_rows, context_lens: HOST arrays of n entries (device pointers and host
 *  counts), copied into the launch. n <= PDA_PACK_MAX_BATCH.
 */
pda_status pda_kv_unpack_blocks_batched(const void* const* ins,
                                        const int32_t* const* block_table_rows,
                                        const int32_t* context_lens, int n, void* k_cache,
                                        void* v_cache, int H_kv, int D, int block_size,
                                        int num_blocks, pda_dtype kv_dtype, int32_t* error_word,
                                        cudaStream_t stream);

/*
 * pda_kv_pack_layers -- pda_kv_pack_blocks of one request over n_layers layers' caches, in
 * one launch.
 *
 * A model keeps one K and one V cache per layer, and a request's blocks have the same ids in
 * every layer (one block table per request). Request-level transfer sends all layers once
 * prefill ends (page on goodput and PD disaggregation, 0539edu.com, sec. 5.4, request
 * granularity); layer-level transfer sends layer N as soon as its prefill is done, hidden
 * behind the computation of the later layers (same page and section, layer granularity;
 * page "Disaggregated LLM Serving: from PD disaggregation to attention offload", sec. 5.6),
 * which is one pda_kv_pack_blocks per layer on a transfer stream. This call is the
 * whole-model form: for layer i < n_layers and t < context_len,
 *      outs[i][t, 0, :, :] = K of token t in k_caches[i],  outs[i][t, 1, :, :] = V.
 *
 *  outs, k_caches, v_caches: HOST arrays of n_layers device pointers, copied into the
 *                 launch; outs[i] is [context_len, 2, H_kv, D] in kv_dtype, dense; every
 *                 layer's caches are [num_blocks, block_size, H_kv, D].
 *  block_table_row device pointer to the request's table row (int32), shared by all layers.
 *  n_layers <= PDA_PACK_MAX_LAYERS (more: PDA_ERR_UNSUPPORTED); 0 or context_len 0 is a
 *  no-op. Errors, bitwise copy and alignment as for pda_kv_pack_blocks.
 */
pda_status pda_kv_pack_layers(void* const* outs, const void* const* k_caches,
                              const void* const* v_caches, int n_layers,
                              const int32_t* block_table_row, int context_len, int H_kv, int D,
                              int block_size, int num_blocks, pda_dtype kv_dtype,
                              int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_unpack_layers -- the receiving side of pda_kv_pack_layers: for layer i and
 * t < context_len, the K row of token t in k_caches[i] = ins[i][t, 0, :, :] and the V row =
 * ins[i][t, 1, :, :]. HOST arrays of n_layers device pointers, copied into the launch;
 * semantics per layer as for pda_kv_unpack_blocks (a bad block id sets
 * PDA_DEVERR_BLOCK_ID and that token is not written in any layer).
 */
pda_status pda_kv_unpack_layers(const void* const* ins, void* const* k_caches,
                                void* const* v_caches, int n_layers,
                                const int32_t* block_table_row, int context_len, int H_kv,
                                int D, int block_size, int num_blocks, pda_dtype kv_dtype,
                                int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_append_block_scales -- pda_kv_append for the E4M3 block scales of an NVFP4 cache.
 *
 * Each decode step's new token brings one scale per 16 elements of its K and V rows (page
 * "From PagedAttention to Prefill-Decode disaggregation", sec. 6.2, NVFP4 KV with block
 * scales); the token of request b goes to slot s = slot_mapping[b], i.e. row s % block_size of
 * block s / block_size (page "Disaggregated LLM Serving: from PD disaggregation to attention
 * offload", sec. 1, the per-step KV write). For b < B and h < H_kv:
 *      k_scales[s / block_size][h][s % block_size][:] = k_new[b][h][:]   (D / 16 bytes)
 * and the same for V.
 *
 *  k_new, v_new     [B, H_kv, D / 16] E4M3 bytes, 4-byte aligned; read only.
 *  k_scales, v_scales [num_blocks, H_kv, block_size, D / 16] (the layout of
 *                   pda_paged_decode_attention_nvfp4), 4-byte aligned; updated in place.
 *  slot_mapping     [B] int32, device; negative = padding (skipped).
 *  D a multiple of 64 (rows move as 4-byte words), else PDA_ERR_UNSUPPORTED. A slot at or
 *  beyond num_blocks * block_size sets PDA_DEVERR_SLOT and is skipped. B = 0 is a no-op.
 */
pda_status pda_kv_append_block_scales(const void* k_new, const void* v_new, void* k_scales,
                                      void* v_scales, const int32_t* slot_mapping, int B,
                                      int H_kv, int D, int block_size, int num_blocks,
                                      int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_pack_block_scales_batched -- pda_kv_pack_blocks_batched for the block scales of an
 * NVFP4 cache: for request i and t < context_lens[i], with block = block_table_rows[i][t /
 * block_size] and offset = t % block_size,
 *      outs[i][t, 0, h, :] = k_scales[block][h][offset][:],
 *      outs[i][t, 1, h, :] = v_scales[block][h][offset][:].
 *
 *  outs[i]          [context_lens[i], 2, H_kv, D / 16] bytes, dense, 4-byte aligned.
 *  outs, block_table_rows, context_lens: HOST arrays of n entries (device pointers and host
 *  counts), copied into the launch. n <= PDA_PACK_MAX_BATCH. A block id out of range sets
 *  PDA_DEVERR_BLOCK_ID and fills that token's scales with 0xFF bytes (an E4M3 NaN).
 *  D a multiple of 64. Bitwise copy.
 */
pda_status pda_kv_pack_block_scales_batched(void* const* outs,
                                            const int32_t* const* block_table_rows,
                                            const int32_t* context_lens, int n,
                                            const void* k_scales, const void* v_scales,
                                            int H_kv, int D, int block_size, int num_blocks,
                                            int32_t* error_word, cudaStream_t stream);

/*
 * pda_kv_unpack_block_scales_batched -- the inverse of pda_kv_pack_block_scales_batched:
 * k_scales[block][h][offset][:] = ins[i][t, 0, h, :] and v_scales[...] = ins[i][t, 1, h, :].
 * A block id out of range sets PDA_DEVERR_BLOCK_ID and that token is not written; other
 * rows are not touched. Arrays, limits and alignment as for the pack.
 */
pda_status pda_kv_unpack_block_scales_batched(const void* const* ins,
                                              const int32_t* const* block_table_rows,
                                              const int32_t* context_lens, int n,
                                              void* k_scales, void* v_scales, int H_kv, int D,
                                              int block_size, int num_blocks,
                                              int32_t* error_word, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PDA_H */
