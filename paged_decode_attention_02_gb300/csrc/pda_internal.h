// pda_internal.h -- host-side helpers shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pda.h"

namespace pda {

// SM count of the current device (cached per device). Returns PDA_ERR_CUDA on failure.
pda_status current_device_sms(int* device, int* num_sms);

// Encodes a 3-D tiled tensor map over a KV cache [num_blocks * block_size, H_kv, D]
// (innermost first: D, H_kv, rows) with box {D, 1, box_rows}: box_rows consecutive cache
// rows of one kv-head (the attention's tile, 16 rows of one block). swizzle_bytes is 0
// (rows land as they are) or 64 / 128 (the shared-memory swizzle of that span, which must
// equal the row's byte width).
pda_status encode_kv_tensor_map(CUtensorMap* tm, const void* base, int num_blocks,
                                int block_size, int H_kv, int D, pda_dtype dtype,
                                int swizzle_bytes, int box_rows);

// A 4-D tiled tensor map over a byte cache [num_blocks * block_size, H_kv, row_bytes] that
// loads the tiles of two adjacent kv-heads (2h', 2h' + 1) with one box: dims {row_bytes,
// rows, 2, H_kv / 2}, box {row_bytes, box_rows, 1 pair}; in shared memory the box is head
// 2h''s box_rows rows followed by head 2h' + 1's, each row swizzled as by
// encode_kv_tensor_map. H_kv must be even.
pda_status encode_kv_pair_tensor_map(CUtensorMap* tm, const void* base, int num_blocks,
                                     int block_size, int H_kv, int row_bytes,
                                     int swizzle_bytes, int box_rows);

inline size_t dtype_bytes(pda_dtype t) {
  return (t == PDA_BF16 || t == PDA_F16) ? 2u : (t == PDA_FP8_E4M3 ? 1u : 4u);
}
// Types a KV cache may hold.
inline bool dtype_ok(int t) {
  return t == PDA_F32 || t == PDA_BF16 || t == PDA_F16 || t == PDA_FP8_E4M3;
}
// Types of q and out.
inline bool float_dtype_ok(int t) { return t == PDA_F32 || t == PDA_BF16 || t == PDA_F16; }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace pda
