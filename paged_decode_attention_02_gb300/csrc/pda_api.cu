// pda_api.cu -- host-side helpers of the C ABI: status names, device SM counts and the
// TMA tensor-map encoder (obtained from the driver through the runtime, no -lcuda).
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "pda_internal.h"

namespace pda {

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices];  // 0 = not yet queried

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

void load_encoder() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}
}  // namespace

pda_status current_device_sms(int* device, int* num_sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PDA_ERR_CUDA;
  *device = dev;
  if (dev >= 0 && dev < kMaxDevices) {
    const int cached = g_sms[dev].load(std::memory_order_relaxed);
    if (cached > 0) {
      *num_sms = cached;
      return PDA_OK;
    }
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    return PDA_ERR_CUDA;
  if (dev >= 0 && dev < kMaxDevices) g_sms[dev].store(sms, std::memory_order_relaxed);
  *num_sms = sms;
  return PDA_OK;
}

pda_status encode_kv_tensor_map(CUtensorMap* tm, const void* base, int num_blocks,
                                int block_size, int H_kv, int D, pda_dtype dtype,
                                int swizzle_bytes, int box_rows) {
  if (swizzle_bytes != 0 && swizzle_bytes != 64 && swizzle_bytes != 128)
    return PDA_ERR_INVALID_ARG;
  if (box_rows <= 0 || box_rows > 256 || block_size % box_rows != 0) return PDA_ERR_INVALID_ARG;
  std::call_once(g_encode_once, load_encoder);
  if (g_encode == nullptr) return PDA_ERR_CUDA;
  const cuuint64_t e = dtype_bytes(dtype);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H_kv),
                              static_cast<cuuint64_t>(num_blocks) * block_size};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * e,
                                 static_cast<cuuint64_t>(H_kv) * D * e};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 1u, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t elem_strides[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt = dtype == PDA_BF16       ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == PDA_F16      ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                 : dtype == PDA_FP8_E4M3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  // With a swizzle the row (box width) must equal the swizzle span: 16-byte chunk c of
  // row r of the box then lands at chunk c ^ (r & 7) (128 B) or c ^ ((r >> 1) & 3) (64 B).
  const CUtensorMapSwizzle swz = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes != 0 && static_cast<cuuint64_t>(D) * e != static_cast<cuuint64_t>(swizzle_bytes))
    return PDA_ERR_INVALID_ARG;
  // L2 fills no wider than a row: rows of one kv-head are H_kv rows apart, and a wider fill
  // drags in the neighbouring heads' rows, which other warps read much later (256-byte
  // fills on 64-byte rows read four times the bytes from DRAM).
  const cuuint64_t row_bytes = static_cast<cuuint64_t>(D) * e;
  const CUtensorMapL2promotion promo = row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                       : row_bytes >= 64  ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B
                                                          : CU_TENSOR_MAP_L2_PROMOTION_NONE;
  const CUresult r = g_encode(tm, dt, 3, const_cast<void*>(base), dims, strides, box,
                              elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PDA_OK : PDA_ERR_INVALID_ARG;
}


pda_status encode_kv_pair_tensor_map(CUtensorMap* tm, const void* base, int num_blocks,
                                     int block_size, int H_kv, int row_bytes,
                                     int swizzle_bytes, int box_rows) {
  std::call_once(g_encode_once, load_encoder);
  if (g_encode == nullptr) return PDA_ERR_CUDA;
  if (box_rows <= 0 || box_rows > 256 || block_size % box_rows != 0) return PDA_ERR_INVALID_ARG;
  if (H_kv % 2 != 0 || (swizzle_bytes != 0 && swizzle_bytes != row_bytes) ||
      (swizzle_bytes != 0 && swizzle_bytes != 64 && swizzle_bytes != 128))
    return PDA_ERR_INVALID_ARG;
  const cuuint64_t X = static_cast<cuuint64_t>(row_bytes);
  // dims, innermost first: a row's bytes, the cache rows, the two heads of a pair, the pairs
  const cuuint64_t dims[4] = {X, static_cast<cuuint64_t>(num_blocks) * block_size, 2,
                              static_cast<cuuint64_t>(H_kv / 2)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(H_kv) * X, X, 2 * X};
  const cuuint32_t box[4] = {static_cast<cuuint32_t>(X), static_cast<cuuint32_t>(box_rows),
                             2u, 1u};
  const cuuint32_t elem_strides[4] = {1u, 1u, 1u, 1u};
  const CUtensorMapSwizzle swz = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                 : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                       : CU_TENSOR_MAP_SWIZZLE_NONE;
  // both heads of a pair are used, so the fill may cover the pair's 2 * row_bytes
  const cuuint64_t pair = 2 * X;
  const CUtensorMapL2promotion promo = pair >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                                       : pair >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B
                                                     : CU_TENSOR_MAP_L2_PROMOTION_L2_64B;
  const CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base),
                              dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swz, promo, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PDA_OK : PDA_ERR_INVALID_ARG;
}

}  // namespace pda

extern "C" const char* pda_status_string(pda_status status) {
  switch (status) {
    case PDA_OK: return "ok";
    case PDA_ERR_INVALID_ARG: return "invalid argument";
    case PDA_ERR_UNSUPPORTED: return "unsupported shape, dtype or size";
    case PDA_ERR_CUDA: return "CUDA runtime error";
    case PDA_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case PDA_ERR_TOO_LARGE: return "sizes need more scratch than the no-allocation entry point has";
  }
  return "unknown status";
}

extern "C" int pda_version(void) { return 1; }

extern "C" pda_status pda_device_sm_count(int* num_sms) {
  if (num_sms == nullptr) return PDA_ERR_INVALID_ARG;
  int dev;
  return pda::current_device_sms(&dev, num_sms);
}
