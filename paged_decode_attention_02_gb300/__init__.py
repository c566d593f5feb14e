"""Decode attention over a paged KV cache for GB300 (sm_103a).

The computation lives in ``libpda.so`` (CUDA kernels behind the C ABI of ``include/pda.h``);
``binding`` marshals torch tensors into it and ``workloads`` draws seeded synthetic inputs.
"""
from .binding import (PdaDeviceError, PdaError, alloc_workspace, check_error, attention_workspace_size, device_sm_count,
                      kv_append, kv_append_block_scales, kv_pack_block_scales_batched,
                      kv_unpack_block_scales_batched, kv_pack_blocks, kv_pack_blocks_batched, kv_pack_layers,
                      kv_unpack_blocks, kv_unpack_blocks_batched, kv_unpack_layers,
                      paged_decode_attention,
                      paged_decode_attention_fp8, paged_decode_attention_nvfp4,
                      paged_decode_attention_noalloc, status_string)

__all__ = ["PdaDeviceError", "PdaError", "alloc_workspace", "check_error", "attention_workspace_size", "device_sm_count",
           "kv_append", "kv_append_block_scales", "kv_pack_block_scales_batched",
           "kv_unpack_block_scales_batched", "kv_pack_blocks", "kv_pack_blocks_batched", "kv_pack_layers",
           "kv_unpack_blocks", "kv_unpack_blocks_batched", "kv_unpack_layers", "paged_decode_attention", "paged_decode_attention_fp8",
           "paged_decode_attention_nvfp4", "paged_decode_attention_noalloc",
           "status_string"]
