"""Thin ctypes binding over ``libpda.so`` (declared in ``include/pda.h``).

Argument marshalling only: shapes, dtypes and devices are read off torch tensors and
passed as plain pointers and sizes; every step of the computation runs in the library's
CUDA kernels. The library must be built (``build_lib.build()``); if it is missing or
fails to load, every call raises, and nothing falls back to another implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build_lib

(PDA_OK, PDA_ERR_INVALID_ARG, PDA_ERR_UNSUPPORTED, PDA_ERR_CUDA, PDA_ERR_WORKSPACE,
 PDA_ERR_TOO_LARGE) = range(6)
PDA_F32, PDA_BF16, PDA_FP8_E4M3, PDA_NVFP4, PDA_F16 = 0, 1, 2, 3, 4
PDA_DEVERR_CONTEXT_LEN, PDA_DEVERR_BLOCK_ID, PDA_DEVERR_SLOT, PDA_DEVERR_TIMEOUT = 1, 2, 4, 8
PDA_PACK_MAX_BATCH = 64
PDA_PACK_MAX_LAYERS = 256
PDA_NOALLOC_SCRATCH_BYTES = 8 << 20

EXPORTED = [
    "pda_status_string", "pda_version", "pda_device_sm_count", "pda_kv_append",
    "pda_attention_workspace_size", "pda_paged_decode_attention", "pda_kv_pack_blocks",
    "pda_kv_pack_blocks_batched", "pda_paged_decode_attention_noalloc",
    "pda_kv_unpack_blocks", "pda_kv_unpack_blocks_batched", "pda_paged_decode_attention_fp8",
    "pda_paged_decode_attention_nvfp4", "pda_kv_pack_layers", "pda_kv_unpack_layers",
    "pda_kv_append_block_scales", "pda_kv_pack_block_scales_batched",
    "pda_kv_unpack_block_scales_batched",
]

_lock = threading.Lock()
_lib = None


class PdaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def lib_path() -> str:
    return build_lib.LIB_PATH


def load():
    """Load libpda.so and declare its C signatures. Raises if the library is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = lib_path()
        if not os.path.exists(path):
            raise RuntimeError(f"libpda.so is not built ({path}); run build_lib.build() first")
        lib = ctypes.CDLL(path)
        P, I, F, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.pda_status_string.argtypes = [I]
        lib.pda_status_string.restype = ctypes.c_char_p
        lib.pda_version.restype = I
        lib.pda_device_sm_count.argtypes = [ctypes.POINTER(I)]
        lib.pda_device_sm_count.restype = I
        lib.pda_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, I, I, P, P]
        lib.pda_kv_append.restype = I
        lib.pda_attention_workspace_size.argtypes = [I, I, I, I, I, I, I, ctypes.POINTER(SZ)]
        lib.pda_attention_workspace_size.restype = I
        lib.pda_paged_decode_attention.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, F,
                                                   I, I, I, I, P, SZ, P, P]
        lib.pda_paged_decode_attention.restype = I
        lib.pda_paged_decode_attention_fp8.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I,
                                                       F, F, F, I, I, I, P, SZ, P, P]
        lib.pda_paged_decode_attention_fp8.restype = I
        lib.pda_paged_decode_attention_nvfp4.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I, I,
                                                         I, I, I, F, F, F, I, I, I, P, SZ, P, P]
        lib.pda_paged_decode_attention_nvfp4.restype = I
        lib.pda_paged_decode_attention_noalloc.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I,
                                                           I, I, F, I, I, I, I, P, P]
        lib.pda_paged_decode_attention_noalloc.restype = I
        lib.pda_kv_pack_blocks.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P]
        lib.pda_kv_pack_blocks.restype = I
        lib.pda_kv_pack_blocks_batched.argtypes = [P, P, P, I, P, P, I, I, I, I, I, P, P]
        lib.pda_kv_pack_blocks_batched.restype = I
        lib.pda_kv_unpack_blocks.argtypes = [P, P, P, P, I, I, I, I, I, I, P, P]
        lib.pda_kv_unpack_blocks.restype = I
        lib.pda_kv_unpack_blocks_batched.argtypes = [P, P, P, I, P, P, I, I, I, I, I, P, P]
        lib.pda_kv_unpack_blocks_batched.restype = I
        # outs/ins, k_caches, v_caches, n_layers, table row, context_len, H_kv, D, bs, NB,
        # dtype, error_word, stream
        lib.pda_kv_pack_layers.argtypes = [P, P, P, I, P, I, I, I, I, I, I, P, P]
        lib.pda_kv_pack_layers.restype = I
        lib.pda_kv_unpack_layers.argtypes = [P, P, P, I, P, I, I, I, I, I, I, P, P]
        lib.pda_kv_unpack_layers.restype = I
        # NVFP4 block scales: news/caches, slots or (bufs, rows, lens, n), H_kv, D, bs, NB, ...
        lib.pda_kv_append_block_scales.argtypes = [P, P, P, P, P, I, I, I, I, I, P, P]
        lib.pda_kv_append_block_scales.restype = I
        lib.pda_kv_pack_block_scales_batched.argtypes = [P, P, P, I, P, P, I, I, I, I, P, P]
        lib.pda_kv_pack_block_scales_batched.restype = I
        lib.pda_kv_unpack_block_scales_batched.argtypes = [P, P, P, I, P, P, I, I, I, I, P, P]
        lib.pda_kv_unpack_block_scales_batched.restype = I
        _lib = lib
        return lib


def status_string(status: int) -> str:
    return load().pda_status_string(int(status)).decode()


class PdaDeviceError(RuntimeError):
    """A kernel reported bad device data (or a timed-out wait) through the error word."""

    NAMES = {PDA_DEVERR_CONTEXT_LEN: "context length out of range",
             PDA_DEVERR_BLOCK_ID: "block id out of range",
             PDA_DEVERR_SLOT: "slot out of range",
             PDA_DEVERR_TIMEOUT: "pipeline wait timed out"}

    def __init__(self, bits: int):
        self.bits = bits
        names = [n for b, n in self.NAMES.items() if bits & b] or [f"bits {bits:#x}"]
        super().__init__("device error: " + ", ".join(names))


def check_error(error_word: torch.Tensor, reset: bool = True):
    """Synchronises, reads a device error word and raises PdaDeviceError if any bit is set
    (and, by default, zeroes it). A host sync: for tests and debugging, not the hot loop."""
    torch.cuda.synchronize(error_word.device)
    bits = int(error_word.item())
    if reset:
        error_word.zero_()
    if bits:
        raise PdaDeviceError(bits)


def _check(status: int, what: str):
    if status != PDA_OK:
        raise PdaError(status, what)


def _dtype(t: torch.Tensor) -> int:
    """float32, bfloat16, float16, or FP8 E4M3 codes (torch.float8_e4m3fn, or uint8 holding
    codes)."""
    if t.dtype == torch.float32:
        return PDA_F32
    if t.dtype == torch.bfloat16:
        return PDA_BF16
    if t.dtype == torch.float16:
        return PDA_F16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return PDA_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}; use float32, bfloat16, float16 or FP8 E4M3 "
                    "codes")


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def device_sm_count() -> int:
    n = ctypes.c_int(0)
    _check(load().pda_device_sm_count(ctypes.byref(n)), "pda_device_sm_count")
    return n.value


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, error_word=None, stream=None):
    """Scatter each request's new K/V (``[B, H_kv, D]``) into its cache slot."""
    NB, bs, H_kv, D = k_cache.shape
    B = slot_mapping.shape[0]
    assert k_new.shape == (B, H_kv, D) and v_new.shape == (B, H_kv, D)
    assert slot_mapping.dtype == torch.int32
    _check(load().pda_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(slot_mapping), B, H_kv, D, bs, NB, _dtype(k_cache),
                                _ptr(error_word), _stream(stream)), "pda_kv_append")


def attention_workspace_size(B, H, H_kv, D, block_size=16, kv_dtype=torch.bfloat16,
                             sm_cap=0) -> int:
    n = ctypes.c_size_t(0)
    dt = {torch.bfloat16: PDA_BF16, torch.float32: PDA_F32, torch.float16: PDA_F16,
          torch.uint8: PDA_FP8_E4M3, torch.float8_e4m3fn: PDA_FP8_E4M3}[kv_dtype]
    _check(load().pda_attention_workspace_size(B, H, H_kv, D, block_size, dt, sm_cap,
                                               ctypes.byref(n)), "pda_attention_workspace_size")
    return n.value


def alloc_workspace(B, H, H_kv, D, block_size=16, kv_dtype=torch.bfloat16, sm_cap=0,
                    device=None) -> torch.Tensor:
    """Workspace for one attention call (torch.uint8 / float8_e4m3fn mean an FP8 cache)."""
    n = attention_workspace_size(B, H, H_kv, D, block_size, kv_dtype, sm_cap)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens,
                           max_context_len: int, scale: float, sm_cap: int = 0, workspace=None,
                           error_word=None, stream=None):
    """``out[b,h] = softmax(scale q[b,h] K^T) V`` over request b's paged history."""
    B, H, D = q.shape
    NB, bs, H_kv, D2 = k_cache.shape
    assert D == D2 and v_cache.shape == k_cache.shape and out.shape == q.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    if workspace is None:
        workspace = alloc_workspace(B, H, H_kv, D, bs, k_cache.dtype, sm_cap, q.device)
    _check(load().pda_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks,
        _ptr(context_lens), int(max_context_len), B, H, H_kv, D, bs, NB, float(scale),
        _dtype(q), _dtype(k_cache), _dtype(out), int(sm_cap), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(error_word), _stream(stream)),
        "pda_paged_decode_attention")
    return out


def paged_decode_attention_fp8(out, q, k_cache, v_cache, block_tables, context_lens,
                               max_context_len: int, scale: float, k_scale: float,
                               v_scale: float, sm_cap: int = 0, workspace=None, error_word=None,
                               stream=None):
    """Attention over an FP8 E4M3 cache: stored code c of K means decode(c) * k_scale."""
    B, H, D = q.shape
    NB, bs, H_kv, D2 = k_cache.shape
    assert D == D2 and v_cache.shape == k_cache.shape and out.shape == q.shape
    assert _dtype(k_cache) == PDA_FP8_E4M3 and _dtype(v_cache) == PDA_FP8_E4M3
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    if workspace is None:
        workspace = alloc_workspace(B, H, H_kv, D, bs, torch.uint8, sm_cap, q.device)
    _check(load().pda_paged_decode_attention_fp8(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks,
        _ptr(context_lens), int(max_context_len), B, H, H_kv, D, bs, NB, float(scale),
        float(k_scale), float(v_scale), _dtype(q), _dtype(out), int(sm_cap), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(error_word), _stream(stream)),
        "pda_paged_decode_attention_fp8")
    return out


def paged_decode_attention_nvfp4(out, q, k_data, v_data, k_block_scales, v_block_scales,
                                 block_tables, context_lens, max_context_len: int, scale: float,
                                 k_scale: float, v_scale: float, sm_cap: int = 0, workspace=None,
                                 error_word=None, stream=None):
    """Attention over an NVFP4 cache: data [NB, bs, H_kv, D/2] uint8 (two E2M1 codes per
    byte, even element low), block scales [NB, H_kv, bs, D/16] uint8 (E4M3, per block and
    head-major)."""
    B, H, D = q.shape
    NB, bs, H_kv, half = k_data.shape
    assert 2 * half == D and v_data.shape == k_data.shape and out.shape == q.shape
    assert tuple(k_block_scales.shape) == (NB, H_kv, bs, D // 16)
    assert v_block_scales.shape == k_block_scales.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    if workspace is None:
        n = ctypes.c_size_t(0)
        _check(load().pda_attention_workspace_size(B, H, H_kv, D, bs, PDA_NVFP4, sm_cap,
                                                   ctypes.byref(n)), "workspace size")
        workspace = torch.empty(max(n.value, 256), dtype=torch.uint8, device=q.device)
    _check(load().pda_paged_decode_attention_nvfp4(
        _ptr(out), _ptr(q), _ptr(k_data), _ptr(v_data), _ptr(k_block_scales),
        _ptr(v_block_scales), _ptr(block_tables), max_blocks, _ptr(context_lens),
        int(max_context_len), B, H, H_kv, D, bs, NB, float(scale), float(k_scale),
        float(v_scale), _dtype(q), _dtype(out), int(sm_cap), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(error_word), _stream(stream)),
        "pda_paged_decode_attention_nvfp4")
    return out


def nvfp4_workspace(B, H, H_kv, D, block_size=16, sm_cap=0, device=None) -> torch.Tensor:
    n = ctypes.c_size_t(0)
    _check(load().pda_attention_workspace_size(B, H, H_kv, D, block_size, PDA_NVFP4, sm_cap,
                                               ctypes.byref(n)), "workspace size")
    return torch.empty(max(n.value, 256), dtype=torch.uint8, device=device or "cuda")


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   max_context_len: int, scale: float, sm_cap: int = 0,
                                   error_word=None, stream=None):
    """``paged_decode_attention`` with the library's fixed scratch instead of a workspace,
    for callers that may not allocate device memory. Calls that overlap on the GPU race."""
    B, H, D = q.shape
    NB, bs, H_kv, D2 = k_cache.shape
    assert D == D2 and v_cache.shape == k_cache.shape and out.shape == q.shape
    assert block_tables.dtype == torch.int32 and context_lens.dtype == torch.int32
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    _check(load().pda_paged_decode_attention_noalloc(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), max_blocks,
        _ptr(context_lens), int(max_context_len), B, H, H_kv, D, bs, NB, float(scale),
        _dtype(q), _dtype(k_cache), _dtype(out), int(sm_cap), _ptr(error_word),
        _stream(stream)), "pda_paged_decode_attention_noalloc")
    return out


def kv_pack_blocks(out, k_cache, v_cache, block_table_row, context_len: int, error_word=None,
                   stream=None):
    """Gather one request's K/V into ``out[context_len, 2, H_kv, D]``."""
    NB, bs, H_kv, D = k_cache.shape
    assert out.shape[0] >= context_len and tuple(out.shape[1:]) == (2, H_kv, D)
    _check(load().pda_kv_pack_blocks(_ptr(out), _ptr(k_cache), _ptr(v_cache),
                                     _ptr(block_table_row), int(context_len), H_kv, D, bs, NB,
                                     _dtype(k_cache), _ptr(error_word), _stream(stream)),
           "pda_kv_pack_blocks")
    return out


def kv_pack_blocks_batched(outs, k_cache, v_cache, block_table_rows, context_lens,
                           error_word=None, stream=None):
    """``kv_pack_blocks`` for several requests in one launch."""
    NB, bs, H_kv, D = k_cache.shape
    n = len(outs)
    assert len(block_table_rows) == n and len(context_lens) == n
    out_arr = (ctypes.c_void_p * max(n, 1))(*[o.data_ptr() for o in outs])
    for o in outs:
        _ptr(o)
    row_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(r).value for r in block_table_rows])
    len_arr = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in context_lens])
    _check(load().pda_kv_pack_blocks_batched(out_arr, row_arr, len_arr, n, _ptr(k_cache),
                                             _ptr(v_cache), H_kv, D, bs, NB, _dtype(k_cache),
                                             _ptr(error_word), _stream(stream)),
           "pda_kv_pack_blocks_batched")
    return outs


def kv_unpack_blocks(packed, k_cache, v_cache, block_table_row, context_len: int,
                     error_word=None, stream=None):
    """Scatter one request's ``[context_len, 2, H_kv, D]`` buffer into its cache blocks."""
    NB, bs, H_kv, D = k_cache.shape
    assert packed.shape[0] >= context_len and tuple(packed.shape[1:]) == (2, H_kv, D)
    _check(load().pda_kv_unpack_blocks(_ptr(packed), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_table_row), int(context_len), H_kv, D, bs,
                                       NB, _dtype(k_cache), _ptr(error_word), _stream(stream)),
           "pda_kv_unpack_blocks")


def kv_unpack_blocks_batched(packed, k_cache, v_cache, block_table_rows, context_lens,
                             error_word=None, stream=None):
    """``kv_unpack_blocks`` for several requests in one launch."""
    NB, bs, H_kv, D = k_cache.shape
    n = len(packed)
    assert len(block_table_rows) == n and len(context_lens) == n
    in_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(x).value for x in packed])
    row_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(r).value for r in block_table_rows])
    len_arr = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in context_lens])
    _check(load().pda_kv_unpack_blocks_batched(in_arr, row_arr, len_arr, n, _ptr(k_cache),
                                               _ptr(v_cache), H_kv, D, bs, NB, _dtype(k_cache),
                                               _ptr(error_word), _stream(stream)),
           "pda_kv_unpack_blocks_batched")


def kv_append_block_scales(k_new, v_new, k_scales, v_scales, slot_mapping, error_word=None,
                           stream=None):
    """Scatter each request's new NVFP4 block scales (``[B, H_kv, D/16]`` uint8) into the
    ``[NB, H_kv, bs, D/16]`` scale caches at its slot."""
    NB, H_kv, bs, S = k_scales.shape
    B = slot_mapping.shape[0]
    assert k_new.shape == (B, H_kv, S) and v_new.shape == (B, H_kv, S)
    assert v_scales.shape == k_scales.shape and slot_mapping.dtype == torch.int32
    _check(load().pda_kv_append_block_scales(_ptr(k_new), _ptr(v_new), _ptr(k_scales),
                                             _ptr(v_scales), _ptr(slot_mapping), B, H_kv,
                                             16 * S, bs, NB, _ptr(error_word),
                                             _stream(stream)), "pda_kv_append_block_scales")


def _scale_arrays(bufs, block_table_rows, context_lens, shape_tail):
    n = len(bufs)
    assert len(block_table_rows) == n and len(context_lens) == n
    for b, L in zip(bufs, context_lens):
        assert b.shape[0] >= int(L) and tuple(b.shape[1:]) == shape_tail
    buf_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(x).value for x in bufs])
    row_arr = (ctypes.c_void_p * max(n, 1))(*[_ptr(r).value for r in block_table_rows])
    len_arr = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in context_lens])
    return n, buf_arr, row_arr, len_arr


def kv_pack_block_scales_batched(outs, k_scales, v_scales, block_table_rows, context_lens,
                                 error_word=None, stream=None):
    """Gather requests' NVFP4 block scales into ``outs[i][len_i, 2, H_kv, D/16]``."""
    NB, H_kv, bs, S = k_scales.shape
    n, o, r, l = _scale_arrays(outs, block_table_rows, context_lens, (2, H_kv, S))
    _check(load().pda_kv_pack_block_scales_batched(o, r, l, n, _ptr(k_scales), _ptr(v_scales),
                                                   H_kv, 16 * S, bs, NB, _ptr(error_word),
                                                   _stream(stream)),
           "pda_kv_pack_block_scales_batched")
    return outs


def kv_unpack_block_scales_batched(packed, k_scales, v_scales, block_table_rows,
                                   context_lens, error_word=None, stream=None):
    """Scatter requests' ``[len_i, 2, H_kv, D/16]`` scale buffers into the scale caches."""
    NB, H_kv, bs, S = k_scales.shape
    n, i, r, l = _scale_arrays(packed, block_table_rows, context_lens, (2, H_kv, S))
    _check(load().pda_kv_unpack_block_scales_batched(i, r, l, n, _ptr(k_scales),
                                                     _ptr(v_scales), H_kv, 16 * S, bs, NB,
                                                     _ptr(error_word), _stream(stream)),
           "pda_kv_unpack_block_scales_batched")


def _layer_arrays(bufs, k_caches, v_caches):
    n = len(bufs)
    assert len(k_caches) == n and len(v_caches) == n
    NB, bs, H_kv, D = k_caches[0].shape
    for k, v in zip(k_caches, v_caches):
        assert tuple(k.shape) == (NB, bs, H_kv, D) == tuple(v.shape)
        assert k.dtype == v.dtype == k_caches[0].dtype
    arr = lambda ts: (ctypes.c_void_p * max(n, 1))(*[_ptr(t).value for t in ts])
    return n, arr(bufs), arr(k_caches), arr(v_caches), (NB, bs, H_kv, D)


def kv_pack_layers(outs, k_caches, v_caches, block_table_row, context_len: int,
                   error_word=None, stream=None):
    """One request's blocks in every layer's caches -> ``outs[i]`` ``[context_len, 2, H_kv,
    D]``, one launch (all layers share the request's block table)."""
    n, out_arr, k_arr, v_arr, (NB, bs, H_kv, D) = _layer_arrays(outs, k_caches, v_caches)
    for o in outs:
        assert o.shape[0] >= context_len and tuple(o.shape[1:]) == (2, H_kv, D)
    _check(load().pda_kv_pack_layers(out_arr, k_arr, v_arr, n, _ptr(block_table_row),
                                     int(context_len), H_kv, D, bs, NB, _dtype(k_caches[0]),
                                     _ptr(error_word), _stream(stream)), "pda_kv_pack_layers")
    return outs


def kv_unpack_layers(packed, k_caches, v_caches, block_table_row, context_len: int,
                     error_word=None, stream=None):
    """The inverse of ``kv_pack_layers``: ``packed[i]`` into layer i's caches, one launch."""
    n, in_arr, k_arr, v_arr, (NB, bs, H_kv, D) = _layer_arrays(packed, k_caches, v_caches)
    for x in packed:
        assert x.shape[0] >= context_len and tuple(x.shape[1:]) == (2, H_kv, D)
    _check(load().pda_kv_unpack_layers(in_arr, k_arr, v_arr, n, _ptr(block_table_row),
                                       int(context_len), H_kv, D, bs, NB, _dtype(k_caches[0]),
                                       _ptr(error_word), _stream(stream)),
           "pda_kv_unpack_layers")
