"""ctypes front end of the fp64 CPU oracle in ``oracle.c``.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use this module. It imports nothing from the CUDA library and the CUDA
library imports nothing from it.

Arrays are NumPy arrays. A bf16 tensor is passed as its raw bits in a ``uint16`` array;
an fp16 tensor as ``float16``; an fp32 tensor as ``float32``. What each function computes, and the page sections it
follows, is stated in ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

ORC_F32, ORC_BF16, ORC_FP8_E4M3, ORC_F16 = 0, 1, 2, 4
ORC_OK, ORC_ERR_ARG, ORC_ERR_DATA = 0, 1, 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile ``oracle.c`` into a shared library with gcc (OpenMP, -O2)."""
    stale = (not os.path.exists(out)) or os.path.getmtime(out) < os.path.getmtime(src)
    if force or stale:
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: str | None = None):
    """Load (building first if needed) the oracle library and declare its signatures."""
    global _lib
    with _lock:
        if path is None and _lib is not None:
            return _lib
        lib_path = path or build()
        lib = ctypes.CDLL(lib_path)
        P, I, F = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        lib.oracle_version.restype = I
        lib.oracle_kv_append.argtypes = [P, P, P, P, P, I, I, I, I, I, I]
        lib.oracle_kv_append.restype = I
        lib.oracle_kv_pack_blocks.argtypes = [P, P, P, P, I, I, I, I, I, I]
        lib.oracle_kv_pack_blocks.restype = I
        lib.oracle_kv_unpack_blocks.argtypes = [P, P, P, P, I, I, I, I, I, I]
        lib.oracle_kv_unpack_blocks.restype = I
        lib.oracle_paged_decode_attention.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, F,
                                                      I, I, F, F, I]
        lib.oracle_decode_e4m3.argtypes = [I]
        lib.oracle_decode_e4m3.restype = ctypes.c_double
        lib.oracle_decode_e2m1.argtypes = [I]
        lib.oracle_decode_e2m1.restype = ctypes.c_double
        lib.oracle_decode_f16.argtypes = [I]
        lib.oracle_decode_f16.restype = ctypes.c_double
        lib.oracle_paged_decode_attention_nvfp4.argtypes = [P, P, P, P, P, P, P, I, P, I, I, I,
                                                            I, I, I, F, I, F, F, I]
        lib.oracle_paged_decode_attention_nvfp4.restype = I
        lib.oracle_paged_decode_attention.restype = I
        lib.oracle_attention_partial.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, I, I, I, I,
                                                 I, F, I, I]
        lib.oracle_attention_partial.restype = I
        lib.oracle_lse_combine.argtypes = [I, P, P, P, I, P]
        lib.oracle_lse_combine.restype = I
        # NVFP4 block-scale caches [num_blocks, H_kv, block_size, row_bytes]
        lib.oracle_kv_append_block_scales.argtypes = [P, P, P, P, P, I, I, I, I, I]
        lib.oracle_kv_append_block_scales.restype = I
        lib.oracle_kv_pack_block_scales.argtypes = [P, P, P, P, I, I, I, I, I]
        lib.oracle_kv_pack_block_scales.restype = I
        lib.oracle_kv_unpack_block_scales.argtypes = [P, P, P, P, I, I, I, I, I]
        lib.oracle_kv_unpack_block_scales.restype = I
        if path is None:
            _lib = lib
        return lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return ORC_F32
    if a.dtype == np.uint16:
        return ORC_BF16
    if a.dtype == np.uint8:
        return ORC_FP8_E4M3
    if a.dtype == np.float16:
        return ORC_F16
    raise TypeError("oracle takes float32, float16, uint16 (bf16 bits) or uint8 (FP8 E4M3 "
                    f"codes) arrays, got {a.dtype}")


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def kv_append(k_new, v_new, k_cache, v_cache, slot_mapping, lib=None) -> int:
    """In-place append of one token per request into the caches; returns the status."""
    lib = lib or load()
    NB, bs, H_kv, D = k_cache.shape
    B = slot_mapping.shape[0]
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    return lib.oracle_kv_append(_ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
                                _ptr(slot_mapping), B, H_kv, D, bs, NB, _dtype_code(k_cache))


def kv_pack_blocks(k_cache, v_cache, block_table_row, context_len: int, lib=None):
    """Gather one request's K/V into a dense ``[L, 2, H_kv, D]`` array; returns (out, status)."""
    lib = lib or load()
    NB, bs, H_kv, D = k_cache.shape
    out = np.zeros((context_len, 2, H_kv, D), dtype=k_cache.dtype)
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    st = lib.oracle_kv_pack_blocks(_ptr(out), _ptr(k_cache), _ptr(v_cache), _ptr(row),
                                   int(context_len), H_kv, D, bs, NB, _dtype_code(k_cache))
    return out, st


def kv_unpack_blocks(packed, k_cache, v_cache, block_table_row, context_len: int, lib=None) -> int:
    """In-place scatter of a dense ``[L, 2, H_kv, D]`` buffer into the caches; returns status."""
    lib = lib or load()
    NB, bs, H_kv, D = k_cache.shape
    assert packed.dtype == k_cache.dtype and packed.shape[1:] == (2, H_kv, D)
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    return lib.oracle_kv_unpack_blocks(_ptr(np.ascontiguousarray(packed)), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(row), int(context_len), H_kv, D, bs,
                                       NB, _dtype_code(k_cache))


def decode_e2m1(code: int, lib=None) -> float:
    """Exact value of one FP4 E2M1 code (0..15)."""
    return (lib or load()).oracle_decode_e2m1(int(code))


def paged_decode_attention_nvfp4(q, k_data, v_data, k_block_scales, v_block_scales,
                                 block_tables, context_lens, scale: float, k_scale: float = 1.0,
                                 v_scale: float = 1.0, num_threads: int = 0, lib=None):
    """fp64 attention over an NVFP4 cache: data [NB, bs, H_kv, D/2] uint8 (two E2M1 codes
    per byte, even element in the low nibble), block scales [NB, H_kv, bs, D/16] uint8
    (E4M3, per block and kv-head). Returns (out[B,H,D] float64, status)."""
    lib = lib or load()
    B, H, D = q.shape
    NB, bs, H_kv, half = k_data.shape
    assert half * 2 == D and k_data.dtype == np.uint8 and v_data.shape == k_data.shape
    assert k_block_scales.shape == (NB, H_kv, bs, D // 16) == v_block_scales.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    out = np.zeros((B, H, D), dtype=np.float64)
    st = lib.oracle_paged_decode_attention_nvfp4(
        _ptr(out), _ptr(q), _ptr(k_data), _ptr(v_data), _ptr(k_block_scales),
        _ptr(v_block_scales), _ptr(bt), bt.shape[1], _ptr(cl), B, H, H_kv, D, bs, NB,
        ctypes.c_float(scale), _dtype_code(q), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
        int(num_threads))
    return out, st


def decode_f16(bits: int, lib=None) -> float:
    """The value of a binary16 bit pattern (exact in double)."""
    return (lib or load()).oracle_decode_f16(int(bits))


def decode_e4m3(code: int, lib=None) -> float:
    """Exact value of one FP8 E4M3 code."""
    return (lib or load()).oracle_decode_e4m3(int(code))


def paged_decode_attention(q, k_cache, v_cache, block_tables, context_lens, scale: float,
                           num_threads: int = 0, lib=None, k_scale: float = 1.0,
                           v_scale: float = 1.0):
    """fp64 decode attention over the paged cache; returns (out[B,H,D] float64, status).
    FP8 caches (uint8 codes) mean code value times k_scale / v_scale."""
    lib = lib or load()
    B, H, D = q.shape
    NB, bs, H_kv, D2 = k_cache.shape
    assert D == D2 and v_cache.shape == k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.zeros((B, H, D), dtype=np.float64)
    st = lib.oracle_paged_decode_attention(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), max_blocks, _ptr(cl), B, H,
        H_kv, D, bs, NB, ctypes.c_float(scale), _dtype_code(q), _dtype_code(k_cache),
        ctypes.c_float(k_scale), ctypes.c_float(v_scale), int(num_threads))
    return out, st


def attention_partial(q, k_cache, v_cache, block_tables, b: int, h: int, t0: int, t1: int,
                      scale: float, lib=None):
    """Unnormalised (m, l, o) of head h of request b over tokens [t0, t1)."""
    lib = lib or load()
    B, H, D = q.shape
    NB, bs, H_kv, _ = k_cache.shape
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    m = np.zeros(1, np.float64)
    l_ = np.zeros(1, np.float64)
    o = np.zeros(D, np.float64)
    st = lib.oracle_attention_partial(_ptr(m), _ptr(l_), _ptr(o), _ptr(q), _ptr(k_cache),
                                      _ptr(v_cache), _ptr(bt), bt.shape[1], b, h, t0, t1, H,
                                      H_kv, D, bs, NB, ctypes.c_float(scale), _dtype_code(q),
                                      _dtype_code(k_cache))
    if st != ORC_OK:
        raise RuntimeError(f"oracle_attention_partial failed with status {st}")
    return float(m[0]), float(l_[0]), o


def lse_combine(m, l_, o, lib=None):
    """Log-sum-exp merge of pieces m[n], l[n], o[n, D] into one normalised row."""
    lib = lib or load()
    m = np.ascontiguousarray(m, np.float64)
    l_ = np.ascontiguousarray(l_, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    n, D = o.shape
    out = np.zeros(D, np.float64)
    st = lib.oracle_lse_combine(n, _ptr(m), _ptr(l_), _ptr(o), D, _ptr(out))
    if st != ORC_OK:
        raise RuntimeError(f"oracle_lse_combine failed with status {st}")
    return out


def kv_append_block_scales(k_new, v_new, k_scales, v_scales, slot_mapping, lib=None) -> int:
    """In-place append of one token's scale rows per request into NVFP4 block-scale caches
    [NB, H_kv, bs, R] (new rows [B, H_kv, R]); returns the status."""
    lib = lib or load()
    NB, H_kv, bs, R = k_scales.shape
    B = slot_mapping.shape[0]
    assert k_new.shape == (B, H_kv, R) == v_new.shape and k_scales.dtype == np.uint8
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int32)
    return lib.oracle_kv_append_block_scales(_ptr(k_new), _ptr(v_new), _ptr(k_scales),
                                             _ptr(v_scales), _ptr(slot_mapping), B, H_kv, R,
                                             bs, NB)


def kv_pack_block_scales(k_scales, v_scales, block_table_row, context_len: int, lib=None):
    """One request's scale rows from block-scale caches [NB, H_kv, bs, R] into a dense
    token-major [L, 2, H_kv, R] buffer; returns (out, status)."""
    lib = lib or load()
    NB, H_kv, bs, R = k_scales.shape
    out = np.zeros((context_len, 2, H_kv, R), dtype=np.uint8)
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    st = lib.oracle_kv_pack_block_scales(_ptr(out), _ptr(k_scales), _ptr(v_scales), _ptr(row),
                                         int(context_len), H_kv, R, bs, NB)
    return out, st


def kv_unpack_block_scales(packed, k_scales, v_scales, block_table_row, context_len: int,
                           lib=None) -> int:
    """The inverse of kv_pack_block_scales, in place; returns the status."""
    lib = lib or load()
    NB, H_kv, bs, R = k_scales.shape
    assert packed.shape[1:] == (2, H_kv, R)
    row = np.ascontiguousarray(block_table_row, dtype=np.int32)
    return lib.oracle_kv_unpack_block_scales(_ptr(np.ascontiguousarray(packed)), _ptr(k_scales),
                                             _ptr(v_scales), _ptr(row), int(context_len),
                                             H_kv, R, bs, NB)
