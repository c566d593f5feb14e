"""Unpaged dense attention in NumPy fp64, for tiny inputs.

TEST INFRASTRUCTURE. This is a second, independent statement of the attention the oracle
computes, with no block table at all: each request's K and V are given as contiguous
``[L, H_kv, D]`` arrays. The test that compares it with ``oracle.c`` builds the contiguous
history first and only then scatters it into a paged pool, so the comparison checks the
oracle's page-table walk (page "From PagedAttention to Prefill-Decode disaggregation",
sec. 2.2 steps 1-2) as well as its softmax.
"""
from __future__ import annotations

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of bf16 bit patterns: they are the upper half of a binary32."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def dense_decode_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """softmax(scale * q K^T) V for one request.

    q: [H, D]; K, V: [L, H_kv, D]; query head h uses kv-head h // (H // H_kv).
    Returns [H, D] float64. L == 0 returns zeros.
    """
    q = np.asarray(q, np.float64)
    K = np.asarray(K, np.float64)
    V = np.asarray(V, np.float64)
    H, D = q.shape
    L, H_kv, _ = K.shape
    out = np.zeros((H, D), np.float64)
    if L == 0:
        return out
    g = H // H_kv
    for h in range(H):
        kh = h // g
        s = np.float64(scale) * (K[:, kh, :] @ q[h])
        w = np.exp(s - s.max())
        out[h] = (w / w.sum()) @ V[:, kh, :]
    return out
