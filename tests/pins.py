"""Pins of the fp64 oracle to facts other than itself.

Each ``pin_*`` function takes an oracle library handle and raises ``AssertionError`` when
the oracle disagrees with what the pages or the mathematics fix. ``test_oracle_pins.py``
runs them on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the oracle
with one planted mistake each and checks that some pin fails.

Facts used:
  - hand-derived closed forms stored under ``tests/golden/``;
  - a context of one token returns that token's V exactly;
  - identical keys (or scale 0) give the mean of V; one dominant key gives its V;
  - permuting physical blocks and rewriting the tables leaves the output bit-identical
    (PagedAttention: blocks need not be contiguous, page "From PagedAttention to
    Prefill-Decode disaggregation", sec. 2.2 step 2);
  - two requests mapped to the same blocks with the same q give identical rows
    (shared prefixes, same page, sec. 2.3);
  - a dense, unpaged NumPy attention over the contiguous history agrees to 1e-12;
  - GQA equals MHA with each kv-head replicated;
  - the log-sum-exp merge of pieces equals the whole;
  - output is linear in V;
  - append then pack gives back the history plus the new token, bit for bit;
  - unpack into freshly scattered blocks then pack gives back the buffer, bit for bit, and
    unpack touches no row outside the request's tokens;
  - every FP8 E4M3 code decodes to the value torch's own float8_e4m3fn conversion gives,
    and to hand-derived values at the format's landmarks; FP8 attention with per-tensor
    scales matches the dense brute force run on torch-decoded, scaled values;
  - every FP4 E2M1 code decodes to the format's table of values; NVFP4 attention matches
    the dense brute force run on values decoded through that table and torch's E4M3;
  - every binary16 bit pattern decodes to NumPy's float16 value, and to hand-derived values
    at the format's landmarks; fp16 attention matches the dense brute force.
"""
from __future__ import annotations

import glob
import json
import math
import os

import numpy as np

from oracle import brute
from oracle import oracle as orc

GOLDEN_DIR = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------- input construction
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 (round to nearest, ties to even); return the bits."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def as_stored(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":  # NumPy's binary16 conversion (round to nearest even)
        return np.ascontiguousarray(x, np.float32).astype(np.float16)
    return np.ascontiguousarray(x, np.float32)


def stored_to_f64(a: np.ndarray) -> np.ndarray:
    return brute.bf16_bits_to_f64(a) if a.dtype == np.uint16 else a.astype(np.float64)


class Paged:
    """Contiguous per-request histories scattered into a paged pool by a random permutation."""

    def __init__(self, rng, lengths, H, H_kv, D, bs, dtype="f32", spare_blocks=3, q=None,
                 hist=None):
        self.lengths = np.asarray(lengths, np.int32)
        B = len(lengths)
        self.B, self.H, self.H_kv, self.D, self.bs, self.dtype = B, H, H_kv, D, bs, dtype
        nblk = [(int(L) + bs - 1) // bs for L in lengths]
        self.NB = sum(nblk) + spare_blocks
        self.max_blocks = max(1, max(nblk) if nblk else 1)
        self.q = as_stored(rng.standard_normal((B, H, D)) if q is None else q, dtype)
        if hist is None:
            hist = [(rng.standard_normal((int(L), H_kv, D)), rng.standard_normal((int(L), H_kv, D)))
                    for L in lengths]
        self.K = [as_stored(k, dtype) for k, _ in hist]
        self.V = [as_stored(v, dtype) for _, v in hist]
        # pool filled with unrelated values, so a wrong read changes the answer
        self.k_cache = as_stored(rng.standard_normal((self.NB, bs, H_kv, D)) * 7.0, dtype)
        self.v_cache = as_stored(rng.standard_normal((self.NB, bs, H_kv, D)) * 7.0, dtype)
        perm = rng.permutation(self.NB).astype(np.int32)
        self.bt = np.full((B, self.max_blocks), -1, np.int32)
        off = 0
        for b, L in enumerate(lengths):
            n = nblk[b]
            self.bt[b, :n] = perm[off:off + n]
            off += n
            for t in range(int(L)):
                blk, row = self.bt[b, t // bs], t % bs
                self.k_cache[blk, row] = self.K[b][t]
                self.v_cache[blk, row] = self.V[b][t]

    def oracle(self, lib, scale):
        return orc.paged_decode_attention(self.q, self.k_cache, self.v_cache, self.bt,
                                          self.lengths, scale, lib=lib)

    def dense(self, scale):
        return np.stack([brute.dense_decode_attention(stored_to_f64(self.q[b]),
                                                      stored_to_f64(self.K[b]),
                                                      stored_to_f64(self.V[b]), scale)
                         for b in range(self.B)])


# ---------------------------------------------------------------- pins
def pin_golden(lib):
    files = sorted(glob.glob(os.path.join(GOLDEN_DIR, "*closed_form*.json")))
    assert files, "no golden fixtures"
    for path in files:
        g = json.load(open(path))
        q = np.array(g["q"], np.float32)
        kc = np.array(g["k_cache"], np.float32)
        vc = np.array(g["v_cache"], np.float32)
        out, st = orc.paged_decode_attention(q, kc, vc, np.array(g["block_tables"], np.int32),
                                             np.array(g["context_lens"], np.int32), g["scale"],
                                             lib=lib)
        assert st == orc.ORC_OK, (path, st)
        err = np.abs(out - np.array(g["expected"])).max()
        assert err <= g["tolerance"], (os.path.basename(path), err)


def pin_ctx1_returns_v(lib):
    rng = np.random.default_rng(11)
    for dtype in ("f32", "bf16"):
        p = Paged(rng, [1, 1, 1], H=4, H_kv=2, D=16, bs=4, dtype=dtype)
        out, st = p.oracle(lib, 0.25)
        assert st == orc.ORC_OK
        for b in range(p.B):
            for h in range(p.H):
                want = stored_to_f64(p.V[b][0, h // 2])
                assert np.array_equal(out[b, h], want), (dtype, b, h)


def pin_identical_keys_mean(lib):
    rng = np.random.default_rng(12)
    L, H_kv, D = 37, 2, 8
    k1 = rng.standard_normal((1, H_kv, D))
    hist = [(np.repeat(k1, L, axis=0), rng.standard_normal((L, H_kv, D)))]
    p = Paged(rng, [L], H=2, H_kv=H_kv, D=D, bs=8, hist=hist)
    out, st = p.oracle(lib, 0.7)
    assert st == orc.ORC_OK
    want = stored_to_f64(p.V[0]).mean(axis=0)
    assert np.abs(out[0] - want).max() <= 1e-12


def pin_scale_zero_mean_and_dominant_key(lib):
    rng = np.random.default_rng(13)
    L, D = 21, 8
    p = Paged(rng, [L], H=1, H_kv=1, D=D, bs=4)
    out, st = p.oracle(lib, 0.0)
    assert st == orc.ORC_OK
    assert np.abs(out[0, 0] - stored_to_f64(p.V[0])[:, 0].mean(axis=0)).max() <= 1e-12
    # one key aligned with q and a large scale: its weight dominates by e^(scale*gap)
    K = np.zeros((L, 1, D))
    K[9, 0, 0] = 1.0
    q = np.zeros((1, 1, D))
    q[0, 0, 0] = 1.0
    hist = [(K, rng.standard_normal((L, 1, D)))]
    p = Paged(rng, [L], H=1, H_kv=1, D=D, bs=4, q=q, hist=hist)
    out, st = p.oracle(lib, 2000.0)  # exp(2000) overflows unless the max is subtracted
    assert st == orc.ORC_OK
    assert np.all(np.isfinite(out))
    assert np.abs(out[0, 0] - stored_to_f64(p.V[0])[9, 0]).max() <= 1e-12


def pin_block_permutation_invariance(lib):
    rng = np.random.default_rng(14)
    for dtype in ("f32", "bf16"):
        p = Paged(rng, [5, 16, 17, 40], H=4, H_kv=2, D=8, bs=4, dtype=dtype)
        out1, _ = p.oracle(lib, 0.3)
        perm = rng.permutation(p.NB)
        inv = np.argsort(perm)
        k2 = np.ascontiguousarray(p.k_cache[perm])
        v2 = np.ascontiguousarray(p.v_cache[perm])
        bt2 = np.where(p.bt >= 0, inv[np.maximum(p.bt, 0)], -1).astype(np.int32)
        out2, _ = orc.paged_decode_attention(p.q, k2, v2, bt2, p.lengths, 0.3, lib=lib)
        assert np.array_equal(out1, out2), dtype


def pin_brute_force(lib):
    rng = np.random.default_rng(15)
    cases = [([1, 17, 33, 100], 2, 2, 64, 16, "f32"),
             ([3, 8, 9, 0, 25], 4, 1, 16, 8, "bf16"),
             ([31, 2, 64], 8, 2, 32, 16, "bf16"),
             ([7, 19], 6, 3, 8, 4, "f32"),
             ([5, 40, 16], 4, 2, 16, 16, "f16"),
             ([2, 33], 8, 8, 8, 32, "f16")]
    for lengths, H, H_kv, D, bs, dtype in cases:
        p = Paged(rng, lengths, H=H, H_kv=H_kv, D=D, bs=bs, dtype=dtype)
        scale = float(np.float32(1.0 / math.sqrt(D)))
        out, st = p.oracle(lib, scale)
        assert st == orc.ORC_OK
        ref = p.dense(scale)
        assert np.abs(out - ref).max() <= 1e-12, (lengths, H, H_kv, D, bs, dtype)


def pin_shared_prefix_rows(lib):
    rng = np.random.default_rng(16)
    p = Paged(rng, [24, 9], H=2, H_kv=1, D=8, bs=4)
    q = p.q.copy()
    q[1] = q[0]
    bt = p.bt.copy()
    bt[1] = bt[0]  # request 1 maps to request 0's blocks
    lens = np.array([24, 24], np.int32)
    out, st = orc.paged_decode_attention(q, p.k_cache, p.v_cache, bt, lens, 0.5, lib=lib)
    assert st == orc.ORC_OK
    assert np.array_equal(out[0], out[1])


def pin_gqa_equals_replicated_mha(lib):
    rng = np.random.default_rng(17)
    H, H_kv, D, bs = 8, 2, 16, 4
    p = Paged(rng, [13, 30], H=H, H_kv=H_kv, D=D, bs=bs)
    out_gqa, _ = p.oracle(lib, 0.25)
    g = H // H_kv
    k_rep = np.ascontiguousarray(np.repeat(p.k_cache, g, axis=2))
    v_rep = np.ascontiguousarray(np.repeat(p.v_cache, g, axis=2))
    out_mha, _ = orc.paged_decode_attention(p.q, k_rep, v_rep, p.bt, p.lengths, 0.25, lib=lib)
    assert np.abs(out_gqa - out_mha).max() <= 1e-13


def pin_split_merge_equals_whole(lib):
    rng = np.random.default_rng(18)
    p = Paged(rng, [50], H=2, H_kv=1, D=8, bs=4)
    whole, _ = p.oracle(lib, 0.4)
    for cuts in ([0, 50], [0, 16, 50], [0, 1, 2, 49, 50], [0, 20, 21, 36, 50]):
        for h in range(2):
            pieces = [orc.attention_partial(p.q, p.k_cache, p.v_cache, p.bt, 0, h, a, b, 0.4,
                                            lib=lib) for a, b in zip(cuts[:-1], cuts[1:])]
            m = [x[0] for x in pieces]
            l_ = [x[1] for x in pieces]
            o = np.stack([x[2] for x in pieces])
            merged = orc.lse_combine(m, l_, o, lib=lib)
            assert np.abs(merged - whole[0, h]).max() <= 1e-13, (cuts, h)


def pin_linear_in_v(lib):
    rng = np.random.default_rng(19)
    L, H_kv, D = 23, 1, 8
    K = rng.standard_normal((L, H_kv, D))
    # small integers, so V1 + V2 is exact in binary32 and linearity is exact up to fp64 rounding
    V1 = rng.integers(-8, 9, (L, H_kv, D)).astype(np.float64)
    V2 = rng.integers(-8, 9, (L, H_kv, D)).astype(np.float64)
    q = rng.standard_normal((1, 1, D))
    outs = []
    for V in (V1, V2, V1 + V2):
        p = Paged(np.random.default_rng(5), [L], H=1, H_kv=1, D=D, bs=4, q=q, hist=[(K, V)])
        outs.append(p.oracle(lib, 0.5)[0])
    assert np.abs(outs[0] + outs[1] - outs[2]).max() <= 1e-12


def pin_error_rows(lib):
    rng = np.random.default_rng(20)
    p = Paged(rng, [5, 9, 0], H=2, H_kv=1, D=4, bs=4)
    out, st = p.oracle(lib, 0.5)
    assert st == orc.ORC_OK
    assert np.all(out[2] == 0.0)  # empty history: zero row
    bt = p.bt.copy()
    bt[1, 1] = p.NB + 5  # block id out of range
    out, st = orc.paged_decode_attention(p.q, p.k_cache, p.v_cache, bt, p.lengths, 0.5, lib=lib)
    assert st == orc.ORC_ERR_DATA and np.all(np.isnan(out[1])) and np.all(np.isfinite(out[0]))
    lens = p.lengths.copy()
    lens[0] = p.max_blocks * p.bs + 1  # longer than the table can hold
    out, st = orc.paged_decode_attention(p.q, p.k_cache, p.v_cache, p.bt, lens, 0.5, lib=lib)
    assert st == orc.ORC_ERR_DATA and np.all(np.isnan(out[0])) and np.all(np.isfinite(out[1]))


def pin_append_then_pack_roundtrip(lib):
    rng = np.random.default_rng(21)
    for dtype in ("f32", "bf16", "f16"):
        H_kv, D, bs = 2, 8, 4
        hist_len = [4, 6, 11]
        p = Paged(rng, [L + 1 for L in hist_len], H=2, H_kv=H_kv, D=D, bs=bs, dtype=dtype)
        # the last position of each request is a fresh slot: overwrite it with garbage first
        new_k = as_stored(rng.standard_normal((3, H_kv, D)), dtype)
        new_v = as_stored(rng.standard_normal((3, H_kv, D)), dtype)
        slots = np.zeros(3, np.int32)
        for b, L in enumerate(hist_len):
            blk, row = p.bt[b, L // bs], L % bs
            slots[b] = blk * bs + row
            p.k_cache[blk, row] = as_stored(np.full((H_kv, D), 99.0), dtype)
            p.v_cache[blk, row] = as_stored(np.full((H_kv, D), -99.0), dtype)
        slots_pad = np.concatenate([slots, [-1]]).astype(np.int32)  # -1 is padding
        nk = np.concatenate([new_k, new_k[:1]])
        nv = np.concatenate([new_v, new_v[:1]])
        st = orc.kv_append(nk, nv, p.k_cache, p.v_cache, slots_pad, lib=lib)
        assert st == orc.ORC_OK
        for b, L in enumerate(hist_len):
            packed, st = orc.kv_pack_blocks(p.k_cache, p.v_cache, p.bt[b], L + 1, lib=lib)
            assert st == orc.ORC_OK
            want = np.stack([np.concatenate([p.K[b][:L], new_k[b:b + 1]]),
                             np.concatenate([p.V[b][:L], new_v[b:b + 1]])], axis=1)
            assert packed.dtype == want.dtype
            assert np.array_equal(packed.view(np.uint8), want.view(np.uint8)), (dtype, b)


def pin_unpack_then_pack_roundtrip(lib):
    rng = np.random.default_rng(22)
    for dtype in ("f32", "bf16", "f16"):
        H_kv, D, bs = 2, 8, 4
        for L in (1, 4, 9, 13):
            NB = (L + bs - 1) // bs + 5
            table = rng.permutation(NB)[:(L + bs - 1) // bs].astype(np.int32)
            packed = as_stored(rng.standard_normal((L, 2, H_kv, D)), dtype)
            kc = as_stored(rng.standard_normal((NB, bs, H_kv, D)), dtype)
            vc = as_stored(rng.standard_normal((NB, bs, H_kv, D)), dtype)
            kc0, vc0 = kc.copy(), vc.copy()
            assert orc.kv_unpack_blocks(packed, kc, vc, table, L, lib=lib) == orc.ORC_OK
            back, st = orc.kv_pack_blocks(kc, vc, table, L, lib=lib)
            assert st == orc.ORC_OK
            assert np.array_equal(back.view(np.uint8), packed.view(np.uint8)), (dtype, L)
            # rows that hold none of the request's tokens are untouched
            touched = np.zeros((NB, bs), bool)
            for t in range(L):
                touched[table[t // bs], t % bs] = True
            assert np.array_equal(kc[~touched].view(np.uint8), kc0[~touched].view(np.uint8))
            assert np.array_equal(vc[~touched].view(np.uint8), vc0[~touched].view(np.uint8))
            # and the rows it wrote are the buffer's, K and V in their places
            t = L - 1
            assert np.array_equal(kc[table[t // bs], t % bs].view(np.uint8),
                                  packed[t, 0].view(np.uint8))
            assert np.array_equal(vc[table[t // bs], t % bs].view(np.uint8),
                                  packed[t, 1].view(np.uint8))


def pin_e4m3_decode(lib):
    import torch

    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.decode_e4m3(c, lib=lib) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    # landmarks of the format, derived by hand
    hand = {0x00: 0.0, 0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x08: 2.0 ** -6,
            0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0xB8: -1.0, 0xFE: -448.0}
    for c, v in hand.items():
        assert orc.decode_e4m3(c, lib=lib) == v, hex(c)
    assert np.isnan(orc.decode_e4m3(0x7F, lib=lib)) and np.isnan(orc.decode_e4m3(0xFF, lib=lib))
    assert np.signbit(orc.decode_e4m3(0x80, lib=lib))


def _fp8_codes(rng, shape):
    """Random E4M3 codes, NaN codes excluded."""
    c = rng.integers(0, 254, size=shape).astype(np.uint8)
    c[c == 0x7F] = 0x7E
    return c


def pin_fp8_attention_brute_force(lib):
    import torch

    rng = np.random.default_rng(23)
    for lengths, H, H_kv, D, bs in (([1, 9, 33, 70], 4, 2, 16, 8), ([5, 40], 8, 1, 32, 16)):
        B = len(lengths)
        k_scale, v_scale = float(np.float32(0.0123)), float(np.float32(0.031))
        nblk = [(L + bs - 1) // bs for L in lengths]
        NB = sum(nblk) + 2
        kc = _fp8_codes(rng, (NB, bs, H_kv, D))
        vc = _fp8_codes(rng, (NB, bs, H_kv, D))
        perm = rng.permutation(NB).astype(np.int32)
        bt = np.full((B, max(nblk)), -1, np.int32)
        off = 0
        for b, n in enumerate(nblk):
            bt[b, :n] = perm[off:off + n]
            off += n
        q = as_stored(rng.standard_normal((B, H, D)), "bf16")
        scale = float(np.float32(1.0 / math.sqrt(D)))
        out, st = orc.paged_decode_attention(q, kc, vc, bt, np.array(lengths, np.int32), scale,
                                             lib=lib, k_scale=k_scale, v_scale=v_scale)
        assert st == orc.ORC_OK
        dec = lambda a: torch.from_numpy(a).view(torch.float8_e4m3fn).to(torch.float64).numpy()
        for b, L in enumerate(lengths):
            rows = [(bt[b, t // bs], t % bs) for t in range(L)]
            K = np.stack([dec(kc[r]) for r in rows]) * k_scale
            V = np.stack([dec(vc[r]) for r in rows]) * v_scale
            ref = brute.dense_decode_attention(stored_to_f64(q[b]), K, V, scale)
            assert np.abs(out[b] - ref).max() <= 1e-12, (lengths, b)


# FP4 E2M1 magnitudes by 3-bit code (sign is the 4th bit), as the format lists them
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def pin_f16_decode(lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([orc.decode_f16(int(b), lib=lib) for b in range(1 << 16)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    # landmarks of the format, derived by hand
    hand = {0x0000: 0.0, 0x3C00: 1.0, 0x3E00: 1.5, 0x4000: 2.0, 0x7BFF: 65504.0,
            0x0400: 2.0 ** -14, 0x0001: 2.0 ** -24, 0x03FF: 1023 * 2.0 ** -24, 0xC000: -2.0,
            0x7C00: math.inf, 0xFC00: -math.inf, 0x3555: 1365 * 2.0 ** -12}
    for b, v in hand.items():
        assert orc.decode_f16(b, lib=lib) == v, hex(b)
    assert np.isnan(orc.decode_f16(0x7E00, lib=lib)) and np.isnan(orc.decode_f16(0xFC01, lib=lib))


def pin_e2m1_decode(lib):
    for c in range(16):
        want = (-1.0 if c & 8 else 1.0) * E2M1_TABLE[c & 7]
        got = orc.decode_e2m1(c, lib=lib)
        assert got == want and np.signbit(got) == bool(c & 8), (c, got, want)


def pin_nvfp4_attention_brute_force(lib):
    import torch

    rng = np.random.default_rng(24)
    table = np.array(E2M1_TABLE)
    for lengths, H, H_kv, D, bs in (([1, 9, 33, 70], 4, 2, 32, 8), ([5, 40], 8, 1, 64, 16)):
        B = len(lengths)
        k_scale, v_scale = float(np.float32(0.9)), float(np.float32(1.3))
        nblk = [(L + bs - 1) // bs for L in lengths]
        NB = sum(nblk) + 2
        kd = rng.integers(0, 256, (NB, bs, H_kv, D // 2)).astype(np.uint8)
        vd = rng.integers(0, 256, (NB, bs, H_kv, D // 2)).astype(np.uint8)
        # block scales: E4M3 codes of 0.25 .. 0.47 (exponent field 5), per block and kv-head
        ks = rng.integers(0x28, 0x30, (NB, H_kv, bs, D // 16)).astype(np.uint8)
        vs = rng.integers(0x28, 0x30, (NB, H_kv, bs, D // 16)).astype(np.uint8)
        perm = rng.permutation(NB).astype(np.int32)
        bt = np.full((B, max(nblk)), -1, np.int32)
        off = 0
        for b, n in enumerate(nblk):
            bt[b, :n] = perm[off:off + n]
            off += n
        q = as_stored(rng.standard_normal((B, H, D)), "bf16")
        scale = float(np.float32(1.0 / math.sqrt(D)))
        out, st = orc.paged_decode_attention_nvfp4(q, kd, vd, ks, vs, bt,
                                                   np.array(lengths, np.int32), scale, k_scale,
                                                   v_scale, lib=lib)
        assert st == orc.ORC_OK

        def dequant(data, sc, tensor_scale):
            lo, hi = data & 15, data >> 4
            codes = np.stack([lo, hi], axis=-1).reshape(*data.shape[:-1], D)  # even: low
            vals = np.where(codes & 8, -1.0, 1.0) * table[codes & 7]
            s = torch.from_numpy(sc).view(torch.float8_e4m3fn).to(torch.float64).numpy()
            return vals * np.repeat(s, 16, axis=-1) * tensor_scale

        for b, L in enumerate(lengths):
            rows = [(bt[b, t // bs], t % bs) for t in range(L)]
            K = np.stack([dequant(kd[r], ks[r[0], :, r[1]], k_scale) for r in rows])
            V = np.stack([dequant(vd[r], vs[r[0], :, r[1]], v_scale) for r in rows])
            ref = brute.dense_decode_attention(stored_to_f64(q[b]), K, V, scale)
            assert np.abs(out[b] - ref).max() <= 1e-12, (lengths, b)


def pin_block_scale_copies(lib):
    """NVFP4 block-scale caches [NB, H_kv, bs, R]: append puts request b's row of kv-head h at
    [slot // bs, h, slot % bs]; pack reads [block, h, row] into the token-major buffer
    [t, 0|1, h]; unpack writes it back. Checked against numpy indexing of that layout."""
    rng = np.random.default_rng(31)
    NB, H_kv, bs, R = 7, 3, 4, 8
    ks = rng.integers(0, 256, (NB, H_kv, bs, R)).astype(np.uint8)
    vs = rng.integers(0, 256, (NB, H_kv, bs, R)).astype(np.uint8)
    k0, v0 = ks.copy(), vs.copy()
    slots = np.array([5, -1, 26, 13], np.int32)  # (1, 1), padding, (6, 2), (3, 1)
    kn = rng.integers(0, 256, (4, H_kv, R)).astype(np.uint8)
    vn = rng.integers(0, 256, (4, H_kv, R)).astype(np.uint8)
    assert orc.kv_append_block_scales(kn, vn, ks, vs, slots, lib=lib) == orc.ORC_OK
    want_k, want_v = k0.copy(), v0.copy()
    for b, sl in enumerate(slots):
        if sl >= 0:
            want_k[sl // bs, :, sl % bs] = kn[b]
            want_v[sl // bs, :, sl % bs] = vn[b]
    assert np.array_equal(ks, want_k) and np.array_equal(vs, want_v)
    table = np.array([6, 1, 3], np.int32)
    L = 10
    packed, st = orc.kv_pack_block_scales(ks, vs, table, L, lib=lib)
    assert st == orc.ORC_OK and packed.shape == (L, 2, H_kv, R)
    for t in range(L):
        blk, off = table[t // bs], t % bs
        assert np.array_equal(packed[t, 0], ks[blk, :, off])
        assert np.array_equal(packed[t, 1], vs[blk, :, off])
    k2, v2 = np.zeros_like(ks), np.zeros_like(vs)
    assert orc.kv_unpack_block_scales(packed, k2, v2, table, L, lib=lib) == orc.ORC_OK
    for t in range(L):
        blk, off = table[t // bs], t % bs
        assert np.array_equal(k2[blk, :, off], ks[blk, :, off])
    touched = np.zeros((NB, bs), bool)
    for t in range(L):
        touched[table[t // bs], t % bs] = True
    assert not k2.transpose(0, 2, 1, 3)[~touched].any()  # nothing else written
    bad = np.array([6, NB + 2, 3], np.int32)
    assert orc.kv_pack_block_scales(ks, vs, bad, L, lib=lib)[1] == orc.ORC_ERR_DATA


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
