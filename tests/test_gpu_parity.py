"""CUDA path against the fp64 oracle, through the C ABI, on seeded inputs.

append and pack are compared bit for bit; attention within max-abs 4e-3 and floored
max-rel 1e-2 (bf16 output) or 1e-4 abs (fp32 output). Small cases compare every output;
the full-size workloads, in the launch configuration the benchmark times, compare sampled
requests (longest, shortest and random ones) that the oracle computes one by one.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import paged_decode_attention_02_gb300 as pda
from gpu_common import (assert_attention_close, fp32_twin, gpu_step, oracle_full_step,
                        oracle_sampled, to_np)
from oracle import oracle as orc
from paged_decode_attention_02_gb300 import binding
from paged_decode_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def variant(base: str, **kw) -> wl.Workload:
    return dataclasses.replace(wl.get(base), **kw)


# ------------------------------------------------------------------ whole workloads
def test_tiny_full_step():
    s = wl.make_step("tiny", device=DEV)
    ref, st, kc, vc = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert np.array_equal(to_np(s.k_cache), kc) and np.array_equal(to_np(s.v_cache), vc)
    assert_attention_close(out, ref, "tiny", strict=True)
    # ctx = 1 returns the appended V exactly (fp32 all the way)
    b1 = int(np.where(s.context_lens_np == 1)[0][0])
    for h in range(s.w.H):
        assert torch.equal(out[b1, h], s.v_new[b1, h // s.w.group])


def test_llama2_7b_b8_every_output():
    s = wl.make_step("llama2_7b_b8", device=DEV)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, "llama2_7b_b8", strict=True)


@pytest.mark.parametrize("name,B", [("llama2_13b_b80", 12), ("gqa_skew_b256", 24),
                                    ("sm_sweep_b128", 16)])
def test_reduced_batch_every_output(name, B):
    s = wl.make_step(name, device=DEV, B=B)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, name, strict=True)


def _sample(s, k=10, seed=0):
    L = s.context_lens_np
    rng = np.random.default_rng(seed)
    picks = {int(np.argmax(L)), int(np.argmin(L))}
    picks |= {int(x) for x in rng.choice(len(L), size=min(k, len(L)), replace=False)}
    return sorted(picks)


@pytest.mark.parametrize("name", ["llama2_13b_b80", "gqa_skew_b256", "sm_sweep_b128"])
def test_full_size_sampled(name):
    s = wl.make_step(name, device=DEV)
    reqs = _sample(s)
    ref, st = oracle_sampled(s, reqs)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out[reqs], ref, name, strict=True)
    assert torch.isfinite(out.float()).all()


def test_full_size_pool_launches_are_bitwise_identical():
    """At full size the headline workload leaves a tenth of each warp's range to chunks that
    warps claim at run time (two per warp here: tiles x 10 % / (100 warps-per-tile-share x 4)
    >= 2). Which warp runs which chunk changes from launch to launch; the pieces merge in
    unit order, so repeated launches must agree bit for bit."""
    s = wl.make_step("gqa_skew_b256", device=DEV)
    tiles = int(((s.context_lens_np.astype(np.int64) + 15) // 16).sum()) * s.w.H_kv
    warps = pda.device_sm_count() * 12
    assert tiles * 10 // (100 * warps * 4) >= 2
    a, err_a = gpu_step(s, append=False)
    b, err_b = gpu_step(s, append=False)
    assert err_a == 0 and err_b == 0
    assert torch.equal(a, b)


_FULL = {}


def _full_step(name):
    """A full-size step of workload ``name`` with the oracle of its sampled requests, shared
    by the capped tests below (one pool on the device at a time). Each GPU step repeats the
    append, which rewrites the same slots with the same values, so the caches stay as the
    oracle saw them."""
    if name not in _FULL:
        _FULL.clear()
        s = wl.make_step(name, device=DEV)
        reqs = _sample(s)
        ref, st = oracle_sampled(s, reqs)
        assert st == 0
        _FULL[name] = (s, reqs, ref)
    return _FULL[name]


def _cap(pct):
    """The SM cap of the benchmark's sweep: ceil(pct % of the SMs)."""
    return int(math.ceil(pct / 100 * pda.device_sm_count()))


@pytest.mark.parametrize("pct", [10, 20, 40, 60])
def test_sm_sweep_full_size_capped_sampled(pct):
    """The SM-fraction sweep at its full 128 requests in the launches the benchmark times:
    4096 (request, kv-head) segments cut over a few hundred workers and merged."""
    s, reqs, ref = _full_step("sm_sweep_b128")
    cap = _cap(pct)
    out, err = gpu_step(s, sm_cap=cap)
    assert err == 0
    assert_attention_close(out[reqs], ref, f"sm_sweep_b128 sm_cap={cap}", strict=True)
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name", ["gqa_skew_b256_fp8", "gqa_skew_b256_nvfp4"])
def test_quantised_full_size_capped_sampled(name):
    """The quantised GQA workloads at full size on 10 % of the SMs (two-kv-head tiles, every
    long segment cut over many workers)."""
    s, reqs, ref = _full_step(name)
    cap = _cap(10)
    out, err = gpu_step(s, sm_cap=cap)
    assert err == 0
    assert_attention_close(out[reqs], ref, f"{name} sm_cap={cap}", strict=True)
    assert torch.isfinite(out.float()).all()


def test_full_size_pack_of_longest_requests():
    _FULL.clear()
    s = wl.make_step("gqa_skew_b256", device=DEV)
    reqs = s.pack_requests
    assert len(reqs) == 8
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_append(s.k_new, s.v_new, s.k_cache, s.v_cache, s.slot_mapping, error_word=err)
    outs = [torch.empty((int(s.context_lens_np[r]), 2, s.w.H_kv, s.w.D), dtype=s.k_cache.dtype,
                        device=DEV) for r in reqs]
    pda.kv_pack_blocks_batched(outs, s.k_cache, s.v_cache, [s.block_tables[r] for r in reqs],
                               [int(s.context_lens_np[r]) for r in reqs], error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # expected: the oracle's pack over host copies of each request's blocks
    bs = s.w.block_size
    for r, o in zip(reqs, outs):
        L = int(s.context_lens_np[r])
        n = (L + bs - 1) // bs
        blocks = torch.from_numpy(s.block_tables_np[r, :n].astype(np.int64)).to(DEV)
        kc = to_np(s.k_cache.index_select(0, blocks)).copy()
        vc = to_np(s.v_cache.index_select(0, blocks)).copy()
        want, st = orc.kv_pack_blocks(kc, vc, np.arange(n, dtype=np.int32), L)
        assert st == 0
        assert np.array_equal(to_np(o).view(np.uint8), want.view(np.uint8)), r


# ------------------------------------------------------------------ shapes and dtypes
SHAPES = [  # (dtype, D, H, H_kv)
    ("bf16", 128, 32, 32), ("bf16", 128, 32, 16), ("bf16", 128, 32, 8), ("bf16", 128, 32, 4),
    ("bf16", 128, 12, 3), ("bf16", 128, 7, 7), ("bf16", 128, 16, 2),
    ("bf16", 64, 16, 16), ("bf16", 64, 16, 8), ("bf16", 64, 16, 4), ("bf16", 64, 16, 2),
    ("f32", 64, 8, 8), ("f32", 64, 8, 2), ("f32", 128, 8, 8), ("f32", 128, 16, 2),
    ("f16", 128, 32, 8), ("f16", 128, 40, 40), ("f16", 128, 12, 3), ("f16", 64, 16, 4),
    ("f16", 64, 8, 8),
    # one kv-head for all query heads (multi-query attention)
    ("bf16", 128, 8, 1), ("bf16", 128, 1, 1), ("f16", 64, 4, 1),
]


@pytest.mark.parametrize("dtype,D,H,H_kv", SHAPES)
def test_shapes_and_groups(dtype, D, H, H_kv):
    w = variant("llama2_13b_b80", dtype=dtype, D=D, H=H, H_kv=H_kv, B=9,
                lengths="uniform:1,700")
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 700, 255], np.int32)
    s = wl.make_step(w, device=DEV, lengths=lens)
    ref, st, kc, vc = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert np.array_equal(to_np(s.k_cache), kc)
    assert_attention_close(out, ref, f"{dtype} D={D} H={H} H_kv={H_kv}", twin=fp32_twin(s))


def test_bf16_inputs_fp32_output():
    s = wl.make_step("llama2_13b_b80", device=DEV, B=6)
    ref, _, _, _ = oracle_full_step(s)
    out, err = gpu_step(s, out_dtype=torch.float32)
    assert err == 0
    assert_attention_close(out, ref, "bf16 in, f32 out")


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.float32])
def test_fp16_step_every_output(out_dtype):
    """fp16 q and caches (the precision the pages' decode kernels ran in), fp16 or fp32
    output, GQA and MHA, with the longest requests split over several workers."""
    for base in ("gqa_skew_b256", "llama2_13b_b80"):
        s = wl.make_step(variant(base, dtype="f16", B=16), device=DEV)
        ref, st, kc, vc = oracle_full_step(s)
        assert st == 0
        out, err = gpu_step(s, out_dtype=out_dtype)
        assert err == 0
        assert np.array_equal(to_np(s.k_cache).view(np.uint8), kc.view(np.uint8))
        assert_attention_close(out, ref, f"{base} fp16 -> {out_dtype}", strict=True)


# ------------------------------------------------------------------ edge cases
def test_empty_and_single_token_histories():
    lens = np.array([0, 1, 0, 2, 1, 16, 0], np.int32)
    s = wl.make_step("llama2_13b_b80", device=DEV, lengths=lens, B=7)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, "empty/single", twin=fp32_twin(s))
    assert (out[lens == 0] == 0).all()
    for b in np.where(lens == 1)[0]:
        assert torch.equal(out[b], s.v_new[b].to(out.dtype))  # exact: p = 1


def test_all_empty_batch():
    s = wl.make_step("llama2_13b_b80", device=DEV, lengths=np.zeros(5, np.int32), B=5)
    out, err = gpu_step(s, append=False)
    assert err == 0 and (out == 0).all()


def test_single_very_long_request_split_over_every_worker():
    w = variant("gqa_skew_b256", B=1)
    s = wl.make_step(w, device=DEV, lengths=np.array([32768], np.int32))
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, "B=1 L=32768", twin=fp32_twin(s))


def _attention_direct(s, out, block_tables, max_context_len):
    """The step's attention through the C ABI with a given table and length bound."""
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if s.w.kv == "nvfp4":
        pda.paged_decode_attention_nvfp4(out, s.q, s.k_cache, s.v_cache, s.k_bscales,
                                         s.v_bscales, block_tables, s.context_lens,
                                         max_context_len, s.scale, s.k_scale, s.v_scale,
                                         error_word=err)
    elif s.w.kv == "fp8":
        pda.paged_decode_attention_fp8(out, s.q, s.k_cache, s.v_cache, block_tables,
                                       s.context_lens, max_context_len, s.scale, s.k_scale,
                                       s.v_scale, error_word=err)
    else:
        pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, block_tables,
                                   s.context_lens, max_context_len, s.scale, error_word=err)
    torch.cuda.synchronize()
    return int(err.item())


@pytest.mark.parametrize("name", ["gqa_skew_b256", "llama2_13b_b80", "gqa_skew_b256_fp8",
                                  "gqa_skew_b256_nvfp4"])
def test_lengths_far_below_the_declared_max(name):
    """A table 2048 blocks wide and max_context_len 32768 let the host size the grid for the
    whole chip, while the lengths hold a few tiles: the kernel keeps the few warps it needs
    (8 tiles each at most), the others leave after the prologue, and the merges run over
    the units that work."""
    lens = np.array([16, 3, 40, 1, 17], np.int32)
    s = wl.make_step(variant(name, B=len(lens)), device=DEV, lengths=lens)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0
    wide = torch.full((s.B, 2048), -1, dtype=torch.int32, device=DEV)
    wide[:, :s.max_blocks] = s.block_tables
    out = torch.empty_like(s.q)
    out32 = torch.empty(s.q.shape, dtype=torch.float32, device=DEV)
    assert _attention_direct(s, out, wide, 32768) == 0
    assert _attention_direct(s, out32, wide, 32768) == 0
    assert_attention_close(out, ref, f"{name} short lengths, max 32768", twin=out32)


def test_many_one_block_requests():
    lens = np.random.default_rng(3).integers(1, 17, size=600).astype(np.int32)
    w = variant("gqa_skew_b256", B=600)
    s = wl.make_step(w, device=DEV, lengths=lens)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, "600 one-block requests", twin=fp32_twin(s))


@pytest.mark.parametrize("name", ["gqa_skew_b256", "gqa_skew_b256_fp8", "gqa_skew_b256_nvfp4"])
def test_largest_batch_every_output(name):
    """The largest batch a call takes (8192 requests of 1 to 48 tokens). Its prefix table
    fills 32 KB of shared memory, so blocks run fewer warps than usual; 65,536 short
    (request, kv-head) segments, many cut by unit boundaries. Every output against the
    oracle."""
    lens = np.random.default_rng(11).integers(1, 49, size=8192).astype(np.int32)
    s = wl.make_step(variant(name, B=8192), device=DEV, lengths=lens)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, f"{name} B=8192", twin=fp32_twin(s))


def test_unused_rows_poisoned_with_nan_are_never_read():
    lens = np.array([5, 16, 17, 40, 1, 100], np.int32)
    s = wl.make_step("llama2_13b_b80", device=DEV, lengths=lens, B=6, poison_unused=True)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0 and np.isfinite(ref).all()
    out, err = gpu_step(s, append=False)
    assert err == 0
    assert_attention_close(out, ref, "poisoned", twin=fp32_twin(s))


def test_shared_prefix_blocks_give_identical_rows():
    s = wl.make_step("llama2_13b_b80", device=DEV, B=4)
    s.block_tables[1] = s.block_tables[0]
    s.block_tables_np[1] = s.block_tables_np[0]
    s.context_lens[1] = s.context_lens[0]
    s.context_lens_np[1] = s.context_lens_np[0]
    s.q[1] = s.q[0]
    out, err = gpu_step(s, append=False)
    assert err == 0
    ref, _, _, _ = oracle_full_step(s, append=False)
    assert np.array_equal(ref[0], ref[1])
    # The two rows may be split at different worker boundaries, so they can differ in the
    # fp32 summation order; both must match the (identical) oracle rows.
    assert_attention_close(out, ref, "shared prefix", twin=fp32_twin(s))


@pytest.mark.parametrize("cap", [1, 2, 15, 30, 61, 91, 152, 1000])
def test_sm_cap_does_not_change_results(cap):
    s = wl.make_step("sm_sweep_b128", device=DEV, B=10)
    ref, _, _, _ = oracle_full_step(s)
    out, err = gpu_step(s, sm_cap=cap)
    assert err == 0
    assert_attention_close(out, ref, f"sm_cap={cap}", twin=fp32_twin(s, cap))


def test_repeat_runs_are_bitwise_identical():
    s = wl.make_step("gqa_skew_b256", device=DEV, B=32)
    a, _ = gpu_step(s, append=False)
    b, _ = gpu_step(s, append=False)
    assert torch.equal(a, b)


# ------------------------------------------------------------------ device-side errors
def test_bad_block_id_gives_nan_rows_and_error_bit():
    lens = np.array([40, 40, 40], np.int32)
    w = variant("gqa_skew_b256", B=3)
    s = wl.make_step(w, device=DEV, lengths=lens)
    s.block_tables[1, 1] = s.num_blocks + 7
    out, err = gpu_step(s, append=False)
    assert err & binding.PDA_DEVERR_BLOCK_ID
    assert torch.isnan(out[1].float()).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(out[2].float()).all()


def test_context_beyond_capacity_gives_nan_rows_and_error_bit():
    lens = np.array([20, 30], np.int32)
    s = wl.make_step("llama2_13b_b80", device=DEV, lengths=lens, B=2)
    s.context_lens[0] = s.max_blocks * 16 + 1
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty_like(s.q)
    pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables, s.context_lens,
                               10 ** 6, s.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.PDA_DEVERR_CONTEXT_LEN
    assert torch.isnan(out[0].float()).all() and torch.isfinite(out[1].float()).all()


def test_context_beyond_declared_max_is_an_error():
    s = wl.make_step("llama2_13b_b80", device=DEV, lengths=np.array([64, 64], np.int32), B=2)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = torch.empty_like(s.q)
    pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables, s.context_lens,
                               32, s.scale, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & binding.PDA_DEVERR_CONTEXT_LEN
    assert torch.isnan(out.float()).all()


def test_append_slot_out_of_range_and_padding():
    s = wl.make_step("tiny", device=DEV)
    before_k = s.k_cache.clone()
    s.slot_mapping[0] = -1                       # padding: skipped silently
    s.slot_mapping[1] = s.num_blocks * 16 + 3    # out of range: error bit, skipped
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_append(s.k_new, s.v_new, s.k_cache, s.v_cache, s.slot_mapping, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == binding.PDA_DEVERR_SLOT
    kc = to_np(before_k).copy()
    vc = to_np(s.v_cache).copy()  # only compared for K below
    sm = s.slot_mapping.cpu().numpy()
    sm_ok = np.where((sm >= 0) & (sm < s.num_blocks * 16), sm, -1).astype(np.int32)
    orc.kv_append(to_np(s.k_new), to_np(s.v_new), kc, vc, sm_ok)
    assert np.array_equal(to_np(s.k_cache), kc)


def test_pack_bad_block_sets_error_and_nan_pattern():
    s = wl.make_step("tiny", device=DEV)
    b = 3
    L = int(s.context_lens_np[b])
    s.block_tables[b, 2] = -5
    out = torch.zeros((L, 2, s.w.H_kv, s.w.D), dtype=s.k_cache.dtype, device=DEV)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_pack_blocks(out, s.k_cache, s.v_cache, s.block_tables[b], L, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == binding.PDA_DEVERR_BLOCK_ID
    bad = to_np(out[32:48]).view(np.uint8)
    assert (bad == 0xFF).all()
    kc, vc = to_np(s.k_cache), to_np(s.v_cache)
    want, _ = orc.kv_pack_blocks(kc, vc, s.block_tables_np[b], 32)
    assert np.array_equal(to_np(out[:32]).view(np.uint8), want.view(np.uint8))


def test_workspace_too_small_is_rejected():
    s = wl.make_step("tiny", device=DEV)
    ws = torch.empty(256, dtype=torch.uint8, device=DEV)
    out = torch.empty_like(s.q)
    with pytest.raises(binding.PdaError) as e:
        pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale, workspace=ws)
    assert e.value.status == binding.PDA_ERR_WORKSPACE


# ------------------------------------------------------------------ two concurrent launches
@pytest.mark.parametrize("ratio", [0.3, 0.5])
def test_local_and_remote_attention_on_two_streams(ratio):
    """The batch split into a 'remote' and a 'local' part, run as two attention launches on
    two streams at once with complementary SM caps (attention offload sharing one GPU)."""
    s = wl.make_step("sm_sweep_b128", device=DEV, B=24)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0
    sms = pda.device_sm_count()
    n_r = int(np.ceil(ratio * s.B))
    cap_r = max(1, int(round(ratio * sms)))
    cap_l = max(1, sms - cap_r)
    parts = [(slice(0, n_r), cap_r), (slice(n_r, s.B), cap_l)]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs, errs, keep = [], [], []
    main = torch.cuda.current_stream()
    for (sl, cap), stream in zip(parts, streams):
        q = s.q[sl].contiguous()
        bt = s.block_tables[sl].contiguous()
        cl = s.context_lens[sl].contiguous()
        out = torch.empty_like(q)
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        ws = pda.alloc_workspace(q.shape[0], s.w.H, s.w.H_kv, s.w.D, 16, q.dtype, cap, DEV)
        keep += [q, bt, cl, ws]
        stream.wait_stream(main)
        with torch.cuda.stream(stream):
            pda.paged_decode_attention(out, q, s.k_cache, s.v_cache, bt, cl,
                                       s.max_context_len, s.scale, sm_cap=cap, workspace=ws,
                                       error_word=err, stream=stream)
        outs.append(out)
        errs.append(err)
    for stream in streams:
        main.wait_stream(stream)
    torch.cuda.synchronize()
    assert all(int(e.item()) == 0 for e in errs)
    assert_attention_close(torch.cat(outs), ref, f"two streams, ratio {ratio}", strict=True)


# ------------------------------------------------------------------ KV unpack
@pytest.mark.parametrize("name,B", [("tiny", None), ("llama2_13b_b80", 6)])
def test_unpack_matches_oracle_bit_for_bit(name, B):
    s = wl.make_step(name, device=DEV, B=B)
    w = s.w
    gen = torch.Generator(device=DEV)
    gen.manual_seed(77)
    kc, vc = to_np(s.k_cache).copy(), to_np(s.v_cache).copy()
    bufs, rows, lens = [], [], []
    for b in range(s.B):
        L = int(s.context_lens_np[b])
        buf = torch.randn((L, 2, w.H_kv, w.D), generator=gen, device=DEV).to(w.torch_dtype)
        bufs.append(buf)
        rows.append(s.block_tables[b])
        lens.append(L)
        assert orc.kv_unpack_blocks(to_np(buf), kc, vc, s.block_tables_np[b], L) == 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_unpack_blocks(bufs[0], s.k_cache, s.v_cache, rows[0], lens[0], error_word=err)
    pda.kv_unpack_blocks_batched(bufs[1:], s.k_cache, s.v_cache, rows[1:], lens[1:],
                                 error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(to_np(s.k_cache), kc) and np.array_equal(to_np(s.v_cache), vc)


def test_full_size_unpack_then_pack_of_longest_requests():
    s = wl.make_step("gqa_skew_b256", device=DEV)
    w = s.w
    reqs = s.pack_requests
    gen = torch.Generator(device=DEV)
    gen.manual_seed(78)
    ins = [torch.randn((int(s.context_lens_np[r]), 2, w.H_kv, w.D), generator=gen,
                       device=DEV).to(w.torch_dtype) for r in reqs]
    rows = [s.block_tables[r] for r in reqs]
    lens = [int(s.context_lens_np[r]) for r in reqs]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_unpack_blocks_batched(ins, s.k_cache, s.v_cache, rows, lens, error_word=err)
    outs = [torch.empty_like(x) for x in ins]
    pda.kv_pack_blocks_batched(outs, s.k_cache, s.v_cache, rows, lens, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for a, b in zip(ins, outs):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_unpack_bad_block_is_skipped_with_error_bit():
    s = wl.make_step("tiny", device=DEV)
    b = 3
    L = int(s.context_lens_np[b])
    s.block_tables[b, 1] = s.num_blocks + 2
    buf = torch.full((L, 2, s.w.H_kv, s.w.D), 7.0, dtype=s.k_cache.dtype, device=DEV)
    before = s.k_cache.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_unpack_blocks(buf, s.k_cache, s.v_cache, s.block_tables[b], L, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == binding.PDA_DEVERR_BLOCK_ID
    kc = to_np(before).copy()
    vc = to_np(s.v_cache).copy()
    bt = s.block_tables[b].cpu().numpy()
    orc.kv_unpack_blocks(to_np(buf), kc, vc, bt, L)  # the oracle skips the same tokens
    assert np.array_equal(to_np(s.k_cache), kc)



# ------------------------------------------------------------------ FP8 E4M3 KV cache
# D = 128: kv-head pairs on the tensor cores for G <= 4 and even H_kv (32/32, 32/16, 32/8),
# one kv-head per tile on the tensor cores for G = 8 (32/4) or odd H_kv with G >= 2 (12/3,
# 6/3), CUDA cores for odd H_kv with G = 1 (5/5); D = 64: CUDA cores.
FP8_SHAPES = [(128, 32, 32), (128, 32, 16), (128, 32, 8), (128, 32, 4), (128, 12, 3),
              (128, 6, 3), (128, 5, 5), (64, 16, 16), (64, 16, 4),
              (128, 8, 1), (128, 2, 1), (128, 1, 1)]  # the last three: one kv-head


@pytest.mark.parametrize("D,H,H_kv", FP8_SHAPES)
def test_fp8_shapes_and_groups(D, H, H_kv):
    w = variant("llama2_13b_b80_fp8", D=D, H=H, H_kv=H_kv, B=9, lengths="uniform:1,700")
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 700, 255], np.int32)
    s = wl.make_step(w, device=DEV, lengths=lens)
    ref, st, kc, vc = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert np.array_equal(to_np(s.k_cache), kc) and np.array_equal(to_np(s.v_cache), vc)
    assert_attention_close(out, ref, f"fp8 D={D} H={H} H_kv={H_kv}", twin=fp32_twin(s))


@pytest.mark.parametrize("name,B", [("llama2_13b_b80_fp8", 10), ("gqa_skew_b256_fp8", 24)])
def test_fp8_reduced_batch_every_output(name, B):
    s = wl.make_step(name, device=DEV, B=B)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, name, strict=True)


def test_fp8_full_size_sampled_and_pack():
    s = wl.make_step("gqa_skew_b256_fp8", device=DEV)
    reqs = _sample(s)
    ref, st = oracle_sampled(s, reqs)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out[reqs], ref, "gqa_skew_b256_fp8", strict=True)
    r = s.pack_requests[0]
    L = int(s.context_lens_np[r])
    packed = torch.empty((L, 2, s.w.H_kv, s.w.D), dtype=torch.uint8, device=DEV)
    pda.kv_pack_blocks(packed, s.k_cache, s.v_cache, s.block_tables[r], L)
    n = (L + 15) // 16
    blocks = torch.from_numpy(s.block_tables_np[r, :n].astype(np.int64)).to(DEV)
    want, st = orc.kv_pack_blocks(to_np(s.k_cache.index_select(0, blocks)).copy(),
                                  to_np(s.v_cache.index_select(0, blocks)).copy(),
                                  np.arange(n, dtype=np.int32), L)
    assert st == 0 and np.array_equal(to_np(packed), want)


def test_fp8_empty_single_and_poisoned_rows():
    lens = np.array([0, 1, 2, 16, 17, 40], np.int32)
    s = wl.make_step("llama2_13b_b80_fp8", device=DEV, lengths=lens, B=6, poison_unused=True)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0 and np.isfinite(ref).all()
    out, err = gpu_step(s, append=False)
    assert err == 0
    assert_attention_close(out, ref, "fp8 edge cases", twin=fp32_twin(s))
    assert (out[0] == 0).all()


def test_fp8_entry_rejects_plain_caches_and_base_entry_rejects_fp8():
    s = wl.make_step("llama2_13b_b80_fp8", device=DEV, B=2)
    out = torch.empty_like(s.q)
    with pytest.raises(binding.PdaError) as e:
        pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale)
    assert e.value.status == binding.PDA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ NVFP4 KV cache
NVFP4_SHAPES = [(128, 32, 32), (128, 32, 8), (128, 32, 16), (128, 16, 2), (128, 64, 8),
                (128, 12, 3), (128, 5, 5), (64, 16, 4), (64, 16, 16),
                (128, 4, 1), (128, 1, 1)]  # the last two: one kv-head


@pytest.mark.parametrize("D,H,H_kv", NVFP4_SHAPES)
def test_nvfp4_shapes_and_groups(D, H, H_kv):
    w = variant("llama2_13b_b80_nvfp4", D=D, H=H, H_kv=H_kv, B=9, lengths="uniform:1,700")
    lens = np.array([1, 15, 16, 17, 31, 32, 33, 700, 255], np.int32)
    s = wl.make_step(w, device=DEV, lengths=lens)
    ksc, vsc = to_np(s.k_bscales).copy(), to_np(s.v_bscales).copy()
    assert orc.kv_append_block_scales(to_np(s.k_new_bscales), to_np(s.v_new_bscales), ksc, vsc,
                                      s.slot_mapping_np) == 0
    ref, st, kc, vc = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert np.array_equal(to_np(s.k_cache), kc) and np.array_equal(to_np(s.v_cache), vc)
    assert np.array_equal(to_np(s.k_bscales), ksc) and np.array_equal(to_np(s.v_bscales), vsc)
    assert_attention_close(out, ref, f"nvfp4 D={D} H={H} H_kv={H_kv}", twin=fp32_twin(s))


@pytest.mark.parametrize("name,B", [("llama2_13b_b80_nvfp4", 10), ("gqa_skew_b256_nvfp4", 24)])
def test_nvfp4_reduced_batch_every_output(name, B):
    s = wl.make_step(name, device=DEV, B=B)
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, name, strict=True)


def test_nvfp4_full_size_sampled():
    s = wl.make_step("gqa_skew_b256_nvfp4", device=DEV)
    reqs = _sample(s)
    ref, st = oracle_sampled(s, reqs)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out[reqs], ref, "gqa_skew_b256_nvfp4", strict=True)


def test_nvfp4_empty_single_and_poisoned_scales():
    lens = np.array([0, 1, 2, 16, 17, 40], np.int32)
    s = wl.make_step("llama2_13b_b80_nvfp4", device=DEV, lengths=lens, B=6, poison_unused=True)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0 and np.isfinite(ref).all()
    out, err = gpu_step(s, append=False)
    assert err == 0
    assert_attention_close(out, ref, "nvfp4 edge cases", twin=fp32_twin(s))
    assert (out[0] == 0).all()


def test_nvfp4_pack_of_data_and_scales_is_bit_exact():
    s = wl.make_step("gqa_skew_b256_nvfp4", device=DEV, B=8)
    reqs = [int(r) for r in np.argsort(-s.context_lens_np)[:4]]
    lens = [int(s.context_lens_np[r]) for r in reqs]
    rows = [s.block_tables[r] for r in reqs]
    kd, vd = to_np(s.k_cache).copy(), to_np(s.v_cache).copy()
    ksc, vsc = to_np(s.k_bscales).copy(), to_np(s.v_bscales).copy()
    data = [torch.empty((L, 2, s.w.H_kv, s.w.D // 2), dtype=torch.uint8, device=DEV)
            for L in lens]
    scales = [torch.empty((L, 2, s.w.H_kv, s.w.D // 16), dtype=torch.uint8, device=DEV)
              for L in lens]
    pda.kv_pack_blocks_batched(data, s.k_cache, s.v_cache, rows, lens)
    pda.kv_pack_block_scales_batched(scales, s.k_bscales, s.v_bscales, rows, lens)
    for i, r in enumerate(reqs):
        want, st = orc.kv_pack_blocks(kd, vd, s.block_tables_np[r], lens[i])
        assert st == 0 and np.array_equal(to_np(data[i]), want), r
        want, st = orc.kv_pack_block_scales(ksc, vsc, s.block_tables_np[r], lens[i])
        assert st == 0 and np.array_equal(to_np(scales[i]), want), r


def test_nvfp4_unpack_scales_inverts_pack_and_touches_nothing_else():
    s = wl.make_step("llama2_13b_b80_nvfp4", device=DEV, B=5)
    reqs = list(range(s.B))
    lens = [int(s.context_lens_np[r]) for r in reqs]
    rows = [s.block_tables[r] for r in reqs]
    packed = [torch.from_numpy(orc.kv_pack_block_scales(to_np(s.k_bscales), to_np(s.v_bscales),
                                                        s.block_tables_np[r], L)[0]).to(DEV)
              for r, L in zip(reqs, lens)]
    k2 = torch.full_like(s.k_bscales, 0x5A)
    v2 = torch.full_like(s.v_bscales, 0xA5)
    kw, vw = to_np(k2).copy(), to_np(v2).copy()
    for r, L, p in zip(reqs, lens, packed):
        assert orc.kv_unpack_block_scales(to_np(p), kw, vw, s.block_tables_np[r], L) == 0
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_unpack_block_scales_batched(packed, k2, v2, rows, lens, error_word=err)
    assert int(err.item()) == 0
    assert np.array_equal(to_np(k2), kw) and np.array_equal(to_np(v2), vw)


def test_nvfp4_scale_calls_edge_cases():
    """Padding and out-of-range slots in the scale append; a bad block id in the scale pack
    (0xFF for its tokens) and unpack (not written); empty requests; D not a multiple of 64."""
    s = wl.make_step("llama2_13b_b80_nvfp4", device=DEV, B=4)
    slots = s.slot_mapping.clone()
    slots[1] = -1
    slots[2] = s.num_blocks * s.w.block_size + 5
    ksc, vsc = to_np(s.k_bscales).copy(), to_np(s.v_bscales).copy()
    assert orc.kv_append_block_scales(to_np(s.k_new_bscales), to_np(s.v_new_bscales), ksc, vsc,
                                      to_np(slots)) != 0  # the oracle flags slot 2 too
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    pda.kv_append_block_scales(s.k_new_bscales, s.v_new_bscales, s.k_bscales, s.v_bscales,
                               slots, error_word=err)
    assert int(err.item()) == binding.PDA_DEVERR_SLOT
    assert np.array_equal(to_np(s.k_bscales), ksc) and np.array_equal(to_np(s.v_bscales), vsc)

    L = int(s.context_lens_np[0])
    row = s.block_tables[0].clone()
    row[0] = s.num_blocks + 7
    out = torch.zeros((L, 2, s.w.H_kv, s.w.D // 16), dtype=torch.uint8, device=DEV)
    err.zero_()
    pda.kv_pack_block_scales_batched([out], s.k_bscales, s.v_bscales, [row], [L], error_word=err)
    assert int(err.item()) == binding.PDA_DEVERR_BLOCK_ID
    n0 = min(L, s.w.block_size)
    assert (out[:n0] == 0xFF).all()
    want, st = orc.kv_pack_block_scales(ksc, vsc, s.block_tables_np[0], L)
    assert st == 0 and np.array_equal(to_np(out[n0:]), want[n0:])

    k2, v2 = torch.zeros_like(s.k_bscales), torch.zeros_like(s.v_bscales)
    err.zero_()
    pda.kv_unpack_block_scales_batched([out], k2, v2, [row], [L], error_word=err)
    assert int(err.item()) == binding.PDA_DEVERR_BLOCK_ID
    kw, vw = np.zeros_like(ksc), np.zeros_like(vsc)
    bad_row = s.block_tables_np[0].copy()
    bad_row[0] = s.num_blocks + 7
    assert orc.kv_unpack_block_scales(to_np(out), kw, vw, bad_row, L) != 0
    assert np.array_equal(to_np(k2), kw) and np.array_equal(to_np(v2), vw)

    pda.kv_pack_block_scales_batched([out], s.k_bscales, s.v_bscales, [row], [0])  # no-op
    pda.kv_pack_block_scales_batched([], s.k_bscales, s.v_bscales, [], [])
    odd = torch.zeros((s.num_blocks, s.w.H_kv, s.w.block_size, 2), dtype=torch.uint8,
                      device=DEV)  # D = 32
    with pytest.raises(binding.PdaError) as e:
        pda.kv_pack_block_scales_batched([out[:, :, :, :2].contiguous()], odd, odd,
                                         [s.block_tables[0]], [L])
    assert e.value.status == binding.PDA_ERR_UNSUPPORTED


# ------------------------------------------------------------------ tensor-core tile step
# FP8 and NVFP4 caches at D = 128 with G >= 2 run their dot products on the tensor cores
# with fp16 operands: q is brought into fp16 range by a power-of-two shift, and a head's
# running maximum may lag the true one by up to 2^8 before the output is rescaled. The
# G = 1 workloads below take the CUDA-core path and check the same edge cases there.
QUANTISED = ["gqa_skew_b256_fp8", "llama2_13b_b80_fp8", "gqa_skew_b256_nvfp4",
             "llama2_13b_b80_nvfp4"]


@pytest.mark.parametrize("name", QUANTISED)
def test_tc_q_far_outside_fp16_range(name):
    """q times 2^20 (|q| up to ~4e6, far above fp16's 65504) with the scale times 2^-20 is
    the same attention; both sides get the scaled inputs."""
    s = wl.make_step(name, device=DEV, B=6)
    s.q.mul_(2.0 ** 20)
    s.scale = float(np.float32(s.scale) * np.float32(2.0 ** -20))
    assert s.q.abs().max().item() > 65504
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, f"{name} q x 2^20", twin=fp32_twin(s))


@pytest.mark.parametrize("name", QUANTISED)
@pytest.mark.parametrize("boost", [8.0, 40.0])
def test_tc_sharp_softmax_rescales(name, boost):
    """A scale `boost` times larger spreads the scores over tens of log2 units, so later
    tiles often raise a head's maximum by more than the allowed lag (output rescaled) and
    others stay within it (probabilities above 1 accumulate unrescaled)."""
    s = wl.make_step(name, device=DEV, B=8)
    s.scale = float(np.float32(s.scale) * np.float32(boost))
    ref, st, _, _ = oracle_full_step(s)
    assert st == 0
    out, err = gpu_step(s)
    assert err == 0
    assert_attention_close(out, ref, f"{name} scale x {boost}", twin=fp32_twin(s))


@pytest.mark.parametrize("kv", ["fp8", "nvfp4", "bf16"])
@pytest.mark.parametrize("H,H_kv", [(64, 8), (16, 8), (8, 8), (12, 3), (7, 7)])
def test_tc_groups_with_ragged_tails(kv, H, H_kv):
    """Group sizes 8 and 2 (tensor cores for quantised caches) and 1, lengths that end at
    every offset of a block (partial tiles mask tokens 1..15 of the last block; the unused
    rows hold NaN, or NaN block scales, so an unmasked one would show). bf16 runs the same
    cases on the CUDA cores."""
    base = {"fp8": "gqa_skew_b256_fp8", "nvfp4": "gqa_skew_b256_nvfp4",
            "bf16": "gqa_skew_b256"}[kv]
    lens = np.array(list(range(1, 17)) + [47, 64, 65, 333], np.int32)
    w = variant(base, H=H, H_kv=H_kv, B=len(lens), lengths="uniform:1,400")
    s = wl.make_step(w, device=DEV, lengths=lens, poison_unused=True)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0 and np.isfinite(ref).all()
    out, err = gpu_step(s, append=False)
    assert err == 0
    assert_attention_close(out, ref, f"{kv} H={H} H_kv={H_kv} ragged", twin=fp32_twin(s))


# ------------------------------------------------------------------ quantised edge cases
# The two-kv-head tiles (every quantised workload) go through the same scheduling, merge
# and error paths as the bf16 kernel with units of two kv-heads and 2G query heads.
@pytest.mark.parametrize("name", ["gqa_skew_b256_fp8", "gqa_skew_b256_nvfp4",
                                  "llama2_13b_b80_nvfp4"])
@pytest.mark.parametrize("cap", [1, 7, 61, 152])
def test_quantised_sm_cap_does_not_change_results(name, cap):
    s = wl.make_step(name, device=DEV, B=10)
    ref, _, _, _ = oracle_full_step(s, append=False)
    out, err = gpu_step(s, append=False, sm_cap=cap)
    assert err == 0
    assert_attention_close(out, ref, f"{name} sm_cap={cap}", twin=fp32_twin(s, cap))


@pytest.mark.parametrize("name", ["gqa_skew_b256_fp8", "llama2_13b_b80_nvfp4"])
def test_quantised_repeat_runs_are_bitwise_identical(name):
    s = wl.make_step(name, device=DEV, B=24)
    a, _ = gpu_step(s, append=False)
    b, _ = gpu_step(s, append=False)
    assert torch.equal(a, b)


@pytest.mark.parametrize("name", ["gqa_skew_b256_fp8", "gqa_skew_b256_nvfp4"])
def test_quantised_bad_block_id_gives_nan_rows_and_error_bit(name):
    lens = np.array([40, 40, 40], np.int32)
    s = wl.make_step(variant(name, B=3), device=DEV, lengths=lens)
    s.block_tables[1, 1] = s.num_blocks + 7
    out, err = gpu_step(s, append=False)
    assert err & binding.PDA_DEVERR_BLOCK_ID
    assert torch.isnan(out[1].float()).all()
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(out[2].float()).all()


@pytest.mark.parametrize("name", ["gqa_skew_b256_fp8", "llama2_13b_b80_nvfp4"])
def test_quantised_single_very_long_request_split_over_every_worker(name):
    """One 20000-token request: every kv-head pair's segment is cut over many workers and
    merged (2G heads per unit)."""
    lens = np.array([20000], np.int32)
    s = wl.make_step(variant(name, B=1, lengths="uniform:1,20000"), device=DEV, lengths=lens)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0
    out, err = gpu_step(s, append=False)
    assert err == 0
    assert_attention_close(out, ref, f"{name} one long request", twin=fp32_twin(s))


# ------------------------------------------------------------------ physical block sizes
# Blocks of 32, 64, 128 or 256 tokens: the attention works in 16-row tiles of one block, a
# block holding block_size / 16 of them; append and pack move whole rows whatever the size.
BLOCK_SIZE_CASES = [("gqa_skew_b256", {}), ("llama2_13b_b80", {}),
                    ("llama2_13b_b80", {"D": 64, "H": 16, "H_kv": 4}),
                    ("tiny", {}), ("gqa_skew_b256", {"dtype": "f16"}),
                    ("gqa_skew_b256_fp8", {}), ("gqa_skew_b256_nvfp4", {}),
                    ("llama2_13b_b80_nvfp4", {}), ("gqa_skew_b256_nvfp4", {"H": 12, "H_kv": 3})]


@pytest.mark.parametrize("bs", [32, 64, 128, 256])
@pytest.mark.parametrize("name,kw", BLOCK_SIZE_CASES)
def test_block_sizes_full_step(name, kw, bs):
    """Append then attention with lengths ending at every kind of offset: inside the first
    tile of a block, at tile and block boundaries, one past them; unused rows poisoned."""
    lens = np.array([1, 15, 16, 17, 31, 32, 33, bs - 1, bs, bs + 1, 3 * bs + 5, 700], np.int32)
    w = variant(name, block_size=bs, B=len(lens), lengths="uniform:1,700", **kw)
    s = wl.make_step(w, device=DEV, lengths=lens, poison_unused=True)
    ksc = vsc = None
    if s.w.kv == "nvfp4":
        ksc, vsc = to_np(s.k_bscales).copy(), to_np(s.v_bscales).copy()
        assert orc.kv_append_block_scales(to_np(s.k_new_bscales), to_np(s.v_new_bscales), ksc,
                                          vsc, s.slot_mapping_np) == 0
    ref, st, kc, vc = oracle_full_step(s)
    assert st == 0 and np.isfinite(ref).all()
    out, err = gpu_step(s)
    assert err == 0
    # bitwise (the poisoned rows hold NaN, which compares unequal as a float)
    assert np.array_equal(to_np(s.k_cache).view(np.uint8), kc.view(np.uint8))
    assert np.array_equal(to_np(s.v_cache).view(np.uint8), vc.view(np.uint8))
    if ksc is not None:
        assert np.array_equal(to_np(s.k_bscales), ksc) and np.array_equal(to_np(s.v_bscales), vsc)
    assert_attention_close(out, ref, f"{name} {kw} block_size={bs}", twin=fp32_twin(s))


@pytest.mark.parametrize("bs", [32, 64])
def test_block_sizes_pack_unpack_and_caps(bs):
    """Pack and unpack of whole requests, and SM-capped attention, over 32- and 64-token
    blocks."""
    s = wl.make_step(variant("gqa_skew_b256", block_size=bs, B=12), device=DEV)
    ref, st, _, _ = oracle_full_step(s, append=False)
    assert st == 0
    for cap in (3, 61, 0):
        out, err = gpu_step(s, append=False, sm_cap=cap)
        assert err == 0
        assert_attention_close(out, ref, f"block_size={bs} sm_cap={cap}",
                               twin=fp32_twin(s, cap))
    kc, vc = to_np(s.k_cache).copy(), to_np(s.v_cache).copy()
    r = int(np.argmax(s.context_lens_np))
    L = int(s.context_lens_np[r])
    packed = torch.empty((L, 2, s.w.H_kv, s.w.D), dtype=s.k_cache.dtype, device=DEV)
    pda.kv_pack_blocks(packed, s.k_cache, s.v_cache, s.block_tables[r], L)
    want, st = orc.kv_pack_blocks(kc, vc, s.block_tables_np[r], L)
    assert st == 0 and np.array_equal(to_np(packed), want)
    k2, v2 = torch.zeros_like(s.k_cache), torch.zeros_like(s.v_cache)
    pda.kv_unpack_blocks(packed, k2, v2, s.block_tables[r], L)
    kw, vw = np.zeros_like(kc), np.zeros_like(vc)
    assert orc.kv_unpack_blocks(want, kw, vw, s.block_tables_np[r], L) == 0
    assert np.array_equal(to_np(k2), kw) and np.array_equal(to_np(v2), vw)


@pytest.mark.parametrize("bs", [8, 24, 48, 512])
def test_unsupported_block_sizes_are_rejected(bs):
    s = wl.make_step(variant("gqa_skew_b256", block_size=bs, B=2), device=DEV)
    with pytest.raises(binding.PdaError) as e:
        pda.alloc_workspace(s.B, s.w.H, s.w.H_kv, s.w.D, bs, s.w.torch_dtype, device=DEV)
    assert e.value.status == binding.PDA_ERR_UNSUPPORTED
