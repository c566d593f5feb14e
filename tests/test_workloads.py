"""The seeded input generator: shapes, ranges, determinism and table structure (CPU)."""
import numpy as np
import pytest
import torch

from paged_decode_attention_02_gb300 import workloads as wl


def test_named_workloads():
    assert [wl.get(i).name for i in range(1, 12)] == [
        "tiny", "llama2_7b_b8", "llama2_13b_b80", "gqa_skew_b256", "sm_sweep_b128",
        "gqa_skew_b256_fp8", "llama2_13b_b80_fp8", "gqa_skew_b256_nvfp4",
        "llama2_13b_b80_nvfp4", "gqa_skew_b256_f16", "gqa_skew_b256_bs64"]


def test_nvfp4_workload_has_codes_and_block_scales():
    s = wl.make_step("llama2_13b_b80_nvfp4", B=2)
    w = s.w
    assert s.k_cache.shape[-1] == w.D // 2 and s.k_bscales.shape[-1] == w.D // 16
    assert s.k_new.shape == (2, w.H_kv, w.D // 2) and s.k_new_bscales.shape == (2, w.H_kv, w.D // 16)
    assert int(s.k_bscales.min()) >= 0x28 and int(s.k_bscales.max()) < 0x30
    assert s.k_bscales.shape == (s.num_blocks, w.H_kv, w.block_size, w.D // 16)


def test_nvfp4_poison_marks_unused_rows_in_head_major_scales():
    s = wl.make_step("llama2_13b_b80_nvfp4", B=2, poison_unused=True)
    bs = s.w.block_size
    used = np.zeros((s.num_blocks, bs), bool)
    for b in range(s.B):
        for t in range(int(s.context_lens_np[b])):
            used[s.block_tables_np[b, t // bs], t % bs] = True
    nan_rows = (s.k_bscales == 0x7F).all(dim=-1).all(dim=1).cpu().numpy()  # [NB, bs]
    assert np.array_equal(nan_rows, ~used)


def test_fp8_workload_shares_lengths_and_tables_with_its_twin():
    a = wl.make_step("gqa_skew_b256_fp8", B=3)
    b = wl.make_step("gqa_skew_b256", B=3)
    assert np.array_equal(a.context_lens_np, b.context_lens_np)
    assert np.array_equal(a.block_tables_np, b.block_tables_np)
    assert a.k_cache.dtype == torch.uint8 and a.q.dtype == torch.bfloat16
    assert not (a.k_cache == 0x7F).any() and not (a.k_cache == 0xFF).any()  # no NaN codes


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_metadata_structure(name):
    w = wl.get(name)
    rng = np.random.default_rng(0)
    L = wl.draw_lengths(w, rng, w.B)
    kind, _, arg = w.lengths.partition(":")
    if kind in ("uniform", "loguniform"):
        lo, hi = (int(x) for x in arg.split(","))
        assert L.min() >= lo and L.max() <= hi
    if name == "tiny":
        assert list(L) == [1, 17, 33, 100]
    NB = wl.pool_blocks(w, L)
    need = int(((L + w.block_size - 1) // w.block_size).sum())
    assert NB >= need


def test_tiny_step_tables_and_slots():
    s = wl.make_step("tiny")
    assert s.num_blocks == 64 and s.q.dtype == torch.float32
    used = s.block_tables_np[s.block_tables_np >= 0]
    assert len(np.unique(used)) == len(used) == 13  # disjoint blocks, 1+2+3+7
    for b, L in enumerate(s.context_lens_np):
        t = L - 1
        assert s.slot_mapping_np[b] == s.block_tables_np[b, t // 16] * 16 + t % 16
    assert s.scale == np.float32(1 / 8)


def test_deterministic_and_seed_sensitive():
    a = wl.make_step("llama2_13b_b80", B=2)
    b = wl.make_step("llama2_13b_b80", B=2)
    c = wl.make_step("llama2_13b_b80", B=2, seed=7)
    assert torch.equal(a.k_cache.view(torch.int16), b.k_cache.view(torch.int16))
    assert np.array_equal(a.block_tables_np, b.block_tables_np)
    assert not torch.equal(a.q.view(torch.int16), c.q.view(torch.int16))


def test_bf16_values_are_rounded_normals():
    s = wl.make_step("llama2_13b_b80", B=2)
    x = s.k_cache.float()
    assert s.k_cache.dtype == torch.bfloat16
    assert abs(x.mean().item()) < 0.01 and abs(x.std().item() - 1) < 0.01


def test_poison_marks_only_unused_rows():
    s = wl.make_step("tiny", poison_unused=True)
    bs = 16
    for b, L in enumerate(s.context_lens_np):
        for t in range(int(L)):
            blk = s.block_tables_np[b, t // bs]
            assert torch.isfinite(s.k_cache[blk, t % bs]).all()
    assert torch.isnan(s.k_cache).any()
