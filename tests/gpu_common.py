"""Shared helpers of the GPU parity tests: host copies for the oracle, the GPU step through
the C ABI, and the attention tolerance check."""
from __future__ import annotations

import numpy as np
import torch

import paged_decode_attention_02_gb300 as pda
from oracle import oracle as orc

# Attention tolerance for bf16 output: max abs error 4e-3, and max of
# |got - ref| / max(|ref|, 1e-2) at most 1e-2 (the floor keeps near-zero outputs from
# turning fp32 accumulation noise into huge ratios).
# Where |ref| > 2.05, rounding even the exact result to bf16 can move it by more than
# 4e-3 (half a bf16 ulp is 2^-8 * 2^floor(log2 |ref|)). There the absolute bound is half a
# bf16 ulp of the reference plus 1e-5 |ref| for the fp32 accumulation that precedes the
# rounding; the relative bound is unchanged everywhere.
ABS_TOL, REL_TOL, REL_FLOOR = 4e-3, 1e-2, 1e-2
# fp32 output: fp32 accumulation and a 2^-22 exp2 approximation; far inside 1e-4.
F32_ABS_TOL = 1e-4


def to_np(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def bf16_half_ulp(x: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 numbers (8 significant bits) at |x|."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 8)


def assert_attention_close(got: torch.Tensor, ref: np.ndarray, what: str = "",
                           strict: bool = False, twin: torch.Tensor | None = None):
    """``strict``: the flat 4e-3 bound everywhere (the named workloads, where |ref| < 2.05).

    Otherwise a bf16 or fp16 output is held to the ulp-aware bound, which on its own would
    let a kernel error of up to about one output ulp pass where |ref| > 2.05. So such a
    check needs ``twin``: the fp32 output of the same launch (same inputs, plan and SM cap).
    The kernel computes the same fp32 values whatever the output type and only rounds them
    at the store, so ``got`` must be exactly ``twin`` rounded to nearest even, and ``twin``
    must match the oracle within the fp32 bound: the whole excess over 4e-3 is then the
    output rounding."""
    if not strict and got.dtype != torch.float32:
        assert twin is not None, f"{what}: a relaxed {got.dtype} check needs its fp32 twin"
        assert twin.dtype == torch.float32 and twin.shape == got.shape
        bits = torch.int16
        assert torch.equal(twin.to(got.dtype).view(bits), got.view(bits)), (
            f"{what}: output is not the fp32 twin rounded to {got.dtype}")
        assert_attention_close(twin, ref, f"{what} (fp32 twin)")
    g = got.detach().double().cpu().numpy()
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(g), nan_ref), f"{what}: NaN pattern differs"
    ok = ~nan_ref
    if not ok.any():
        return
    err = np.abs(g[ok] - ref[ok])
    rel = err / np.maximum(np.abs(ref[ok]), REL_FLOOR)
    r = ref[ok]
    if got.dtype == torch.float32:
        bound = np.full_like(r, F32_ABS_TOL)
    elif strict:
        bound = np.full_like(r, ABS_TOL)
    else:
        bound = np.maximum(ABS_TOL, bf16_half_ulp(r) + 1e-5 * np.abs(r))
    worst = int(np.argmax(err - bound))
    assert err[worst] <= bound[worst], (
        f"{what}: abs err {err[worst]:.3e} > bound {bound[worst]:.3e} at |ref| {abs(r[worst]):.3f}")
    assert rel.max() <= REL_TOL, f"{what}: max rel err {rel.max():.3e} > {REL_TOL}"


def _oracle_attention(s, q, kc, vc, bt, lens, ksc=None, vsc=None, num_threads=0):
    if s.w.kv == "nvfp4":
        return orc.paged_decode_attention_nvfp4(q, kc, vc, ksc, vsc, bt, lens, s.scale,
                                                s.k_scale, s.v_scale, num_threads=num_threads)
    return orc.paged_decode_attention(q, kc, vc, bt, lens, s.scale, num_threads=num_threads,
                                      k_scale=s.k_scale, v_scale=s.v_scale)


def oracle_full_step(s, append: bool = True, num_threads: int = 0):
    """fp64 oracle of the whole step on host copies taken before the GPU runs. For NVFP4
    the new tokens' block scales are appended into the per-block scale caches as well."""
    kc, vc = to_np(s.k_cache).copy(), to_np(s.v_cache).copy()
    ksc = vsc = None
    if s.w.kv == "nvfp4":
        ksc, vsc = to_np(s.k_bscales).copy(), to_np(s.v_bscales).copy()
    if append:
        assert orc.kv_append(to_np(s.k_new), to_np(s.v_new), kc, vc, s.slot_mapping_np) == 0
        if ksc is not None:
            assert orc.kv_append_block_scales(to_np(s.k_new_bscales), to_np(s.v_new_bscales),
                                              ksc, vsc, s.slot_mapping_np) == 0
    ref, st = _oracle_attention(s, to_np(s.q), kc, vc, s.block_tables_np, s.context_lens_np,
                                ksc, vsc, num_threads)
    return ref, st, kc, vc


def oracle_sampled(s, reqs, append: bool = True):
    """Oracle of requests ``reqs`` only: their blocks are fetched into a small host pool
    (renumbered), so full-size workloads need not be copied whole. Call before the GPU
    step mutates the caches."""
    bs = s.w.block_size
    reqs = list(reqs)
    nblk = [(int(s.context_lens_np[r]) + bs - 1) // bs for r in reqs]
    used = sorted({int(s.block_tables_np[r, j]) for r, n in zip(reqs, nblk) for j in range(n)})
    pos = {b: i for i, b in enumerate(used)}
    idx = torch.tensor(used if used else [0], dtype=torch.long, device=s.k_cache.device)
    kc = to_np(s.k_cache.index_select(0, idx)).copy()
    vc = to_np(s.v_cache.index_select(0, idx)).copy()
    ksc = vsc = None
    if s.w.kv == "nvfp4":
        ksc = to_np(s.k_bscales.index_select(0, idx)).copy()
        vsc = to_np(s.v_bscales.index_select(0, idx)).copy()
    mb = max(1, max(nblk) if nblk else 1)
    bt = np.full((len(reqs), mb), -1, np.int32)
    for i, (r, n) in enumerate(zip(reqs, nblk)):
        bt[i, :n] = [pos[int(b)] for b in s.block_tables_np[r, :n]]
    lens = s.context_lens_np[reqs].astype(np.int32)
    if append:
        slots = np.full(len(reqs), -1, np.int32)
        for i, r in enumerate(reqs):
            sl = int(s.slot_mapping_np[r])
            if sl >= 0:
                slots[i] = pos[sl // bs] * bs + sl % bs
        st = orc.kv_append(to_np(s.k_new[reqs]), to_np(s.v_new[reqs]), kc, vc, slots)
        assert st == 0
        if ksc is not None:
            st = orc.kv_append_block_scales(to_np(s.k_new_bscales[reqs]),
                                            to_np(s.v_new_bscales[reqs]), ksc, vsc, slots)
            assert st == 0
    return _oracle_attention(s, to_np(s.q[reqs]).copy(), kc, vc, bt, lens, ksc, vsc)


def gpu_step(s, append: bool = True, sm_cap: int = 0, out_dtype=None, workspace=None):
    """kv_append then paged_decode_attention through the C ABI; returns (out, error word)."""
    err = torch.zeros(1, dtype=torch.int32, device=s.q.device)
    if append:
        pda.kv_append(s.k_new, s.v_new, s.k_cache, s.v_cache, s.slot_mapping, error_word=err)
        if s.w.kv == "nvfp4":
            pda.kv_append_block_scales(s.k_new_bscales, s.v_new_bscales, s.k_bscales,
                                       s.v_bscales, s.slot_mapping, error_word=err)
    out = torch.empty(s.q.shape, dtype=out_dtype or s.q.dtype, device=s.q.device)
    if s.w.kv == "nvfp4":
        pda.paged_decode_attention_nvfp4(out, s.q, s.k_cache, s.v_cache, s.k_bscales,
                                         s.v_bscales, s.block_tables, s.context_lens,
                                         s.max_context_len, s.scale, s.k_scale, s.v_scale,
                                         sm_cap=sm_cap, workspace=workspace, error_word=err)
    elif s.w.kv == "fp8":
        pda.paged_decode_attention_fp8(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                       s.context_lens, s.max_context_len, s.scale, s.k_scale,
                                       s.v_scale, sm_cap=sm_cap, workspace=workspace,
                                       error_word=err)
    else:
        pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale, sm_cap=sm_cap,
                                   workspace=workspace, error_word=err)
    torch.cuda.synchronize()
    return out, int(err.item())


def fp32_twin(s, sm_cap: int = 0) -> torch.Tensor:
    """The attention of step ``s`` again with fp32 output, in the same launch configuration
    (run after the step's own append, which it does not repeat)."""
    out, err = gpu_step(s, append=False, sm_cap=sm_cap, out_dtype=torch.float32)
    assert err == 0
    return out
