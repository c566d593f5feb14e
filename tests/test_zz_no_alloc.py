"""The no-allocation attention entry point against the workspace entry point.

``pda_paged_decode_attention_noalloc`` serves callers that may not allocate device memory
when they run (a plugin whose host framework owns all device memory, or a serving loop
that forbids allocation after start-up): its scratch is a fixed array inside the library.
This file runs last, so a run that stops at its first failure has run everything else.
Calls go through the C ABI directly (ctypes), two in a row on different inputs, so the
second call also shows that what the first left in the shared scratch does not leak.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_decode_attention_02_gb300 as pda
from gpu_common import assert_attention_close, oracle_full_step
from paged_decode_attention_02_gb300 import binding
from paged_decode_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(lib, out, s, err, sm_cap=0):
    w = s.w
    dt = binding.PDA_BF16 if w.dtype == "bf16" else binding.PDA_F32
    return lib.pda_paged_decode_attention_noalloc(
        _p(out), _p(s.q), _p(s.k_cache), _p(s.v_cache), _p(s.block_tables), s.max_blocks,
        _p(s.context_lens), s.max_context_len, s.B, w.H, w.H_kv, w.D, w.block_size,
        s.num_blocks, ctypes.c_float(s.scale), dt, dt, dt, sm_cap, _p(err),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return binding.load()


def test_noalloc_matches_workspace_entry_point_on_two_calls(lib):
    """Calls of alternating shapes, each one's counters lying where the previous one left
    partial results. Every output is held to the oracle (strict bound) and to the workspace
    entry point within the same tolerance. The no-allocation call always splits the work
    statically (the workspace call may leave a share to chunks claimed at run time, which
    rounds differently in the last bits), so its own results must repeat bit for bit: a
    repeat that differs would be scratch leaking from the call before."""
    steps = [wl.make_step("gqa_skew_b256", device="cuda", B=48),
             wl.make_step("llama2_13b_b80", device="cuda", B=20)]
    oracle = [oracle_full_step(s, append=False)[0] for s in steps]
    first = {}
    for i, (s, want) in enumerate(zip(steps + steps, oracle + oracle)):
        ref = torch.empty_like(s.q)
        pda.paged_decode_attention(ref, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale)
        out = torch.full_like(s.q, float("nan"))
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        st = _noalloc(lib, out, s, err)
        torch.cuda.synchronize()
        assert st == binding.PDA_OK, binding.status_string(st)
        assert int(err.item()) == 0
        assert_attention_close(out, want, f"noalloc {s.w.name} vs oracle", strict=True)
        assert_attention_close(out, ref.double().cpu().numpy(),
                               f"noalloc {s.w.name} vs workspace entry point", strict=True)
        key = i % len(steps)
        if key in first:
            assert torch.equal(out, first[key]), "a repeated call differs: scratch leaked"
        else:
            first[key] = out


def test_noalloc_rejects_sizes_beyond_its_scratch(lib):
    # A GQA group of 8 at D = 128 needs about 10 MB of scratch on a full GB300.
    w = wl.Workload("g8", 9, B=4, H=64, H_kv=8, D=128, block_size=16, dtype="bf16",
                    lengths="uniform:16,64", pool="scaled:1.25")
    need = pda.attention_workspace_size(4, 64, 8, 128, 16, torch.bfloat16, 0)
    s = wl.make_step(w, device="cuda")
    out = torch.zeros_like(s.q)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = _noalloc(lib, out, s, err)
    torch.cuda.synchronize()
    if need > binding.PDA_NOALLOC_SCRATCH_BYTES:
        assert st == binding.PDA_ERR_TOO_LARGE
        assert (out == 0).all()  # nothing was launched
    else:  # a smaller GPU: the same call fits and must be right
        assert st == binding.PDA_OK
        ref = torch.empty_like(s.q)
        pda.paged_decode_attention(ref, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale)
        assert_attention_close(out, ref.double().cpu().numpy(), "noalloc g8", strict=True)
