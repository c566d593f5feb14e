"""Decode steps replayed from bucketed CUDA graphs against the fp64 oracle."""
import numpy as np
import pytest
import torch

from gpu_common import assert_attention_close, to_np
from oracle import oracle as orc
from paged_decode_attention_02_gb300 import binding
from paged_decode_attention_02_gb300 import graphs as pg
from paged_decode_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_bucket_sizes():
    assert pg.bucket_sizes(20, 8, True) == [0, 8, 16, 20]
    assert pg.bucket_sizes(16, 8, False) == [8, 16]


def test_graph_replays_match_oracle_with_padding_and_two_streams():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    cases = [(5, 3), (8, 8), (16, 0), (1, 15), (0, 7)]
    B = sum(a + b for a, b in cases)  # each case takes fresh requests
    s = wl.make_step("sm_sweep_b128", device="cuda", B=B)
    w = s.w
    g = pg.DecodeStepGraphs(s.k_cache, s.v_cache, w.H, s.max_blocks, max_local=16,
                            max_remote=16, interval=8, scale=s.scale, remote_sm_cap=46)
    g.capture()
    # the eager warm-up inside capture() appended every row with slot -1 only: caches are
    # untouched, so host copies taken now are the oracle's starting point
    kc, vc = to_np(s.k_cache).copy(), to_np(s.v_cache).copy()
    nxt = 0
    for n_l, n_r in cases:
        assert nxt + n_l + n_r <= s.B  # checked on the host before any device indexing
        reqs = list(range(nxt, nxt + n_l + n_r))
        nxt += n_l + n_r

        def part(sel):
            return {"q": s.q[sel], "k_new": s.k_new[sel], "v_new": s.v_new[sel],
                    "slot_mapping": s.slot_mapping[sel], "block_tables": s.block_tables[sel],
                    "context_lens": s.context_lens[sel]} if len(sel) else None

        local, remote = part(reqs[:n_l]), part(reqs[n_l:])
        out_l, out_r = g.run(local, remote)
        torch.cuda.synchronize()
        assert int(g.err.item()) == 0
        assert orc.kv_append(to_np(s.k_new[reqs]), to_np(s.v_new[reqs]), kc, vc,
                             s.slot_mapping_np[reqs]) == 0
        ref, st = orc.paged_decode_attention(to_np(s.q[reqs]), kc, vc, s.block_tables_np[reqs],
                                             s.context_lens_np[reqs], s.scale)
        assert st == 0
        got = torch.cat([out_l, out_r]) if n_l and n_r else (out_l if n_l else out_r)
        assert_attention_close(got.clone(), ref, f"graph ({n_l}, {n_r})", strict=True)
    assert np.array_equal(to_np(s.k_cache), kc) and np.array_equal(to_np(s.v_cache), vc)
