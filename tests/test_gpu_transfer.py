"""Request-level and layer-level KV transfer staging (pack over layers, layer-by-layer pack on
a transfer stream, layer-by-layer unpack on the decode side) against the oracle's pack."""
import dataclasses

import numpy as np
import pytest
import torch

import paged_decode_attention_02_gb300 as pda
from gpu_common import assert_attention_close, oracle_full_step, to_np
from oracle import oracle as orc
from paged_decode_attention_02_gb300 import binding
from paged_decode_attention_02_gb300 import transfer as tr
from paged_decode_attention_02_gb300 import workloads as wl

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def layered(name="llama2_13b_b80", B=4, n_layers=5, seed=11):
    """A step of `name` plus n_layers caches of the same geometry and block table, each with
    its own seeded contents (layer 0 is the step's own cache)."""
    s = wl.make_step(name, device=DEV, B=B)
    g = torch.Generator(device="cpu").manual_seed(seed)
    ks, vs = [s.k_cache], [s.v_cache]
    for _ in range(n_layers - 1):
        ks.append(torch.randn(s.k_cache.shape, generator=g).to(s.k_cache.dtype).to(DEV))
        vs.append(torch.randn(s.v_cache.shape, generator=g).to(s.v_cache.dtype).to(DEV))
    return s, ks, vs


def oracle_pack(kc, vc, s, r):
    out, st = orc.kv_pack_blocks(to_np(kc).copy(), to_np(vc).copy(), s.block_tables_np[r],
                                 int(s.context_lens_np[r]))
    assert st == 0
    return out


def test_pack_layers_is_per_layer_pack_bit_for_bit():
    s, ks, vs = layered()
    for r in range(s.B):
        L = int(s.context_lens_np[r])
        outs = [torch.empty((L, 2, s.w.H_kv, s.w.D), dtype=ks[0].dtype, device=DEV)
                for _ in ks]
        pda.kv_pack_layers(outs, ks, vs, s.block_tables[r], L)
        for i in range(len(ks)):
            assert np.array_equal(to_np(outs[i]), oracle_pack(ks[i], vs[i], s, r)), (r, i)


def test_unpack_layers_inverts_pack_layers_and_touches_nothing_else():
    s, ks, vs = layered(B=3, n_layers=4)
    r = int(np.argmax(s.context_lens_np))
    L = int(s.context_lens_np[r])
    outs = [torch.empty((L, 2, s.w.H_kv, s.w.D), dtype=ks[0].dtype, device=DEV) for _ in ks]
    pda.kv_pack_layers(outs, ks, vs, s.block_tables[r], L)
    k2 = [torch.zeros_like(k) for k in ks]
    v2 = [torch.zeros_like(v) for v in vs]
    pda.kv_unpack_layers(outs, k2, v2, s.block_tables[r], L)
    for i in range(len(ks)):
        kc = np.zeros_like(to_np(ks[i]))
        vc = np.zeros_like(kc)
        assert orc.kv_unpack_blocks(to_np(outs[i]), kc, vc, s.block_tables_np[r], L) == 0
        assert np.array_equal(to_np(k2[i]), kc) and np.array_equal(to_np(v2[i]), vc)


def test_pack_layers_limits_empty_and_bad_block():
    s, ks, vs = layered(B=2, n_layers=2)
    L = int(s.context_lens_np[0])
    out = torch.empty((L, 2, s.w.H_kv, s.w.D), dtype=ks[0].dtype, device=DEV)
    n = binding.PDA_PACK_MAX_LAYERS + 1
    with pytest.raises(binding.PdaError) as e:
        pda.kv_pack_layers([out] * n, [ks[0]] * n, [vs[0]] * n, s.block_tables[0], L)
    assert e.value.status == binding.PDA_ERR_UNSUPPORTED
    pda.kv_pack_layers([out, out], ks, vs, s.block_tables[0], 0)  # no-op
    row = s.block_tables[0].clone()
    row[0] = s.num_blocks + 3
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    outs = [torch.zeros((L, 2, s.w.H_kv, s.w.D), dtype=ks[0].dtype, device=DEV) for _ in ks]
    pda.kv_pack_layers(outs, ks, vs, row, L, error_word=err)
    assert int(err.item()) == binding.PDA_DEVERR_BLOCK_ID
    n0 = min(L, s.w.block_size)
    for i in range(len(ks)):
        assert (outs[i][:n0].view(torch.uint8) == 0xFF).all()
        good = oracle_pack(ks[i], vs[i], s, 0)
        assert np.array_equal(to_np(outs[i][n0:]), good[n0:])


def test_layerwise_pack_waits_for_each_layer_behind_slow_compute():
    """Each layer's final token is appended on the compute stream behind a long GEMM, then
    layer_done(); the transfer stream must pack the appended rows of every layer."""
    s, ks, vs = layered(B=4, n_layers=6)
    reqs = list(range(s.B))
    sent = {}

    def send(layer, bufs, stream):  # the hand-off runs on the transfer stream after the pack
        with torch.cuda.stream(stream):
            sent[layer] = [b.clone() for b in bufs]

    lw = tr.LayerwisePack(ks, vs, [s.block_tables[r] for r in reqs],
                          [int(s.context_lens_np[r]) for r in reqs], send=send)
    a = torch.randn(4096, 4096, device=DEV, dtype=torch.bfloat16)
    g = torch.Generator(device="cpu").manual_seed(5)
    news = []
    for i in range(lw.n_layers):
        for _ in range(3):
            a = (a @ a).clamp_(-1, 1)  # keeps the compute stream busy before the append
        kn = torch.randn(s.k_new.shape, generator=g).to(s.k_new.dtype).to(DEV)
        vn = torch.randn(s.v_new.shape, generator=g).to(s.v_new.dtype).to(DEV)
        news.append((kn, vn))
        pda.kv_append(kn, vn, ks[i], vs[i], s.slot_mapping)
        lw.layer_done(i)
    lw.wait()
    torch.cuda.synchronize()
    for i in range(lw.n_layers):
        kc, vc = to_np(ks[i]).copy(), to_np(vs[i]).copy()  # final caches (with the append)
        for r in reqs:
            want, st = orc.kv_pack_blocks(kc, vc, s.block_tables_np[r], int(s.context_lens_np[r]))
            assert st == 0 and np.array_equal(to_np(lw.outs[i][r]), want), (i, r)
            assert np.array_equal(to_np(sent[i][r]), want), (i, r, "sent")
        # the appended token is the last packed row of each request
        r = reqs[0]
        L = int(s.context_lens_np[r])
        assert torch.equal(lw.outs[i][r][L - 1, 0], news[i][0][r])


def test_layerwise_unpack_then_decode_each_layer():
    """Decode side: each layer's buffer is unpacked into zeroed caches on a transfer stream;
    attention of that layer waits only for its own layer and matches the oracle."""
    s, ks, vs = layered(B=3, n_layers=3)
    r_all = list(range(s.B))
    outs = [[oracle_pack(ks[i], vs[i], s, r) for r in r_all] for i in range(len(ks))]
    k2 = [torch.zeros_like(k) for k in ks]
    v2 = [torch.zeros_like(v) for v in vs]
    recv = [tr.LayerwiseUnpack(k2, v2, s.block_tables[r], int(s.context_lens_np[r]))
            for r in r_all]
    # one transfer stream for the decode side: every request's unpacker shares it
    for u in recv[1:]:
        u.stream = recv[0].stream
    ws = pda.alloc_workspace(s.B, s.w.H, s.w.H_kv, s.w.D, s.w.block_size, s.w.torch_dtype)
    keep = []  # received buffers stay alive until the end (read on the transfer stream)
    for i in range(len(ks)):
        for r, u in zip(r_all, recv):
            buf = torch.from_numpy(outs[i][r]).view(ks[0].dtype).to(DEV)  # "arrives"
            landed = torch.cuda.Event()
            landed.record()
            keep.append(buf)
            u.arrived(i, buf, landed)
        recv[-1].wait_layer(i)
        out = torch.empty_like(s.q)
        pda.paged_decode_attention(out, s.q, k2[i], v2[i], s.block_tables, s.context_lens,
                                   s.max_context_len, s.scale, workspace=ws)
        ref, st, _, _ = oracle_full_step(dataclasses.replace(s, k_cache=ks[i], v_cache=vs[i]),
                                         append=False)
        assert st == 0
        assert_attention_close(out, ref, f"layer {i}", strict=True)
    torch.cuda.synchronize()
