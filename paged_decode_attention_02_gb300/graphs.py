"""Decode steps captured as CUDA graphs over buckets of (local batch, offloaded batch).

A decode instance that offloads part of its attention runs, per layer, a variable number
of local and of offloaded requests. Capturing a graph per exact pair of sizes is too many
graphs and shapes change every step, so graphs are captured for a grid of bucket sizes and
each step replays the smallest graph whose buckets hold both counts (review of "Injecting
Adrenaline into LLM Serving", sec. 3.2.2, the two-dimensional CUDA graph, and sec. 3.2.1 on
keeping host work off the per-layer critical path). Padding rows get context length 0 and
slot -1, which the kernels treat as an empty request (zero output, no append).

One captured step is: ``kv_append`` of every row, attention of the local rows on the SMs
left to them, and attention of the offloaded rows on a second stream confined to
``remote_sm_cap`` SMs, running at the same time (the offloaded requests model the
attention executor sharing a GPU with other work, sec. 3.3). Everything runs in the
library's kernels; this module only stages inputs into static buffers and replays graphs.
"""
from __future__ import annotations

import bisect

import torch

from . import binding


def bucket_sizes(max_n: int, interval: int, with_zero: bool) -> list:
    """0 (optional), interval, 2*interval, ..., and max_n itself."""
    sizes = list(range(interval, max_n, interval)) + [max_n]
    return ([0] if with_zero else []) + sorted(set(s for s in sizes if s > 0))


class DecodeStepGraphs:
    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, H: int, max_blocks: int,
                 max_local: int, max_remote: int, interval: int, scale: float,
                 remote_sm_cap: int, dtype=None):
        self.k_cache, self.v_cache = k_cache, v_cache
        NB, bs, H_kv, D = k_cache.shape
        self.H, self.H_kv, self.D, self.bs, self.max_blocks = H, H_kv, D, bs, max_blocks
        self.scale = float(scale)
        self.dtype = dtype or k_cache.dtype
        dev = k_cache.device
        self.device = dev
        self.sms = binding.device_sm_count()
        self.remote_cap = max(1, min(int(remote_sm_cap), self.sms - 1))
        self.local_cap = self.sms - self.remote_cap
        self.local_sizes = bucket_sizes(max_local, interval, with_zero=True)
        self.remote_sizes = bucket_sizes(max_remote, interval, with_zero=True)
        n = max_local + max_remote
        self.q = torch.zeros((n, H, D), dtype=self.dtype, device=dev)
        self.k_new = torch.zeros((n, H_kv, D), dtype=k_cache.dtype, device=dev)
        self.v_new = torch.zeros((n, H_kv, D), dtype=k_cache.dtype, device=dev)
        self.slots = torch.full((n,), -1, dtype=torch.int32, device=dev)
        self.tables = torch.zeros((n, max_blocks), dtype=torch.int32, device=dev)
        self.lens = torch.zeros((n,), dtype=torch.int32, device=dev)
        self.out = torch.zeros((n, H, D), dtype=self.dtype, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.side = torch.cuda.Stream(dev)
        self.ws = {}
        self.graphs = {}

    # ---------------------------------------------------------------- capture
    def _views(self, bl: int, br: int):
        rows_l = slice(0, bl)
        rows_r = slice(bl, bl + br)
        return rows_l, rows_r

    def _workspace(self, role: str, n: int, cap: int) -> torch.Tensor:
        # the local and the offloaded launch of one step run at the same time: never share
        key = (role, n, cap)
        if key not in self.ws:
            self.ws[key] = binding.alloc_workspace(n, self.H, self.H_kv, self.D, self.bs,
                                                   self.k_cache.dtype, cap, self.device)
        return self.ws[key]

    def _step(self, bl: int, br: int):
        """The work of one bucket, issued on the current stream (and the side stream)."""
        main = torch.cuda.current_stream(self.device)
        n = bl + br
        if n == 0:
            return
        binding.kv_append(self.k_new[:n], self.v_new[:n], self.k_cache, self.v_cache,
                          self.slots[:n], error_word=self.err, stream=main)
        max_ctx = self.max_blocks * self.bs
        rows_l, rows_r = self._views(bl, br)
        if br:
            self.side.wait_stream(main)
            binding.paged_decode_attention(
                self.out[rows_r], self.q[rows_r], self.k_cache, self.v_cache,
                self.tables[rows_r], self.lens[rows_r], max_ctx, self.scale,
                sm_cap=self.remote_cap, workspace=self._workspace("remote", br, self.remote_cap),
                error_word=self.err, stream=self.side)
        if bl:
            cap = self.local_cap if br else 0
            binding.paged_decode_attention(
                self.out[rows_l], self.q[rows_l], self.k_cache, self.v_cache,
                self.tables[rows_l], self.lens[rows_l], max_ctx, self.scale, sm_cap=cap,
                workspace=self._workspace("local", bl, cap), error_word=self.err, stream=main)
        if br:
            main.wait_stream(self.side)

    def capture(self):
        """Captures one graph per bucket pair. Call once, outside any other capture."""
        # run every bucket once eagerly first: one-time library set-up happens here
        for bl in self.local_sizes:
            for br in self.remote_sizes:
                self._step(bl, br)
        torch.cuda.synchronize(self.device)
        pool = torch.cuda.graph_pool_handle()
        for bl in self.local_sizes:
            for br in self.remote_sizes:
                if bl + br == 0:
                    continue
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, pool=pool):
                    self._step(bl, br)
                self.graphs[(bl, br)] = g
        torch.cuda.synchronize(self.device)
        self.err.zero_()
        return self

    # ---------------------------------------------------------------- replay
    def bucket(self, n_local: int, n_remote: int):
        i = bisect.bisect_left(self.local_sizes, n_local)
        j = bisect.bisect_left(self.remote_sizes, n_remote)
        if i == len(self.local_sizes) or j == len(self.remote_sizes):
            raise ValueError(f"({n_local}, {n_remote}) exceeds the captured buckets")
        return self.local_sizes[i], self.remote_sizes[j]

    def stage(self, local: dict, remote: dict):
        """Copies one step's inputs into the rows of the smallest fitting bucket and pads the
        rest as empty; returns the bucket. In a model, the tables, lengths and slots change
        once per step, while each layer's q and new K/V would be written straight into
        ``self.q``, ``self.k_new`` and ``self.v_new`` by the layer before."""
        n_l = local["q"].shape[0] if local else 0
        n_r = remote["q"].shape[0] if remote else 0
        bl, br = self.bucket(n_l, n_r)
        for start, part, nb in ((0, local, bl), (bl, remote, br)):
            if nb == 0:
                continue
            n = part["q"].shape[0] if part else 0
            self.lens[start:start + nb].zero_()
            self.slots[start:start + nb].fill_(-1)
            if n == 0:
                continue
            self.q[start:start + n].copy_(part["q"], non_blocking=True)
            self.k_new[start:start + n].copy_(part["k_new"], non_blocking=True)
            self.v_new[start:start + n].copy_(part["v_new"], non_blocking=True)
            self.slots[start:start + n].copy_(part["slot_mapping"], non_blocking=True)
            t = part["block_tables"]
            self.tables[start:start + n, :t.shape[1]].copy_(t, non_blocking=True)
            self.lens[start:start + n].copy_(part["context_lens"], non_blocking=True)
        return bl, br

    def replay(self, bucket):
        """One layer of the staged step: replays the bucket's graph."""
        self.graphs[bucket].replay()

    def outputs(self, bucket, n_local: int, n_remote: int):
        bl, _ = bucket
        return self.out[:n_local], self.out[bl:bl + n_remote]

    def run(self, local: dict, remote: dict):
        """Stage one step and replay it once. Returns (local out, remote out) as views of
        the static output buffer."""
        bucket = self.stage(local, remote)
        self.replay(bucket)
        n_l = local["q"].shape[0] if local else 0
        n_r = remote["q"].shape[0] if remote else 0
        return self.outputs(bucket, n_l, n_r)
