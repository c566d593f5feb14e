"""KV transfer staging between a prefill and a decode instance: request-level and layer-level.

Request level: once prefill has finished every layer, one ``kv_pack_layers`` launch gathers
the request's blocks of all layers into per-layer dense buffers (page on goodput and PD
disaggregation, 0539edu.com, sec. 5.4, request granularity). Layer level: as soon as layer N
of the prefill is done, layer N's blocks are packed on a transfer stream while layer N + 1
computes, so the staging hides behind compute (same section, layer granularity; page
"Disaggregated LLM Serving: from PD disaggregation to attention offload", sec. 5.6, and its
Splitwise paragraph). The decode side mirrors it: layer N is unpacked into the freshly
allocated blocks as soon as its buffer is there, and decode of layer N may start then.

Ordering uses CUDA events only: ``layer_done(n)`` records an event on the compute stream and
makes the transfer stream wait for it before the pack of layer n, so the pack reads the
layer's final KV without any host synchronisation (capturable into CUDA graphs).

The pages' rule for choosing (small prompts request-level, large prompts layer-level, the
batch's token count being known when prefill starts) gives no threshold;
``choose_granularity`` takes it as an argument.
"""
from __future__ import annotations

import torch

from . import binding


def choose_granularity(num_tokens: int, layer_threshold_tokens: int) -> str:
    """``"layer"`` for prompts of at least ``layer_threshold_tokens`` tokens, else
    ``"request"`` (small prompts: the whole KV is small and per-layer launches and
    synchronisation cost more than they hide)."""
    return "layer" if num_tokens >= layer_threshold_tokens else "request"


class LayerwisePack:
    """Stages requests' KV layer by layer on a transfer stream.

    k_caches, v_caches: per-layer caches ``[num_blocks, block_size, H_kv, D]`` (same
    geometry and dtype in every layer); block_table_rows: per request, its device int32 table
    row (shared by all layers); context_lens: per request, host token counts; outs:
    ``outs[layer][request]`` dense ``[len, 2, H_kv, D]`` buffers (allocated if None).
    """

    def __init__(self, k_caches, v_caches, block_table_rows, context_lens, outs=None,
                 transfer_stream: torch.cuda.Stream | None = None, error_word=None,
                 send=None):
        assert len(k_caches) == len(v_caches) and len(k_caches) > 0
        self.k_caches, self.v_caches = list(k_caches), list(v_caches)
        self.rows = list(block_table_rows)
        self.lens = [int(x) for x in context_lens]
        assert len(self.rows) == len(self.lens) <= binding.PDA_PACK_MAX_BATCH
        dev = self.k_caches[0].device
        _, _, H_kv, D = self.k_caches[0].shape
        dt = self.k_caches[0].dtype
        if outs is None:
            outs = [[torch.empty((L, 2, H_kv, D), dtype=dt, device=dev) for L in self.lens]
                    for _ in self.k_caches]
        self.outs = outs
        self.stream = transfer_stream or torch.cuda.Stream(device=dev)
        self.error_word = error_word
        # send(layer, buffers, stream): enqueues the hand-off of a packed layer (a copy to the
        # NIC's staging memory, a peer copy, ...) on the transfer stream after its pack
        self.send = send
        self.layer_events = [torch.cuda.Event() for _ in self.k_caches]  # layer n packed
        self._ready = [torch.cuda.Event() for _ in self.k_caches]  # layer n computed

    @property
    def n_layers(self) -> int:
        return len(self.k_caches)

    def layer_done(self, layer: int, compute_stream: torch.cuda.Stream | None = None):
        """Layer ``layer``'s KV is final on ``compute_stream``: pack it on the transfer stream
        once the compute stream reaches this point. Returns at once (no host sync)."""
        cs = compute_stream or torch.cuda.current_stream(self.k_caches[0].device)
        self._ready[layer].record(cs)
        self.stream.wait_event(self._ready[layer])
        if any(self.lens):
            binding.kv_pack_blocks_batched(self.outs[layer], self.k_caches[layer],
                                           self.v_caches[layer], self.rows, self.lens,
                                           error_word=self.error_word, stream=self.stream)
        if self.send is not None:
            self.send(layer, self.outs[layer], self.stream)
        self.layer_events[layer].record(self.stream)

    def wait(self, stream: torch.cuda.Stream | None = None):
        """Make ``stream`` (default: current) wait until every layer is packed."""
        s = stream or torch.cuda.current_stream(self.k_caches[0].device)
        s.wait_event(self.layer_events[-1])


def pack_request_level(outs, k_caches, v_caches, block_table_row, context_len: int,
                       error_word=None, stream=None):
    """Request-level staging: every layer of one request in one launch, after prefill."""
    return binding.kv_pack_layers(outs, k_caches, v_caches, block_table_row, context_len,
                                  error_word=error_word, stream=stream)


class LayerwiseUnpack:
    """The decode side: unpack layer n into the request's new blocks once its buffer has
    arrived (``arrived(n)``, an event on the stream that delivered it), and let decode of
    layer n start as soon as that layer is in place (``wait_layer``)."""

    def __init__(self, k_caches, v_caches, block_table_row, context_len: int,
                 transfer_stream: torch.cuda.Stream | None = None, error_word=None):
        self.k_caches, self.v_caches = list(k_caches), list(v_caches)
        self.row, self.len = block_table_row, int(context_len)
        dev = self.k_caches[0].device
        self.stream = transfer_stream or torch.cuda.Stream(device=dev)
        self.error_word = error_word
        self.layer_events = [torch.cuda.Event() for _ in self.k_caches]

    def arrived(self, layer: int, packed: torch.Tensor, event: torch.cuda.Event | None = None):
        """``packed`` holds layer ``layer``'s ``[len, 2, H_kv, D]`` buffer (complete once
        ``event`` fires, if given): scatter it on the transfer stream."""
        if event is not None:
            self.stream.wait_event(event)
        if self.len:
            binding.kv_unpack_blocks(packed, self.k_caches[layer], self.v_caches[layer],
                                     self.row, self.len, error_word=self.error_word,
                                     stream=self.stream)
        self.layer_events[layer].record(self.stream)

    def wait_layer(self, layer: int, stream: torch.cuda.Stream | None = None):
        """Make ``stream`` (default: current) wait until layer ``layer`` is unpacked."""
        s = stream or torch.cuda.current_stream(self.k_caches[0].device)
        s.wait_event(self.layer_events[layer])
