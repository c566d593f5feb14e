"""Seeded synthetic inputs for the decode step over a paged KV cache.

This module only draws inputs: context lengths, block tables, slot mappings and N(0,1)
tensors. It holds none of the attention, append or pack arithmetic, and both the CUDA
path and the CPU oracle take their inputs from it.

Shapes follow the pages' workloads: the Adrenaline evaluation uses Llama-2 7B (32 heads
of 128) and 13B (40 heads of 128) with decode batches up to the 80 of its attention-share
figure (review of "Injecting Adrenaline into LLM Serving", sec. 2.2 and sec. 5.1), and the
paged layout is PagedAttention's (page "From PagedAttention to Prefill-Decode
disaggregation", sec. 2.2). The ShareGPT / OpenThoughts traces those pages measure on
are not available; the length distributions below stand in for them.

Recipe (one per named workload):
  - lengths, block tables and slots are drawn with NumPy from
    ``SeedSequence(1000 + index).spawn(3)`` (lengths, tables, values);
  - block tables: every request's blocks are a disjoint slice of one random permutation
    of the pool, so a request's blocks are scattered and out of order; unused table
    entries are -1;
  - q, the pool's K and V, and the appended token's K/V are N(0,1) drawn in fp32 by a
    ``torch.Generator`` seeded from the third stream, on the device the caller asks for,
    then rounded to the workload's dtype (round-to-nearest-even for bf16 and fp16);
  - FP8 workloads store E4M3 codes of value / scale (per-tensor scales, K and V apart;
    torch's float8_e4m3fn rounding), drawn with the seeds of their bf16 twin so the
    lengths and tables are the same;
  - NVFP4 workloads store random E2M1 code bytes and random E4M3 block scales in
    [0.25, 0.47) (per-tensor scales 0.9 for K, 1.3 for V), also on their twin's seeds; the
    cache's scales are laid out [num_blocks, H_kv, block_size, D/16];
  - context lengths count the tokens after this step's append, so the appended token is
    the last position each request attends to; ``slot_mapping[b]`` points at it.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

KV_BLOCK_SIZE = 16


@dataclass(frozen=True)
class Workload:
    name: str
    index: int
    B: int
    H: int
    H_kv: int
    D: int
    block_size: int
    dtype: str  # "f32", "bf16" or "f16": q, K/V and output
    lengths: str  # recipe name, see draw_lengths
    pool: str  # "fixed:<n>" or "scaled:<factor>"
    pack_top: int = 0  # number of longest requests whose KV is packed each step
    sm_caps_pct: tuple = field(default_factory=tuple)  # SM-fraction sweep, % of SMs
    description: str = ""
    kv: str = ""  # "": the cache holds `dtype`; "fp8": FP8 E4M3 codes; "nvfp4": E2M1 + scales
    k_scale: float = 1.0  # value of one K code unit (FP8 caches)
    v_scale: float = 1.0
    seed_of: int = 0  # draw with another workload's seeds (same lengths and tables)

    @property
    def group(self) -> int:
        return self.H // self.H_kv

    @property
    def torch_dtype(self):
        return {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[self.dtype]

    @property
    def elem_bytes(self) -> int:
        """Bytes of one q / out element."""
        return 4 if self.dtype == "f32" else 2

    @property
    def kv_elem_bytes(self) -> float:
        """Bytes of one stored K (or V) element, block scales included for NVFP4."""
        if self.kv == "nvfp4":
            return 0.5 + 1 / 16
        return 1 if self.kv == "fp8" else self.elem_bytes

    @property
    def kv_torch_dtype(self):
        return torch.uint8 if self.kv in ("fp8", "nvfp4") else self.torch_dtype


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", 1, B=4, H=2, H_kv=2, D=64, block_size=16, dtype="f32",
                 lengths="list:1,17,33,100", pool="fixed:64",
                 description="tiny paged decode attention, fp32, plus one appended token per request"),
        Workload("llama2_7b_b8", 2, B=8, H=32, H_kv=32, D=128, block_size=16, dtype="bf16",
                 lengths="const:1024", pool="fixed:4096",
                 description="Llama-2-7B single-layer decode, batch 8, context 1024"),
        Workload("llama2_13b_b80", 3, B=80, H=40, H_kv=40, D=128, block_size=16, dtype="bf16",
                 lengths="uniform:128,4096", pool="scaled:1.25",
                 description="Llama-2-13B single-layer decode, batch 80, context U[128,4096]"),
        Workload("gqa_skew_b256", 4, B=256, H=32, H_kv=8, D=128, block_size=16, dtype="bf16",
                 lengths="loguniform:16,32768", pool="scaled:1.25", pack_top=8,
                 description="GQA 32/8, batch 256, context log-uniform [16,32768], "
                             "plus a pack of the 8 longest requests"),
        Workload("sm_sweep_b128", 5, B=128, H=32, H_kv=32, D=128, block_size=16, dtype="bf16",
                 lengths="uniform:512,2048", pool="scaled:1.25",
                 sm_caps_pct=(10, 20, 40, 60, 100),
                 description="Llama-2-7B shape, batch 128, context U[512,2048], SM-fraction sweep"),
        Workload("gqa_skew_b256_fp8", 6, B=256, H=32, H_kv=8, D=128, block_size=16,
                 dtype="bf16", lengths="loguniform:16,32768", pool="scaled:1.25", pack_top=8,
                 kv="fp8", k_scale=0.03, v_scale=0.05, seed_of=4,
                 description="gqa_skew_b256 with an FP8 E4M3 KV cache (per-tensor scales)"),
        Workload("llama2_13b_b80_fp8", 7, B=80, H=40, H_kv=40, D=128, block_size=16,
                 dtype="bf16", lengths="uniform:128,4096", pool="scaled:1.25", kv="fp8",
                 k_scale=0.03, v_scale=0.05, seed_of=3,
                 description="llama2_13b_b80 with an FP8 E4M3 KV cache (per-tensor scales)"),
        Workload("gqa_skew_b256_nvfp4", 8, B=256, H=32, H_kv=8, D=128, block_size=16,
                 dtype="bf16", lengths="loguniform:16,32768", pool="scaled:1.25", pack_top=8,
                 kv="nvfp4", k_scale=0.9, v_scale=1.3, seed_of=4,
                 description="gqa_skew_b256 with an NVFP4 KV cache"),
        Workload("llama2_13b_b80_nvfp4", 9, B=80, H=40, H_kv=40, D=128, block_size=16,
                 dtype="bf16", lengths="uniform:128,4096", pool="scaled:1.25", kv="nvfp4",
                 k_scale=0.9, v_scale=1.3, seed_of=3,
                 description="llama2_13b_b80 with an NVFP4 KV cache"),
        Workload("gqa_skew_b256_f16", 10, B=256, H=32, H_kv=8, D=128, block_size=16,
                 dtype="f16", lengths="loguniform:16,32768", pool="scaled:1.25", pack_top=8,
                 seed_of=4, description="gqa_skew_b256 in fp16 (q, caches and output)"),
        Workload("gqa_skew_b256_bs64", 11, B=256, H=32, H_kv=8, D=128, block_size=64,
                 dtype="bf16", lengths="loguniform:16,32768", pool="scaled:1.25", pack_top=8,
                 seed_of=4, description="gqa_skew_b256 over 64-token physical blocks"),
    ]
}


def get(name_or_index) -> Workload:
    if isinstance(name_or_index, int) or str(name_or_index).isdigit():
        idx = int(name_or_index)
        for w in WORKLOADS.values():
            if w.index == idx:
                return w
        raise KeyError(name_or_index)
    return WORKLOADS[name_or_index]


def _streams(w: Workload, seed: int | None):
    ss = np.random.SeedSequence(1000 + (w.seed_of or w.index) if seed is None else seed)
    return ss.spawn(3)


def draw_lengths(w: Workload, rng: np.random.Generator, B: int) -> np.ndarray:
    kind, _, arg = w.lengths.partition(":")
    if kind == "list":
        vals = [int(x) for x in arg.split(",")]
        return np.array([vals[i % len(vals)] for i in range(B)], np.int32)
    if kind == "const":
        return np.full(B, int(arg), np.int32)
    lo, hi = (int(x) for x in arg.split(","))
    if kind == "uniform":
        return rng.integers(lo, hi, size=B, endpoint=True).astype(np.int32)
    if kind == "loguniform":
        x = np.exp(rng.uniform(math.log(lo), math.log(hi), size=B))
        return np.clip(np.floor(x), lo, hi).astype(np.int32)
    raise ValueError(w.lengths)


def pool_blocks(w: Workload, lengths: np.ndarray) -> int:
    need = int(sum((int(L) + w.block_size - 1) // w.block_size for L in lengths))
    kind, _, arg = w.pool.partition(":")
    if kind == "fixed":
        return max(int(arg), need)
    return max(int(math.ceil(float(arg) * need)), need, 1)


@dataclass
class Step:
    """One decode step's inputs. Tensors live on ``device``; metadata also as NumPy."""
    w: Workload
    B: int
    num_blocks: int
    max_blocks: int
    context_lens_np: np.ndarray
    block_tables_np: np.ndarray
    slot_mapping_np: np.ndarray
    q: torch.Tensor
    k_cache: torch.Tensor
    v_cache: torch.Tensor
    k_new: torch.Tensor
    v_new: torch.Tensor
    block_tables: torch.Tensor
    context_lens: torch.Tensor
    slot_mapping: torch.Tensor
    scale: float
    pack_requests: list
    k_scale: float = 1.0
    v_scale: float = 1.0
    # NVFP4: block scales of the caches ([NB, H_kv, bs, D/16] E4M3 bytes, per block and
    # head-major) and of the new tokens ([B, H_kv, D/16]);
    # k_cache / v_cache / k_new / v_new then hold the packed E2M1 codes ([..., H_kv, D/2])
    k_bscales: torch.Tensor | None = None
    v_bscales: torch.Tensor | None = None
    k_new_bscales: torch.Tensor | None = None
    v_new_bscales: torch.Tensor | None = None

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens_np.max()) if self.B else 0


def _randn(shape, gen: torch.Generator, device, dtype, chunk: int = 1 << 28,
           scale_by: float = 1.0, to=None) -> torch.Tensor:
    """N(0,1) drawn in fp32, times scale_by, rounded to dtype (or to `to`, stored as raw
    bytes when `to` is an 8-bit float type), in chunks to bound the fp32 temporary."""
    store = torch.uint8 if to is not None else dtype
    out = torch.empty(shape, dtype=store, device=device)
    flat = out.view(-1)
    n = flat.numel()
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        x = torch.randn(e - s, generator=gen, device=device, dtype=torch.float32)
        if scale_by != 1.0:
            x = x * scale_by
        flat[s:e] = x.to(to).view(torch.uint8) if to is not None else x.to(dtype)
    return out


def make_step(w: Workload | str, device="cpu", B: int | None = None, seed: int | None = None,
              lengths: np.ndarray | None = None, poison_unused: bool = False) -> Step:
    """Draw one decode step of workload ``w``.

    ``B`` overrides the batch (fewer requests of the same recipe), ``lengths`` overrides the
    drawn context lengths, and ``poison_unused`` fills every cache row that holds no valid
    token (unused blocks and the tails of last blocks) with NaN, so that a read outside a
    request's history shows up in its output.
    """
    if isinstance(w, str):
        w = get(w)
    s_len, s_tab, s_val = _streams(w, seed)
    rng_len = np.random.default_rng(s_len)
    rng_tab = np.random.default_rng(s_tab)
    B = w.B if B is None else int(B)
    L = draw_lengths(w, rng_len, B) if lengths is None else np.asarray(lengths, np.int32)
    assert L.shape == (B,)
    bs = w.block_size
    nblk = (L.astype(np.int64) + bs - 1) // bs
    NB = pool_blocks(w, L)
    max_blocks = max(1, int(nblk.max()) if B else 1)
    perm = rng_tab.permutation(NB).astype(np.int32)
    bt = np.full((B, max_blocks), -1, np.int32)
    off = 0
    for b in range(B):
        n = int(nblk[b])
        bt[b, :n] = perm[off:off + n]
        off += n
    slots = np.full(B, -1, np.int32)
    for b in range(B):
        if L[b] > 0:
            t = int(L[b]) - 1
            slots[b] = bt[b, t // bs] * bs + t % bs

    gen = torch.Generator(device=device)
    gen.manual_seed(int(np.random.default_rng(s_val).integers(0, 2**62)))
    dt = w.torch_dtype
    q = _randn((B, w.H, w.D), gen, device, dt)
    nv = {}
    if w.kv == "nvfp4":
        # random E2M1 code pairs (every byte is valid) and E4M3 block scales in [0.25, 0.47)
        # (exponent field 5), so element values are of order 1
        def codes(shape):
            return torch.randint(0, 256, shape, generator=gen, device=device, dtype=torch.int32
                                 ).to(torch.uint8)

        def bscales(shape):
            return torch.randint(0x28, 0x30, shape, generator=gen, device=device,
                                 dtype=torch.int32).to(torch.uint8)

        half, nsc = w.D // 2, w.D // 16
        k_cache = codes((NB, bs, w.H_kv, half))
        v_cache = codes((NB, bs, w.H_kv, half))
        k_new = codes((B, w.H_kv, half))
        v_new = codes((B, w.H_kv, half))
        # cache scales per block, head-major: [NB, H_kv, bs, D/16]
        nv = dict(k_bscales=bscales((NB, w.H_kv, bs, nsc)),
                  v_bscales=bscales((NB, w.H_kv, bs, nsc)),
                  k_new_bscales=bscales((B, w.H_kv, nsc)), v_new_bscales=bscales((B, w.H_kv, nsc)))
    elif w.kv == "fp8":
        # N(0,1) values stored as E4M3 codes of value / scale (round to nearest even)
        def kvt(shape, sc):
            return _randn(shape, gen, device, torch.float32, scale_by=1.0 / sc,
                          to=torch.float8_e4m3fn)
        k_cache = kvt((NB, bs, w.H_kv, w.D), w.k_scale)
        v_cache = kvt((NB, bs, w.H_kv, w.D), w.v_scale)
        k_new = kvt((B, w.H_kv, w.D), w.k_scale)
        v_new = kvt((B, w.H_kv, w.D), w.v_scale)
    else:
        k_cache = _randn((NB, bs, w.H_kv, w.D), gen, device, dt)
        v_cache = _randn((NB, bs, w.H_kv, w.D), gen, device, dt)
        k_new = _randn((B, w.H_kv, w.D), gen, device, dt)
        v_new = _randn((B, w.H_kv, w.D), gen, device, dt)
    if poison_unused:
        valid = np.zeros(NB * bs, bool)
        for b in range(B):
            for t in range(int(L[b])):
                valid[bt[b, t // bs] * bs + t % bs] = True
        bad = torch.from_numpy(~valid).to(device).view(NB, bs)
        nan = 0x7F if w.kv == "fp8" else float("nan")  # 0x7F is the E4M3 NaN code
        if w.kv == "nvfp4":  # E2M1 has no NaN: poison the rows' block scales instead
            nv["k_bscales"].permute(0, 2, 1, 3)[bad] = 0x7F
            nv["v_bscales"].permute(0, 2, 1, 3)[bad] = 0x7F
        else:
            k_cache[bad] = nan
            v_cache[bad] = nan

    order = np.argsort(-L.astype(np.int64), kind="stable")
    pack = [int(b) for b in order[: w.pack_top]] if w.pack_top else []
    return Step(
        w=w, B=B, num_blocks=NB, max_blocks=max_blocks, context_lens_np=L,
        block_tables_np=bt, slot_mapping_np=slots, q=q, k_cache=k_cache, v_cache=v_cache,
        k_new=k_new, v_new=v_new,
        block_tables=torch.from_numpy(bt).to(device),
        context_lens=torch.from_numpy(L).to(device),
        slot_mapping=torch.from_numpy(slots).to(device),
        scale=float(np.float32(1.0 / math.sqrt(w.D))),
        pack_requests=pack,
        k_scale=float(np.float32(w.k_scale)),
        v_scale=float(np.float32(w.v_scale)),
        **nv,
    )
