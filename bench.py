#!/usr/bin/env python
"""Benchmark of one decode step over a paged KV cache on GB300.

A step is the whole hot path on one batch: ``kv_append`` of each request's new token,
``paged_decode_attention`` (partial kernel + log-sum-exp combine) over every request's
history, and ``kv_pack_blocks`` of the longest requests into contiguous transfer buffers.
The default workload is ``gqa_skew_b256`` (B=256, H=32, H_kv=8, D=128, bf16, context
log-uniform in [16, 32768], pack of the 8 longest), the largest of the five synthetic
workloads and the only one that exercises every step.

Prints one JSON line. ``value`` is algorithmic GB/s of the step (bytes every kernel must
move at least once, see ``step_bytes``) over the device time of the step, inputs resident
in HBM, L2 flushed between steps. ``e2e`` is the same metric with the step's inputs copied
from pinned host memory and its outputs copied back inside the timed region.
``roofline`` reports the attention call against the measured HBM copy bandwidth.
``cpu_baseline`` is the fp64 CPU oracle timed on a bounded sample of the same workload.
``--impl reference`` times only that oracle (the CPU reference arm).

Multi-GPU: every rank runs an independent replica of the workload (requests shard with no
exchange), so ``value`` is the sum over ranks and ``scaling`` is "weak".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import shutil
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

HEADLINE = "gqa_skew_b256"
METRIC = "paged decode-attn HBM GB/s (% of GB300 peak) and decode tokens/s per layer"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0  # GB300's HBM3e rate as the task names it (~8 TB/s)
ATTN_SOURCES = ["paged_decode_attention_02_gb300/csrc/decode_attention.cu",
                "paged_decode_attention_02_gb300/csrc/pda_device.cuh",
                "paged_decode_attention_02_gb300/csrc/warp_attn_tc.cuh",
                "paged_decode_attention_02_gb300/csrc/work_units.h",
                "paged_decode_attention_02_gb300/csrc/pda_api.cu"]


# ------------------------------------------------------------------ bytes
def step_bytes(s, pack_reqs) -> dict:
    """Algorithmic bytes: each element the op must read or write, once.

    attention: K and V of every history token and kv-head (once, even under GQA), q and
    out, the block-table entries in use and the context lengths. Workspace traffic, the
    unused tail of each last block and unused pool blocks are not counted.
    append: the new K/V read and written, plus the slot ids.
    pack: the packed requests' K/V read and written, plus their table entries.
    """
    w = s.w
    e, e_kv = w.elem_bytes, w.kv_elem_bytes
    L = s.context_lens_np.astype(np.int64)
    bs = w.block_size
    nblk = (L + bs - 1) // bs
    kv_tok = int(round(2 * w.H_kv * w.D * e_kv))  # NVFP4: codes and block scales
    attn = int(L.sum()) * kv_tok + 2 * s.B * w.H * w.D * e + int(nblk.sum()) * 4 + s.B * 4
    append = 2 * s.B * kv_tok + s.B * 4
    pl = np.array([int(L[r]) for r in pack_reqs], np.int64)
    pack = int(pl.sum()) * kv_tok * 2 + int(((pl + bs - 1) // bs).sum()) * 4
    return {"attention": attn, "append": append, "pack": pack,
            "step": attn + append + pack, "tokens": int(L.sum())}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments and trailing blanks, so that editing a comment
    does not change the kernel's hash."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_sha() -> str:
    """Hash of the attention kernel's code (its sources without comments, and the build
    options), which names the kernel an ncu summary under profiles/ was taken on."""
    h = hashlib.sha256()
    h.update(os.environ.get("PDA_NVCC_DEFINES", "").encode())  # build options change the code
    for p in ATTN_SOURCES:
        with open(os.path.join(ROOT, p), encoding="utf-8") as f:
            h.update(strip_comments(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, algorithmic_bytes: int):
    """DRAM bytes per full-size attention launch, from the committed ncu summary of the
    workload if it was taken on the current kernel source, else None. The capture runs a
    reduced batch of the same recipe (a few GB on the device at most); its DRAM bytes over
    its algorithmic bytes (``dram_traffic_ratio``) scale the full launch's algorithmic bytes,
    since both grow with the tokens streamed."""
    path = os.path.join(ROOT, "profiles", f"attn_partial_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_sha = re.search(r"kernel_sha:\s*([0-9a-f]+)", text)
    m_r = re.search(r"dram_traffic_ratio:\s*([0-9.]+)", text)
    if not m_sha or not m_r or m_sha.group(1) != kernel_sha():
        return None
    return int(round(float(m_r.group(1)) * algorithmic_bytes))


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 200 ms while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            self.proc = subprocess.Popen(
                [exe, f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self._t.join(timeout=2)

    def summary(self):
        if self.proc is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


class L2Flush:
    """Evicts L2 before a timed step: writes a buffer twice the size of L2, then reads a
    second one, so the timed kernels find neither their inputs nor dirty lines (whose
    write-back they would otherwise pay for) in L2."""

    def __init__(self, l2_bytes: int, dev):
        import torch
        n = max(2 * l2_bytes, 1 << 20) // 4
        self.w = torch.empty(n, dtype=torch.float32, device=dev)
        self.r = torch.ones(n, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.sink)


def attention(s, out, sm_cap, workspace, error_word=None, stream=None):
    """One attention call through the C ABI (the FP8 entry point for FP8 caches)."""
    import paged_decode_attention_02_gb300 as pda
    if s.w.kv == "nvfp4":
        return pda.paged_decode_attention_nvfp4(out, s.q, s.k_cache, s.v_cache, s.k_bscales,
                                                s.v_bscales, s.block_tables, s.context_lens,
                                                s.max_context_len, s.scale, s.k_scale,
                                                s.v_scale, sm_cap=sm_cap, workspace=workspace,
                                                error_word=error_word, stream=stream)
    if s.w.kv == "fp8":
        return pda.paged_decode_attention_fp8(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                              s.context_lens, s.max_context_len, s.scale,
                                              s.k_scale, s.v_scale, sm_cap=sm_cap,
                                              workspace=workspace, error_word=error_word,
                                              stream=stream)
    return pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                      s.context_lens, s.max_context_len, s.scale, sm_cap=sm_cap,
                                      workspace=workspace, error_word=error_word, stream=stream)


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return ws, rank, local


def dist_max(x: float, ws: int) -> float:
    """The largest of every rank's x (the slowest rank's time decides a replica run)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(bytes_per_step: float, t_step_max: float, ws: int) -> float:
    """Whole-job GB/s of N independent replicas: every rank moved bytes_per_step in each
    step, and the job's step time is the slowest rank's."""
    return ws * bytes_per_step / t_step_max / 1e9


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def kv_arrays(s):
    """Per stored array pair of a step: (cache K, cache V, new K, new V, append, batched pack,
    batched unpack) -- the K/V rows, and for NVFP4 also the block scales, which have their
    own calls (per-block head-major layout). The three calls share one argument order."""
    import paged_decode_attention_02_gb300 as pda
    arrays = [(s.k_cache, s.v_cache, s.k_new, s.v_new, pda.kv_append, pda.kv_pack_blocks_batched,
               pda.kv_unpack_blocks_batched)]
    if s.w.kv == "nvfp4":
        arrays.append((s.k_bscales, s.v_bscales, s.k_new_bscales, s.v_new_bscales,
                       pda.kv_append_block_scales, pda.kv_pack_block_scales_batched,
                       pda.kv_unpack_block_scales_batched))
    return arrays


def workspace_for(s, sm_cap):
    import paged_decode_attention_02_gb300 as pda
    w = s.w
    if w.kv == "nvfp4":
        return pda.binding.nvfp4_workspace(s.B, w.H, w.H_kv, w.D, w.block_size, sm_cap,
                                           s.q.device)
    return pda.alloc_workspace(s.B, w.H, w.H_kv, w.D, w.block_size, w.kv_torch_dtype, sm_cap,
                               s.q.device)


# ------------------------------------------------------------------ oracle (CPU) timing
def _np(t):
    import torch
    t = t.detach().cpu().contiguous()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def oracle_pass(s, threads: int):
    """One oracle pass over a step on host arrays: append, attention, pack. Returns seconds."""
    from oracle import oracle as orc
    kc, vc = _np(s.k_cache).copy(), _np(s.v_cache).copy()
    q, kn, vn = _np(s.q), _np(s.k_new), _np(s.v_new)
    nvfp4 = s.w.kv == "nvfp4"
    if nvfp4:  # codes and block scales are appended and packed apart
        ksc, vsc = _np(s.k_bscales).copy(), _np(s.v_bscales).copy()
        ksn, vsn = _np(s.k_new_bscales), _np(s.v_new_bscales)
    t0 = time.perf_counter()
    orc.kv_append(kn, vn, kc, vc, s.slot_mapping_np)
    if nvfp4:
        orc.kv_append_block_scales(ksn, vsn, ksc, vsc, s.slot_mapping_np)
        orc.paged_decode_attention_nvfp4(q, kc, vc, ksc, vsc, s.block_tables_np,
                                         s.context_lens_np, s.scale, s.k_scale, s.v_scale,
                                         num_threads=threads)
    else:
        orc.paged_decode_attention(q, kc, vc, s.block_tables_np, s.context_lens_np, s.scale,
                                   num_threads=threads, k_scale=s.k_scale, v_scale=s.v_scale)
    for r in s.pack_requests:
        orc.kv_pack_blocks(kc, vc, s.block_tables_np[r], int(s.context_lens_np[r]))
        if nvfp4:
            orc.kv_pack_block_scales(ksc, vsc, s.block_tables_np[r], int(s.context_lens_np[r]))
    return time.perf_counter() - t0


def oracle_sample(w, seconds: float, threads: int):
    """A step of workload w with as many requests as the oracle processes in ~`seconds`."""
    from paged_decode_attention_02_gb300 import workloads as wl
    probe_B = min(w.B, 8)
    probe = wl.make_step(w, device="cpu", B=probe_B)
    t = max(oracle_pass(probe, threads), 1e-3)
    per_tok = t / max(1, int(probe.context_lens_np.sum()))
    mean_tok = max(1.0, float(probe.context_lens_np.mean()))
    B = int(min(w.B, max(probe_B, seconds / per_tok / mean_tok)))
    return probe if B == probe_B else wl.make_step(w, device="cpu", B=B)


def oracle_legs(w, seconds: float = 2.0, max_B: int = 12) -> dict:
    """The fp64 oracle on a bounded sample of workload w (its first max_B requests, drawn by
    the same recipe on the host): all host cores, repeated for about `seconds`, and one
    pass on one core."""
    from paged_decode_attention_02_gb300 import workloads as wl

    threads = cpu_threads()
    sample = wl.make_step(w, device="cpu", B=min(w.B, max_B))
    b = step_bytes(sample, sample.pack_requests)
    reps, t = 0, 0.0
    while t < seconds or reps == 0:
        t += oracle_pass(sample, threads)
        reps += 1
    t1 = oracle_pass(sample, 1)
    return {"sample": f"B={sample.B} ({b['tokens']} tokens)",
            "all_cores": {"GBps": round(b["step"] * reps / t / 1e9, 4), "threads": threads,
                          "s_per_pass": round(t / reps, 3)},
            "one_core": {"GBps": round(b["step"] / t1 / 1e9, 4), "threads": 1,
                         "s_per_pass": round(t1, 3)}}


def cpu_threads() -> int:
    return int(os.environ.get("OMP_NUM_THREADS", os.cpu_count() or 1))


# ------------------------------------------------------------------ our arm
def run_ours(args, ws, rank, local):
    import torch

    import paged_decode_attention_02_gb300 as pda
    from paged_decode_attention_02_gb300 import build_lib
    from paged_decode_attention_02_gb300 import workloads as wl

    build_lib.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = wl.get(args.config)
    s = wl.make_step(w, device=dev, B=args.batch)
    pack_reqs = s.pack_requests
    nb = step_bytes(s, pack_reqs)
    stream = torch.cuda.current_stream(dev)

    out = torch.empty_like(s.q)
    cap = args.sm_cap
    wsp = workspace_for(s, cap)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    # the codes, and for NVFP4 also the block scales, each appended and packed by its calls
    arrays = kv_arrays(s)
    pack_rows = [s.block_tables[r] for r in pack_reqs]
    pack_lens = [int(s.context_lens_np[r]) for r in pack_reqs]
    packs_of = [[torch.empty((L, 2) + tuple(kn.shape[1:]), dtype=kc.dtype, device=dev)
                 for L in pack_lens] for kc, _, kn, _, _, _, _ in arrays]
    packs = [p for group in packs_of for p in group]
    launches_per_step = len(arrays) + 1 + (len(arrays) if pack_reqs else 0)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        for kc, vc, kn, vn, append, _, _ in arrays:
            append(kn, vn, kc, vc, s.slot_mapping, error_word=err)
        if ev:
            ev[1].record(stream)
        attention(s, out, cap, wsp, error_word=err)
        if ev:
            ev[2].record(stream)
        if pack_reqs:
            for (kc, vc, _, _, _, pack, _), group in zip(arrays, packs_of):
                pack(group, kc, vc, pack_rows, pack_lens, error_word=err)
        if ev:
            ev[3].record(stream)

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = L2Flush(l2, dev)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier(ws)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        for k in range(args.steps):
            flush()
            step(evs[k])
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        barrier(ws)
    t_append = np.mean([e[0].elapsed_time(e[1]) for e in evs]) * 1e-3
    t_attn = np.mean([e[1].elapsed_time(e[2]) for e in evs]) * 1e-3
    t_pack = np.mean([e[2].elapsed_time(e[3]) for e in evs]) * 1e-3
    t_step = np.mean([e[0].elapsed_time(e[3]) for e in evs]) * 1e-3
    t_step_max = dist_max(t_step, ws)

    # ---- end to end: per-step inputs from pinned host memory, results back to host.
    # A serving loop overlaps the copy-out of step k (attention output and packed KV, about
    # 1 GB, bound by the ~190 GB/s device-to-host link) with the compute of step k + 1: two
    # sets of output buffers, the copies on their own stream; step k waits only for the
    # copy-out that last used its buffer set. Timed over the whole loop (inputs larger than
    # L2, so no flush inside it).
    d_in = [s.q] + [t for _, _, kn, vn, _, _, _ in arrays for t in (kn, vn)] + [
        s.slot_mapping, s.block_tables, s.context_lens]
    h_in = [x.detach().cpu().pin_memory() for x in d_in]
    outs2 = [out, torch.empty_like(out)]
    packs2 = [packs_of, [[torch.empty_like(p) for p in group] for group in packs_of]]
    h_out2 = [[torch.empty(out.shape, dtype=out.dtype).pin_memory()] + [
        torch.empty(p.shape, dtype=p.dtype).pin_memory() for p in packs] for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in h_in)
    d2h = sum(x.numel() * x.element_size() for x in h_out2[0])
    copy_stream = torch.cuda.Stream(dev)
    computed = [torch.cuda.Event() for _ in range(2)]
    copied = [torch.cuda.Event() for _ in range(2)]
    for e in copied:
        e.record(stream)

    def e2e_step(k):
        b = k % 2
        stream.wait_event(copied[b])  # buffer set b is free again
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        for kc, vc, kn, vn, append, _, _ in arrays:
            append(kn, vn, kc, vc, s.slot_mapping, error_word=err)
        attention(s, outs2[b], cap, wsp, error_word=err)
        if pack_reqs:
            for (kc, vc, _, _, _, pack, _), group in zip(arrays, packs2[b]):
                pack(group, kc, vc, pack_rows, pack_lens, error_word=err)
        computed[b].record(stream)
        copy_stream.wait_event(computed[b])
        with torch.cuda.stream(copy_stream):
            d_out = [outs2[b]] + [p for group in packs2[b] for p in group]
            for d, h in zip(d_out, h_out2[b]):
                h.copy_(d, non_blocking=True)
        copied[b].record(copy_stream)

    for k in range(max(2, args.warmup)):
        e2e_step(k)
    torch.cuda.synchronize()
    barrier(ws)
    torch.cuda.synchronize()
    e_start, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_start.record(stream)
    for k in range(args.steps):
        e2e_step(k)
    for e in copied:
        stream.wait_event(e)
    e_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    t_e2e = dist_max(e_start.elapsed_time(e_end) * 1e-3 / args.steps, ws)
    if int(err.item()) != 0:
        raise RuntimeError(f"device error word {int(err.item())} during timing")

    # ---- unpack (the receiving side of the transfer): write the packed buffers back into
    # their own blocks, which leaves the cache unchanged
    t_unpack = None
    if pack_reqs:
        uev = []
        for _ in range(args.warmup + args.steps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush()
            a.record(stream)
            for (kc, vc, _, _, _, _, unpack), group in zip(arrays, packs_of):
                unpack(group, kc, vc, pack_rows, pack_lens, error_word=err)
            b.record(stream)
            uev.append((a, b))
        torch.cuda.synchronize()
        t_unpack = float(np.mean([a.elapsed_time(b) for a, b in uev[args.warmup:]])) * 1e-3

    peak, peak_src = hbm_peak()
    attn_gbs = nb["attention"] / t_attn / 1e9
    traffic = (profiled_traffic(w.name, nb["attention"])
               if (args.batch is None and cap == 0) else None)
    res = {
        "metric": METRIC,
        "value": round(replica_value(nb["step"], t_step_max, ws), 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_step_max * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        # arithmetic type: fp32 on the CUDA cores; quantised caches at D = 128 multiply fp16
        # operands (exact codes, split probabilities) on the tensor cores into fp32
        "dtype": "f16 mma, f32 accumulate" if (w.kv and w.D == 128) else "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "B": s.B, "H": w.H, "H_kv": w.H_kv, "D": w.D,
                   "block_size": w.block_size, "kv_dtype": w.kv or w.dtype,
                   "context_tokens": nb["tokens"], "pack_requests": len(pack_reqs),
                   "sm_cap": cap, "parallelism": f"replicas x{ws}",
                   "l2": f"flushed before every step: wrote, then read, a {2 * l2 >> 20} MiB "
                         f"buffer (no dirty lines left); KV set {nb['attention'] / 1e9:.2f} GB "
                         f"> L2 as well"},
        "attention": {"us": round(t_attn * 1e6, 2), "GBps": round(attn_gbs, 1),
                      "frac_of_peak": round(attn_gbs / peak, 4),
                      "decode_tokens_per_s_per_layer": round(s.B / t_attn, 1),
                      "bytes": nb["attention"]},
        "append": {"us": round(t_append * 1e6, 2),
                   "GBps": round(nb["append"] / t_append / 1e9, 2), "bytes": nb["append"]},
        "pack": {"us": round(t_pack * 1e6, 2),
                 "GBps": round(nb["pack"] / t_pack / 1e9, 1) if t_pack > 0 else None,
                 "bytes": nb["pack"]},
        "unpack": ({"us": round(t_unpack * 1e6, 2), "GBps": round(nb["pack"] / t_unpack / 1e9, 1),
                    "bytes": nb["pack"], "note": "not part of the step"} if t_unpack else None),
        "roofline": {"bound": "hbm", "achieved": round(attn_gbs, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(attn_gbs / peak, 4),
                     "traffic": traffic, "kernel": "attn_partial_kernel (one launch per call; "
                     "cut segments are merged inside it)", "peak_source": peak_src},
        "e2e": {"value": round(replica_value(nb["step"], t_e2e, ws), 2), "unit": "GB/s",
                "ms_per_step": round(t_e2e * 1e3, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "note": "inputs copied in from pinned memory and output + packed KV copied "
                        "out every step; copy-out of step k overlaps step k+1 (two buffer "
                        "sets, copy stream)"},
        "gpu_launches": launches_per_step * args.steps,
        "wall_s_timed": round(t_wall, 4),
        "clocks": clk.summary(),
    }

    if args.sweeps and ws == 1:
        res["workloads"] = sweep_workloads(args, dev, flush, peak)
        res["kv_transfer_staging"] = transfer_legs(dev)
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        threads = cpu_threads()
        sample = oracle_sample(w, args.cpu_seconds, threads)
        sb = step_bytes(sample, sample.pack_requests)
        reps, t_cpu = 0, 0.0
        while t_cpu < args.cpu_seconds or reps == 0:
            t_cpu += oracle_pass(sample, threads)
            reps += 1
        t_one = oracle_pass(sample, 1)  # the same sample on one core
        res["cpu_baseline"] = {
            "value": round(sb["step"] * reps / t_cpu / 1e9, 4), "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "value_one_core": round(sb["step"] / t_one / 1e9, 4),
            "sample": f"{w.name} recipe with B={sample.B} ({sb['tokens']} tokens, pack of "
                      f"{len(sample.pack_requests)}), fp64 C oracle, {reps} pass(es) on "
                      f"{threads} threads in {t_cpu:.1f} s; one pass on 1 thread in "
                      f"{t_one:.1f} s"}
    # last key of the line, so that a reader who sees only the tail still gets every workload
    res["per_config"] = per_config(w, s.B, res["attention"], res.get("workloads"), peak)
    return res


def per_config(w, B, headline_attn, workloads, peak) -> dict:
    """Attention alone on each named workload, compact: us per layer (one attention launch),
    decode tokens/s per layer (B / t), algorithmic GB/s, and its fraction of the measured
    copy peak and of the nominal 8 TB/s HBM3e rate; the SM-fraction workload at each cap."""
    from paged_decode_attention_02_gb300 import workloads as wl

    def entry(r):
        return {"us": r["us"], "tok_s": r["decode_tokens_per_s_per_layer"], "GBps": r["GBps"],
                "frac": r["frac_of_peak"], "frac_8TB": round(r["GBps"] / NOMINAL_HBM_GBS, 4)}

    res = {"peak_GBps": peak, "nominal_GBps": NOMINAL_HBM_GBS}
    res[w.name] = dict(entry(headline_attn), B=B)
    for name, r in (workloads or {}).items():
        if name == "single_request":
            res[name] = {n: {"us": v["us"], "context_len": v["context_len"]}
                         for n, v in r.items()}
            continue
        caps = wl.get(name).sm_caps_pct
        if not caps:
            res[name] = entry(r["all_sms"])
            continue
        sub = {}
        for key, v in r.items():
            if key == "all_sms":
                sub["100%"] = entry(v)
            elif key.startswith("sm_cap_"):
                n = int(key[len("sm_cap_"):])
                pct = [p for p in caps if p < 100 and math.ceil(p / 100 * _sms()) == n]
                sub[f"{pct[0] if pct else '?'}% ({n} SMs)"] = dict(entry(v), GBps_per_SM=round(
                    v["GBps"] / n, 1))
        res[name] = sub
    return res


def _sms() -> int:
    import paged_decode_attention_02_gb300 as pda
    return pda.device_sm_count()


def transfer_legs(dev, n_layers: int = 40, prompts=(2048, 8192), reps: int = 5) -> dict:
    """KV transfer staging of one prefilled request, request level against layer level.

    Geometry of llama2-13b (40 layers, 40 kv-heads, D = 128, bf16); the prompt's blocks are
    scattered over a per-layer pool. Each layer's prefill compute is stood in for by one bf16
    GEMM with that layer's projection and MLP flops (2 * T * 5120 * 61952; a library GEMM,
    not part of the measured kernels). Staging a layer = packing its blocks into a dense
    buffer (our kernel) and handing that buffer on: a device-to-host copy into pinned memory
    on the copy engine stands in for the send to the decode instance. Times, from the first
    GEMM on the compute stream: compute alone; compute, then pack and send of every layer
    (request level: one ``kv_pack_layers`` launch); compute with layer n packed and sent on a
    transfer stream right after GEMM n (layer level). Reported: each total and the staging
    time it leaves exposed beyond compute alone (medians of ``reps`` runs)."""
    import torch

    from paged_decode_attention_02_gb300 import transfer as tr

    H_kv, D, hidden, ffn_out = 40, 128, 5120, 61952
    g = torch.Generator(device="cpu").manual_seed(1234)
    gd = torch.Generator(device=dev).manual_seed(1234)  # bulk data drawn on the device

    def randn(*shape):
        return torch.randn(*shape, generator=gd, device=dev, dtype=torch.bfloat16)

    W = randn(hidden, ffn_out) * 0.01
    res = {"n_layers": n_layers, "geometry": "llama2-13b (H_kv=40, D=128, bf16)",
           "compute_stand_in": "bf16 GEMM [T,5120]x[5120,61952] per layer (cuBLAS)",
           "send_stand_in": "device-to-host copy of each packed layer into pinned memory"}
    main = torch.cuda.current_stream(dev)
    for T in prompts:
        nblk = (T + 15) // 16
        pool = nblk + 64
        row = torch.randperm(pool, generator=g)[:nblk].to(torch.int32).to(dev)
        ks = [randn(pool, 16, H_kv, D) for _ in range(n_layers)]
        vs = [randn(pool, 16, H_kv, D) for _ in range(n_layers)]
        X = randn(T, hidden)
        Y = torch.empty(T, ffn_out, dtype=torch.bfloat16, device=dev)
        outs = [torch.empty(T, 2, H_kv, D, dtype=torch.bfloat16, device=dev)
                for _ in range(n_layers)]
        host = torch.empty(T, 2, H_kv, D, dtype=torch.bfloat16).pin_memory()  # reused

        def send(layer, bufs, stream):
            with torch.cuda.stream(stream):
                host.copy_(bufs[0], non_blocking=True)

        lw = tr.LayerwisePack(ks, vs, [row], [T], outs=[[o] for o in outs], send=send)

        def run(mode):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(main)
            for i in range(n_layers):
                torch.matmul(X, W, out=Y)
                if mode == "layer":
                    lw.layer_done(i, main)
            if mode == "request":
                tr.pack_request_level(outs, ks, vs, row, T, stream=main)
                for i in range(n_layers):
                    send(i, [outs[i]], main)
            if mode == "layer":
                lw.wait(main)
            b.record(main)
            return a, b

        times = {}
        for mode in ("compute", "request", "layer"):
            run(mode)  # warm-up
            torch.cuda.synchronize()
            evs = [run(mode) for _ in range(reps)]
            torch.cuda.synchronize()
            times[mode] = float(np.median([x.elapsed_time(y) for x, y in evs]))
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        ev[0].record(main)
        tr.pack_request_level(outs, ks, vs, row, T, stream=main)
        ev[1].record(main)
        for i in range(n_layers):
            send(i, [outs[i]], main)
        ev[2].record(main)
        torch.cuda.synchronize()
        t_pack, t_send = ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])
        layer_bytes = T * 2 * H_kv * D * 2
        res[f"T={T}"] = {
            "compute_ms": round(times["compute"], 3),
            "request_level_ms": round(times["request"], 3),
            "layer_level_ms": round(times["layer"], 3),
            "exposed_request_level_ms": round(times["request"] - times["compute"], 3),
            "exposed_layer_level_ms": round(times["layer"] - times["compute"], 3),
            "pack_all_layers_ms": round(t_pack, 3),
            "pack_GBps": round(2 * n_layers * layer_bytes / (t_pack * 1e-3) / 1e9, 1),
            "send_all_layers_ms": round(t_send, 3),
            "send_GBps": round(n_layers * layer_bytes / (t_send * 1e-3) / 1e9, 1)}
        del ks, vs, outs, lw, X, Y, host
        torch.cuda.empty_cache()
    return res


def sweep_workloads(args, dev, flush, peak):
    """Attention alone on the other full-size workloads, and the SM-fraction sweep."""
    import torch

    import paged_decode_attention_02_gb300 as pda
    from paged_decode_attention_02_gb300 import workloads as wl

    out_all = {}
    sms = pda.device_sm_count()
    stream = torch.cuda.current_stream(dev)

    def time_attention(s, cap, nb):
        out = torch.empty_like(s.q)
        wsp = workspace_for(s, cap)
        for _ in range(5):  # 5 warm-up launches, then the median of sweep_iters (50)
            flush()
            attention(s, out, cap, wsp)
        ts = []
        for _ in range(args.sweep_iters):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush()
            a.record(stream)
            attention(s, out, cap, wsp)
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        t = float(np.median([a.elapsed_time(b) for a, b in ts])) * 1e-3
        gbs = nb / t / 1e9
        return {"us": round(t * 1e6, 2), "GBps": round(gbs, 1),
                "frac_of_peak": round(gbs / peak, 4),
                "decode_tokens_per_s_per_layer": round(s.B / t, 1)}

    # One decode step of a single request (its latency, not bandwidth, is what matters):
    # the first request of the 13B-shape and GQA recipes.
    single = {}
    for name in ("llama2_13b_b80", "gqa_skew_b256"):
        s = wl.make_step(wl.get(name), device=dev, B=1)
        r = time_attention(s, 0, step_bytes(s, [])["attention"])
        single[name] = dict(r, context_len=int(s.context_lens_np[0]))
        del s
    out_all["single_request"] = single

    for name in ("tiny", "llama2_7b_b8", "llama2_13b_b80", "sm_sweep_b128", "llama2_13b_b80_fp8",
                 "gqa_skew_b256_fp8", "llama2_13b_b80_nvfp4", "gqa_skew_b256_nvfp4",
                 "gqa_skew_b256_f16", "gqa_skew_b256_bs64"):
        if name == args.config:
            continue
        w = wl.get(name)
        s = wl.make_step(w, device=dev)
        nb = step_bytes(s, [])
        caps = [0] + [int(math.ceil(p / 100 * sms)) for p in w.sm_caps_pct if p < 100]
        res_w = {}
        for cap in caps:
            key = "all_sms" if cap == 0 else f"sm_cap_{cap}"
            res_w[key] = time_attention(s, cap, nb["attention"])
        res_w["bytes"] = nb["attention"]
        if not args.no_cpu_baseline:
            res_w["oracle"] = oracle_legs(w)
        if name == "llama2_7b_b8":
            res_w["host_overhead_per_layer"] = graph_legs(args, s, sms)
        if w.sm_caps_pct:
            res_w["two_streams"] = overlap_legs(args, s, nb["attention"], sms, flush, peak,
                                                res_w["all_sms"]["us"])
        out_all[name] = res_w
        del s
        torch.cuda.empty_cache()
    return out_all


def graph_legs(args, s, sms):
    """Host cost of issuing one decode step (append + attention) per layer, eager through
    the C ABI against a replay of a bucketed CUDA graph, on the Llama-2-7B batch-8 shape of
    the pages' per-layer example. Host us = wall time to issue the step (no sync inside the
    loop); GPU us = device time of the step from CUDA events."""
    import torch

    import paged_decode_attention_02_gb300 as pda
    from paged_decode_attention_02_gb300 import graphs as pg

    dev = s.q.device
    main = torch.cuda.current_stream(dev)
    out = torch.empty_like(s.q)
    ws = pda.alloc_workspace(s.B, s.w.H, s.w.H_kv, s.w.D, s.w.block_size, s.w.torch_dtype, 0,
                             dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    n = 200

    def eager():
        pda.kv_append(s.k_new, s.v_new, s.k_cache, s.v_cache, s.slot_mapping, error_word=err)
        pda.paged_decode_attention(out, s.q, s.k_cache, s.v_cache, s.block_tables,
                                   s.context_lens, s.max_context_len, s.scale, workspace=ws,
                                   error_word=err)

    def measure(fn):
        for _ in range(10):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(main)
        t0 = time.perf_counter()
        for _ in range(n):
            fn()
        host = (time.perf_counter() - t0) / n
        b.record(main)
        torch.cuda.synchronize()
        return {"host_us": round(host * 1e6, 2), "gpu_us": round(a.elapsed_time(b) * 1e3 / n, 2)}

    res = {"eager_per_layer": measure(eager)}
    g = pg.DecodeStepGraphs(s.k_cache, s.v_cache, s.w.H, s.max_blocks, max_local=s.B,
                            max_remote=s.B, interval=max(1, s.B // 2), scale=s.scale,
                            remote_sm_cap=max(1, int(round(0.3 * sms)))).capture()
    part = {"q": s.q, "k_new": s.k_new, "v_new": s.v_new, "slot_mapping": s.slot_mapping,
            "block_tables": s.block_tables, "context_lens": s.context_lens}
    n_r = max(1, int(round(0.3 * s.B)))
    loc = {k: v[n_r:] for k, v in part.items()}
    rem = {k: v[:n_r] for k, v in part.items()}
    for key, (lp, rp) in {"all_local": (part, None),
                          f"{n_r}_of_{s.B}_offloaded": (loc, rem)}.items():
        res[f"graph_stage_per_step_{key}"] = measure(lambda: g.stage(lp, rp))
        bucket = g.stage(lp, rp)
        res[f"graph_replay_per_layer_{key}"] = measure(lambda: g.replay(bucket))
    res["note"] = ("the step's inputs are staged once per step; each layer replays a graph. "
                   "The pages' per-layer figure for this shape (whole layer, A100, vLLM): "
                   "380 us GPU, 1137 us CPU")
    return res


def overlap_legs(args, s, attn_bytes, sms, flush, peak, t_single_us):
    """Local + offloaded attention sharing one GPU: the batch is split into a remote part
    (the first `ratio` of the requests) and a local part, run as two concurrent launches on
    two streams whose SM caps split the GPU in the same ratio. Reports the time of both
    together against one launch of the whole batch on every SM."""
    import torch

    import paged_decode_attention_02_gb300 as pda

    w = s.w
    dev = s.q.device
    main = torch.cuda.current_stream(dev)
    res = {}
    for ratio in (0.3, 0.5, 0.7):
        n_r = int(math.ceil(ratio * s.B))
        cap_r = max(1, int(round(ratio * sms)))
        parts = [(slice(0, n_r), cap_r), (slice(n_r, s.B), max(1, sms - cap_r))]
        legs = []
        for sl, cap in parts:
            q = s.q[sl].contiguous()
            legs.append(dict(q=q, bt=s.block_tables[sl].contiguous(),
                             cl=s.context_lens[sl].contiguous(), out=torch.empty_like(q),
                             cap=cap, stream=torch.cuda.Stream(dev),
                             ws=pda.alloc_workspace(q.shape[0], w.H, w.H_kv, w.D, w.block_size,
                                                    w.torch_dtype, cap, dev)))

        def run():
            for g in legs:
                g["stream"].wait_stream(main)
                pda.paged_decode_attention(g["out"], g["q"], s.k_cache, s.v_cache, g["bt"],
                                           g["cl"], s.max_context_len, s.scale, sm_cap=g["cap"],
                                           workspace=g["ws"], stream=g["stream"])
            for g in legs:
                main.wait_stream(g["stream"])

        for _ in range(3):
            flush()
            run()
        ts = []
        for _ in range(args.sweep_iters):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            flush()
            a.record(main)
            run()
            b.record(main)
            ts.append((a, b))
        torch.cuda.synchronize()
        t = float(np.median([a.elapsed_time(b) for a, b in ts])) * 1e-3
        gbs = attn_bytes / t / 1e9
        res[f"remote_{int(ratio * 100)}pct"] = {
            "remote_requests": n_r, "remote_sms": cap_r, "local_sms": sms - cap_r,
            "us": round(t * 1e6, 2), "GBps": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4),
            "vs_one_launch": round(t_single_us / (t * 1e6), 4)}
    return res


# ------------------------------------------------------------------ reference arm
def run_reference(args, ws, rank):
    """The fp64 CPU oracle on the host cores, on a bounded sample of the same workload."""
    from paged_decode_attention_02_gb300 import workloads as wl

    if rank != 0:
        return None
    w = wl.get(args.config)
    threads = cpu_threads()
    per_step = min(10.0, args.ref_budget_s / max(1, args.steps + args.warmup))
    sample = oracle_sample(w, per_step, threads)
    sb = step_bytes(sample, sample.pack_requests)
    for _ in range(args.warmup):
        oracle_pass(sample, threads)
    times = [oracle_pass(sample, threads) for _ in range(args.steps)]
    t = float(np.mean(times))
    v = round(sb["step"] / t / 1e9, 4)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": sample.B, "H": w.H, "H_kv": w.H_kv, "D": w.D,
                   "block_size": w.block_size, "kv_dtype": w.kv or w.dtype,
                   "context_tokens": sb["tokens"], "pack_requests": len(sample.pack_requests)},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": f"{w.name} recipe with B={sample.B} of {w.B} requests "
                                   f"({sb['tokens']} tokens) per step"},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE, help="workload name or index (1-5)")
    ap.add_argument("--batch", type=int, default=None, help="fewer requests (profiling only)")
    ap.add_argument("--sm-cap", type=int, default=0, help="SMs the attention may use (0: all)")
    ap.add_argument("--no-sweeps", dest="sweeps", action="store_false")
    ap.add_argument("--sweep-iters", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-budget-s", type=float, default=120.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    launched = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != launched:
        print(f"bench.py --gpus {args.gpus}: one process per GPU is needed; launch it as "
              f"python -m torch.distributed.run --nproc-per-node {args.gpus} bench.py "
              f"--gpus {args.gpus} ... (this process sees WORLD_SIZE={launched})",
              file=sys.stderr)
        sys.exit(2)
    ws, rank, local = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, ws, rank)
    else:
        res = run_ours(args, ws, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
