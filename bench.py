#!/usr/bin/env python3
"""Benchmark of the paged decode step (KV GB/s, % of measured HBM peak, KV tokens/s).

One step = the whole hot path over one batch: copy-on-write block copies (when the
workload has them), slot mapping + cache write of every new token (one fused launch),
then decode
attention (plan, split-KV attention, merge) and chunked-prefill attention (when the
workload has a prefill batch).  Default workload: the Llama-3.1-8B-shaped GQA decode
layer (256 sequences, 32 query / 8 KV heads, head dim 128, bf16, block size 16,
lognormal context lengths).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line on rank 0.  `value` is KV bytes read per step / device time per step
(GB/s) with every input resident in HBM; `e2e` repeats the measurement through the same
C-ABI calls with the step's inputs copied from pinned host memory and the output copied
back inside the timed region.  The reference arm (`--impl reference`) times the CPU
oracle on the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import multiprocessing as mp
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "paged decode attention KV GB/s and % of GB300 HBM peak; KV tokens/s"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
# Vendor figure, context only (the roofline uses the measured copy): NVIDIA's public GB300
# NVL72 specification gives up to 576 TB/s of HBM3e bandwidth over its 72 GPUs, 8 TB/s each.
NOMINAL_HBM_GBS = 8000.0
DECODE_SRC = os.path.join(ROOT, "paged_kv_cache_53_gb300", "csrc", "pa_decode.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_traffic.json")
# end-to-end pass: steps shorter than this replay a captured CUDA graph (see run_ours)
GRAPH_STEP_MS = 0.1
# bytes written between steps of the L2-flushed passes (L2: 129 MB)
FLUSH_BYTES = 512 << 20
# GPU cycles of the sleep queued ahead of each back-to-back pass (~100 us): the host
# enqueues the pass's first calls meanwhile, so that the pass does not start with the GPU
# waiting for them.
PASS_LEAD_CYCLES = 200_000


# ------------------------------------------------------------------ accounting
def kv_bytes(step: W.Step) -> int:
    """K and V bytes one decode over the step reads: each context token's K and V row for
    every KV head, once."""
    sh = step.shape
    return int(step.decode.context_lens.astype(np.int64).sum()) * 2 * sh.num_kv_heads * \
        sh.head_dim * sh.elem_bytes


def shared_prefix_saving(step: W.Step):
    """(tokens, blocks) that a decode attending the shared prefix once does not read
    again: the prefix of every sharer after the first."""
    if step.shared_prefix is None:
        return 0, 0
    _, plen, sharers = step.shared_prefix
    extra = max(0, len(sharers) - 1)
    return extra * plen, extra * (plen // step.shape.block_size)


def decode_algorithmic_bytes(step: W.Step, out_bytes: int, shared: bool = False) -> int:
    """Algorithmic HBM bytes of one decode call: KV rows, q, the output, the block-table
    entries walked and the context lengths.  With `shared`, the shared prefix's KV rows
    and block entries count once."""
    sh, b = step.shape, step.decode
    blocks = int(((b.context_lens.astype(np.int64) + sh.block_size - 1) // sh.block_size).sum())
    q = b.num_seqs * sh.num_q_heads * sh.head_dim * sh.elem_bytes
    o = b.num_seqs * sh.num_q_heads * sh.head_dim * out_bytes
    kv = kv_bytes(step)
    if shared:
        tok, blk = shared_prefix_saving(step)
        kv -= tok * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
        blocks -= blk
    return kv + q + o + 4 * blocks + 4 * b.num_seqs


def prefill_useful_flops(step: W.Step) -> int:
    """Causal attention flops of one prefill call: q.k and p.v over every visible
    position of every query token, for every query head (4 * D per pair)."""
    sh, b = step.shape, step.prefill
    q = b.query_lens.astype(np.int64)
    ctx0 = b.context_lens.astype(np.int64) - q
    visible = int((q * ctx0 + q * (q + 1) // 2).sum())
    return 4 * sh.head_dim * sh.num_q_heads * visible


def prefill_algorithmic_bytes(step: W.Step, out_bytes: int) -> int:
    """Bytes a prefill call must move at least: every context position's K and V row of
    its KV head once, the query rows in and the output rows out, the block-table entries
    and lengths."""
    sh, b = step.shape, step.prefill
    ctx = b.context_lens.astype(np.int64)
    kv = int(ctx.sum()) * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
    rows = b.num_new_tokens * sh.num_q_heads * sh.head_dim
    tables = int(((ctx + sh.block_size - 1) // sh.block_size).sum()) * 4 + 8 * b.num_seqs
    return kv + rows * (sh.elem_bytes + out_bytes) + tables


def measured_peaks(kind: str = "hbm"):
    """HBM GB/s, or bf16 dense TFLOP/s (burst or sustained), from the driver's
    measurements."""
    key, fallback = {"hbm": ("hbm_gbs", FALLBACK_HBM_GBS),
                     "tensor": ("bf16_tflops", 1900.0),
                     "tensor_sustained": ("bf16_tflops_sustained", 1700.0)}[kind]
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p[key]), "measured"
    except Exception:
        return fallback, "fallback"


def kernel_source_hash() -> str:
    """Hash of the sources that define the decode kernels (their file, the device helpers
    and the shared declarations): recorded ncu traffic is only reported while it holds."""
    h = hashlib.sha256()
    d = os.path.dirname(DECODE_SRC)
    for f in ("pa_decode.cu", "pa_device.cuh", "pa_internal.h", "pa_launch.h"):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """ncu DRAM bytes per decode-kernel launch for this workload, if they were taken on
    the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
        e = rec.get(workload)
        if e and e.get("source_hash") == kernel_source_hash():
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ ranks
def replica_step(workload: str, rank: int, world: int) -> W.Step:
    """The step rank `rank` serves: the named workload, reseeded per rank so that each
    replica holds its own batch (sequences are independent; no data crosses ranks)."""
    step = W.NAMED[workload]()
    if world > 1:
        step = W.replace(step, seed=step.seed + 1000 * rank)
    return step


def slowest_over_ranks(values, world: int, device=None):
    """Element-wise maximum over all ranks of per-rank times: the slowest rank sets the
    job's time.  The only collective of the bench, outside the timed region."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu().tolist()]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 50):
        self.index = index
        self.period_ms = period_ms
        self.proc = None

    def __enter__(self):
        self.first = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        if self.proc is not None:
            # the timed region starts only once the sampler is up and has read the GPU
            # once, so that its start-up does not fall inside it
            import select
            ready, _, _ = select.select([self.proc.stdout], [], [], 10.0)
            if ready:
                self.first.append(self.proc.stdout.readline())
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            # the sample taken before the timed region is left out
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx,
                "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------------ our arm
def run_ours(args, rank, world, local_rank):
    import torch
    import paged_kv_cache_53_gb300 as pa
    import paged_kv_cache_53_gb300.build as pabuild

    pabuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    step = replica_step(args.workload, rank, world)
    sh = step.shape
    vals = W.make_values(step, dev)
    kc, vc = vals["k_cache"], vals["v_cache"]
    tdt = kc.dtype
    stream = torch.cuda.current_stream(dev)

    meta = {}
    for kind in ("decode", "prefill"):
        b = getattr(step, kind)
        if b is None:
            continue
        meta[kind] = {
            "bt": torch.from_numpy(b.block_tables).to(dev),
            "ctx": torch.from_numpy(b.context_lens).to(dev),
            "cu": torch.from_numpy(b.cu_q_lens).to(dev),
            "slots": torch.empty(b.num_new_tokens, dtype=torch.int64, device=dev),
        }
    pairs = torch.from_numpy(step.cow_pairs).to(dev) if step.cow_pairs is not None else None
    d, p = step.decode, step.prefill
    share = d is not None and step.shared_prefix is not None and args.share_prefix == "on"
    # a plain decode batch takes the fused step call (cache write + decode)
    fused_decode = d is not None and not share and args.decode_append == "on"
    # a batch with both kinds takes the mixed-step call (decode and prefill side by side)
    mixed = fused_decode and p is not None and args.mixed_step == "on"
    if d is not None:
        out_dec = torch.empty((d.num_seqs, sh.num_q_heads, sh.head_dim), dtype=tdt, device=dev)
        if share:
            pblocks, plen, sharers = step.shared_prefix
            meta["decode"]["pblocks"] = torch.from_numpy(pblocks).to(dev)
            meta["decode"]["sharers"] = torch.from_numpy(sharers).to(dev)
            nbytes = pa.decode_shared_prefix_workspace_bytes(
                d.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, d.max_ctx,
                sh.block_size, len(sharers), plen)
        else:
            nbytes = pa.decode_workspace_bytes(d.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                               sh.head_dim, d.max_ctx, sh.block_size)
        ws_dec = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    if p is not None:
        out_pre = torch.empty((p.num_new_tokens, sh.num_q_heads, sh.head_dim), dtype=tdt,
                              device=dev)
        nbytes = pa.prefill_workspace_bytes(p.num_seqs, p.num_new_tokens, p.max_q,
                                            sh.num_q_heads, sh.num_kv_heads, sh.head_dim,
                                            p.max_ctx, sh.block_size)
        ws_pre = torch.empty(max(16, nbytes), dtype=torch.uint8, device=dev)
    q_in = {kind: vals[f"q_{kind}"] for kind in meta}
    launches_per_step = 0

    # a step's inputs and outputs: per batch kind the query, new K/V and table tensors
    resident_io = {kind: {"q": q_in[kind], "kn": vals[f"k_new_{kind}"],
                          "vn": vals[f"v_new_{kind}"], **m} for kind, m in meta.items()}
    resident_io["out"] = {"decode": out_dec if d is not None else None,
                          "prefill": out_pre if p is not None else None}

    def one_step(ev=None, io=None):
        """The whole hot path over one batch; ev = (decode start/end, prefill start/end);
        io = the step's input and output tensors (the resident ones by default)."""
        nonlocal launches_per_step
        io = io or resident_io
        n = 0
        if pairs is not None:
            pa.copy_blocks([kc], [vc], pairs)
            n += 1
        if mixed and ev is None:
            # decode and prefill side by side in one call (the per-call pass runs them as
            # separate calls, so that each has a duration of its own)
            md, mp = io["decode"], io["prefill"]
            pa.mixed_step(
                kc, vc, step.scale,
                decode=dict(out=io["out"]["decode"], q=md["q"], k_new=md["kn"], v_new=md["vn"],
                            block_tables=md["bt"], context_lens=md["ctx"], max_ctx=d.max_ctx,
                            workspace=ws_dec, slots=meta["decode"]["slots"]),
                prefill=dict(out=io["out"]["prefill"], q=mp["q"], k_new=mp["kn"], v_new=mp["vn"],
                             block_tables=mp["bt"], cu_q_lens=mp["cu"], context_lens=mp["ctx"],
                             max_q=p.max_q, max_ctx=p.max_ctx, workspace=ws_pre,
                             slots=meta["prefill"]["slots"]))  # the current stream (captured)
            launches_per_step = n + 7  # decode: cache write, plan, attend, merge; prefill: 3
            return
        for kind in meta:  # slot mapping + cache write, fused
            if kind == "decode" and fused_decode:
                continue  # written by pa_decode_append below
            b, m = getattr(step, kind), io[kind]
            pa.cache_append(m["kn"], m["vn"], kc, vc, m["bt"], m["cu"], m["ctx"], b.max_q,
                            meta[kind]["slots"])
            n += 1
        if d is not None:
            if ev is not None:
                ev[0].record(stream)
            md = io["decode"]
            if fused_decode:
                pa.decode_append(io["out"]["decode"], md["q"], md["kn"], md["vn"], kc, vc,
                                 md["bt"], md["ctx"], d.max_ctx, step.scale, ws_dec,
                                 slots=meta["decode"]["slots"])
                n += 4  # cache write, plan, attend, merge
            elif share:
                pa.decode_shared_prefix(io["out"]["decode"], md["q"], kc, vc, md["bt"], md["ctx"],
                                        d.max_ctx, md["pblocks"], plen, md["sharers"],
                                        step.scale, ws_dec)
                n += 4  # plan, shared prefix, attend, merge
            else:
                pa.decode(io["out"]["decode"], md["q"], kc, vc, md["bt"], md["ctx"], d.max_ctx,
                          step.scale, ws_dec)
                n += 3  # plan, attend, merge
            if ev is not None:
                ev[1].record(stream)
        if p is not None:
            if ev is not None:
                ev[2].record(stream)
            mp = io["prefill"]
            pa.prefill_chunk(io["out"]["prefill"], mp["q"], kc, vc, mp["bt"], mp["cu"], mp["ctx"],
                             p.max_q, p.max_ctx, step.scale, ws_pre)
            if ev is not None:
                ev[3].record(stream)
            n += 2  # plan, attention
        launches_per_step = n

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # warm-up
    for _ in range(args.warmup):
        one_step()
    barrier()
    if pa.get_status() != 0:
        raise RuntimeError("library status word set during warm-up")

    # timed region: inputs resident in HBM.  Two passes of k steps each, under one clock
    # sampler.  The first gives the step time and records nothing between kernels: an event
    # recorded between two launches ends the programmatic-dependent-launch overlap of the
    # kernels on either side of it, which costs ~8 us per step here.  The second records
    # events around each library call, for the per-call durations of the roofline.
    # Every pass times exactly k steps between a barrier and a synchronisation on both
    # sides; passes repeat until --min-timed-s seconds have gone by, so that the clock
    # sampler (one sample per 50 ms) sees the GPU under load, and the median pass is
    # reported.  Then, in turn: passes with events around each library call (per-call
    # durations), and passes whose steps are each preceded by a write of FLUSH_BYTES
    # (outside the events) so that no step finds the previous one's data in L2.
    k = args.steps
    mk = lambda: torch.cuda.Event(enable_timing=True)
    evs = [(mk(), mk(), mk(), mk()) for _ in range(k)]
    fevs = [(mk(), mk()) for _ in range(k)]
    t0, t1, t2, t3 = mk(), mk(), mk(), mk()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_read = torch.ones(FLUSH_BYTES // 8, dtype=torch.int32, device=dev)
    pass_ms, dec_list, pre_list, evented_list, flushed_list = [], [], [], [], []

    def timed_passes(body, seconds, min_passes=3):
        t_start = time.perf_counter()
        n = 0
        while n < min_passes or time.perf_counter() - t_start < seconds:
            barrier()
            body()
            barrier()
            n += 1
        return n

    # each pass is queued behind a short sleep kernel, outside its events, so that the host
    # has queued the first steps when the pass starts (with few steps per pass, the GPU
    # would otherwise wait one step's host latency inside the timed region)
    def plain_pass():
        torch.cuda._sleep(PASS_LEAD_CYCLES)
        t0.record(stream)
        for i in range(k):
            one_step()
        t1.record(stream)
        torch.cuda.synchronize(dev)
        pass_ms.append(t0.elapsed_time(t1))

    def evented_pass():
        torch.cuda._sleep(PASS_LEAD_CYCLES)
        t2.record(stream)
        for i in range(k):
            one_step(evs[i])
        t3.record(stream)
        torch.cuda.synchronize(dev)
        evented_list.append(t2.elapsed_time(t3) / k)
        if d is not None:
            dec_list.extend(e[0].elapsed_time(e[1]) for e in evs)
        if p is not None:
            pre_list.extend(e[2].elapsed_time(e[3]) for e in evs)

    def flushed_pass():
        for i in range(k):
            # the write evicts the step's data; the read then replaces the dirty lines the
            # write left with clean ones, so that no write-back falls inside the next step
            flush.fill_(i & 0xff)
            flush_read.max()
            fevs[i][0].record(stream)
            one_step()
            fevs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        flushed_list.extend(e[0].elapsed_time(e[1]) for e in fevs)

    with ClockSampler(local_rank) as clocks:
        n_plain = timed_passes(plain_pass, args.min_timed_s)
        step_launches = launches_per_step
        n_evented = timed_passes(evented_pass, args.min_timed_s / 4)
        n_flushed = timed_passes(flushed_pass, args.min_timed_s / 4)
    total_ms = float(np.median(pass_ms))
    evented_ms = float(np.median(evented_list))
    dec_ms = float(np.mean(dec_list)) if d is not None else 0.0
    pre_ms = float(np.mean(pre_list)) if p is not None else 0.0
    flushed_ms = float(np.mean(flushed_list))
    del flush, flush_read
    if pa.get_status() != 0:
        raise RuntimeError("library status word set during the timed region")

    # end to end: every step's inputs copied from pinned host memory and its outputs copied
    # back, through a copy stream, with two sets of device buffers so that step i+1's
    # inputs and step i-1's outputs move while step i computes (a serving loop's overlap)
    in_names = {kind: [n for n in ("q", "kn", "vn", "bt", "ctx", "cu", "pblocks", "sharers")
                       if n in resident_io[kind]] for kind in meta}
    out_kinds = [kk for kk in ("decode", "prefill") if resident_io["out"][kk] is not None]

    def packed(tensors, device, pin):
        """One byte buffer holding every tensor at a 256-byte-aligned offset, and views of
        it with the tensors' shapes and dtypes (so that one copy moves them all)."""
        offs, total = [], 0
        for t in tensors:
            offs.append(total)
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
        if pin:
            buf = buf.pin_memory()
        views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                 for o, t in zip(offs, tensors)]
        return buf, views

    in_list = [(kind, n) for kind in in_names for n in in_names[kind]]
    in_src = [resident_io[kind][n] for kind, n in in_list]
    h_buf, h_views = packed(in_src, "cpu", True)
    for v, t in zip(h_views, in_src):
        v.copy_(t.cpu())
    h_in = {kind: {} for kind in in_names}
    for (kind, n), v in zip(in_list, h_views):
        h_in[kind][n] = v
    out_src = [resident_io["out"][kk] for kk in out_kinds]
    d_io, d_bufs, d_outbufs, h_outbufs = [], [], [], []
    for _ in range(2):
        dbuf, dviews = packed(in_src, dev, False)
        io = {kind: {} for kind in in_names}
        for (kind, n), v in zip(in_list, dviews):
            io[kind][n] = v
        obuf, oviews = packed(out_src, dev, False)
        io["out"] = {"decode": None, "prefill": None}
        for kk, v in zip(out_kinds, oviews):
            io["out"][kk] = v
        d_io.append(io)
        d_bufs.append(dbuf)
        d_outbufs.append(obuf)
        h_outbufs.append(packed(out_src, "cpu", True)[0])
    h2d = sum(t.numel() * t.element_size() for h in h_in.values() for t in h.values())
    d2h = sum(t.numel() * t.element_size() for t in out_src)
    ke = max(1, min(k, args.e2e_steps))
    copy_stream = torch.cuda.Stream(dev)
    ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    drained = [torch.cuda.Event(), torch.cuda.Event()]

    def h2d_step(bi):
        with torch.cuda.stream(copy_stream):
            d_bufs[bi].copy_(h_buf, non_blocking=True)
            ready[bi].record(copy_stream)

    # Steps shorter than GRAPH_STEP_MS: the step's launches captured once per buffer set and
    # replayed every step (inputs are read from the buffers at replay time), so that the
    # host keeps ahead of them.  Longer steps are launched directly: each graph replay
    # starts only once the previous one has ended, where direct launches let the next
    # step's first kernel be set up while the previous one finishes.
    graphs = []
    use_graphs = args.graphs == "on" or (args.graphs == "auto" and total_ms / k < GRAPH_STEP_MS)
    if use_graphs:
        for bi in range(2):
            d_bufs[bi].copy_(h_buf)
            one_step(io=d_io[bi])  # the library's one-time set-up happens outside capture
        torch.cuda.synchronize(dev)
        for bi in range(2):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one_step(io=d_io[bi])
            graphs.append(g)
        torch.cuda.synchronize(dev)
        if pa.get_status() != 0:
            raise RuntimeError("library status word set while capturing the step")
    barrier()
    e0, e1 = mk(), mk()
    e0.record(copy_stream)
    for i in range(min(2, ke)):
        h2d_step(i)
    for i in range(ke):
        bi = i % 2
        stream.wait_event(ready[bi])
        if i >= 2:
            stream.wait_event(drained[bi])  # step i-2's outputs have left this buffer
        if graphs:
            graphs[bi].replay()
        else:
            one_step(io=d_io[bi])
        done[bi].record(stream)
        with torch.cuda.stream(copy_stream):
            copy_stream.wait_event(done[bi])
            h_outbufs[bi].copy_(d_outbufs[bi], non_blocking=True)
            drained[bi].record(copy_stream)
        if i + 2 < ke:
            h2d_step(bi)  # after this buffer's outputs left, on the same copy stream
    e1.record(copy_stream)
    barrier()
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / ke
    e2e_how = ("per step: one packed host-to-device copy of the inputs and one device-to-host "
               "copy of the outputs on a copy stream, overlapping the neighbouring steps' "
               "compute (two buffer sets); the step's launches " +
               ("replayed from a CUDA graph" if graphs else "issued from the host"))

    step_ms = total_ms / k
    step_ms, dec_ms, pre_ms, e2e_ms, evented_ms, flushed_ms = slowest_over_ranks(
        [step_ms, dec_ms, pre_ms, e2e_ms, evented_ms, flushed_ms], world, device=dev)

    config = {
        "workload": step.name, "num_q_heads": sh.num_q_heads, "num_kv_heads": sh.num_kv_heads,
        "head_dim": sh.head_dim, "block_size": sh.block_size,
        "cow_copies": int(step.cow_pairs.shape[0]) if step.cow_pairs is not None else 0,
        "parallelism": f"replicas x{world}",
        "timing": (f"step: median of {n_plain} passes of exactly k steps (repeated for at "
                   f"least {args.min_timed_s:g} s), no event between kernels; per-call "
                   f"durations: {n_evented} passes of k steps with events around each call "
                   f"({evented_ms:.5f} ms per step there); L2-flushed: {n_flushed} passes whose "
                   f"steps each follow a {FLUSH_BYTES >> 20} MiB write and a "
                   f"{FLUSH_BYTES >> 21} MiB read outside the events"
                   + ("; the step is one pa_mixed_step call (decode and prefill side by side), "
                      "the per-call pass runs them as separate calls" if mixed else "")),
        "l2_flush": (f"value: inputs larger than L2, no flush between steps; "
                     f"value_l2_flushed: a {FLUSH_BYTES >> 20} MiB write then a "
                     f"{FLUSH_BYTES >> 21} MiB read before every step (events around each step, "
                     "compare with value_evented, which has the events but no flush)"),
    }
    if share:
        config["shared_prefix"] = {"sharers": int(len(sharers)), "prefix_len": int(plen),
                                   "attended": "once per KV head for all sharers"}
    res = {"metric": METRIC, "n_gpus": world, "steps": k, "warmup": args.warmup,
           "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": sh.dtype, "data": "synthetic", "config": config}
    if p is not None:
        flops = prefill_useful_flops(step)
        tpeak, tkind = measured_peaks("tensor")
        pre = {"ms_per_call": round(pre_ms, 5), "useful_gflop": round(flops / 1e9, 2),
               "achieved": round(flops / (pre_ms * 1e-3) / 1e12, 1), "peak": tpeak,
               "peak_kind": tkind, "unit": "TFLOP/s",
               "frac": round(flops / (pre_ms * 1e-3) / 1e12 / tpeak, 4),
               "timing": "CUDA events around each call",
               "tokens": p.num_new_tokens, "max_ctx": p.max_ctx}
        config["prefill_tokens"] = p.num_new_tokens
    if d is not None:
        kvb = kv_bytes(step)
        kv_tokens = int(d.context_lens.astype(np.int64).sum())
        peak, peak_kind = measured_peaks()
        alg = decode_algorithmic_bytes(step, out_dec.element_size(), shared=share)
        if fused_decode:  # the call also reads the new K/V rows, writes them and the slots
            alg += 2 * 2 * d.num_seqs * sh.num_kv_heads * sh.head_dim * sh.elem_bytes + 8 * d.num_seqs
        # a step that is the decode call alone (no copies, no prefill): its back-to-back time
        # is the call's duration as a serving loop sees it; the evented per-call time also
        # carries the lost launch overlap an event between two calls costs
        sole = p is None and pairs is None and fused_decode
        launch_ms = step_ms if sole else dec_ms
        achieved = alg / (launch_ms * 1e-3) / 1e9
        config.update({"num_seqs": d.num_seqs, "kv_tokens_per_step": kv_tokens,
                       "kv_bytes_per_step": kvb, "max_ctx": d.max_ctx,
                       "l2": f"inputs larger than L2: {kvb / 1e9:.2f} GB of KV read per step "
                             "vs 0.13 GB L2"})
        if step.shared_prefix is not None:
            # blocks held once but read by many sequences: the metric counts every reader
            # (logical bytes); the unique bytes are what must come from HBM at least
            tok, _ = shared_prefix_saving(step)
            ukv = kvb - tok * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
            config.update({
                "unique_kv_bytes_per_step": int(ukv),
                "value_kind": "effective (logical bytes, every reader counted; L2-assisted)",
                "l2": f"{kvb / 1e9:.2f} GB logical, {ukv / 1e9:.3f} GB unique KV per step "
                      "vs 0.13 GB L2"})
        res.update({
            "value": round(world * kvb / (step_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "value_l2_flushed": round(world * kvb / (flushed_ms * 1e-3) / 1e9, 1),
            "value_evented": round(world * kvb / (evented_ms * 1e-3) / 1e9, 1),
            "kv_tokens_per_s": round(world * kv_tokens / (step_ms * 1e-3), 1),
            "hbm_frac_of_measured": round(kvb / (step_ms * 1e-3) / 1e9 / peak, 4),
            "hbm_frac_of_nominal": round(kvb / (step_ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
            "e2e": {"value": round(world * kvb / (e2e_ms * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 5), "steps": ke,
                    "how": e2e_how},
            "roofline": {"bound": "hbm",
                         "kernel": ("pa_decode_shared_prefix (plan + shared prefix + attend + "
                                    "merge)" if share else
                                    "pa_decode_append (cache write + plan + attend + merge)"
                                    if fused_decode else "pa_decode (plan + attend + merge)"),
                         "achieved": round(achieved, 1), "peak": peak, "peak_kind": peak_kind,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": None if share else recorded_traffic(args.workload),
                         "algorithmic_bytes": alg,
                         "ms_per_launch": round(launch_ms, 5),
                         "ms_per_launch_evented": round(dec_ms, 5),
                         "timing": ("back-to-back steps (the step is this one call), CUDA "
                                    "events at the pass edges" if sole else
                                    "CUDA events around each call")},
        })
        if p is not None:
            res["prefill"] = pre
            # the step's roofline: the decode call at HBM bandwidth plus the prefill call at
            # the slower of its tensor-core and HBM times
            pf_bytes = prefill_algorithmic_bytes(step, out_pre.element_size())
            t_dec = alg / (peak * 1e9)
            t_pf = max(pre["useful_gflop"] * 1e9 / (pre["peak"] * 1e12), pf_bytes / (peak * 1e9))
            res["step_roofline"] = {
                "ms": round((t_dec + t_pf) * 1e3, 5), "decode_ms": round(t_dec * 1e3, 5),
                "prefill_ms": round(t_pf * 1e3, 5), "prefill_algorithmic_bytes": pf_bytes,
                "frac": round((t_dec + t_pf) * 1e3 / step_ms, 4),
                "how": "decode algorithmic bytes / measured HBM GB/s + max(prefill useful "
                       "flops / measured bf16 TFLOP/s, prefill bytes / measured HBM GB/s), "
                       "over the measured step time"}
    else:  # a prefill-only workload: useful causal TFLOP/s against the tensor roofline
        flops = prefill_useful_flops(step)
        res.update({
            "metric": "chunked-prefill attention useful TFLOP/s",
            "value": round(world * flops / (step_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
            "value_l2_flushed": round(world * flops / (flushed_ms * 1e-3) / 1e12, 1),
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 1), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 5), "steps": ke,
                    "how": e2e_how},
            "roofline": dict(pre, bound="tensor", kernel="pa_prefill_chunk",
                             traffic=recorded_traffic(args.workload)),
        })
    res["clocks"] = clocks.summary()
    res["gpu_launches"] = step_launches * k
    return res, step


# ------------------------------------------------------------------ secondary calls
def _device_inputs(step: W.Step, dev):
    import torch
    vals = W.make_values(step, dev)
    meta = {}
    for kind in ("decode", "prefill"):
        b = getattr(step, kind)
        if b is None:
            continue
        meta[kind] = {"bt": torch.from_numpy(b.block_tables).to(dev),
                      "ctx": torch.from_numpy(b.context_lens).to(dev),
                      "cu": torch.from_numpy(b.cu_q_lens).to(dev)}
    return vals, meta


def _time_call(call, seconds: float, stream, dev, per_pass: int = 20, warmup: int = 5):
    """Device time of `call` (ms), in alternating passes of `per_pass` calls repeated until
    `seconds` have passed, clocks sampled meanwhile: back-to-back passes with one event pair
    around the whole pass (as a serving loop issues its calls: each call's first kernels
    start while the previous call's last ones drain) give the median pass time per call;
    each such pass is queued behind a short sleep kernel, outside its events, so that the
    host has queued its first calls when it starts (else a pass of short calls starts
    with the GPU idle for the host's latency of one call); evented passes, an event pair
    around each call (which ends that overlap), give the mean per-call time.  Returns
    (back-to-back ms, evented ms, calls timed, clocks)."""
    import torch
    mk = lambda: torch.cuda.Event(enable_timing=True)
    for _ in range(warmup):
        call()
    torch.cuda.synchronize(dev)
    evs = [(mk(), mk()) for _ in range(per_pass)]
    t0, t1 = mk(), mk()
    times, passes = [], []
    with ClockSampler(dev.index or 0) as clocks:
        t_start = time.perf_counter()
        while not times or time.perf_counter() - t_start < seconds:
            torch.cuda._sleep(PASS_LEAD_CYCLES)
            t0.record(stream)
            for _ in range(per_pass):
                call()
            t1.record(stream)
            for a, b in evs:
                a.record(stream)
                call()
                b.record(stream)
            torch.cuda.synchronize(dev)
            passes.append(t0.elapsed_time(t1) / per_pass)
            times.extend(a.elapsed_time(b) for a, b in evs)
    return (float(np.median(passes)), float(np.mean(times)), len(times) + per_pass * len(passes),
            clocks.summary())


def run_extras(args, dev):
    """The hot path's other calls on their own workloads, each timed alone after the
    headline (pools built one at a time and freed in turn): the chunked prefill of the
    mixed workload against the tensor roofline, the prefix-sharing decode against HBM on
    its unique bytes, and the OPT-13B-shaped decode step against HBM."""
    import torch
    import paged_kv_cache_53_gb300 as pa
    stream = torch.cuda.current_stream(dev)
    hbm, hbm_kind = measured_peaks()
    tpeak, tkind = measured_peaks("tensor")
    tsus = measured_peaks("tensor_sustained")[0]
    out = {}
    seconds = args.extra_timed_s

    # chunked prefill: 8 chunks of 512 tokens over 0..16,384 tokens of paged context
    step = W.mixed_prefill_only()
    sh, p = step.shape, step.prefill
    vals, meta = _device_inputs(step, dev)
    kc, vc, m = vals["k_cache"], vals["v_cache"], meta["prefill"]
    pa.cache_append(vals["k_new_prefill"], vals["v_new_prefill"], kc, vc, m["bt"], m["cu"],
                    m["ctx"], p.max_q)
    o = torch.empty((p.num_new_tokens, sh.num_q_heads, sh.head_dim), dtype=kc.dtype, device=dev)
    ws = torch.empty(max(16, pa.prefill_workspace_bytes(p.num_seqs, p.num_new_tokens, p.max_q,
                                                        sh.num_q_heads, sh.num_kv_heads,
                                                        sh.head_dim, p.max_ctx, sh.block_size)),
                     dtype=torch.uint8, device=dev)
    ms, ms_ev, n, clk = _time_call(lambda: pa.prefill_chunk(o, vals["q_prefill"], kc, vc, m["bt"],
                                                     m["cu"], m["ctx"], p.max_q, p.max_ctx,
                                                     step.scale, ws), seconds, stream, dev)
    flops = prefill_useful_flops(step)
    tf = flops / (ms * 1e-3) / 1e12
    out["prefill_call"] = {
        "workload": step.name, "call": "pa_prefill_chunk", "ms_per_call": round(ms, 5),
        "ms_per_call_evented": round(ms_ev, 5), "calls_timed": n, "clocks": clk,
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": tpeak,
                     "peak_kind": f"{tkind} bf16 dense, burst", "unit": "TFLOP/s",
                     "frac": round(tf / tpeak, 4), "frac_of_sustained": round(tf / tsus, 4),
                     "useful_gflop": round(flops / 1e9, 2), "traffic": None}}
    del vals, meta, kc, vc, m, o, ws
    torch.cuda.empty_cache()

    # prefix sharing: 128 sequences on one 2,048-token prefix + 8 groups of 4 samples
    step = W.prefix_sharing_cow()
    sh, d = step.shape, step.decode
    vals, meta = _device_inputs(step, dev)
    kc, vc, m = vals["k_cache"], vals["v_cache"], meta["decode"]
    pa.copy_blocks([kc], [vc], torch.from_numpy(step.cow_pairs).to(dev))
    pa.cache_append(vals["k_new_decode"], vals["v_new_decode"], kc, vc, m["bt"], m["cu"],
                    m["ctx"], 1)
    pblocks, plen, sharers = step.shared_prefix
    pb_t, sh_t = torch.from_numpy(pblocks).to(dev), torch.from_numpy(sharers).to(dev)
    o = torch.empty((d.num_seqs, sh.num_q_heads, sh.head_dim), dtype=kc.dtype, device=dev)
    ws = torch.empty(pa.decode_shared_prefix_workspace_bytes(
        d.num_seqs, sh.num_q_heads, sh.num_kv_heads, sh.head_dim, d.max_ctx, sh.block_size,
        len(sharers), plen), dtype=torch.uint8, device=dev)
    ms, ms_ev, n, clk = _time_call(lambda: pa.decode_shared_prefix(o, vals["q_decode"], kc, vc, m["bt"],
                                                            m["ctx"], d.max_ctx, pb_t, plen,
                                                            sh_t, step.scale, ws),
                            seconds, stream, dev)
    alg = decode_algorithmic_bytes(step, o.element_size(), shared=True)
    gbs = alg / (ms * 1e-3) / 1e9
    out["shared_prefix_call"] = {
        "workload": step.name, "call": "pa_decode_shared_prefix", "ms_per_call": round(ms, 5),
        "ms_per_call_evented": round(ms_ev, 5), "calls_timed": n, "clocks": clk,
        "logical_kv_gbs": round(kv_bytes(step) / (ms * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                     "peak_kind": hbm_kind, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "algorithmic_bytes": alg, "traffic": None,
                     "how": "unique bytes: the shared prefix's K/V and block entries once"}}
    del vals, meta, kc, vc, m, o, ws, pb_t, sh_t
    torch.cuda.empty_cache()

    # OPT-13B-shaped decode step (MHA, 40 heads, fp16): cache write + decode in one call
    step = W.opt13b_decode()
    sh, d = step.shape, step.decode
    vals, meta = _device_inputs(step, dev)
    kc, vc, m = vals["k_cache"], vals["v_cache"], meta["decode"]
    o = torch.empty((d.num_seqs, sh.num_q_heads, sh.head_dim), dtype=kc.dtype, device=dev)
    ws = torch.empty(pa.decode_workspace_bytes(d.num_seqs, sh.num_q_heads, sh.num_kv_heads,
                                               sh.head_dim, d.max_ctx, sh.block_size),
                     dtype=torch.uint8, device=dev)
    ms, ms_ev, n, clk = _time_call(lambda: pa.decode_append(o, vals["q_decode"], vals["k_new_decode"],
                                                     vals["v_new_decode"], kc, vc, m["bt"],
                                                     m["ctx"], d.max_ctx, step.scale, ws),
                            seconds, stream, dev)
    alg = decode_algorithmic_bytes(step, o.element_size())
    alg += 2 * 2 * d.num_seqs * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
    gbs = alg / (ms * 1e-3) / 1e9
    out["opt13b_decode_call"] = {
        "workload": step.name, "call": "pa_decode_append", "ms_per_call": round(ms, 5),
        "ms_per_call_evented": round(ms_ev, 5), "calls_timed": n, "clocks": clk,
        "kv_gbs": round(kv_bytes(step) / (ms * 1e-3) / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": hbm,
                     "peak_kind": hbm_kind, "unit": "GB/s", "frac": round(gbs / hbm, 4),
                     "algorithmic_bytes": alg, "traffic": None}}
    del vals, meta, kc, vc, m, o, ws
    torch.cuda.empty_cache()
    if pa.get_status() != 0:
        raise RuntimeError("library status word set while timing the secondary calls")
    return out


# ------------------------------------------------------------------ swap (pre-emption)
def run_swap(args, local_rank):
    """pa_swap_blocks bandwidth: a scattered set of blocks of a Llama-3.1-8B-shaped layer
    (8 KV heads, head dim 128, block 16, bf16: 64 KiB of K+V per block) moved device ->
    page-locked host and back, against one contiguous copy of the same bytes each way
    (the host link's practical peak)."""
    import torch
    import paged_kv_cache_53_gb300 as pa
    import paged_kv_cache_53_gb300.build as pabuild

    pabuild.build()
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    nb_dev, nb_host, h_kv, bs, d = 16384, args.swap_blocks, 8, 16, 128
    g = torch.Generator(device=dev).manual_seed(53_010)
    kc = W.randn((nb_dev, h_kv, bs, d), "bf16", dev, g)
    vc = W.randn((nb_dev, h_kv, bs, d), "bf16", dev, g)
    hk = torch.empty((nb_host, h_kv, bs, d), dtype=torch.bfloat16).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    rng = np.random.default_rng(53_010)
    dev_ids = rng.permutation(nb_dev)[:nb_host].astype(np.int32)
    out_pairs = torch.from_numpy(np.stack([dev_ids, np.arange(nb_host, dtype=np.int32)], 1)).to(dev)
    in_pairs = torch.from_numpy(np.stack([np.arange(nb_host, dtype=np.int32),
                                          rng.permutation(nb_dev)[:nb_host].astype(np.int32)],
                                         1)).to(dev)
    nbytes = 2 * nb_host * h_kv * bs * d * 2  # K and V
    stream = torch.cuda.current_stream(dev)
    mk = lambda: torch.cuda.Event(enable_timing=True)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        a, b = mk(), mk()
        a.record(stream)
        for _ in range(args.steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        return a.elapsed_time(b) / args.steps

    with ClockSampler(local_rank) as clocks:
        t_out = timed(lambda: pa.swap_blocks([kc], [vc], [hk], [hv], out_pairs))
        t_in = timed(lambda: pa.swap_blocks([hk], [hv], [kc], [vc], in_pairs))
        flat_d = kc[:nb_host]
        flat_h = hk
        t_d2h = timed(lambda: (flat_h.copy_(flat_d, non_blocking=True),
                               hv.copy_(vc[:nb_host], non_blocking=True)))
        t_h2d = timed(lambda: (flat_d.copy_(flat_h, non_blocking=True),
                               vc[:nb_host].copy_(hv, non_blocking=True)))
    if pa.get_status() != 0:
        raise RuntimeError("library status word set during the swap measurement")
    gbs = lambda ms: round(nbytes / (ms * 1e-3) / 1e9, 1)
    return {
        "metric": "swap GB/s (device <-> page-locked host, scattered blocks)",
        "value": gbs(t_out), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"swap {nb_host} blocks of 8x16x128 bf16 K+V, one layer",
                   "bytes_per_direction": nbytes},
        "swap_out_ms": round(t_out, 4), "swap_in_ms": round(t_in, 4),
        "swap_out_gbs": gbs(t_out), "swap_in_gbs": gbs(t_in),
        "contiguous_copy_d2h_gbs": gbs(t_d2h), "contiguous_copy_h2d_gbs": gbs(t_h2d),
        "frac_of_contiguous_copy": {"out": round(t_d2h / t_out, 4), "in": round(t_h2d / t_in, 4)},
        "gpu_launches": 2 * args.steps, "clocks": clocks.summary(),
    }


# ------------------------------------------------------------------ block manager (host)
def _blockmgr_trace(bm, n_steps: int, rng_seed: int = 53_020):
    """One serving-like trace through a block manager: 128 requests on a shared
    2,048-token system prompt (prefix caching) plus 8 prompts with 4 samples each, then
    `n_steps` decode steps in which every sequence appends one token and the step's
    copy-on-write pairs, tables and slots are emitted; every 64 steps 16 requests finish
    and 16 new ones arrive.  Returns seconds spent in the decode steps."""
    import time
    rng = np.random.default_rng(rng_seed)
    system = rng.integers(0, 50_000, 2048).tolist()
    live, nxt = [], 0
    for _ in range(128):
        bm.add_sequence(nxt, system + rng.integers(0, 50_000, int(rng.integers(1, 513))).tolist())
        live.append(nxt)
        nxt += 1
    for _ in range(8):
        parent = nxt
        bm.add_sequence(parent, rng.integers(0, 50_000, int(rng.integers(1, 513))).tolist())
        live.append(parent)
        nxt += 1
        for _ in range(3):
            bm.fork(parent, nxt)
            live.append(nxt)
            nxt += 1
    width = 256
    tok = rng.integers(0, 50_000, size=len(live)).tolist()
    t = 0.0
    for step in range(n_steps):
        t0 = time.perf_counter()
        bm.append_tokens_batch(live, tok[:len(live)])
        bm.take_copies()
        bm.block_tables(live, width)
        bm.slot_mapping(live, [1] * len(live))
        t += time.perf_counter() - t0
        if step % 64 == 63:
            for s in live[:16]:
                bm.free_sequence(s)
            live = live[16:]
            for _ in range(16):
                bm.add_sequence(nxt, system + rng.integers(0, 50_000, int(rng.integers(1, 513))).tolist())
                live.append(nxt)
                nxt += 1
    return t


def run_blockmgr(args):
    """Host bookkeeping per decode step of 160 sequences: the C++ block manager against
    the reference block manager on the same trace."""
    import paged_kv_cache_53_gb300.build as pabuild
    pabuild.build()
    from paged_kv_cache_53_gb300.block_manager import BlockManager
    from oracle.block_manager import BlockManager as RefManager  # the reference arm
    nb, steps = 40_000, args.steps
    t_ours = _blockmgr_trace(BlockManager(nb, 16, prefix_caching=True), steps)
    ref_steps = max(1, min(steps, 64))
    t_ref = _blockmgr_trace(RefManager(nb, 16, prefix_caching=True), ref_steps)
    us = lambda t, n: round(t / n * 1e6, 2)
    return {
        "metric": "block manager host time per decode step (160 sequences)",
        "value": us(t_ours, steps), "unit": "us/step", "higher_is_better": False,
        "n_gpus": 0, "steps": steps, "warmup": 0, "dtype": "int32", "data": "synthetic",
        "config": {"workload": "128 requests on a 2,048-token shared prompt + 8 x 4 samples, "
                               "one token each per step, block 16, prefix caching on",
                   "per_step": "append 160 tokens, take copy pairs, emit tables and slots"},
        "cpu_baseline": {"value": us(t_ref, ref_steps), "unit": "us/step", "cores": 1,
                         "kind": "oracle", "sample": f"{ref_steps} steps of the same trace"},
    }


# ------------------------------------------------------------------ oracle (CPU) timing
def _oracle_worker(payload):
    """Runs the oracle decode over one chunk of sequences; returns (seconds, kv tokens)."""
    import oracle
    (q, kc, vc, tables, ctx, scale, dtype) = payload
    t = time.perf_counter()
    oracle.decode_attention(q, kc, vc, tables, ctx, scale, dtype)
    return time.perf_counter() - t, int(ctx.astype(np.int64).sum())


def _oracle_payload(step: W.Step, seqs, gen):
    """The listed sequences of the workload with a pool of just their blocks (random
    values, same shapes and lengths), tables renumbered into that pool."""
    import torch  # noqa: F401
    sh, d = step.shape, step.decode
    ctx = d.context_lens[seqs].astype(np.int32)
    nblk = (ctx.astype(np.int64) + sh.block_size - 1) // sh.block_size
    total = int(nblk.sum())
    kc = W.to_numpy(W.randn((total, sh.num_kv_heads, sh.block_size, sh.head_dim), sh.dtype,
                            "cpu", gen))
    vc = W.to_numpy(W.randn((total, sh.num_kv_heads, sh.block_size, sh.head_dim), sh.dtype,
                            "cpu", gen))
    q = W.to_numpy(W.randn((len(seqs), sh.num_q_heads, sh.head_dim), sh.dtype, "cpu", gen))
    tables = np.full((len(seqs), int(nblk.max())), -1, dtype=np.int32)
    start = 0
    for i, n in enumerate(nblk):
        tables[i, :n] = np.arange(start, start + n)
        start += n
    return (q, kc, vc, tables, ctx, step.scale, sh.dtype)


class OraclePool:
    """A spawned pool of single-threaded workers (started with spawn, so it is safe
    after CUDA is initialised)."""

    def __init__(self, n):
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                               "MKL_NUM_THREADS")}
        for k in keep:
            os.environ[k] = "1"
        try:
            self.pool = mp.get_context("spawn").Pool(n)
            self.pool.map(_noop, range(n))
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def close(self):
        self.pool.close()
        self.pool.join()


def _noop(_):
    import oracle  # noqa: F401
    return 0


def host_cores():
    return min(len(os.sched_getaffinity(0)), 16)


def _oracle_full_pass(name: str):
    """Run in a spawned single-threaded worker: the whole decode batch of workload `name`
    (every sequence, random values of the same shapes and lengths) through the oracle.
    Returns (seconds of oracle work, KV bytes read); generating the inputs is not timed."""
    import torch
    step = W.NAMED[name]()
    gen = torch.Generator().manual_seed(step.seed)
    payload = _oracle_payload(step, list(range(step.decode.num_seqs)), gen)
    secs, toks = _oracle_worker(payload)
    sh = step.shape
    return secs, toks * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes


def single_thread_oracle(names=("opt13b_decode", "llama8b_gqa_decode")):
    """One full single-threaded oracle pass over each named decode workload."""
    pool = OraclePool(1)
    res = {}
    try:
        for name in names:
            secs, nbytes = pool.pool.apply(_oracle_full_pass, (name,))
            res[name] = {"seconds": round(secs, 3), "value": round(nbytes / secs / 1e9, 4),
                         "unit": "GB/s", "kv_bytes": int(nbytes)}
    finally:
        pool.close()
    return res


def _oracle_chunk_pass(args):
    """Run in a spawned single-threaded worker: worker k of n takes every n-th sequence of
    workload `name`'s decode batch, builds its inputs, waits until wall-clock time t_go (so
    that all workers compute at once) and runs the oracle.  Returns (start, end, kv tokens)
    of the oracle's work, in wall-clock seconds."""
    import torch
    name, k, n, t_go = args
    step = W.NAMED[name]()
    gen = torch.Generator().manual_seed(step.seed + 1000 + k)
    payload = _oracle_payload(step, list(range(step.decode.num_seqs))[k::n], gen)
    wait = t_go - time.time()
    if wait > 0:
        time.sleep(wait)
    t0 = time.time()
    _, toks = _oracle_worker(payload)
    return t0, time.time(), toks


def all_core_oracle(cores, names=("opt13b_decode", "llama8b_gqa_decode")):
    """One full oracle pass over each named decode workload on `cores` single-threaded
    workers at once (the batch's sequences dealt round-robin); wall seconds from the first
    worker's start to the last one's end."""
    pool = OraclePool(cores)
    res = {}
    try:
        for name in names:
            t_go = time.time() + 3.0  # after every worker has built its inputs
            out = pool.pool.map(_oracle_chunk_pass, [(name, k, cores, t_go) for k in range(cores)],
                                chunksize=1)
            wall = max(o[1] for o in out) - min(o[0] for o in out)
            sh = W.NAMED[name]().shape
            nbytes = sum(o[2] for o in out) * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
            res[name] = {"seconds": round(wall, 3), "value": round(nbytes / wall / 1e9, 4),
                         "unit": "GB/s", "kv_bytes": int(nbytes), "cores": cores}
    finally:
        pool.close()
    return res


# ---- all-core oracle runs with the inputs resident in the workers ----
_W = {}  # per-worker state of a SyncOraclePool worker (a spawned process)


def _sync_pool_init(barrier, counter):
    _W["barrier"] = barrier
    with counter.get_lock():
        _W["k"] = counter.value
        counter.value += 1


def _oracle_sync_task(args):
    """Worker k of n: builds its share (every n-th of the listed sequences) of workload
    `name`'s decode batch once, waits until all n workers are ready (so that each holds
    exactly one task of the round and all compute at once), then runs the oracle over it
    `reps` times.  Returns (start, end, kv tokens) of the oracle's work, wall-clock."""
    import torch
    name, n, reps, seqs = args
    k = _W["k"]
    key = (name, n, len(seqs), seqs[0] if seqs else -1, seqs[-1] if seqs else -1)
    if _W.get("key") != key:
        step = W.NAMED[name]()
        gen = torch.Generator().manual_seed(step.seed + 1000 + k)
        mine = list(seqs)[k::n]
        _W["payload"] = _oracle_payload(step, mine, gen) if mine else None
        _W["key"] = key
    _W["barrier"].wait(timeout=600)
    t0 = time.time()
    toks = 0
    for _ in range(reps):
        if _W["payload"] is not None:
            toks += _oracle_worker(_W["payload"])[1]
    return t0, time.time(), toks


class SyncOraclePool:
    """n spawned single-threaded workers, each holding its share of the inputs between
    rounds, started together by a barrier: a round's wall time is the oracle's own, with no
    inter-process transfer of inputs inside it."""

    def __init__(self, n):
        ctx = mp.get_context("spawn")
        self.n = n
        keep = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                               "MKL_NUM_THREADS")}
        for k in keep:
            os.environ[k] = "1"
        try:
            self.pool = ctx.Pool(n, initializer=_sync_pool_init,
                                 initargs=(ctx.Barrier(n), ctx.Value("i", 0)))
        finally:
            for k, v in keep.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, name, seqs, reps=1):
        out = self.pool.map(_oracle_sync_task, [(name, self.n, reps, seqs)] * self.n,
                            chunksize=1)
        return max(o[1] for o in out) - min(o[0] for o in out), sum(o[2] for o in out)

    def close(self):
        self.pool.close()
        self.pool.join()


def oracle_sequences(step: W.Step, budget_s: float, cores: int):
    """The decode batch's sequences worth about `budget_s` seconds of oracle work per core
    (the cost of one token measured on one sequence first; the whole batch if it is
    cheaper), and how many times to run them."""
    import torch
    d = step.decode
    gen = torch.Generator().manual_seed(step.seed)
    order = np.random.default_rng(7).permutation(d.num_seqs)
    secs, toks = _oracle_worker(_oracle_payload(step, [int(order[0])], gen))
    want = budget_s * cores * max(1, toks) / max(secs, 1e-9)
    seqs, tok = [], 0
    for s in order:
        if seqs and tok >= want:
            break
        seqs.append(int(s))
        tok += int(d.context_lens[s])
    reps = max(1, int(round(want / max(tok, 1))))
    return sorted(seqs), tok, reps


def cpu_baseline(name: str, step: W.Step, budget_s: float):
    cores = min(host_cores(), step.decode.num_seqs)
    seqs, tok, reps = oracle_sequences(step, budget_s, cores)
    pool = SyncOraclePool(cores)
    try:
        pool.run(name, seqs, 1)  # builds every worker's inputs (untimed)
        wall, toks = pool.run(name, seqs, reps)
    finally:
        pool.close()
    sh = step.shape
    kvb = toks * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
    desc = (f"{len(seqs)} of {step.decode.num_seqs} sequences ({tok} of "
            f"{int(step.decode.context_lens.sum())} KV tokens) of the same workload, {reps}x, "
            f"held by {cores} spawned single-threaded float64 numpy oracle workers started "
            "together (inputs built before the timed round)")
    single = single_thread_oracle()
    single["how"] = ("one full pass of each workload's whole decode batch by one spawned "
                     "single-threaded worker, wall seconds of the oracle's work (input "
                     "generation excluded)")
    allc = all_core_oracle(cores)
    allc["how"] = ("one full pass of each workload's whole decode batch by all workers at "
                   "once (every worker builds its share of the inputs first), wall seconds "
                   "from the first worker's start to the last one's end")
    return {"value": round(kvb / wall / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle", "sample": desc, "seconds": round(wall, 2),
            "single_thread": single, "all_core": allc}


def run_reference(args, world):
    step = W.NAMED[args.workload]()
    cores = min(host_cores(), step.decode.num_seqs)
    per_step = min(2.0, max(0.02, args.ref_total_s / max(1, args.steps + args.warmup)))
    seqs, tok, reps = oracle_sequences(step, per_step, cores)
    pool = SyncOraclePool(cores)
    try:
        pool.run(args.workload, seqs, 1)  # builds every worker's inputs (untimed)
        for _ in range(args.warmup):
            pool.run(args.workload, seqs, reps)
        runs = [pool.run(args.workload, seqs, reps) for _ in range(args.steps)]
    finally:
        pool.close()
    wall = float(np.mean([r[0] for r in runs]))
    sh = step.shape
    kvb = runs[0][1] * 2 * sh.num_kv_heads * sh.head_dim * sh.elem_bytes
    gbs = kvb / wall / 1e9
    workers = cores
    desc = (f"{len(seqs)} of {step.decode.num_seqs} sequences ({tok} of "
            f"{int(step.decode.context_lens.sum())} KV tokens) of the same workload, {reps}x "
            f"per step, held by {cores} spawned single-threaded float64 numpy oracle workers "
            "started together (inputs built before the timed steps)")
    full = kv_bytes(step)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(full / (gbs * 1e9) * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": step.name, "parallelism": "host cores",
                   "sample_seconds_per_step": round(wall, 3)},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": workers,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(W.NAMED), default="llama8b_gqa_decode")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="the k-step timed pass repeats until this many seconds have passed")
    ap.add_argument("--extra-timed-s", type=float, default=0.5,
                    help="seconds of timed calls for each secondary call")
    ap.add_argument("--extras", choices=["on", "off"], default="on",
                    help="on: after the headline, time the prefill, shared-prefix and "
                         "OPT-13B-shaped decode calls on their own workloads")
    ap.add_argument("--mixed-step", choices=["on", "off"], default="on",
                    help="on: a batch of decodes and prefill chunks in one pa_mixed_step call "
                         "(the two side by side on disjoint SMs); off: the calls in turn")
    ap.add_argument("--decode-append", choices=["on", "off"], default="on",
                    help="on: a plain decode batch's cache write and decode in one call "
                         "(pa_decode_append); off: pa_cache_append then pa_decode")
    ap.add_argument("--share-prefix", choices=["on", "off"], default="on",
                    help="workloads with a shared prefix: attend it once for all sharers "
                         "(pa_decode_shared_prefix) or per sequence (pa_decode)")
    ap.add_argument("--cpu-budget-s", type=float, default=2.0,
                    help="seconds per core of oracle work for the cpu_baseline sample")
    ap.add_argument("--ref-total-s", type=float, default=120.0,
                    help="wall seconds the reference arm's timed steps may take in total")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--op", choices=["step", "swap", "blockmgr"], default="step",
                    help="step: the hot path over --workload; swap: pa_swap_blocks bandwidth; "
                         "blockmgr: host block-manager time per decode step")
    ap.add_argument("--swap-blocks", type=int, default=8192)
    ap.add_argument("--graphs", choices=["auto", "on", "off"], default="auto",
                    help="end-to-end steps: replay a captured CUDA graph (on), issue the "
                         "launches from the host (off), or graphs only for steps shorter "
                         "than %.2f ms (auto)" % GRAPH_STEP_MS)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.op == "blockmgr":
        if rank == 0 and args.impl == "ours":
            print(json.dumps(run_blockmgr(args)), flush=True)
        elif rank == 0:
            print(json.dumps({"impl": "reference", "unavailable":
                              "the block-manager measurement reports the reference manager "
                              "in its cpu_baseline"}))
        return 0

    if args.op == "swap":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the swap measurement has no oracle arm (a plain copy)"}))
            return 0
        if rank == 0:
            print(json.dumps(run_swap(args, local_rank)), flush=True)
        return 0

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, world)), flush=True)
        return 0

    # the oracle's worker pool is spawned, so it may start after the GPU is in use
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res, step = run_ours(args, rank, world, local_rank)
    if args.extras == "on" and world == 1 and args.workload == "llama8b_gqa_decode":
        import torch
        res.update(run_extras(args, torch.device("cuda", local_rank)))
    if rank == 0 and not args.no_cpu_baseline and world == 1 and step.decode is not None:
        res["cpu_baseline"] = cpu_baseline(args.workload, step, args.cpu_budget_s)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
