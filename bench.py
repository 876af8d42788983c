#!/usr/bin/env python3
"""Benchmark of the paged decode-attention hot path on GB300.

One step = the whole decode path over one batch: append the step's new K/V
and run paged decode attention with split-KV partitions and their log-sum-exp
merge.  A decode-only batch does both in one call (paged_attention_decode_append:
the decode kernel writes each sequence's new row itself); a mixed batch first
appends its rows through slot_mapping (kv_reshape_and_cache), then runs its
causal chunks (paged_attention_prefill_chunk) and the decodes
(paged_attention_decode).  The two-call form of a decode-only step is reported
alongside (rows.two_call_step).
The metric is KV-read throughput: the logical K+V bytes the attention reads
(sum over sequences of ctx * n_kv * 128 * 2 * 2) per second, with sequences/s
and tokens/s alongside.  The step time is taken over the whole timed loop, with
no event between its steps (an event between two launches costs them their
programmatic-dependent overlap); the per-kernel times come from a separate
pass with CUDA events around each call.  On one GPU the line also carries
`configs`: the same measurement on the other workloads of the five
configurations (70B-shaped long contexts, the head-sharing sweep, the mixed
continuous batch with its prefill chunk, the tiny batch), each with its own
clock record.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own batch
(weak scaling, no collective on the data path); the time is the max over ranks.
``--impl reference`` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_95_gb300 import workloads as W  # noqa: E402

METRIC = "paged decode attn: KV-read HBM GB/s (% of GB300 peak); sequences/s"
DEFAULT_WORKLOAD = "llama3_8b_b64"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ---- distributed plumbing (host side only) ---------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(world_size, backend):
    if world_size <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(value: float, dist, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---- clocks during the timed region -----------------------------------------------

class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons every 100 ms."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, window=None):
        """Median SM clock, max clock and throttle reasons of the samples inside
        `window` (t0, t1) (default: the marked one), +-0.1 s."""
        window = window or self.window
        rows = []
        for ts, line in list(self.samples):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if window and window[0] - 0.1 <= r[0] <= window[1] + 0.1]
        use = inside if inside else rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in use:
            for name, flag in zip(names, r[3][5:9]):
                if flag.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": sorted(reasons), "samples": len(use), "samples_in_timed_region": len(inside)}


# ---- the oracle on host cores (reference arm and cpu_baseline) -----------------------

def oracle_step(wl: W.Workload, batch: W.Batch):
    import oracle  # test infrastructure: only this arm and the cpu_baseline leg call it
    kc, vc = oracle.kv_reshape_and_cache(wl.new_key, wl.new_value, wl.k_cache, wl.v_cache, wl.slot_mapping)
    return oracle.paged_attention(batch.q, batch.cu_q_lens, kc, vc, batch.block_tables, batch.context_lens,
                                  wl.scale, n_q=wl.n_q)


def subset_workload(wl: W.Workload, nseq: int):
    """The first ``nseq`` sequences of the decode batch (their append tokens too)."""
    b = wl.decode
    sub = W.Batch(q=b.q[:nseq], cu_q_lens=b.cu_q_lens[:nseq + 1], block_tables=b.block_tables[:nseq],
                  context_lens=b.context_lens[:nseq])
    w2 = W.Workload(name=wl.name, n_q=wl.n_q, n_kv=wl.n_kv, head_dim=wl.head_dim, block_size=wl.block_size,
                    num_blocks=wl.num_blocks, poison_block=wl.poison_block, k_cache=wl.k_cache, v_cache=wl.v_cache,
                    new_key=wl.new_key[:nseq], new_value=wl.new_value[:nseq], slot_mapping=wl.slot_mapping[:nseq],
                    scale=wl.scale, decode=sub)
    return w2


def time_oracle(wl: W.Workload, budget_s: float, min_reps: int = 1):
    """Time the oracle on a bounded sample of the workload; returns (GB/s, seqs/s, desc, threads, reps)."""
    import oracle
    threads = oracle.num_threads()
    nseq = wl.decode.num_seqs
    # calibrate on a small sample, then size the sample to the budget
    probe = subset_workload(wl, max(1, nseq // 16))
    t0 = time.perf_counter()
    oracle_step(probe, probe.decode)
    tp = time.perf_counter() - t0
    per_seq = tp / probe.decode.num_seqs
    take = int(max(1, min(nseq, budget_s / max(per_seq, 1e-9))))
    sample = subset_workload(wl, take)
    reps, elapsed = 0, 0.0
    while reps < min_reps or elapsed < 0.5 * budget_s:
        t0 = time.perf_counter()
        oracle_step(sample, sample.decode)
        elapsed += time.perf_counter() - t0
        reps += 1
        if elapsed > budget_s:
            break
    per_step = elapsed / reps
    kv = wl.kv_read_bytes(sample.decode)
    desc = (f"{take} of {nseq} sequences of {wl.name} (append + decode attention, fp64 oracle), "
            f"{reps} repetition(s), {per_step:.3f} s each")
    return kv / per_step / 1e9, take / per_step, desc, threads, reps, per_step


# ---- our arm ------------------------------------------------------------------------

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dist = init_dist(world, "nccl")
    from paged_kv_cache_95_gb300 import build as B
    B.build()
    from paged_kv_cache_95_gb300 import pagedkv as P
    P.load_library()

    wl = W.shard_for_rank(args.workload, rank, world)
    batch = wl.decode
    dev = torch.device("cuda", local)

    def up_bf16(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)

    def up_i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    k_cache, v_cache = up_bf16(wl.k_cache), up_bf16(wl.v_cache)
    new_k, new_v, slots = up_bf16(wl.new_key), up_bf16(wl.new_value), up_i32(wl.slot_mapping)
    q, tables, lens = up_bf16(batch.q), up_i32(batch.block_tables), up_i32(batch.context_lens)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    chunk = wl.chunk  # causal prefill chunks of a mixed batch (None for decode-only workloads)
    if chunk is not None:
        cq, ccu, ctab, clen = (up_bf16(chunk.q), up_i32(chunk.cu_q_lens), up_i32(chunk.block_tables),
                               up_i32(chunk.context_lens))
        cout = torch.empty(cq.shape, dtype=torch.bfloat16, device=dev)
        cws = torch.zeros(256, dtype=torch.uint8, device=dev)
        cmax = int(chunk.q_lens.max())
        chunk_flops = _chunk_flops(chunk, wl)
    desc = P.cache_desc(k_cache)
    ws_bytes = P.paged_attention_workspace_size(batch.num_seqs, wl.n_q, batch.max_blocks_per_seq, 0, desc)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    kv_bytes = wl.kv_read_bytes(batch)
    chunk_kv_bytes = wl.kv_read_bytes(chunk) if chunk is not None else 0
    pool_bytes = 2 * k_cache.numel() * 2

    stream = torch.cuda.current_stream(dev)
    # Decode-only batches run the step as one call that appends each sequence's new
    # row inside the decode kernel; a mixed batch appends its chunk rows first.
    fused = chunk is None

    def step(ev=None):
        """One step; `ev` (four CUDA events) splits it into append / chunk / decode."""
        if ev is not None:
            ev[0].record(stream)
        if not fused:
            P.kv_reshape_and_cache(new_k, new_v, k_cache, v_cache, slots)
        if ev is not None:
            ev[1].record(stream)
        if chunk is not None:
            P.paged_attention_prefill_chunk(cout, cq, ccu, cmax, k_cache, v_cache, ctab, clen, wl.scale,
                                            workspace=cws)
        if ev is not None:
            ev[2].record(stream)
        if fused:
            P.paged_attention_decode_append(out, q, new_k, new_v, k_cache, v_cache, tables, lens, wl.scale,
                                            workspace=ws)
        else:
            P.paged_attention_decode(out, q, k_cache, v_cache, tables, lens, wl.scale, workspace=ws)
        if ev is not None:
            ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)

    # The clock sampler runs for the whole bench; each timed region marks its window.
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist)
    torch.cuda.synchronize(dev)
    # A batch whose bytes fit in L2 twice over is timed step by step with L2 flushed
    # (a write larger than L2, then a read) between steps, outside each step's events;
    # a larger one back to back between two events, with nothing recorded in between
    # (an event between two launches would cost them their programmatic-dependent overlap).
    small = kv_bytes + chunk_kv_bytes < 2 * L2_BYTES
    flush = _L2Flush(torch, dev) if small else None
    w0 = time.time()
    total_ms = _timed_loop(torch, stream, step, args.steps, flush)
    w1 = time.time()
    barrier(dist)
    clocks.mark(w0, w1)
    t_max = max_over_ranks(total_ms / 1e3, dist, device=dev)
    ms_per_step = t_max / args.steps * 1e3
    value = world * (kv_bytes + chunk_kv_bytes) * args.steps / t_max / 1e9

    # Per-kernel times from a separate sampled pass (events between the calls).
    nsample = max(20, min(args.steps, 100))
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(nsample)]
    for e in evs:
        if flush is not None:
            flush()
        step(e)
    torch.cuda.synchronize(dev)
    append_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    prefill_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs) if chunk is not None else None
    decode_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
    st = int(ws[:4].view(torch.int32).item()) & 0xFFFFFFFF
    if st:
        raise RuntimeError(f"device status word set during the bench: {st:#x}")

    # ---- end to end through the public API with host buffers ----
    # Every step uploads its inputs from pinned host memory and reads its result
    # back.  A copy stream moves step i+1's inputs and step i's result while step i
    # computes (two device buffer sets, ordered by events), as a serving loop would;
    # all of those copies fall inside the timed region.
    dev_in = [q, new_k, new_v, slots, tables, lens] + ([cq, ccu, ctab, clen] if chunk is not None else [])
    skip_in = {3} if fused else set()  # the slot mapping is not an input of the one-call step
    # A step's inputs travel as one pinned host buffer and one copy (each tensor at a
    # 256-byte offset, viewed in place on both sides): one host call per step instead
    # of one per tensor, so the host keeps ahead of the GPU.
    offs, off = [], 0
    for k_, x in enumerate(dev_in):
        offs.append(off)
        if k_ not in skip_in:
            off += -(-x.numel() * x.element_size() // 256) * 256
    packed_bytes = off

    def views(buf):
        return [buf[o:o + x.numel() * x.element_size()].view(x.dtype).view(x.shape) if k_ not in skip_in else x
                for k_, (o, x) in enumerate(zip(offs, dev_in))]

    h_buf = torch.empty(packed_bytes, dtype=torch.uint8).pin_memory()
    for hv, x in zip(views(h_buf), dev_in):
        if hv is not x:
            hv.copy_(x.cpu())
    d_buf = [torch.empty(packed_bytes, dtype=torch.uint8, device=dev) for _ in range(2)]
    d_set = [views(b) for b in d_buf]
    d_out = [torch.empty_like(out) for _ in range(2)]
    h_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    d_cout = [torch.empty_like(cout) for _ in range(2)] if chunk is not None else None
    hc_out = [torch.empty(cout.shape, dtype=cout.dtype).pin_memory() for _ in range(2)] if chunk is not None else None
    bi = packed_bytes  # the one copy per step: the step's input tensors, each padded to 256 bytes
    bo = h_out[0].numel() * h_out[0].element_size() + (hc_out[0].numel() * hc_out[0].element_size()
                                                        if chunk is not None else 0)
    copy = torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in range(2)]    # set s's inputs are on the device
    ev_comp = [torch.cuda.Event() for _ in range(2)]  # set s's step is computed (inputs free, outputs ready)
    ev_down = [torch.cuda.Event() for _ in range(2)]  # set s's outputs are back on the host (buffers free)

    def upload(i):
        s_ = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(ev_comp[s_])
            d_buf[s_].copy_(h_buf, non_blocking=True)
            ev_up[s_].record(copy)

    def compute(i):
        s_ = i % 2
        d = d_set[s_]
        stream.wait_event(ev_up[s_])
        stream.wait_event(ev_down[s_])
        if fused:
            P.paged_attention_decode_append(d_out[s_], d[0], d[1], d[2], k_cache, v_cache, d[4], d[5], wl.scale,
                                            workspace=ws)
        else:
            P.kv_reshape_and_cache(d[1], d[2], k_cache, v_cache, d[3])
            if chunk is not None:
                P.paged_attention_prefill_chunk(d_cout[s_], d[6], d[7], cmax, k_cache, v_cache, d[8], d[9], wl.scale,
                                                workspace=cws)
            P.paged_attention_decode(d_out[s_], d[0], k_cache, v_cache, d[4], d[5], wl.scale, workspace=ws)
        ev_comp[s_].record(stream)

    def download(i):
        s_ = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(ev_comp[s_])
            h_out[s_].copy_(d_out[s_], non_blocking=True)
            if chunk is not None:
                hc_out[s_].copy_(d_cout[s_], non_blocking=True)
            ev_down[s_].record(copy)

    def e2e_run(n):
        upload(0)
        for i in range(n):
            if i + 1 < n:
                upload(i + 1)
            compute(i)
            download(i)
        stream.wait_event(ev_down[(n - 1) % 2])

    e2e_run(max(args.warmup, 2))
    torch.cuda.synchronize(dev)
    barrier(dist)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # The host enqueues the first steps while the GPU waits (outside the events): a
    # step's copies and events take the host about as long as the GPU takes to run
    # it, so the head start is sized to the step count (≈ 145 µs of GPU spin per
    # step, at most 20 steps) -- without it a short run measures the host's start.
    torch.cuda._sleep(300000 * min(args.steps, 20))
    e0.record(stream)
    copy.wait_event(e0)
    e2e_run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3, dist, device=dev)
    e2e_value = world * (kv_bytes + chunk_kv_bytes) * args.steps / e2e_t / 1e9
    # the result read back in the last step is the device-resident loop's result, bit for bit
    if not torch.equal(h_out[(args.steps - 1) % 2], out.cpu()):
        raise RuntimeError("end-to-end result differs from the device-resident step's result")

    # [kv_cache_write] + (prefill chunk) + paged decode (with the append when fused) + split-KV merge
    nparts = P.paged_attention_decode_partitions(batch.num_seqs, wl.n_q, batch.max_blocks_per_seq, 0, desc)
    launches_per_step = (1 if fused else 2) + (1 if chunk is not None else 0) + (1 if nparts > 1 else 0)

    # the next hot-path rows on the same batch (single-GPU runs; outside the timed region)
    fp8_chunk = None
    if chunk is not None:
        def fp8_chunk(k8, v8, ks, vs):
            """The causal chunks over the FP8 copy of the pool."""
            ms = _time_events(torch, stream, lambda: P.paged_attention_prefill_chunk(
                cout, cq, ccu, cmax, k8, v8, ctab, clen, wl.scale, workspace=cws, k_scale=ks, v_scale=vs), 200)
            return {"avg_launch_ms": round(ms, 5), "tflops": round(chunk_flops / ms / 1e9, 2),
                    "frac_of_bf16": round(chunk_flops / ms / 1e9 / _bf16_peak()[0], 4),
                    "time_vs_bf16_cache": round(ms / prefill_ms, 3)}
    # rows are timed back to back; compare them with the back-to-back step (decode-only batches)
    rows = _row_variants(P, torch, dev, wl, batch, k_cache, v_cache, new_k, new_v, slots, q, tables, lens,
                         ms_per_step if fused else decode_ms, kv_bytes, steps=200, fused=fused,
                         fp8_chunk=fp8_chunk) if world == 1 else None

    if rows is not None and chunk is not None:
        # the causal chunks under a 512-token window (each row sees its newest 512 keys)
        pw = 512
        mpw = _time_events(torch, stream, lambda: P.paged_attention_prefill_chunk(
            cout, cq, ccu, cmax, k_cache, v_cache, ctab, clen, wl.scale, workspace=cws, window=pw), 200)
        fw = _chunk_flops(chunk, wl, window=pw)
        rows["window_prefill"] = {"window": pw, "algorithmic_flops": fw, "avg_launch_ms": round(mpw, 5),
                                  "tflops": round(fw / mpw / 1e9, 2), "frac_of_bf16": round(fw / mpw / 1e9 / _bf16_peak()[0], 4),
                                  "time_vs_unwindowed": round(mpw / prefill_ms, 3)}
    # the other workloads of the five configurations, each timed the same way (one GPU)
    configs = None
    if world == 1 and args.configs:
        del h_buf, d_buf, d_set, d_out, h_out, d_cout, hc_out
        torch.cuda.empty_cache()
        configs = _config_rows(P, torch, dev, clocks, skip=args.workload)
    clocks.stop()

    if rank == 0:
        peak, peak_src = measured_peaks()
        # The dominant kernel's launch time: a decode-only step is one call (the decode
        # kernel with the append, then the merge), so the timed region itself gives it
        # (events around the whole loop); with other kernels in the step (the mixed
        # batch) the sampled pass with events around each call does.
        roof_ms = ms_per_step if fused else decode_ms
        achieved = kv_bytes / (roof_ms / 1e3) / 1e9
        cpu = None
        if world == 1:
            gbs, sps, sdesc, threads, reps, per_step = time_oracle(wl, budget_s=args.cpu_budget)
            cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sdesc}
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic",
            "impl": "ours",
            "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
            "sequences_per_s": round(world * batch.num_seqs * args.steps / t_max, 1),
            "tokens_per_s": round(world * batch.num_seqs * args.steps / t_max, 1),
            "config": dict(_config(wl, batch, kv_bytes + chunk_kv_bytes, pool_bytes, world),
                           partitions_per_sequence=nparts),
            "roofline": {"bound": "hbm",
                         "kernel": ("paged_attention_decode_append (decode kernel with the step's append + split-KV "
                                    "merge kernel)") if fused else
                         "paged_attention_decode (decode kernel + split-KV merge kernel)",
                         "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s",
                         "traffic": _profiled_traffic(args.workload),
                         "bytes_per_launch": kv_bytes, "avg_launch_ms": round(roof_ms, 5),
                         "append_avg_ms": round(append_ms, 5),
                         "timing": ("CUDA events around the timed loop / steps (one step = one call: the decode "
                                    "kernel with the append, then the merge kernel)") if fused else
                         f"CUDA events around each call on {nsample} steps after the timed loop",
                         "avg_call_ms_events_each_call": round(decode_ms, 5)},
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo, "ms_per_step": round(e2e_t / args.steps * 1e3, 5)},
            "prefill": None if chunk is None else _prefill_report(chunk_flops, prefill_ms, chunk, wl),
            "rows": rows,
            "configs": configs,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


class _L2Flush:
    """Evicts L2 between steps: a write larger than L2, then a read of another
    buffer that large, so the written (dirty) lines are written back before the
    next step rather than during it."""

    def __init__(self, torch, dev):
        self.buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        self.rd = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty((), dtype=torch.float32, device=dev)
        self.torch = torch

    def __call__(self):
        self.buf.zero_()
        self.torch.sum(self.rd, 0, out=self.sink)


def _head_start_cycles(steps):
    """GPU spin (cycles) that lets the host enqueue up to 20 steps before a timed region
    (a longer spin slowed a 10000-step loop by 12%)."""
    return 200000 + 150000 * min(steps, 20)


def _timed_loop(torch, stream, fn, steps, flush=None):
    """Total ms of `steps` calls of fn().  Without `flush`: back to back between two
    events.  With it: L2 flushed before every call, outside per-call events."""
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # Keep the GPU busy (outside the events) while the host enqueues the first steps,
        # so the timed region starts with launches queued, not with host launch latency:
        # ≈ 70 µs of spin per step, for up to 20 steps, covers the host's call overhead
        # (a 20-step run otherwise measures the host's start as much as the GPU).
        torch.cuda._sleep(_head_start_cycles(steps))
        a.record(stream)
        for _ in range(steps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev)


def _config_rows(P, torch, dev, clocks, skip=None):
    """Throughput of the five configurations' other workloads on one GPU.

    Structure (contexts, block tables, slots, shared prefix) is each workload's
    own (workloads.py, structure only); q, K/V and the new rows are N(0,1) draws
    rounded to bf16 from a seeded device generator, so building a 1.3 GB pool
    takes milliseconds instead of the host draw's minute.  Each row's timed
    region is sized to about 0.3 s so the clock sampler sees it."""
    peak, _ = measured_peaks()
    bpeak, _ = _bf16_peak()
    stream = torch.cuda.current_stream(dev)
    res = {}
    for name in ("llama3_70b_b8_32k", "llama3_70b_b1_128k", "sweep_mha", "sweep_gqa", "sweep_mqa", "mixed", "tiny"):
        if name == skip:
            continue
        wl = W.make_workload(name, values=False)
        g = torch.Generator(device=dev)
        g.manual_seed(W._FAMILY_SEED[name])

        def randn(*shape):
            return torch.randn(shape, generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)

        def i32(a):
            return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

        b = wl.decode
        B = b.num_seqs
        q = randn(B, wl.n_q, wl.head_dim)  # drawn first: the sweep's three variants share it
        shape = (wl.num_blocks, wl.n_kv, wl.block_size, wl.head_dim)
        kc, vc = randn(*shape), randn(*shape)
        tab, ln = i32(b.block_tables), i32(b.context_lens)
        nk, nv = randn(B, wl.n_kv, wl.head_dim), randn(B, wl.n_kv, wl.head_dim)
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        desc = P.cache_desc(kc)
        ws = torch.zeros(P.paged_attention_workspace_size(B, wl.n_q, b.max_blocks_per_seq, 0, desc),
                         dtype=torch.uint8, device=dev)
        nparts = P.paged_attention_decode_partitions(B, wl.n_q, b.max_blocks_per_seq, 0, desc)
        ctx = b.context_lens.astype(np.int64)
        dec_bytes = int(ctx.sum()) * wl.n_kv * wl.head_dim * 2 * 2
        row = {"n_q": wl.n_q, "n_kv": wl.n_kv, "num_seqs": B, "context_min": int(ctx.min()),
               "context_max": int(ctx.max()), "partitions_per_sequence": nparts}
        ch = wl.chunk
        if ch is None:
            def step():
                P.paged_attention_decode_append(out, q, nk, nv, kc, vc, tab, ln, wl.scale, workspace=ws)
            step_bytes = dec_bytes
        else:
            rows_c = int(ch.cu_q_lens[-1])
            cq, ccu, ctab, clen = (randn(rows_c, wl.n_q, wl.head_dim), i32(ch.cu_q_lens), i32(ch.block_tables),
                                   i32(ch.context_lens))
            cout = torch.empty(cq.shape, dtype=torch.bfloat16, device=dev)
            cws = torch.zeros(256, dtype=torch.uint8, device=dev)
            cmax = int(ch.q_lens.max())
            tk, tv = randn(len(wl.slot_mapping), wl.n_kv, wl.head_dim), randn(len(wl.slot_mapping), wl.n_kv,
                                                                             wl.head_dim)
            sl = i32(wl.slot_mapping)
            step_bytes = dec_bytes + wl.kv_read_bytes(ch)

            def step(ev=None):
                if ev is not None:
                    ev[0].record(stream)
                P.kv_reshape_and_cache(tk, tv, kc, vc, sl)
                if ev is not None:
                    ev[1].record(stream)
                P.paged_attention_prefill_chunk(cout, cq, ccu, cmax, kc, vc, ctab, clen, wl.scale, workspace=cws)
                if ev is not None:
                    ev[2].record(stream)
                P.paged_attention_decode(out, q, kc, vc, tab, ln, wl.scale, workspace=ws)
                if ev is not None:
                    ev[3].record(stream)
        small = step_bytes < 2 * L2_BYTES
        flush = _L2Flush(torch, dev) if small else None
        for _ in range(5):
            step()
        torch.cuda.synchronize()
        probe = _timed_loop(torch, stream, step, 5, flush) / 5
        steps = int(min(20000, max(20, 0.3 / max(probe * 1e-3 * (1.0 if flush is None else 3.0), 1e-6))))
        w0 = time.time()
        total = _timed_loop(torch, stream, step, steps, flush)
        w1 = time.time()
        ms = total / steps
        row.update({"steps": steps, "step_ms": round(ms, 5),
                    "l2": "flushed before every step" if small else "inputs larger than L2; back to back"})
        if ch is None:
            row.update({"kv_read_bytes": dec_bytes, "gbs": round(dec_bytes / ms / 1e6, 2),
                        "frac_of_hbm": round(dec_bytes / ms / 1e6 / peak, 4),
                        "sequences_per_s": round(B / ms * 1e3, 1), "step": "paged_attention_decode_append"})
        else:
            evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(4)) for _ in range(100)]
            for e in evs:
                step(e)
            torch.cuda.synchronize()
            t_app = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
            t_pre = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
            t_dec = statistics.mean(e[2].elapsed_time(e[3]) for e in evs)
            flops = _chunk_flops(ch, wl)
            shared = len(wl.shared_prefix_seqs)
            uniq = dec_bytes - max(0, shared - 1) * 1024 * wl.n_kv * wl.head_dim * 2 * 2
            row.update({"step": "kv_reshape_and_cache + paged_attention_prefill_chunk + paged_attention_decode",
                        "kv_read_bytes": step_bytes, "gbs": round(step_bytes / ms / 1e6, 2),
                        "append_ms": round(t_app, 5),
                        "prefill": {"ms": round(t_pre, 5), "algorithmic_flops": flops,
                                    "tflops": round(flops / t_pre / 1e9, 2),
                                    "frac_of_bf16": round(flops / t_pre / 1e9 / bpeak, 4)},
                        "decode": {"ms": round(t_dec, 5), "logical_bytes": dec_bytes, "unique_bytes": uniq,
                                   "gbs_logical": round(dec_bytes / t_dec / 1e6, 2),
                                   "frac_of_hbm_unique": round(uniq / t_dec / 1e6 / peak, 4)}})
        if name.startswith("llama3_70b"):  # the FP8 cache on the same batch
            nb_ = wl.num_blocks
            k8 = torch.empty(shape, dtype=torch.uint8, device=dev)
            v8 = torch.empty_like(k8)
            ks = torch.empty(shape[:3], dtype=torch.float32, device=dev)
            vs = torch.empty_like(ks)
            all_slots = torch.arange(nb_ * wl.block_size, dtype=torch.int32, device=dev)
            P.kv_reshape_and_cache_fp8(kc.permute(0, 2, 1, 3).reshape(-1, wl.n_kv, wl.head_dim).contiguous(),
                                       vc.permute(0, 2, 1, 3).reshape(-1, wl.n_kv, wl.head_dim).contiguous(),
                                       k8, v8, ks, vs, all_slots)
            ws8 = torch.zeros(P.paged_attention_workspace_size(B, wl.n_q, b.max_blocks_per_seq, 0, P.cache_desc(k8)),
                              dtype=torch.uint8, device=dev)
            m8 = _time_events(torch, stream, lambda: P.paged_attention_decode(out, q, k8, v8, tab, ln, wl.scale,
                                                                              workspace=ws8, k_scale=ks, v_scale=vs),
                              200)
            b8 = int(ctx.sum()) * wl.n_kv * (2 * wl.head_dim + 2 * 4)
            row["fp8_decode"] = {"bytes_per_launch": b8, "avg_launch_ms": round(m8, 5),
                                 "gbs": round(b8 / m8 / 1e6, 2), "frac_of_hbm": round(b8 / m8 / 1e6 / peak, 4)}
            # verify k = 16 draft positions per sequence, bf16 and FP8 caches (the library's route)
            kv16 = 16
            q16 = randn(B * kv16, wl.n_q, wl.head_dim)
            o16 = torch.empty(q16.shape, dtype=torch.bfloat16, device=dev)
            lib = P.load_library()
            for tag, kk, vv, sk, sv in (("verify_k16", kc, vc, None, None), ("fp8_verify_k16", k8, v8, ks, vs)):
                w16 = P.paged_attention_verify(o16, q16, kv16, kk, vv, tab, ln, wl.scale, k_scale=sk, v_scale=sv)
                mv = _time_events(torch, stream, lambda: P.paged_attention_verify(
                    o16, q16, kv16, kk, vv, tab, ln, wl.scale, workspace=w16, k_scale=sk, v_scale=sv), 50)
                on_pre = lib.paged_attention_verify_on_prefill(B, kv16, wl.n_q, ctypes.byref(P.cache_desc(kk)))
                row[tag] = {"q_per_seq": kv16, "avg_launch_ms": round(mv, 5),
                            "tokens_per_s": round(B * kv16 / mv * 1e3, 1),
                            "kernel": "tcgen05 prefill kernel" if on_pre == 1 else "decode kernel",
                            "workspace_bytes": int(w16.numel())}
            del k8, v8, ks, vs, ws8, all_slots, q16, o16
        row["clocks"] = clocks.summary((w0, w1))
        st = int(ws[:4].view(torch.int32).item()) & 0xFFFFFFFF
        if st:
            raise RuntimeError(f"device status word set during the {name} row: {st:#x}")
        res[name] = row
        del kc, vc, q, out, ws
        flush = None
        torch.cuda.empty_cache()
    return res


def _time_events(torch, stream, fn, steps, warmup=3):
    """Mean ms per call of fn() over `steps` calls back to back (two CUDA events on
    `stream` around the whole run, the queue filled first), as the headline loop is
    timed: an event between two calls would cost them their programmatic-dependent
    overlap."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(_head_start_cycles(steps))
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / steps


def _row_variants(P, torch, dev, wl, batch, k_cache, v_cache, new_k, new_v, slots, q, tables, lens, decode_ms,
                  kv_bytes, steps, fused=False, fp8_chunk=None):
    """FP8 cache, sliding window and host block manager on the bench batch
    (``fp8_chunk``: times the workload's prefill chunks over the FP8 pool)."""
    peak, _ = measured_peaks()
    stream = torch.cuda.current_stream(dev)
    B = batch.num_seqs
    ctx = batch.context_lens.astype(np.int64)
    res = {}

    # FP8 (E4M3) pool: the bf16 pool quantised slot by slot by the library's own FP8 append
    nb, n_kv, bs, d = k_cache.shape
    k8 = torch.empty((nb, n_kv, bs, d), dtype=torch.uint8, device=dev)
    v8 = torch.empty_like(k8)
    ks = torch.empty((nb, n_kv, bs), dtype=torch.float32, device=dev)
    vs = torch.empty_like(ks)
    all_slots = torch.arange(nb * bs, dtype=torch.int32, device=dev)
    P.kv_reshape_and_cache_fp8(k_cache.permute(0, 2, 1, 3).reshape(nb * bs, n_kv, d).contiguous(),
                               v_cache.permute(0, 2, 1, 3).reshape(nb * bs, n_kv, d).contiguous(), k8, v8, ks, vs,
                               all_slots)
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    desc8 = P.cache_desc(k8)
    ws8 = torch.zeros(P.paged_attention_workspace_size(B, wl.n_q, batch.max_blocks_per_seq, 0, desc8),
                      dtype=torch.uint8, device=dev)
    ms8 = _time_events(torch, stream, lambda: P.paged_attention_decode(out, q, k8, v8, tables, lens, wl.scale,
                                                                       workspace=ws8, k_scale=ks, v_scale=vs), steps)
    ms8_app = _time_events(torch, stream, lambda: P.kv_reshape_and_cache_fp8(new_k, new_v, k8, v8, ks, vs, slots),
                           steps)
    b8 = int(ctx.sum()) * n_kv * (2 * d + 2 * 4)  # codes of K and V plus their two fp32 scales
    res["fp8_decode"] = {
        "cache": "E4M3 codes + fp32 scale per token and KV head", "bytes_per_launch": b8,
        "avg_launch_ms": round(ms8, 5), "gbs": round(b8 / ms8 / 1e6, 2), "frac_of_hbm": round(b8 / ms8 / 1e6 / peak, 4),
        "sequences_per_s": round(B / ms8 * 1e3, 1), "speedup_vs_bf16_decode": round(decode_ms / ms8, 3),
        "append_avg_ms": round(ms8_app, 5)}
    if fp8_chunk is not None:
        res["fp8_prefill"] = fp8_chunk(k8, v8, ks, vs)
    # FP8 verify with k = 16 draft positions: G * 16 columns per KV head (the FP8 prefill
    # kernel where it is faster than ceil(G * 16 / 8) decode CTAs per KV head)
    k16 = 16
    q16 = torch.randn((B * k16, wl.n_q, d), device=dev).to(torch.bfloat16)
    out16 = torch.empty(q16.shape, dtype=torch.bfloat16, device=dev)
    ws16 = P.paged_attention_verify(out16, q16, k16, k8, v8, tables, lens, wl.scale, k_scale=ks, v_scale=vs)
    ms16 = _time_events(torch, stream, lambda: P.paged_attention_verify(
        out16, q16, k16, k8, v8, tables, lens, wl.scale, workspace=ws16, k_scale=ks, v_scale=vs), steps)
    res["fp8_verify_k16"] = {"q_per_seq": k16, "bytes_per_launch": b8, "avg_launch_ms": round(ms16, 5),
                             "tokens_per_s": round(B * k16 / ms16 * 1e3, 1),
                             "time_vs_one_fp8_decode": round(ms16 / ms8, 3)}

    # sliding window of 1024 tokens: only the visible keys' blocks are read
    win = 1024
    wsw = torch.zeros(P.paged_attention_workspace_size(B, wl.n_q, batch.max_blocks_per_seq, 0, P.cache_desc(k_cache)),
                      dtype=torch.uint8, device=dev)
    msw = _time_events(torch, stream, lambda: P.paged_attention_decode(out, q, k_cache, v_cache, tables, lens,
                                                                       wl.scale, workspace=wsw, window=win), steps)
    bw = int(np.minimum(ctx, win).sum()) * n_kv * 2 * d * 2
    res["window_decode"] = {"window": win, "bytes_per_launch": bw, "avg_launch_ms": round(msw, 5),
                            "gbs": round(bw / msw / 1e6, 2), "frac_of_hbm": round(bw / msw / 1e6 / peak, 4),
                            "sequences_per_s": round(B / msw * 1e3, 1)}

    # multi-token verify: k = 4 draft positions per sequence (causal among them), same K/V bytes as the decode
    kv, gv = 4, wl.n_q // n_kv  # draft positions, group size
    qv = torch.randn((B * kv, wl.n_q, d), device=dev).to(torch.bfloat16)
    outv = torch.empty(qv.shape, dtype=torch.bfloat16, device=dev)
    wsv = P.paged_attention_verify(outv, qv, kv, k_cache, v_cache, tables, lens, wl.scale)
    msv = _time_events(torch, stream, lambda: P.paged_attention_verify(outv, qv, kv, k_cache, v_cache, tables, lens,
                                                                       wl.scale, workspace=wsv), steps)
    res["verify_k4"] = {"q_per_seq": kv, "bytes_per_launch": kv_bytes, "avg_launch_ms": round(msv, 5),
                        "gbs": round(kv_bytes / msv / 1e6, 2), "frac_of_hbm": round(kv_bytes / msv / 1e6 / peak, 4),
                        "tokens_per_s": round(B * kv / msv * 1e3, 1),
                        "time_vs_one_decode": round(msv / decode_ms, 3),
                        "path": "decode kernel" if gv * kv <= 32 or gv > 16 or 128 % gv else
                        "tcgen05 prefill kernel"}

    # host block manager: one decode step of this batch = one appended token per sequence + table emission
    reps = 200
    bm = P.BlockManager(nb + B * (reps // 16 + 2))
    for i, c in enumerate(ctx):
        bm.add(i)
        bm.append(i, int(c))
    ids = np.arange(B, dtype=np.int64)
    width = batch.max_blocks_per_seq + reps // 16 + 2
    t0 = time.perf_counter()
    for _ in range(reps):
        bm.append_batch(ids)
        bm.block_tables(ids, width)
    host_us = (time.perf_counter() - t0) / reps * 1e6
    res["block_manager"] = {"sequences": B, "us_per_step": round(host_us, 2),
                            "note": "host C++ through ctypes: one batched append of a token per sequence + "
                                    "block-table emission"}
    bm.close()

    if fused:  # the same step as two calls: append kernel, then decode (+ merge), both back to back
        out2 = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        ws2 = torch.zeros(P.paged_attention_workspace_size(B, wl.n_q, batch.max_blocks_per_seq, 0,
                                                           P.cache_desc(k_cache)), dtype=torch.uint8, device=dev)

        def two_calls():
            P.kv_reshape_and_cache(new_k, new_v, k_cache, v_cache, slots)
            P.paged_attention_decode(out2, q, k_cache, v_cache, tables, lens, wl.scale, workspace=ws2)

        def one_call():
            P.paged_attention_decode_append(out2, q, new_k, new_v, k_cache, v_cache, tables, lens, wl.scale,
                                            workspace=ws2)
        ms2 = _time_events(torch, stream, two_calls, steps)
        ms1 = _time_events(torch, stream, one_call, steps)
        res["two_call_step"] = {"append_then_decode_ms": round(ms2, 5), "one_call_ms": round(ms1, 5),
                                "one_call_speedup": round(ms2 / ms1, 3)}
    return res


def _chunk_flops(chunk, wl, window: int = 0) -> int:
    """Algorithmic flops of the causal chunks: 4 * n_q * d per visible (query, key) pair
    (row i at position c + i sees c + i + 1 keys, at most `window` of them under a window)."""
    pairs = 0
    for ql, ctx in zip(chunk.q_lens.tolist(), chunk.context_lens.tolist()):
        c = ctx - ql
        pairs += sum(min(c + i + 1, window) if window > 0 else c + i + 1 for i in range(ql))
    return 4 * wl.n_q * wl.head_dim * pairs


def _bf16_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured burst bf16 (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s"


def _prefill_report(flops, ms, chunk, wl):
    peak, src = _bf16_peak()
    tflops = flops / (ms / 1e3) / 1e12
    return {"kernel": "prefill_chunk_kernel (tcgen05)", "algorithmic_flops": flops, "avg_launch_ms": round(ms, 5),
            "tflops": round(tflops, 2), "peak_tflops": peak, "frac": round(tflops / peak, 4), "peak_source": src,
            "rows": int(chunk.cu_q_lens[-1]), "kv_read_bytes": wl.kv_read_bytes(chunk)}


def _config(wl, batch, kv_bytes, pool_bytes, world):
    lens = batch.context_lens
    return {"workload": wl.name, "batch_per_gpu": batch.num_seqs, "global_batch": batch.num_seqs * world,
            "n_q": wl.n_q, "n_kv": wl.n_kv, "head_dim": wl.head_dim, "block_size": wl.block_size,
            "context_min": int(lens.min()), "context_max": int(lens.max()), "context_mean": float(lens.mean()),
            "kv_read_bytes_per_step": kv_bytes, "pool_bytes": pool_bytes, "out_dtype": "bf16",
            "partition": "auto", "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
            "l2": (f"inputs larger than L2: {kv_bytes / 1e6:.0f} MB read per step vs 129 MB L2; no flush"
                   if kv_bytes >= 2 * L2_BYTES else
                   f"{kv_bytes / 1e6:.1f} MB read per step fits in L2 (129 MB) twice over: L2 flushed by a "
                   f"{2 * L2_BYTES / 1e6:.0f} MB write and a {2 * L2_BYTES / 1e6:.0f} MB read before every step, "
                   f"outside the step's events")}


def kernel_source_hash() -> str:
    """Hash of the decode kernel's sources (a profile is stale once they change)."""
    import hashlib
    h = hashlib.sha256()
    for name in ("decode.cu", "decode_core.cuh", "ptx.cuh", "launch.h"):
        with open(os.path.join(ROOT, "paged_kv_cache_95_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _profiled_traffic(workload):
    """dram read+write bytes per decode launch from the committed ncu summary, or
    None when there is none or the kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"decode_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != kernel_source_hash():
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


# ---- reference arm (the oracle on host cores) -----------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return  # rank 0 alone runs the CPU reference
    wl = W.make_workload(args.workload)
    import oracle
    threads = oracle.num_threads()
    nseq = wl.decode.num_seqs
    # size the per-step sample so that warmup + steps fit the budget
    probe = subset_workload(wl, max(1, nseq // 16))
    t0 = time.perf_counter()
    oracle_step(probe, probe.decode)
    per_seq = (time.perf_counter() - t0) / probe.decode.num_seqs
    budget = args.ref_budget / max(1, args.steps + args.warmup)
    take = int(max(1, min(nseq, budget / max(per_seq, 1e-9))))
    sample = subset_workload(wl, take)
    for _ in range(args.warmup):
        oracle_step(sample, sample.decode)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle_step(sample, sample.decode)
        times.append(time.perf_counter() - t0)
    t = sum(times)
    kv = wl.kv_read_bytes(sample.decode)
    value = kv * args.steps / t / 1e9
    sdesc = f"{take} of {nseq} sequences of {wl.name} per step (append + decode attention, fp64 oracle)"
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
        "config": dict(_config(wl, sample.decode, kv, 2 * wl.k_cache.nbytes, 1),
                       l2="fp64 oracle on the host cores (no GPU, no L2 flush)"),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sdesc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "sequences_per_s": round(take * args.steps / t, 3),
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=W.WORKLOAD_NAMES)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--ref-budget", type=float, default=120.0, help="seconds of oracle time for --impl reference")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the rows of the other workloads (one GPU only)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
