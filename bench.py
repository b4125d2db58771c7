#!/usr/bin/env python
"""Decode-step benchmark: KV append + paged decode attention (+ split-K reduce).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl ours|reference]

Prints ONE JSON line (rank 0).  A step is one pass of the whole hot path over
one batch: for every layer, the paged KV append of the new token of each
sequence, the split-K paged decode attention and the split-K reduce.  The
default workload is the large-batch long-context one (128 sequences, contexts
U[4097, 32769], Qwen3-8B attention shape, bf16, ~17 GB pool): it reads ~10.4 GB
per step, far more than the 129 MB L2, so no flush is needed between steps.

With the default workload the line also carries ``rows``: the other four
decode workloads (tiny fp32 MHA, GPT-2 12 layers, Qwen3-8B single stream 36
layers, the continuous-batching mix) and the 8K-token chunked prefill, each
measured in the same process with its own timing, roofline, clocks and
oracle parity (every sequence and layer for the decode rows).  Rows whose
bytes fit in L2 are timed step by step with L2 flushed in between.

``--impl reference`` times the CPU fp64 oracle instead (the baseline arm), on
a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_xs_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode-attn KV GB/s & % of GB300 HBM peak; sequence-steps/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "paged_kv_cache_xs_gb300", "csrc", "paged_decode.cu")


# ------------------------------------------------------------------ byte accounting

def step_bytes(cfg: wl.DecodeConfig, context_lens: torch.Tensor, window: int = 0) -> dict:
    """Algorithmic bytes of one layer of the decode step (per the cost model:
    K and V read once per KV head, not per query head; with a sliding window
    only the tokens inside it)."""
    s = torch.tensor([], dtype=cfg.dtype).element_size()
    n = context_lens.to(torch.int64).clamp(min=0)
    if window > 0:
        n = n.clamp(max=window)
    kv = int(n.sum()) * cfg.Hkv * cfg.D * 2 * s
    q = cfg.B * cfg.Hq * cfg.D * s
    out = cfg.B * cfg.Hq * cfg.D * s
    append = 2 * cfg.B * cfg.Hkv * cfg.D * s * 2
    tables = int(((n + cfg.block_size - 1) // cfg.block_size).sum()) * 4 + 4 * cfg.B
    attn = kv + q + tables
    return {"kv": kv, "attn": attn, "step": attn + out + append}


def hbm_peak() -> tuple[float, str]:
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak(sustained: bool) -> tuple[float, str]:
    """Dense bf16 tensor peak, TFLOP/s: the measured cuBLAS figure (burst for a
    kernel timed alone, sustained for one timed inside a long loop)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        return float(peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else 1900.0), "fallback"


def kernel_traffic(workload: str, variant: str = "") -> int | None:
    """Per-launch DRAM bytes of the attention kernel from the committed ncu
    summary of this workload (and launch variant, e.g. "_sinks_w4096"), if
    it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", f"paged_decode_attn_{workload}{variant}.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    sha = hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]
    m_sha = re.search(r"kernel_source_sha256_16:\s*([0-9a-f]+)", text)
    m_tr = re.search(r"dram_bytes_per_full_launch:\s*([0-9]+)", text)
    if not m_sha or not m_tr or m_sha.group(1) != sha:
        return None
    return int(m_tr.group(1))


# ------------------------------------------------------------------ clocks

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu_index = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        self.marks = []

    def mark(self):
        self.marks.append(time.time())

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]),
                             "power": float(parts[3]) if parts[3] not in ("[N/A]", "") else None,
                             "hw": parts[5], "hw_th": parts[6], "sw_th": parts[7],
                             "pcap": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        load = [r for r in rows if r["power"] is None or r["power"] > 0] or rows
        reasons = set()
        for r in load:
            if r["hw"] == "Active":
                reasons.add("hw_slowdown")
            if r["hw_th"] == "Active":
                reasons.add("hw_thermal_slowdown")
            if r["sw_th"] == "Active":
                reasons.add("sw_thermal_slowdown")
            if r["pcap"] == "Active":
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in load),
                "sm_max_mhz": max(r["max"] for r in load), "reasons": sorted(reasons),
                "samples": len(load),
                "power_w_max": max((r["power"] for r in load if r["power"] is not None),
                                   default=None)}


# ------------------------------------------------------------------ distributed

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
        return rank, world, local, dist
    return rank, world, local, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle leg

def oracle_sample(w: wl.DecodeWorkload, seqs: list[int], layer: int = 0):
    """CPU inputs for the oracle on a subset of sequences: the pre-append
    pages those sequences use (renumbered), their q and new rows."""
    bt = w.block_tables[seqs].cpu()
    lens = w.context_lens[seqs].cpu()
    ids, rows = [], []
    for i in range(len(seqs)):
        p = (int(lens[i]) + 15) // 16
        rows.append(list(range(len(ids), len(ids) + p)))
        ids.extend(bt[i, :p].tolist())
    nbt = torch.full((len(seqs), max(len(r) for r in rows)), -1, dtype=torch.int32)
    for i, r in enumerate(rows):
        nbt[i, :len(r)] = torch.tensor(r, dtype=torch.int32)
    idx = torch.tensor(ids, dtype=torch.long, device=w.k_cache.device)
    sel = torch.tensor(seqs, dtype=torch.long, device=w.q.device)
    return dict(q=w.q[layer].index_select(0, sel).cpu(),
                k_new=w.k_new[layer].index_select(0, sel).cpu(),
                v_new=w.v_new[layer].index_select(0, sel).cpu(),
                k_cache=w.k_cache[layer].index_select(0, idx).cpu(),
                v_cache=w.v_cache[layer].index_select(0, idx).cpu(),
                block_tables=nbt, context_lens=lens, scale=w.scale)


def oracle_step(sample: dict, threads: int, sinks=None, window: int = 0):
    """Append + attention of the sampled sequences in the oracle (with sinks
    and a window: the gpt-oss variant's oracle)."""
    import oracle
    slots = oracle.slot_mapping(sample["block_tables"], sample["context_lens"], 16,
                                sample["k_cache"].shape[0])
    kc, vc = oracle.kv_append(sample["k_new"], sample["v_new"], sample["k_cache"],
                              sample["v_cache"], slots)
    if sinks is not None or window > 0:
        return oracle.paged_decode_sinks(sample["q"], kc, vc, sample["block_tables"],
                                         sample["context_lens"], sample["scale"],
                                         sinks=None if sinks is None else sinks.cpu(),
                                         window=window, nthreads=threads)
    return oracle.paged_decode(sample["q"], kc, vc, sample["block_tables"],
                               sample["context_lens"], sample["scale"], nthreads=threads)


def sample_bytes(cfg, sample, window: int = 0) -> int:
    sub = wl.DecodeConfig(**{**cfg.__dict__, "B": len(sample["context_lens"])})
    return step_bytes(sub, sample["context_lens"], window)["step"]


def pick_sample(w: wl.DecodeWorkload, target_s: float, threads: int, seed: int = 0):
    """Choose a seeded subset of sequences whose oracle step takes about
    target_s seconds on `threads` cores (calibrated on two sequences)."""
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(w.cfg.B, generator=g).tolist()
    cal = oracle_sample(w, order[:min(2, w.cfg.B)])
    t0 = time.perf_counter()
    oracle_step(cal, threads)
    dt = max(time.perf_counter() - t0, 1e-3)
    tokens_cal = int(cal["context_lens"].sum())
    lens = w.context_lens.cpu()
    chosen, tok = [], 0
    budget = target_s / dt * tokens_cal
    for b in order:
        if chosen and tok + int(lens[b]) > budget:
            break
        chosen.append(b)
        tok += int(lens[b])
    return sorted(chosen)


def cpu_baseline(w: wl.DecodeWorkload, target_s: float, gpu_out: torch.Tensor | None = None,
                 sinks=None, window: int = 0):
    """The oracle timed on the host cores on a seeded sample of the workload.
    With gpu_out (layer 0's output of the timed steps, [B, Hq, D]) it also
    returns the largest absolute difference between the GPU output and the
    oracle's on the sampled sequences, against the stated tolerance."""
    threads = len(os.sched_getaffinity(0))
    seqs = pick_sample(w, target_s, threads)
    sample = oracle_sample(w, seqs)
    t0 = time.perf_counter()
    ref = oracle_step(sample, threads, sinks, window)
    dt = time.perf_counter() - t0
    parity = None
    if gpu_out is not None:
        sel = torch.tensor(seqs, dtype=torch.long, device=gpu_out.device)
        got = gpu_out.index_select(0, sel).cpu().double()
        tol = 1e-2 if w.cfg.dtype == torch.bfloat16 else 1e-5
        err = float((got - ref).abs().max()) if got.numel() else 0.0
        parity = {"max_abs_err": err, "tolerance": tol, "ok": bool(err <= tol),
                  "sequences": len(seqs), "reference": "fp64 CPU oracle, same seeded sample"}
    gbs = sample_bytes(w.cfg, sample, window) / dt / 1e9
    # The same oracle on one core, on a smaller sample of its own (a few seconds).
    seqs1 = pick_sample(w, min(target_s, 10.0) / 3.0, 1, seed=1)
    sample1 = oracle_sample(w, seqs1)
    t1 = time.perf_counter()
    oracle_step(sample1, 1, sinks, window)
    dt1 = time.perf_counter() - t1
    gbs1 = sample_bytes(w.cfg, sample1, window) / dt1 / 1e9
    line = {"value": round(gbs, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "seconds": round(dt, 3),
            "sample": f"{len(seqs)} of {w.cfg.B} sequences (seeded), all {w.cfg.Hq} query heads, "
                      f"1 layer: append + fp64 attention over {int(sample['context_lens'].sum())} "
                      f"tokens",
            "single_core": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                            "seconds": round(dt1, 3),
                            "sample": f"{len(seqs1)} of {w.cfg.B} sequences (seeded), "
                                      f"{int(sample1['context_lens'].sum())} tokens"}}
    return line, parity


# ------------------------------------------------------------------ arms

def run_reference(args, rank, world, dist):
    """The oracle as the baseline arm: each step is the fp64 CPU oracle on a
    bounded sample of the workload."""
    if rank != 0:
        return
    cfg = wl.CONFIGS[args.config]
    dev = torch.device("cuda:0") if torch.cuda.is_available() else torch.device("cpu")
    w = wl.make_workload(cfg, device=dev, layers=1)
    threads = len(os.sched_getaffinity(0))
    seqs = pick_sample(w, args.ref_step_seconds, threads)
    sample = oracle_sample(w, seqs)
    del w
    for _ in range(args.warmup):
        oracle_step(sample, threads)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(sample, threads)
    dt = (time.perf_counter() - t0) / args.steps
    gbs = sample_bytes(cfg, sample) / dt / 1e9
    sample_desc = (f"{len(seqs)} of {cfg.B} sequences (seeded) per step, all {cfg.Hq} query heads, "
                   f"1 layer")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
                   "block_size": cfg.block_size, "layers": cfg.layers, "sample": sample_desc},
        "seq_steps_per_s": round(len(seqs) / dt, 3),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample_desc},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


L2_BYTES = 129 * 1024 * 1024  # L2 of one GB300


def measure_decode(args, cfg: wl.DecodeConfig, rank, world, local, dist, *, steps: int,
                   warmup: int, load_seconds: float, sinks_on: bool = False, window: int = 0,
                   partition_tokens: int = 0, with_e2e: bool = True):
    """Time exactly `steps` decode steps of workload `cfg` on this rank
    (weak scaling: every rank its own seeded batch of the same shape) and
    return what the JSON line reports: the slowest rank's time per step, the
    per-launch time of the step kernel, clocks sampled under load, the
    end-to-end time through host buffers (with_e2e) and the objects the
    oracle leg needs (workload, outputs).  A step whose bytes are under the
    L2 size is timed step by step with L2 flushed in between."""
    from paged_kv_cache_xs_gb300.step import CapturedStep, PagedDecodeStep

    dev = torch.device(f"cuda:{local}")
    w = wl.make_workload(cfg, device=dev, seed=cfg.seed + 7919 * rank)
    L = cfg.layers
    sinks = None
    if sinks_on:
        g = torch.Generator(device=dev).manual_seed(cfg.seed + 17)
        sinks = torch.randn(cfg.Hq, generator=g, device=dev).to(cfg.dtype)
    lens_cpu = w.context_lens.cpu()
    win_tokens = int(lens_cpu.clamp(max=window).sum()) if window > 0 else w.total_context_tokens
    fused = args.fused == "on"
    step = PagedDecodeStep(cfg.B, cfg.Hq, cfg.Hkv, cfg.D, w.max_blocks_per_seq, cfg.dtype, dev,
                           total_context_tokens=win_tokens,
                           max_context_len=min(w.max_context_len, window or 1 << 30),
                           partition_tokens=partition_tokens or None,
                           sinks=sinks, window=window, fused=fused)
    out = torch.empty(L, cfg.B, cfg.Hq, cfg.D, dtype=cfg.dtype, device=dev)  # every layer's output
    stream = torch.cuda.current_stream()
    by = step_bytes(cfg, lens_cpu, window)
    bytes_per_step = by["step"] * L

    # Early reads: each launch reads lengths, tables and its first pages while
    # the launch before it (the previous layer's, or the previous step's on
    # these same lengths) finishes; neither writes what is read early.
    early = fused and args.early_reads == "on"

    def one_step(ev=None):
        cur = torch.cuda.current_stream()
        for layer in range(L):
            if fused:  # append + attention + combine: one launch
                step.run(out[layer], w.q[layer], w.k_new[layer], w.v_new[layer],
                         w.k_cache[layer], w.v_cache[layer], w.block_tables, w.context_lens,
                         w.scale, early_reads=early)
                continue
            step.append(w.k_new[layer], w.v_new[layer], w.k_cache[layer], w.v_cache[layer],
                        w.block_tables, w.context_lens)
            if ev is not None:
                ev[layer][0].record(cur)
            step.attend(out[layer], w.q[layer], w.k_cache[layer], w.v_cache[layer],
                        w.block_tables, w.context_lens, w.scale)
            if ev is not None:
                ev[layer][1].record(cur)
            step.reduce(out[layer], w.context_lens)

    # A multi-layer step replays as one CUDA graph (CapturedStep), its
    # launches chained by programmatic dependent launch; a one-layer step is
    # launched directly, where consecutive steps chain the same way.
    use_graph = args.graph == "on" or (args.graph == "auto" and L > 1)
    graph = None
    graph_ev = None
    if use_graph:
        # One CUDA graph per step (all layers).  In the three-launch form the
        # attention launches are bracketed by event-record nodes so their
        # device time is measured; the one-launch step is timed whole.
        if not fused:
            try:
                graph_ev = [[torch.cuda.Event(enable_timing=True, external=True)
                             for _ in range(2)] for _ in range(L)]
            except TypeError:  # a torch without external events: time the graph only
                graph_ev = None
        graph = CapturedStep(lambda: one_step(graph_ev))

    def run_step(ev=None):
        if graph is not None:
            graph.replay()
        else:
            one_step(ev)

    # Inputs smaller than L2 could be served from it by the previous step:
    # flush it (write a buffer twice its size) before every timed step.
    flush_buf = None
    if bytes_per_step < L2_BYTES:
        flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)

    clocks = ClockSampler(local)
    # Warm-up, then keep the GPU loaded for a while so the clock sampler sees it.
    for _ in range(warmup):
        run_step()
    torch.cuda.synchronize()
    t_load = time.time()
    while time.time() - t_load < load_seconds:
        for _ in range(4):
            run_step()
        torch.cuda.synchronize()

    # ---- timed region: exactly `steps` steps
    attn_ev = None if (graph is not None or fused) else [
        [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(L)]
        for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    if flush_buf is None:
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for k in range(steps):
            run_step(None if attn_ev is None else attn_ev[k])
        end.record(stream)
        torch.cuda.synchronize()
        elapsed_ms = start.elapsed_time(end)
    else:
        step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
        for k in range(steps):
            flush_buf.fill_(k)
            step_ev[k][0].record(stream)
            run_step(None if attn_ev is None else attn_ev[k])
            step_ev[k][1].record(stream)
        torch.cuda.synchronize()
        elapsed_ms = sum(a.elapsed_time(b) for a, b in step_ev)
    barrier(dist)
    if attn_ev is not None:
        attn_ms = [e[0].elapsed_time(e[1]) for ev in attn_ev for e in ev]
    elif graph_ev is not None:  # the last replay's attention launches
        attn_ms = [e[0].elapsed_time(e[1]) for e in graph_ev]
    else:
        attn_ms = [elapsed_ms / (steps * L)]
    clock_info = clocks.stop()
    assert step.error_flags() == 0, f"device error flags {step.error_flags()}"
    l2_flushed = flush_buf is not None
    del flush_buf

    max_ms = max_over_ranks(elapsed_ms, dist)
    ms_per_step = max_ms / steps
    res = dict(w=w, out=out, step=step, sinks=sinks, by=by, L=L, fused=fused, early=early,
               graph=graph is not None, bytes_per_step=bytes_per_step, ms_per_step=ms_per_step,
               value=world * bytes_per_step / (ms_per_step * 1e-3) / 1e9,
               seq_steps=world * cfg.B * L / (ms_per_step * 1e-3), attn_ms=attn_ms,
               clocks=clock_info, l2_flushed=l2_flushed, e2e=None,
               cluster=step.cluster_size(fused))
    if not with_e2e:
        return res

    # ---- e2e: the same step fed from pinned host buffers: every step copies that
    # step's inputs (all layers' q and new K/V rows, block tables, lengths) to the
    # device, runs the step (the same graph or launches), and reads every layer's
    # output back.  The KV pools are device-resident state.
    dev_in = (w.q, w.k_new, w.v_new, w.block_tables, w.context_lens)
    host_in = tuple(t.cpu().pin_memory() for t in dev_in)
    hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        for d, h in zip(dev_in, host_in):
            d.copy_(h, non_blocking=True)
        run_step()
        hout.copy_(out, non_blocking=True)
        torch.cuda.current_stream().synchronize()

    for _ in range(2):
        e2e_step()
    barrier(dist)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(steps):
        e2e_step()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist) / steps
    res["e2e"] = {"value": round(world * bytes_per_step / e2e_s / 1e9, 2), "unit": "GB/s",
                  "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "ms_per_step": round(e2e_s * 1e3, 4)}
    return res


def split_config(m: dict) -> dict:
    """How the step kernel split the work: one cluster of `cluster_size` CTAs
    per (sequence, KV head), or the persistent grid's partitions."""
    if m["cluster"]:
        return {"kernel": "cluster", "cluster_size": m["cluster"]}
    return {"kernel": "persistent", "partition_tokens": m["step"].partition_tokens,
            "max_partitions": m["step"].max_partitions}


def decode_roofline(m: dict, traffic=None) -> dict:
    """Roofline object of the step kernel: algorithmic bytes per launch over
    the average launch time, against the measured HBM copy peak."""
    peak, peak_kind = hbm_peak()
    attn_avg_ms = statistics.mean(m["attn_ms"])
    # The fused launch also appends the new rows and writes the output.
    launch_bytes = m["by"]["step"] if m["fused"] else m["by"]["attn"]
    gbs = launch_bytes / (attn_avg_ms * 1e-3) / 1e9
    kernel = "paged_decode_cluster_kernel" if m["cluster"] else "paged_decode_kernel"
    return {"kernel": kernel, "bound": "hbm", "achieved": round(gbs, 1),
            "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_kind": peak_kind,
            "traffic": traffic, "algorithmic_bytes_per_launch": launch_bytes,
            "avg_launch_ms": round(attn_avg_ms, 4)}


def oracle_parity_all(w: wl.DecodeWorkload, out: torch.Tensor, sinks=None, window: int = 0):
    """Every sequence of every layer of the timed output against the oracle
    (append + fp64 attention from the same pools), on all host cores."""
    threads = len(os.sched_getaffinity(0))
    tol = 1e-2 if w.cfg.dtype == torch.bfloat16 else 1e-5
    seqs = list(range(w.cfg.B))
    worst = 0.0
    for layer in range(w.cfg.layers):
        ref = oracle_step(oracle_sample(w, seqs, layer), threads, sinks, window)
        got = out[layer].cpu().double()
        worst = max(worst, float((got - ref).abs().max()) if got.numel() else 0.0)
    return {"max_abs_err": worst, "tolerance": tol, "ok": bool(worst <= tol),
            "sequences": w.cfg.B, "layers": w.cfg.layers,
            "reference": "fp64 CPU oracle, every sequence and layer of the timed output"}


def decode_row(args, idx: int, rank, world, local, dist) -> dict:
    """One workload measured in the same process as the headline line, for
    its `rows` object: the same timing, roofline, clocks and oracle parity."""
    cfg = wl.CONFIGS[idx]
    m = measure_decode(args, cfg, rank, world, local, dist, steps=args.row_steps,
                       warmup=args.warmup, load_seconds=args.row_load_seconds, with_e2e=False)
    peak, peak_kind = hbm_peak()
    row = {
        "workload": cfg.name, "value": round(m["value"], 2), "unit": "GB/s",
        "ms_per_step": round(m["ms_per_step"], 5), "steps": args.row_steps,
        "seq_steps_per_s": round(m["seq_steps"], 1),
        "pct_of_hbm_peak": {"of_measured": round(100 * m["value"] / world / peak, 2),
                            "of_nominal_8TBps": round(100 * m["value"] / world / NOMINAL_HBM_GBS,
                                                      2), "peak_kind": peak_kind},
        "roofline": decode_roofline(m, kernel_traffic(cfg.name) if m["fused"] else None),
        "dtype": "bf16" if cfg.dtype == torch.bfloat16 else "f32",
        "config": {"B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D, "layers": m["L"],
                   "context_tokens": m["w"].total_context_tokens,
                   **split_config(m),
                   "l2": ("flushed before every timed step (a write of twice the L2 size); "
                          "each step timed by its own events") if m["l2_flushed"] else
                         f"inputs larger than L2 ({m['bytes_per_step'] / 1e9:.3f} GB per step)"},
        "gpu_launches": args.row_steps * m["L"] * m["step"].launches_per_step(m["fused"]),
        "cuda_graph": m["graph"], "fused_step": m["fused"], "early_reads": m["early"],
        "clocks": m["clocks"],
    }
    if rank == 0 and not args.no_cpu_baseline:
        row["parity"] = oracle_parity_all(m["w"], m["out"])
    del m
    torch.cuda.empty_cache()
    return row


def run_ours(args, rank, world, local, dist):
    from paged_kv_cache_xs_gb300 import build as xsbuild
    from paged_kv_cache_xs_gb300 import ops

    xsbuild.build()
    ops.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = wl.CONFIGS[args.config]
    if args.batch:
        # The same length distribution with fewer sequences and a pool of
        # just the pages they need (a small case for counter captures).
        cfg = dataclasses.replace(cfg, B=args.batch, pool="needed", pool_arg=1,
                                  name=f"{cfg.name}_b{args.batch}")
    m = measure_decode(args, cfg, rank, world, local, dist, steps=args.steps, warmup=args.warmup,
                       load_seconds=args.load_seconds, sinks_on=args.sinks, window=args.window,
                       partition_tokens=args.partition_tokens, with_e2e=True)
    w, step, sinks, L = m["w"], m["step"], m["sinks"], m["L"]
    fused, early = m["fused"], m["early"]
    line = None
    if rank == 0:
        peak, peak_kind = hbm_peak()
        value = m["value"]
        # The committed DRAM counters were taken on the one-launch step at the
        # heuristic's partition, plain or with sinks and a window (a summary per
        # variant); any other form of the launch reports none.
        variant = (f"_sinks_w{args.window}" if sinks is not None else f"_w{args.window}") \
            if (sinks is not None or args.window > 0) else ""
        traffic = kernel_traffic(cfg.name, variant) if fused and not args.partition_tokens \
            else None
        l2 = ("flushed before every timed step (a write of twice the L2 size); each step timed "
              "by its own events") if m["l2_flushed"] else \
            f"inputs larger than L2 ({m['bytes_per_step'] / 1e9:.2f} GB read per step)"
        line = {
            "metric": METRIC,
            "value": round(value, 2),
            "unit": "GB/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(m["ms_per_step"], 4),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16" if cfg.dtype == torch.bfloat16 else "f32",
            "data": "synthetic (seeded; lengths, shuffled block order and N(0,1) values drawn "
                    "per the workload recipe)",
            "config": {"workload": cfg.name, "B": cfg.B, "Hq": cfg.Hq, "Hkv": cfg.Hkv,
                       "D": cfg.D, "block_size": cfg.block_size, "layers": L,
                       "pool_blocks": w.num_blocks, "context_tokens": w.total_context_tokens,
                       "max_context_len": w.max_context_len,
                       **split_config(m),
                       "sinks": bool(args.sinks), "window": args.window, "l2": l2,
                       "parallelism": f"replicas x{world} (independent batches, no collective)"},
            "seq_steps_per_s": round(m["seq_steps"], 1),
            "pct_of_hbm_peak": {"of_measured": round(100 * value / world / peak, 2),
                                "of_nominal_8TBps": round(100 * value / world / NOMINAL_HBM_GBS,
                                                          2),
                                "peak_kind": peak_kind},
            "roofline": decode_roofline(m, traffic),
            "e2e": m["e2e"],
            "gpu_launches": args.steps * L * step.launches_per_step(fused),
            "cuda_graph": m["graph"],
            "fused_step": fused,
            "early_reads": early,
            "clocks": m["clocks"],
        }
        if not args.no_cpu_baseline:
            # The oracle of the step that ran (with sinks / a window: the gpt-oss
            # variant's), timed on the host and compared with layer 0's output.
            line["cpu_baseline"], parity = cpu_baseline(w, args.cpu_seconds, gpu_out=m["out"][0],
                                                        sinks=sinks, window=args.window)
            line["parity"] = parity
    # The other workloads (and the chunked prefill) measured in this same
    # process, each with its own timing, roofline, clocks and oracle parity.
    want_rows = args.rows == "on" or (args.rows == "auto" and args.config == 4 and
                                      not args.sinks and args.window == 0 and
                                      not args.partition_tokens and not args.batch)
    if want_rows:
        del m, w, step
        torch.cuda.empty_cache()
        rows = {}
        for idx in (0, 1, 2, 3):
            row = decode_row(args, idx, rank, world, local, dist)
            rows[row["workload"]] = row
        # The chunked prefills: 8K tokens in 1K chunks, and 32K in 4K chunks
        # (~7 ms a prefill: fewer timed steps, each still after an L2 flush).
        for tokens, chunk, steps in ((8192, 1024, args.row_steps),
                                     (32768, 4096, max(10, args.row_steps // 10))):
            pre = prefill_measure(args, rank, world, local, dist, tokens=tokens, chunk=chunk,
                                  steps=steps, load_seconds=args.row_load_seconds,
                                  cpu_seconds=args.row_cpu_seconds)
            if pre is not None:
                rows[pre["config"]["workload"]] = pre
        if line is not None:
            line["rows"] = rows
    if line is not None:
        print(json.dumps(line), flush=True)


def run_swap(args, rank, world, local, dist):
    """KV swap row: whole blocks between the device pool and a pinned host
    swap pool (swap-out, swap-in), against the plain DMA rate of the same bytes."""
    from paged_kv_cache_xs_gb300 import build as xsbuild
    from paged_kv_cache_xs_gb300 import ops

    xsbuild.build()
    ops.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = wl.CONFIGS[args.config]
    nb = 262144 if args.config == 4 else 65536
    n = args.swap_blocks
    shape = (nb, cfg.Hkv, cfg.block_size, cfg.D)
    kd = torch.empty(shape, dtype=cfg.dtype, device=dev).normal_()
    vd = torch.empty(shape, dtype=cfg.dtype, device=dev).normal_()
    kh = torch.empty((n,) + shape[1:], dtype=cfg.dtype).pin_memory()
    vh = torch.empty((n,) + shape[1:], dtype=cfg.dtype).pin_memory()
    g = torch.Generator().manual_seed(cfg.seed)
    blocks = torch.randperm(nb, generator=g)[:n]
    out_map = torch.stack([blocks, torch.arange(n)], 1).to(torch.int64).to(dev)
    in_map = torch.stack([torch.arange(n), blocks], 1).to(torch.int64).to(dev)
    moved = 2 * n * kd[0].numel() * kd.element_size()          # K + V bytes per direction
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(fn, reps):  # slowest rank's time per call
        for _ in range(args.warmup):
            fn()
        barrier(dist)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return max_over_ranks(e0.elapsed_time(e1) / reps, dist)

    clocks = ClockSampler(local)
    t_out = timed(lambda: ops.xs_kv_swap(kd, vd, kh, vh, out_map, err_flag=err), args.steps)
    t_in = timed(lambda: ops.xs_kv_swap(kh, vh, kd, vd, in_map, err_flag=err), args.steps)
    clock_info = clocks.stop()
    assert int(err.item()) == 0
    # Reference: one contiguous DMA copy of the same bytes each way.
    flat_d = torch.empty(moved // 2, dtype=torch.uint8, device=dev)
    flat_h = torch.empty(moved // 2, dtype=torch.uint8).pin_memory()
    t_d2h = timed(lambda: flat_h.copy_(flat_d, non_blocking=True), args.steps) * 2
    t_h2d = timed(lambda: flat_d.copy_(flat_h, non_blocking=True), args.steps) * 2
    if rank != 0:
        return
    gbs = lambda ms: moved / (ms * 1e-3) / 1e9
    line = {
        "metric": "KV swap GB/s (device pool <-> pinned host swap pool)",
        "value": round(world * gbs((t_out + t_in) / 2), 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_out + t_in, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if cfg.dtype == torch.bfloat16 else "f32", "data": "synthetic",
        "config": {"workload": f"{cfg.name}_swap", "blocks_per_direction": n,
                   "block_bytes": kd[0].numel() * kd.element_size(), "pool_blocks": nb},
        "swap_out_gbs": round(gbs(t_out), 2), "swap_in_gbs": round(gbs(t_in), 2),
        "dma_copy_d2h_gbs": round(gbs(t_d2h), 2), "dma_copy_h2d_gbs": round(gbs(t_h2d), 2),
        # Bound by the host link, not HBM: the peak is the plain DMA copy of the
        # same bytes over that link, measured in this run (both directions).
        "roofline": {"kernel": "kv_swap_kernel", "bound": "link",
                     "achieved": round(gbs((t_out + t_in) / 2), 2),
                     "peak": round(gbs((t_d2h + t_h2d) / 2), 2), "unit": "GB/s",
                     "frac": round((t_d2h + t_h2d) / (t_out + t_in), 4),
                     "peak_kind": "DMA copy (cudaMemcpyAsync) of the same bytes, this run",
                     "traffic": None},
        "gpu_launches": 2 * args.steps,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = swap_cpu_baseline(kd, vd, kh, vh, blocks,
                                                                 args.cpu_seconds)
    print(json.dumps(line), flush=True)


def swap_cpu_baseline(kd, vd, kh, vh, blocks, target_s: float):
    """The oracle's swap-out (block copies between two host pools) timed on a
    seeded sample of the swapped blocks, repeated for about target_s / 4
    seconds; and a bit-exact check of the GPU's swap-out of those blocks
    against the oracle's."""
    import oracle
    g = torch.Generator().manual_seed(11)
    n = blocks.numel()
    pick = torch.randperm(n, generator=g)[:min(n, 1024)]
    src_k = kd.index_select(0, blocks[pick].to(kd.device)).cpu()
    src_v = vd.index_select(0, blocks[pick].to(vd.device)).cpu()
    m = len(pick)
    mapping = torch.stack([torch.arange(m), torch.arange(m)], 1).to(torch.int64)
    dst_k, dst_v = torch.zeros_like(src_k), torch.zeros_like(src_v)
    reps, t0 = 0, time.perf_counter()
    while True:
        ek, ev = oracle.kv_swap(src_k, src_v, dst_k, dst_v, mapping)
        reps += 1
        dt = time.perf_counter() - t0
        if dt >= target_s / 4:
            break
    moved = 2 * m * src_k[0].numel() * src_k.element_size()
    got_k, got_v = kh[pick], vh[pick]
    exact = bool(torch.equal(got_k.view(torch.int16), ek.view(torch.int16)) and
                 torch.equal(got_v.view(torch.int16), ev.view(torch.int16)))
    base = {"value": round(moved * reps / dt / 1e9, 3), "unit": "GB/s", "cores": 1,
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"{m} of {n} swapped blocks (seeded), K and V, host pool to host pool, "
                      f"{reps} repetitions"}
    parity = {"bit_exact": exact, "blocks": m, "reference": "oracle swap-out of the same blocks"}
    return base, parity


def run_alloc(args, rank, world, local, dist):
    """Device page allocator row: every step, one launch advances each of the
    workload's sequences by one token and pops a free block for each token
    that starts a page; the oracle replays the same steps on its own copy."""
    from paged_kv_cache_xs_gb300 import build as xsbuild
    from paged_kv_cache_xs_gb300 import ops

    xsbuild.build()
    ops.load()
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    cfg = wl.CONFIGS[args.config]
    bs = cfg.block_size
    gen = torch.Generator().manual_seed(cfg.seed + 7919 * rank)
    hist = wl.draw_history(cfg, gen)                      # tokens already in the cache
    nsteps = args.warmup + args.steps
    width = int((hist.max() + nsteps + bs - 1) // bs) + 1  # room for every step's growth
    pages = [(int(n) + bs - 1) // bs for n in hist.tolist()]
    need = sum(pages) + cfg.B * ((nsteps + bs - 1) // bs + 1)
    nb = max(2 * need, 1024)
    perm = torch.randperm(nb, generator=gen).to(torch.int32)
    bt = torch.full((cfg.B, width), -1, dtype=torch.int32)
    pos = 0
    for b, p in enumerate(pages):
        bt[b, :p] = perm[pos:pos + p]
        pos += p
    stack, top0 = perm[pos:].clone(), nb - pos
    dbt, dlens = bt.to(dev), hist.to(dev)
    dstack = stack.to(dev)
    dtop = torch.tensor([top0], dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    step = lambda: ops.xs_block_alloc_decode(dbt, dlens, dstack, dtop, block_size=bs,
                                             err_flag=err)
    # Eager warm-up, then the K timed steps as one CUDA graph (the allocator
    # runs inside a captured decode step; eager launches from Python would
    # time the host's launch path instead).  Capture executes nothing.
    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(args.steps):
            step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist)
    torch.cuda.synchronize()
    e0.record()
    graph.replay()
    e1.record()
    torch.cuda.synchronize()
    clock_info = clocks.stop()
    if clock_info is not None:
        clock_info["note"] = "the timed replay is shorter than the sampling interval"
    us = max_over_ranks(e0.elapsed_time(e1) * 1e3 / args.steps, dist)  # slowest rank
    assert int(err.item()) == 0, f"device error flags {int(err.item())}"
    if rank != 0:
        return
    line = {
        "metric": "device page allocation (sequence-steps/s; one launch per decode step)",
        "value": round(world * cfg.B / (us * 1e-6), 1), "unit": "sequence-steps/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us / 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": f"{cfg.name}_alloc", "B": cfg.B, "block_size": bs,
                   "pool_blocks": nb, "max_blocks_per_seq": width},
        "roofline": {"kernel": "block_alloc_decode_kernel", "bound": "latency",
                     "achieved": round(us, 3), "peak": None, "unit": "us per launch",
                     "note": "a few hundred bytes per launch (lengths, popped ids, table "
                             "entries): one dependent load / atomic / store chain; "
                             "no bandwidth or compute roofline applies", "traffic": None},
        "gpu_launches": args.steps,
        "cuda_graph": True,
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = alloc_cpu_baseline(
            bt, hist, stack, top0, nsteps, bs, dbt.cpu(), dlens.cpu(), int(dtop.item()))
    print(json.dumps(line), flush=True)


def alloc_cpu_baseline(bt, lens, stack, top, nsteps: int, bs: int, gbt, glens, gtop: int):
    """The oracle's allocation over the same steps from the same state, timed
    on one host core, and compared with the device's result.  Which popped
    block went to which sequence depends on the order of the atomics, so what
    is unique is compared (lengths, stack top, the set of blocks in use), and
    every table must hold each block once and cover its length."""
    import oracle
    obt, olens, otop = bt, lens, top
    t0 = time.perf_counter()
    for _ in range(nsteps):
        obt, olens, otop, _ = oracle.block_alloc_decode(obt, olens, bs, stack, otop)
    dt = time.perf_counter() - t0
    B = lens.numel()
    used_gpu = sorted(int(x) for x in gbt[gbt >= 0].tolist())
    used_cpu = sorted(int(x) for x in obt[obt >= 0].tolist())
    covered = all(int((gbt[b] >= 0).sum()) == (max(int(glens[b]), 0) + bs - 1) // bs
                  for b in range(B))
    exact = bool(torch.equal(glens, olens) and gtop == otop and used_gpu == used_cpu and
                 len(set(used_gpu)) == len(used_gpu) and covered)
    base = {"value": round(B * nsteps / dt, 1), "unit": "sequence-steps/s", "cores": 1,
            "kind": "oracle", "seconds": round(dt, 3),
            "sample": f"all {B} sequences, {nsteps} steps"}
    parity = {"exact": exact, "steps": nsteps,
              "compared": "lengths, stack top and the set of blocks in use equal the oracle's; "
                          "no block twice; every table covers its length"}
    return base, parity


def run_prefill(args, rank, world, local, dist):
    """Chunked-prefill row: one Qwen3-8B-shaped sequence prefilled in chunks
    (append + causal paged attention per chunk), timed per chunk."""
    from paged_kv_cache_xs_gb300 import build as xsbuild
    from paged_kv_cache_xs_gb300 import ops

    xsbuild.build()
    ops.load()
    torch.cuda.set_device(torch.device(f"cuda:{local}"))
    line = prefill_measure(args, rank, world, local, dist, tokens=args.prefill_tokens,
                           chunk=args.prefill_chunk, steps=args.steps,
                           load_seconds=args.load_seconds, cpu_seconds=args.cpu_seconds,
                           impl=args.prefill_impl)
    if line is not None:
        print(json.dumps(line), flush=True)


def prefill_measure(args, rank, world, local, dist, *, tokens: int, chunk: int, steps: int,
                    load_seconds: float, cpu_seconds: float, impl: str = "tensor"):
    """Time `steps` prefills of one Qwen3-8B-shaped sequence of `tokens`
    tokens in `chunk`-token chunks; returns the line (rank 0) or None."""
    from paged_kv_cache_xs_gb300 import ops

    dev = torch.device(f"cuda:{local}")
    Hq, Hkv, D, bs = 32, 8, 128, 16
    dtype = torch.bfloat16
    total = tokens
    pages = (total + bs - 1) // bs
    g = torch.Generator(device=dev).manual_seed(2000 + rank)
    ids = torch.randperm(pages * 2, generator=g, device=dev)[:pages].to(torch.int32)
    kc = torch.empty(pages * 2, Hkv, bs, D, dtype=dtype, device=dev).normal_(generator=g)
    vc = torch.empty_like(kc).normal_(generator=g)
    ks = torch.randn(Hkv, total, D, generator=g, device=dev).to(dtype)
    vs = torch.randn(Hkv, total, D, generator=g, device=dev).to(dtype)
    q = torch.randn(total, Hq, D, generator=g, device=dev).to(dtype)
    wss = {}
    tensor = impl == "tensor"
    nchunks = (total + chunk - 1) // chunk
    ks_c = [ks[:, s0:s0 + chunk].contiguous() for s0 in range(0, total, chunk)]
    vs_c = [vs[:, s0:s0 + chunk].contiguous() for s0 in range(0, total, chunk)]
    out = torch.empty(total, Hq, D, dtype=dtype, device=dev)
    # XS_PREFILL_OVERLAP: chunk c + 1's append and the start of its attention
    # run beside chunk c's attention (the launches follow one another with
    # nothing between them on the stream).
    overlap = tensor and args.prefill_overlap == "on"

    def prefill_all(ev=None):
        ov = overlap and ev is None  # (events between the launches would serialise them)
        for c, start in enumerate(range(0, total, chunk)):
            T = min(chunk, total - start)
            ops.xs_prefill_append(ks_c[c], vs_c[c], kc, vc, ids, start, overlap=ov)
            if ev is not None:
                ev[c][0].record()
            if tensor:
                ops.xs_paged_prefill_tc(out[start:start + T], q[start:start + T], kc, vc, ids,
                                        start, D ** -0.5, overlap=ov)
            else:
                ws = wss.get(T)
                if ws is None:
                    ws = wss[T] = ops.DecodeWorkspace(T, Hq, Hkv, D, pages, dev,
                                                      total_context_tokens=T * (start + T),
                                                      max_context_len=total, fused=False)
                ops.xs_paged_prefill(out[start:start + T], ws.part_o, ws.part_m, ws.part_l,
                                     q[start:start + T], kc, vc, ids, start, D ** -0.5,
                                     ws.partition_tokens, ws.max_partitions,
                                     work_counters=ws.work)
            if ev is not None:
                ev[c][1].record()

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        prefill_all()
    torch.cuda.synchronize()
    t_load = time.time()
    while time.time() - t_load < load_seconds:  # >= ~1 s under load for the clock sampler
        prefill_all()
        torch.cuda.synchronize()
    # The sequence's pages fit in L2: flush it (write a buffer twice its
    # size) before every timed prefill, each timed by its own events.
    flush_buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev)
    step_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(steps)]
    barrier(dist)
    torch.cuda.synchronize()
    for k in range(steps):
        flush_buf.fill_(k)
        step_ev[k][0].record()
        prefill_all()
        step_ev[k][1].record()
    torch.cuda.synchronize()
    ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in step_ev) / steps, dist)  # slowest rank
    clock_info = clocks.stop()
    # The attention launches alone, bracketed by events (one more pass,
    # without overlap).
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(nchunks)]
    flush_buf.fill_(-1)
    prefill_all(ev)
    torch.cuda.synchronize()
    attn_ms = sum(a.elapsed_time(b) for a, b in ev)
    del flush_buf
    if rank != 0:
        return None
    # Causal attention flops: 4 * D per (query head, query token, key) pair.
    pairs = total * (total + 1) / 2
    flop = 4 * D * Hq * pairs
    tflops = flop / (ms * 1e-3) / 1e12
    attn_tflops = flop / (attn_ms * 1e-3) / 1e12
    if tensor:
        peak, peak_kind = bf16_peak(sustained=False)
        # With overlap the attention launches run beside the appends and one
        # another, so they have no time of their own: the roofline takes the
        # whole prefill's (appends included), the stricter figure.
        achieved = tflops if overlap else attn_tflops
        roof = {"kernel": "prefill_tc_kernel", "bound": "tensor", "achieved": round(achieved, 1),
                "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                "peak_kind": peak_kind, "traffic": None,
                "algorithmic_flop": flop, "attention_ms": round(attn_ms, 4),
                "time": "the whole prefill per step (appends included; chunks overlapped)"
                        if overlap else "the attention launches alone",
                "note": "tcgen05.mma (M=128) with TMEM accumulators, bf16 operands; K/V pages by TMA"}
    else:
        roof = {"kernel": "paged_decode_kernel (prefill mode)", "bound": "alu",
                "achieved": round(attn_tflops, 2), "unit": "TFLOP/s",
                "attention_ms": round(attn_ms, 4),
                "note": "fp32 CUDA-core FMA path (the decode kernel in prefill mode)"}
    line = {
        "metric": "chunked prefill attention over the paged cache (tokens/s, TFLOP/s)",
        "value": round(world * total / (ms * 1e-3), 1), "unit": "tokens/s", "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"qwen3_8b_prefill_{total}_chunk{chunk}", "tokens": total,
                   "chunk": chunk, "Hq": Hq, "Hkv": Hkv, "D": D, "impl": impl,
                   "overlap": overlap,
                   "l2": "flushed before every timed prefill (a write of twice the L2 "
                         "size); each prefill timed by its own events"},
        "attention_tflops": round(tflops, 2),
        "roofline": roof,
        "gpu_launches": steps * nchunks * (2 if tensor else 3),
        "clocks": clock_info,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = prefill_cpu_baseline(
            q, kc, vc, ids, out, total, flop, cpu_seconds)
    return line


def prefill_cpu_baseline(q, kc, vc, ids, out, total: int, total_flop: float, target_s: float):
    """The fp64 oracle's chunked-prefill attention on the host cores, timed on
    the last n query tokens of the sequence (the rows with the longest
    contexts; n calibrated on one row for about target_s seconds), reported as
    the whole sequence's tokens/s at the oracle's measured flop rate; and the
    max-abs difference of the GPU's output rows against the oracle's."""
    import oracle
    threads = len(os.sched_getaffinity(0))
    Hq, D = q.shape[1], q.shape[2]
    kc_h, vc_h, ids_h = kc.cpu(), vc.cpu(), ids.cpu()
    scale = D ** -0.5

    def rows_flop(s0, n):  # 4 D flop per (query head, query token, attended key)
        return 4 * D * Hq * sum(p + 1 for p in range(s0, s0 + n))

    t0 = time.perf_counter()
    oracle.paged_prefill(q[total - 1:].cpu(), kc_h, vc_h, ids_h, total - 1, scale, nthreads=threads)
    dt1 = max(time.perf_counter() - t0, 1e-4)
    n = max(1, min(total, int(target_s / dt1)))
    s0 = total - n
    t0 = time.perf_counter()
    ref = oracle.paged_prefill(q[s0:].cpu(), kc_h, vc_h, ids_h, s0, scale, nthreads=threads)
    dt = time.perf_counter() - t0
    rate = rows_flop(s0, n) / dt  # flop/s
    err = float((out[s0:].cpu().double() - ref).abs().max())
    base = {"value": round(total / (total_flop / rate), 2), "unit": "tokens/s", "cores": threads,
            "kind": "oracle", "tflops": round(rate / 1e12, 5), "seconds": round(dt, 3),
            "sample": f"query tokens {s0}..{total - 1} of {total} (all {Hq} heads), fp64; "
                      f"value = the whole sequence at the sample's flop rate"}
    parity = {"max_abs_err": err, "tolerance": 1e-2, "ok": bool(err <= 1e-2), "rows": n,
              "reference": "fp64 CPU oracle on the same rows"}
    return base, parity


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=4,
                    help="workload index (0-4); default: the large-batch long-context one")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["decode", "swap", "prefill", "alloc"], default="decode",
                    help="decode: the decode step (default); swap: KV block swap to pinned "
                         "host; prefill: chunked prefill into the paged cache; alloc: the "
                         "device page allocator")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--prefill-chunk", type=int, default=1024)
    ap.add_argument("--prefill-overlap", choices=["on", "off"], default="on",
                    help="launch chunks with XS_PREFILL_OVERLAP (tensor path): chunk c + 1's "
                         "append and attention start beside chunk c's attention")
    ap.add_argument("--prefill-impl", choices=["tensor", "cuda-core"], default="tensor",
                    help="prefill attention: tensor-core kernel or the decode kernel in prefill mode")
    ap.add_argument("--swap-blocks", type=int, default=16384,
                    help="blocks per swap direction for --op swap")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sinks", action="store_true",
                    help="gpt-oss variant: random per-head sink logits in the softmax")
    ap.add_argument("--window", type=int, default=0,
                    help="gpt-oss variant: sliding window of the last W tokens (0 = all)")
    ap.add_argument("--fused", choices=["on", "off"], default="on",
                    help="on: each layer's step is one launch (append + attention + combine); "
                         "off: three launches")
    ap.add_argument("--early-reads", choices=["on", "off"], default="on",
                    help="on: one-launch steps read lengths, tables and first pages before the "
                         "previous launch completes (XS_STEP_EARLY_READS)")
    ap.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                    help="replay each step as one CUDA graph (auto: when the workload has "
                         "more than one layer)")
    ap.add_argument("--batch", type=int, default=0,
                    help="draw the workload with this many sequences (same length "
                         "distribution, pool of the pages needed); 0 = the workload's own")
    ap.add_argument("--partition-tokens", type=int, default=0,
                    help="split-K partition size (multiple of 16); 0 = the library's heuristic")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target duration of the CPU oracle baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=2.0,
                    help="target duration of one reference-arm step")
    ap.add_argument("--load-seconds", type=float, default=1.0,
                    help="untimed load before the timed region (clock sampling)")
    ap.add_argument("--rows", choices=["auto", "on", "off"], default="auto",
                    help="also measure workloads 0-3 and the 8K/1K chunked prefill in the same "
                         "process and report them under 'rows' (auto: with the default "
                         "long-batch decode line)")
    ap.add_argument("--row-steps", type=int, default=200,
                    help="timed steps of each extra row (enough that the first launch's "
                         "host-side start, a few us before the GPU has work, is a small share "
                         "of a row whose launches are tens of us)")
    ap.add_argument("--row-load-seconds", type=float, default=0.4,
                    help="untimed load before each extra row's timed region")
    ap.add_argument("--row-cpu-seconds", type=float, default=3.0,
                    help="target duration of the prefill row's oracle sample")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least 3 untimed warm-up steps
    rank, world, local, dist = dist_setup(args.gpus)
    try:
        if args.impl == "reference":
            run_reference(args, rank, world, dist)
        elif args.op == "swap":
            run_swap(args, rank, world, local, dist)
        elif args.op == "prefill":
            run_prefill(args, rank, world, local, dist)
        elif args.op == "alloc":
            run_alloc(args, rank, world, local, dist)
        else:
            run_ours(args, rank, world, local, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
