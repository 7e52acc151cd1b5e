#!/usr/bin/env python3
"""Benchmark of one decode step over a paged BF16 KV cache on GB300.

A step is one pass of the whole hot path over one batch of synthetic input:
kv_append of every sequence's new token into its page slot, then paged decode
attention (split-context pass + merge) for every sequence, per layer.

Default workload: batch 256 x context 2048, 1 layer, 32 query / 8 KV heads,
head_dim 64, 16-token pages, 32768 shuffled pages (1 GiB of BF16 K/V, larger
than L2, so no flush is needed).  Smaller workloads (--config) flush L2 between
steps by writing a buffer twice the L2 size.

Prints ONE JSON line (rank 0).  `value` is whole-job algorithmic HBM bytes per
second (GB/s) with inputs resident; `e2e` is the same metric through the
library's public calls with the step's inputs copied from pinned host memory and
the output copied back inside the timed region.  `--impl reference` times the
FP64 CPU oracle on the host cores instead (a deliberately slow baseline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time
from concurrent.futures import ThreadPoolExecutor
from contextlib import contextmanager

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
METRIC = "paged decode attention HBM GB/s and % of GB300 peak; sequence-layers/s"
APPEND_BYTES_PER_TOKEN = 2 * 1024 * 2 + 4   # read K and V rows (1 KiB each), write them, read the slot


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=None)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--config", choices=["bandwidth", "llama_step", "ragged", "tiny", "trace", "prefill"],
                   default="bandwidth")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    p.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg (profiling runs)")
    p.add_argument("--ctas", type=int, default=0, help="CTAs of the split-context pass (0 = the library's choice)")
    p.add_argument("--step", choices=["fused", "separate"], default="fused",
                   help="fused: pkv_decode_step (append + attention in one launch); separate: kv_append, then "
                        "paged_decode_attention")
    p.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                   help="replay each step as a CUDA graph (auto: on for the launch-bound workloads)")
    p.add_argument("--nvtx", action="store_true", help="NVTX ranges around the bench phases and steps")
    p.add_argument("--overlap", choices=["auto", "on", "off"], default="auto",
                   help="launch each layer's fused step with PKV_OVERLAP_PREVIOUS, so it starts while the "
                        "previous layer's finishes (auto: on for multi-layer fused steps)")
    return p.parse_args()


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the job's time is its slowest rank's); the value
    itself when not distributed.  Works with NCCL (CUDA tensor) and gloo (CPU tensor)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank_step: int, world: int, ms_per_step_max: float) -> float:
    """Whole-job throughput: every rank runs its own replica of the workload (no data-path
    exchange), so the job moves world x the bytes in the slowest rank's time."""
    return world * bytes_per_rank_step / (ms_per_step_max * 1e-3) / 1e9


def make_workload(name: str):
    from workloads import configs
    return configs.CONFIGS[name]()


def step_bytes(wl) -> tuple[int, int]:
    """(attention bytes per layer, append bytes per layer) of one step."""
    seqs_with_tokens = int(np.sum(wl.context_lens > 0))
    return wl.algorithmic_bytes(), seqs_with_tokens * APPEND_BYTES_PER_TOKEN


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


NVTX = False  # --nvtx: name the bench phases and steps for a profiler's range filters


@contextmanager
def nvtx(name: str):
    """An NVTX range around a phase (warm-up, timed steps, end-to-end, CPU baseline) when --nvtx
    is given, so a capture can be limited to it (ncu --nvtx --nvtx-include "timed/")."""
    if not NVTX:
        yield
        return
    import torch
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


def committed_traffic(record: str, source: str, workload: str):
    """Per-launch DRAM bytes of a kernel from a committed ncu summary (profiles/<record>), if it
    was taken on the current kernel source (csrc/<source>) and on this workload; else None."""
    path = os.path.join(ROOT, "profiles", record)
    src = os.path.join(ROOT, "paged_kv_cache_180_gb300", "csrc", source)
    try:
        with open(path) as f:
            rec = json.load(f)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
        if rec.get("kernel_source_sha256") != sha or rec.get("workload_name") != workload:
            return None
        return rec.get("traffic_bytes_per_launch_full_workload")
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples taken every 100 ms while running."""

    QUERY = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines: list[tuple[float, str]] = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu_index), "-lms", "100"], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        rows = []
        for ts, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((ts, parts))
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        note = None
        if not inside:  # timed region shorter than the sampling period: nearest sample
            inside = [min(rows, key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))]
            note = "timed region shorter than the 100 ms sampling period; nearest sample"

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[2]) for _, p in inside if num(p[2]) is not None]
        mx = [num(p[3]) for _, p in inside if num(p[3]) is not None]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for _, p in inside:
            for name, val in zip(names, p[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        out = {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
               "reasons": sorted(reasons), "samples": len(inside),
               "power_w_max": max((num(p[4]) or 0.0) for _, p in inside)}
        if note:
            out["note"] = note
        return out


# ---------------------------------------------------------------------------
def cpu_oracle_run(wl, threads: int, reps: int = 3):
    """Times the FP64 oracle (as it stands) on the host: append of every token of the
    sampled sequences into its own pool, then attention, threaded over sequences."""
    import oracle
    seqs = list(range(wl.num_seqs))
    pool = oracle.Pool(wl.num_pages)
    q = wl.q(0)
    bt = np.ascontiguousarray(wl.block_tables[:, 0, :])
    lens = np.ascontiguousarray(wl.context_lens)
    kv = {}
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for s, res in zip(seqs, ex.map(lambda s: wl.kv_tokens(s, 0), seqs)):
            kv[s] = res
    slots = {s: wl.slot_mapping(s, 0, 0, int(lens[s])) for s in seqs}

    def one(s):
        k, v = kv[s]
        oracle.kv_append(pool, k, v, slots[s])
        out, err = oracle.paged_decode_attention(pool, q[s:s + 1], bt[s:s + 1], lens[s:s + 1], wl.scale,
                                                 wl.max_context)
        return err

    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        with ThreadPoolExecutor(max_workers=threads) as ex:
            errs = list(ex.map(one, seqs))
        times.append(time.perf_counter() - t0)
        assert not any(errs)
    return statistics.median(times), len(seqs)


def cpu_baseline(wl):
    threads = os.cpu_count() or 1
    t, nseq = cpu_oracle_run(wl, threads)
    attn, app = step_bytes(wl)
    return {"value": round((attn + app) / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"the whole {wl.name} step ({nseq} sequences, 1 layer: append of every token into the "
                      f"oracle's own pool + FP64 attention), median of 3 passes, threaded over sequences",
            "seconds_per_step": round(t, 4), "seq_layers_per_s": round(nseq / t, 2)}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = make_workload(args.config)
    steps = args.steps if args.steps is not None else 3
    warmup = args.warmup if args.warmup is not None else 1
    threads = os.cpu_count() or 1
    import oracle
    oracle.build()
    for _ in range(warmup):
        cpu_oracle_run(wl, threads, reps=1)
    times = [cpu_oracle_run(wl, threads, reps=1)[0] for _ in range(steps)]
    t = sum(times) / len(times)
    attn, app = step_bytes(wl)
    value = (attn + app) / t / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 K/V/q)",
            "config": {"workload": wl.name, "num_seqs": wl.num_seqs, "layers": wl.num_layers,
                       "context_lens": ("2048 each" if wl.name == "bandwidth" else "per workload"),
                       "q_heads": 32, "kv_heads": 8, "head_dim": 64, "page_tokens": 16,
                       "pool_pages": wl.num_pages, "parallelism": "host threads", "l2": "n/a (CPU)"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"each step: the whole {wl.name} step (append + FP64 attention of every "
                                       f"sequence) on the host cores"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "seq_layers_per_s": round(wl.num_seqs * wl.num_layers / t, 2)}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def run_native(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen

    wl = make_workload(args.config)
    L = wl.num_layers
    steps = args.steps if args.steps is not None else (10000 if wl.name == "bandwidth" else 2000)
    warmup = args.warmup if args.warmup is not None else 20

    # ---- resident state: the pool holds every token but each sequence's decode token ----
    pool = pkv.KVPool(wl.num_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for layer in range(L):
        k, v, slots = torch_gen.workload_kv(wl, layer, dev, upto_offset=1)
        if slots.numel():
            pkv.kv_append(pool, k, v, slots, status)
        del k, v, slots
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables)).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    q = [torch_gen.workload_q(wl, layer, dev) for layer in range(L)]
    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    dec = [tuple(to_dev(a) for a in wl.decode_tokens(layer)) for layer in range(L)]
    out = torch.empty(wl.num_seqs, 32, 64, dtype=torch.float32, device=dev)
    ws = pkv.decode_workspace(wl.num_seqs, device=dev)
    blocks = wl.max_blocks
    stride = L * blocks
    stream = torch.cuda.current_stream(dev)
    ctas, attn_launches = pkv.decode_plan(wl.num_seqs, wl.max_context)
    if args.ctas:
        ctas = args.ctas

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    pool_bytes = wl.num_pages * 32768
    flush_w = flush_r = None
    if pool_bytes < 2 * l2:
        # Between steps: write a buffer twice the L2 size, then read another one, so
        # the timed kernels start with none of their inputs (and no dirty lines) in L2.
        flush_w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
        flush_r = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)

    def flush():
        if flush_w is not None:
            flush_w.zero_()
            flush_r.max()

    fused = args.step == "fused"
    # the layers' steps read disjoint pages, so each may start while the previous one finishes
    overlap = fused and (args.overlap == "on" or (args.overlap == "auto" and L > 1))

    def step(e_marks=None, attention_only=False):
        for layer in range(L):
            kn, vn, sn = dec[layer]
            bt_l = bt.view(-1)[layer * blocks:]
            if e_marks is not None:
                e_marks[0].record(stream)
            if fused and not attention_only:
                if e_marks is not None:
                    e_marks[1].record(stream)
                pkv.decode_step(pool, kn, vn, sn, out, q[layer], bt_l, stride, lens, wl.max_context, wl.scale, ws,
                                status, overlap_previous=overlap and layer > 0)
            else:
                if not attention_only:
                    pkv.kv_append(pool, kn, vn, sn, status)
                if e_marks is not None:
                    e_marks[1].record(stream)
                pkv.paged_decode_attention(pool, out, q[layer], bt_l, stride, lens, wl.max_context, wl.scale, ws,
                                           status, num_ctas=args.ctas)
            if e_marks is not None:
                e_marks[2].record(stream)
                e_marks = e_marks[3:]

    use_graph = args.graph == "on" or (args.graph == "auto" and wl.name != "bandwidth")
    with nvtx("warmup"):
        for _ in range(warmup):
            step()
        torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    graphs = None
    if use_graph:
        # whole step, and attention only (for the per-kernel roofline), each one graph
        graphs = []
        for attention_only in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(attention_only=attention_only)
            graphs.append(g)
        for _ in range(3):
            graphs[0].replay()
            graphs[1].replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)

    # ---- timed region: device time of every step, CUDA events on the launching stream ----
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.time()
    append_ms, attn_ms, step_ms = [], [], []
    if graphs is None:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3 * L)] for _ in range(steps)]
        with nvtx("timed"):
            for i in range(steps):
                flush()
                with nvtx(f"step {i}"):
                    step(ev[i])
            torch.cuda.synchronize()
        for i in range(steps):
            tot = 0.0
            for layer in range(L):
                e0, e1, e2 = ev[i][3 * layer:3 * layer + 3]
                a_, b_ = e0.elapsed_time(e1), e1.elapsed_time(e2)
                append_ms.append(a_)
                attn_ms.append(b_ / 1.0)
                tot += a_ + b_
            step_ms.append(tot)
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * steps)]
        with nvtx("timed"):
            for i in range(steps):
                flush()
                ev[i][0].record(stream)
                graphs[0].replay()
                ev[i][1].record(stream)
        with nvtx("timed attention only"):
            for i in range(steps):
                flush()
                ev[steps + i][0].record(stream)
                graphs[1].replay()
                ev[steps + i][1].record(stream)
            torch.cuda.synchronize()
        step_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
        attn_ms = [ev[steps + i][0].elapsed_time(ev[steps + i][1]) / L for i in range(steps)]
        append_ms = [max(0.0, step_ms[i] / L - attn_ms[i]) for i in range(steps)]
    t_wall1 = time.time()
    if world > 1:
        dist.barrier()
    time.sleep(0.25)
    sampler.stop()
    clocks = sampler.summary(t_wall0, t_wall1)
    ms = sum(step_ms) / steps
    ms_max = max_over_ranks(ms, dev)

    attn_b, app_b = step_bytes(wl)
    bytes_step = (attn_b + app_b) * L
    value = whole_job_gbs(bytes_step, world, ms_max)
    attn_avg_s = (sum(attn_ms) / len(attn_ms)) * 1e-3
    # dominant kernel: the fused step kernel (attention + append bytes) or the attention kernel
    kernel_b = attn_b + app_b if (fused and graphs is None) else attn_b
    achieved = kernel_b / attn_avg_s / 1e9
    peak, peak_kind = measured_peak()

    # ---- end to end through the public calls with host buffers ----
    e2e = None
    if not args.no_e2e:
        # Every input of a step (tables, lengths, and per layer q, new K/V rows, slots) sits in
        # one pinned host buffer, and every layer's output goes to one pinned host buffer.  The
        # tables and lengths (read once per page) are copied to the device; q, the new rows and
        # the slots are passed as mapped host pointers and the output is written straight to
        # host memory, so the kernel itself moves them over the host link.
        parts = [bt, lens] + [x for layer in range(L) for x in (q[layer], *dec[layer])]
        offs, total = [], 0
        for x in parts:
            offs.append(total)
            total += (x.numel() * x.element_size() + 255) // 256 * 256
        h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
        copied = offs[2]  # the tables and lengths lead the buffer
        d_in = torch.empty(copied, dtype=torch.uint8, device=dev)
        h_views = []
        for x, o in zip(parts, offs):
            nb = x.numel() * x.element_size()
            h_views.append(h_in[o:o + nb].view(x.dtype).view(x.shape))
            h_views[-1].copy_(x.cpu())
        d_bt = d_in[offs[0]:offs[0] + bt.numel() * 4].view(torch.int32).view(bt.shape)
        d_lens = d_in[offs[1]:offs[1] + lens.numel() * 4].view(torch.int32).view(lens.shape)
        h_q = [h_views[2 + 4 * layer] for layer in range(L)]
        h_dec = [tuple(h_views[3 + 4 * layer:6 + 4 * layer]) for layer in range(L)]
        h_out = torch.empty((L,) + tuple(out.shape), dtype=out.dtype).pin_memory()
        h2d = total
        d2h = h_out.numel() * 4

        def e2e_body():
            d_in.copy_(h_in[:copied], non_blocking=True)
            for layer in range(L):
                kn, vn, sn = h_dec[layer]
                bt_l = d_bt.view(-1)[layer * blocks:]
                if fused:
                    pkv.decode_step(pool, kn, vn, sn, h_out[layer], h_q[layer], bt_l, stride, d_lens, wl.max_context,
                                    wl.scale, ws, status, overlap_previous=overlap and layer > 0)
                else:
                    pkv.kv_append(pool, kn, vn, sn, status)
                    pkv.paged_decode_attention(pool, h_out[layer], h_q[layer], bt_l, stride, d_lens, wl.max_context,
                                               wl.scale, ws, status, num_ctas=args.ctas)

        # the step's copy and launches are replayed as one CUDA graph
        e2e_body()
        torch.cuda.synchronize()
        g_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_e2e):
            e2e_body()
        stream = torch.cuda.current_stream(dev)

        def e2e_step():
            g_e2e.replay()
            stream.synchronize()

        e2e_steps = max(3, min(steps, 200))
        for _ in range(3):
            e2e_step()
        ts = []
        with nvtx("e2e"):
            for _ in range(e2e_steps):
                if flush_w is not None:
                    flush()
                    torch.cuda.synchronize()
                t0 = time.perf_counter()
                e2e_step()
                ts.append(time.perf_counter() - t0)
        t_e2e = max_over_ranks(sum(ts) / len(ts), dev)
        # the last layer's output through host memory equals the device-resident run's, bit for bit
        e2e_same = bool(torch.equal(h_out[L - 1], out.cpu()))
        e2e = {"value": round(whole_job_gbs(bytes_step, world, t_e2e * 1e3), 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(t_e2e * 1e3, 4), "matches_device_run": e2e_same,
               "how": "host wall clock per step, one CUDA graph replay + stream synchronize: H2D copy of the "
                      "tables and lengths from pinned memory; q, new K/V rows and slots read by the kernel from "
                      "mapped pinned host memory; every layer's output written to pinned host memory"}

    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"

    line = None
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16 in, f32 accumulate/out", "data": "synthetic (seeded N(0,1) bf16)",
            "config": {"workload": wl.name, "num_seqs": wl.num_seqs, "layers": L,
                       "context_lens": ("2048 each" if wl.name == "bandwidth" else "per workload"),
                       "q_heads": 32, "kv_heads": 8, "head_dim": 64, "page_tokens": 16,
                       "pool_pages": wl.num_pages, "parallelism": f"replicas x{world}",
                       "l2": ("inputs larger than L2 (1 GiB pool)" if flush_w is None else
                              "L2 flushed between steps (write of a 2x L2 buffer, then read of another)"),
                       "timing": ("CUDA graph replay per step (whole step; attention-only graph for the "
                                  "per-kernel figure)" if graphs is not None else "CUDA events around each kernel"),
                       "split_ctas": ctas},
            "seq_layers_per_s": round(world * wl.num_seqs * L / (ms_max * 1e-3), 1),
            "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                            "nominal_8TBps": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": committed_traffic("decode_attention_traffic.json", "decode_attention.cu", wl.name),
                         "kernel": ("pkv_decode_step (append + split-context attention + merge, one launch)"
                                    if (fused and graphs is None) else
                                    "paged_decode_attention (split-context attention + merge, one launch)"),
                         "algorithmic_bytes_per_launch": kernel_b, "avg_launch_us": round(attn_avg_s * 1e6, 3),
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s"},
            "kernel_us": ({"decode_step": round(1e3 * sum(attn_ms) / len(attn_ms), 3)} if (fused and graphs is None)
                          else {("kv_append" if graphs is None else "append (step minus attention)"):
                                round(1e3 * sum(append_ms) / len(append_ms), 3),
                                "paged_decode_attention": round(1e3 * sum(attn_ms) / len(attn_ms), 3)}),
            "step_kind": args.step, "overlap_previous": bool(overlap),
            "clocks": clocks,
            "gpu_launches": steps * L * ((0 if fused else 1) + attn_launches)
                            + (steps * L * attn_launches if graphs is not None else 0),
            "e2e": e2e,
        }
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    # CPU baseline (the oracle as it stands), rank 0 at N=1 only, on the machine's host cores.
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            with nvtx("cpu_baseline"):
                line["cpu_baseline"] = cpu_baseline(wl)
        print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
def run_trace(args):
    """Continuous-batching trace: 32 slots, 1 layer, 1000 steps planned by the library's
    scheduler (prompts U[16, 512], new-token budgets U[1, 512], 4096-page pool).  Each step
    appends its tokens (admitted prompts + one per decoding slot) and attends over every slot.
    Plans and inputs are prepared before timing; each step's device time is taken with CUDA
    events after an L2 flush (write of a 2x L2 buffer, then read of another)."""
    import torch
    import paged_kv_cache_180_gb300 as pkv
    from workloads import configs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    tr = configs.trace()
    steps = min(args.steps if args.steps is not None else tr.num_steps, tr.num_steps)
    warmup = args.warmup if args.warmup is not None else 3

    sched = pkv.Scheduler(tr.num_pages, 1, 16, tr.max_context, tr.num_slots, tr.free_order)
    for rid in range(tr.num_requests):
        sched.submit(rid, int(tr.prompt_lens[rid]), int(tr.new_budgets[rid]))
    t0 = time.perf_counter()
    plans = [sched.step() for _ in range(steps)]
    host_plan_us = (time.perf_counter() - t0) / steps * 1e6
    stats = sched.stats()

    # device inputs of every step
    def to_dev(a):
        a = np.ascontiguousarray(a)
        if a.dtype == np.uint16:
            return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(a).to(dev)

    per_step = []
    attn_bytes = app_bytes = seq_layers = 0
    for i, pl in enumerate(plans):
        reqs, pos = pl["append_request"], pl["append_position"]
        ks, vs, j = [], [], 0
        while j < len(reqs):
            e = j
            while e + 1 < len(reqs) and reqs[e + 1] == reqs[j] and pos[e + 1] == pos[e] + 1:
                e += 1
            k, v = tr.request_kv(int(reqs[j]), int(pos[j]), int(pos[e]) + 1)
            ks.append(k)
            vs.append(v)
            j = e + 1
        lens = pl["context_lens"]
        q = np.zeros((tr.num_slots, 32, 64), np.uint16)
        if len(pl["decode_slot"]):
            q[pl["decode_slot"]] = tr.step_q(i, pl["decode_slot"])
        bt = np.ascontiguousarray(pl["block_tables"][:, 0, :])
        n_app = len(reqs)
        per_step.append(dict(
            k=to_dev(np.concatenate(ks)) if n_app else None, v=to_dev(np.concatenate(vs)) if n_app else None,
            slots=to_dev(pl["append_slot_mapping"][0]) if n_app else None, q=to_dev(q), bt=to_dev(bt),
            lens=to_dev(lens)))
        live = lens > 0
        attn_bytes += int(lens.sum()) * 2048 + int(live.sum()) * 4096 + 4 * int(np.ceil(lens[live] / 16).sum()) \
            + 4 * tr.num_slots
        app_bytes += n_app * APPEND_BYTES_PER_TOKEN
        seq_layers += int(live.sum())
    pool = pkv.KVPool(tr.num_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pkv.decode_workspace(tr.num_slots, device=dev)
    out = torch.empty(tr.num_slots, 32, 64, dtype=torch.float32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def run_step(x):
        if x["k"] is not None:
            pkv.kv_append(pool, x["k"], x["v"], x["slots"], status)
        pkv.paged_decode_attention(pool, out, x["q"], x["bt"], x["bt"].shape[1], x["lens"], tr.max_context, 0.125,
                                   ws, status)

    for x in per_step[:warmup]:       # warm-up on the first steps (replayed again below)
        run_step(x)
    pool.buffer.zero_()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in per_step]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    tw0 = time.time()
    for x, (e0, e1) in zip(per_step, ev):
        flush_w.zero_()
        flush_r.max()
        e0.record(stream)
        run_step(x)
        e1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dev)
    value = whole_job_gbs(attn_bytes + app_bytes, world, total_ms)
    if rank == 0:
        line = {"metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world, "steps": steps,
                "warmup": warmup, "ms_per_step": round(total_ms / steps, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 accumulate/out",
                "data": "synthetic (seeded N(0,1) bf16; seeded request trace)",
                "config": {"workload": "trace", "slots": tr.num_slots, "layers": 1, "pool_pages": tr.num_pages,
                           "requests": tr.num_requests, "prompt": "U[16, 512]", "new_tokens": "U[1, 512]",
                           "parallelism": f"replicas x{world}",
                           "l2": "L2 flushed before every step (write of a 2x L2 buffer, then read of another)",
                           "timing": "CUDA events around each step's append + attention"},
                "seq_layers_per_s": round(world * seq_layers / (total_ms * 1e-3), 1),
                "host_plan_us_per_step": round(host_plan_us, 2),
                "scheduler_stats": stats,
                "clocks": sampler.summary(tw0, tw1),
                "gpu_launches": sum((1 if x["k"] is not None else 0) + 1 for x in per_step)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0



# ---------------------------------------------------------------------------
def run_prefill(args):
    """Paged prefill: 16 sequences x 512-token prompts (the pages' longest prompt), 1 layer.
    A step appends every prompt token (kv_append) and runs causal paged prefill attention.
    Tensor-bound: the roofline counts the causal flops, 4 * head_dim * q_heads * sum_i (p_i + 1)
    (QK^T and PV, 2 flops per multiply-add), against the measured bf16 tensor peak."""
    import torch
    import paged_kv_cache_180_gb300 as pkv
    from workloads import configs, torch_gen

    local = int(os.environ.get("LOCAL_RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    nseq, plen = 16, 512
    wl = configs.custom(187, [plen] * nseq, name="prefill")
    steps = args.steps if args.steps is not None else 500
    warmup = args.warmup if args.warmup is not None else 10
    pool = pkv.KVPool(wl.num_pages, device=dev)
    k, v, slots = torch_gen.workload_kv(wl, 0, dev)
    n = wl.num_seqs * wl.num_q_heads * wl.head_dim * plen
    q = torch_gen.normal_bf16(rng_key("prefill-q"), 0, n, dev).view(nseq * plen, 32, 64)
    qs = torch.arange(0, (nseq + 1) * plen, plen, dtype=torch.int32, device=dev)
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables[:, 0, :])).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    out = torch.empty(nseq * plen, 32, 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    flush_r = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    # after the append the attention kernel may start its set-up early (it reads the pages only
    # once the append has completed); alone (attention-only figure) it is launched plainly
    overlap = args.overlap != "off"

    def attend(after_append=False):
        pkv.paged_prefill_attention(pool, out, q, qs, bt, bt.shape[1], lens, plen, wl.max_context, wl.scale, status,
                                    overlap_previous=overlap and after_append)

    def step(attention_only=False):
        if not attention_only:
            pkv.kv_append(pool, k, v, slots, status)
        attend(after_append=not attention_only)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # Each step replays as a CUDA graph (whole step, and attention alone for the per-kernel
    # figure), so host-side call overhead never shows up as device idle time.
    use_graph = args.graph != "off"
    graphs = None
    if use_graph:
        graphs = []
        for attention_only in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(attention_only=attention_only)
            graphs.append(g)
        for _ in range(3):
            graphs[0].replay()
            graphs[1].replay()
        torch.cuda.synchronize()
        stream = torch.cuda.current_stream(dev)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    tw0 = time.time()
    if graphs is None:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for e in ev:
            flush_w.zero_()
            flush_r.max()
            e[0].record(stream)
            pkv.kv_append(pool, k, v, slots, status)
            e[1].record(stream)
            attend()
            e[2].record(stream)
        torch.cuda.synchronize()
        app_ms = [e[0].elapsed_time(e[1]) for e in ev]
        att_ms = [e[1].elapsed_time(e[2]) for e in ev]
        all_ms = [a + b for a, b in zip(app_ms, att_ms)]
    else:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * steps)]
        for i in range(2 * steps):
            flush_w.zero_()
            flush_r.max()
            ev[i][0].record(stream)
            graphs[0 if i < steps else 1].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        all_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
        att_ms = [ev[steps + i][0].elapsed_time(ev[steps + i][1]) for i in range(steps)]
        app_ms = [max(0.0, a - b) for a, b in zip(all_ms, att_ms)]
    tw1 = time.time()
    time.sleep(0.25)
    sampler.stop()
    step_ms = max_over_ranks(sum(all_ms) / steps, dev)
    flops = 4 * 64 * 32 * nseq * (plen * (plen + 1) // 2)
    att_s = sum(att_ms) / steps * 1e-3
    tflops = flops / att_s / 1e12
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        pass
    peak = float(peaks.get("bf16_tflops", 1900.0))
    if rank == 0:
        line = {"metric": "paged prefill attention TFLOP/s (causal) and % of the bf16 tensor peak",
                "value": round(world * flops / (step_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s", "n_gpus": world,
                "steps": steps, "warmup": warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, f32 accumulate/out",
                "data": "synthetic (seeded N(0,1) bf16)",
                "config": {"workload": "prefill", "num_seqs": nseq, "prompt_tokens": plen, "layers": 1,
                           "overlap_previous": bool(overlap),
                           "q_heads": 32, "kv_heads": 8, "head_dim": 64, "page_tokens": 16,
                           "l2": "L2 flushed between steps (write of a 2x L2 buffer, then read of another)",
                           "timing": ("CUDA graph replay per step (whole step; attention-only graph for the "
                                      "per-kernel figure)" if graphs is not None else "CUDA events around each kernel")},
                "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                             "frac": round(tflops / peak, 4),
                             "traffic": committed_traffic("prefill_attention_traffic.json", "prefill_attention.cu",
                                                          wl.name),
                             "kernel": "paged_prefill_kernel (tcgen05.mma M128 N64, TMEM accumulators, P as bf16 hi + lo)",
                             "algorithmic_flops_per_launch": flops,
                             "avg_launch_us": round(att_s * 1e6, 3),
                             "peak_source": "measured bf16_tflops (MEASURED_PEAKS.json, cuBLAS burst)"},
                "kernel_us": {("kv_append (all prompt tokens)" if graphs is None else "kv_append (step minus attention)"):
                              round(1e3 * sum(app_ms) / steps, 3),
                              "paged_prefill_attention": round(att_s * 1e6, 3)},
                "clocks": sampler.summary(tw0, tw1), "gpu_launches": 2 * steps + (steps if graphs is not None else 0)}
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def rng_key(tag: str) -> int:
    from workloads import rng
    return rng.stream_key(187, tag)



def main():
    global NVTX
    args = parse_args()
    NVTX = args.nvtx
    if args.impl == "reference":
        return run_reference(args)
    if args.config == "trace":
        return run_trace(args)
    if args.config == "prefill":
        return run_prefill(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
