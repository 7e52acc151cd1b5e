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
the output copied back inside the timed region.  With the default workload at one
GPU the line also carries `other_configs`: the tiny, 16-layer Llama, ragged,
continuous-batching trace and paged-prefill workloads measured in the same run,
each with its kernel time, roofline fraction and CPU baseline.  `--impl
reference` times the FP64 CPU oracle on the host cores instead (a deliberately
slow baseline).
"""
from __future__ import annotations

import argparse
import ctypes
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
FALLBACK_BF16_TFLOPS = 1900.0
METRIC = "paged decode attention HBM GB/s and % of GB300 peak; sequence-layers/s"
APPEND_BYTES_PER_TOKEN = 2 * 1024 * 2 + 4   # read K and V rows (1 KiB each), write them, read the slot
LEAD_SPIN_CYCLES = 4_000_000                 # about 2 ms of GPU spin before the first timed step


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
    p.add_argument("--no-other-configs", action="store_true",
                   help="measure only the chosen workload (no other_configs; profiling runs)")
    p.add_argument("--ctas", type=int, default=0, help="CTAs of the split-context pass (0 = the library's choice)")
    p.add_argument("--step", choices=["fused", "separate"], default="fused",
                   help="fused: pkv_decode_step (append + attention in one launch); separate: kv_append, then "
                        "paged_decode_attention")
    p.add_argument("--graph", choices=["auto", "on", "off"], default="auto",
                   help="replay each step as a CUDA graph (auto: on for the launch-bound workloads)")
    p.add_argument("--nvtx", action="store_true", help="NVTX ranges around the bench phases and steps")
    p.add_argument("--prefill-shape", default="16,512", metavar="SEQS,TOKENS",
                   help="prompts of the prefill workload (default 16 x 512; another shape is reported under "
                        "its own workload name, e.g. prefill_4x2048)")
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


def measured_tensor_peak():
    """bf16 dense tensor peak (TFLOP/s): the measured cuBLAS burst figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the platform string)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


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
# CPU baselines: the oracle as it stands, on the host cores.
# ---------------------------------------------------------------------------
class OracleDecodeStep:
    """Host inputs of one decode step of ``wl`` for the oracle: per (layer, sequence) unit the K/V
    of every token and their slots (drawn before timing), one oracle pool, the queries and tables.
    A unit appends its tokens into the pool and attends for its sequence at its layer."""

    def __init__(self, wl, threads: int):
        import oracle
        self.oracle = oracle
        self.wl = wl
        self.pool = oracle.Pool(wl.num_pages)
        self.units = [(layer, s) for layer in range(wl.num_layers) for s in range(wl.num_seqs)
                      if wl.context_lens[s] > 0 and wl.has_pages(s)]
        self.q = [wl.q(layer) for layer in range(wl.num_layers)]
        self.bt = [np.ascontiguousarray(wl.block_tables[:, layer, :]) for layer in range(wl.num_layers)]
        self.lens = np.ascontiguousarray(wl.context_lens)
        self.kv = {}
        with ThreadPoolExecutor(max_workers=threads) as ex:
            for u, res in zip(self.units, ex.map(lambda u: wl.kv_tokens(u[1], u[0]), self.units)):
                self.kv[u] = res
        self.slots = {(layer, s): wl.slot_mapping(s, layer, 0, int(self.lens[s])) for layer, s in self.units}

    def one(self, unit) -> int:
        layer, s = unit
        k, v = self.kv[unit]
        self.oracle.kv_append(self.pool, k, v, self.slots[unit])
        _, err = self.oracle.paged_decode_attention(self.pool, self.q[layer][s:s + 1], self.bt[layer][s:s + 1],
                                                    self.lens[s:s + 1], self.wl.scale, self.wl.max_context)
        return err

    def run(self, threads: int, units=None) -> float:
        units = self.units if units is None else units
        t0 = time.perf_counter()
        if threads == 1:
            errs = [self.one(u) for u in units]
        else:
            with ThreadPoolExecutor(max_workers=threads) as ex:
                errs = list(ex.map(self.one, units))
        t = time.perf_counter() - t0
        assert not any(errs)
        return t


def single_thread_seconds(run_units, units, full_seconds_threaded: float, threads: int, budget_s: float = 3.0):
    """One-thread time of all ``units``, measured on a leading sample of them sized to take about
    ``budget_s`` (estimated from the threaded time) and scaled by the unit count.  Returns
    (seconds for all units, units timed)."""
    n = len(units)
    est_one = max(full_seconds_threaded * threads, 1e-9)
    k = max(1, min(n, int(math.ceil(n * budget_s / est_one))))
    t = run_units(units[:k])
    return t * n / k, k


def cpu_baseline(wl, reps: int = 3):
    """The oracle on the whole step (append + FP64 attention of every sequence and layer), threaded
    over (layer, sequence) on all host cores, plus a one-thread figure on a sample of the units."""
    threads = os.cpu_count() or 1
    prep = OracleDecodeStep(wl, threads)
    times = [prep.run(threads) for _ in range(reps)]
    t = statistics.median(times)
    one_t, k = single_thread_seconds(lambda us: prep.run(1, us), prep.units, t, threads)
    attn, app = step_bytes(wl)
    b = (attn + app) * wl.num_layers
    n_units = len(prep.units)
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"the whole {wl.name} step ({wl.num_seqs} sequences x {wl.num_layers} layers: append of every "
                      f"token into the oracle's own pool + FP64 attention), median of {reps} passes, threaded over "
                      f"(layer, sequence)",
            "seconds_per_step": round(t, 5), "seq_layers_per_s": round(n_units / t, 2),
            "single_thread": {"value": round(b / one_t / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "seconds_per_step": round(one_t, 5),
                              "sample": f"{k} of {n_units} (layer, sequence) units on one thread, scaled to the "
                                        f"whole step"}}


def cpu_baseline_trace(tr, host_steps, step_bytes_list, sample_steps: int = 200, one_thread_steps: int = 50):
    """The oracle replaying the first ``sample_steps`` steps of the continuous-batching trace: each
    step appends its tokens into the oracle's pool and attends over every live slot (threaded over
    slots); the one-thread figure replays the first ``one_thread_steps`` again on a fresh pool."""
    import oracle
    threads = os.cpu_count() or 1
    n = min(sample_steps, len(host_steps))

    def replay(count: int, nthreads: int) -> float:
        pool = oracle.Pool(tr.num_pages)
        ex = ThreadPoolExecutor(max_workers=nthreads) if nthreads > 1 else None
        t0 = time.perf_counter()
        for x in host_steps[:count]:
            if x["k"] is not None:
                assert oracle.kv_append(pool, x["k"], x["v"], x["slots"]) == 0
            live = [s for s in range(tr.num_slots) if x["lens"][s] > 0]

            def one(s, x=x, pool=pool):
                return oracle.paged_decode_attention(pool, x["q"][s:s + 1], x["bt"][s:s + 1], x["lens"][s:s + 1],
                                                     0.125, tr.max_context)[1]
            errs = list(ex.map(one, live)) if ex is not None else [one(s) for s in live]
            assert not any(errs)
        t = time.perf_counter() - t0
        if ex is not None:
            ex.shutdown()
        return t

    t = replay(n, threads)
    k = min(one_thread_steps, n)
    t1 = replay(k, 1)
    b = sum(step_bytes_list[:n])
    b1 = sum(step_bytes_list[:k])
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"the trace's first {n} steps (appends + FP64 attention over the live slots), threaded "
                      f"over slots", "seconds_per_step": round(t / n, 6),
            "single_thread": {"value": round(b1 / t1 / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "seconds_per_step": round(t1 / k, 6), "sample": f"the first {k} steps on one thread"}}


def cpu_baseline_prefill(wl, q_bits, plen: int, flops: int):
    """The oracle's causal paged prefill attention on the host: every sequence's prompt (threaded
    over sequences), and one sequence on one thread scaled to the whole batch."""
    import oracle
    threads = os.cpu_count() or 1
    pool = oracle.Pool(wl.num_pages)
    for s in range(wl.num_seqs):
        k, v = wl.kv_tokens(s, 0)
        assert oracle.kv_append(pool, k, v, wl.slot_mapping(s, 0, 0, int(wl.context_lens[s]))) == 0
    bt = np.ascontiguousarray(wl.block_tables[:, 0, :])
    qs1 = np.array([0, plen], dtype=np.int32)

    def one(s):
        _, err = oracle.paged_prefill_attention(pool, np.ascontiguousarray(q_bits[s * plen:(s + 1) * plen]), qs1,
                                                bt[s:s + 1], wl.context_lens[s:s + 1], wl.scale, wl.max_context)
        return err

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as ex:
        errs = list(ex.map(one, range(wl.num_seqs)))
    t = time.perf_counter() - t0
    assert not any(errs)
    t0 = time.perf_counter()
    assert one(0) == 0
    t1 = (time.perf_counter() - t0) * wl.num_seqs
    return {"value": round(flops / t / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"the whole prefill step's attention ({wl.num_seqs} prompts of {plen} tokens, FP64), "
                      f"threaded over sequences", "seconds_per_step": round(t, 5),
            "single_thread": {"value": round(flops / t1 / 1e12, 6), "unit": "TFLOP/s", "cores": 1,
                              "seconds_per_step": round(t1, 5),
                              "sample": "one prompt on one thread, scaled to the batch"}}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    if args.config in ("trace", "prefill"):
        print(json.dumps({"impl": "reference", "unavailable": "the reference arm times the decode workloads; the "
                          f"{args.config} workload's oracle is timed as cpu_baseline of the native line"}))
        return 0
    wl = make_workload(args.config)
    steps = args.steps if args.steps is not None else 3
    warmup = args.warmup if args.warmup is not None else 1
    threads = os.cpu_count() or 1
    import oracle
    oracle.build()
    prep = OracleDecodeStep(wl, threads)
    for _ in range(warmup):
        prep.run(threads)
    times = [prep.run(threads) for _ in range(steps)]
    t = sum(times) / len(times)
    attn, app = step_bytes(wl)
    value = (attn + app) * wl.num_layers / t / 1e9
    line = {"metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus, "steps": steps,
            "warmup": warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded N(0,1) bf16 K/V/q)",
            "config": {"workload": wl.name, "num_seqs": wl.num_seqs, "layers": wl.num_layers,
                       "context_lens": ("2048 each" if wl.name == "bandwidth" else "per workload"),
                       "q_heads": 32, "kv_heads": 8, "head_dim": 64, "page_tokens": 16,
                       "pool_pages": wl.num_pages, "parallelism": "host threads", "l2": "n/a (CPU)"},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "cpu_model": cpu_model(),
                             "sample": f"each step: the whole {wl.name} step (append + FP64 attention of every "
                                       f"sequence) on the host cores"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "seq_layers_per_s": round(len(prep.units) / t, 2)}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU measurements
# ---------------------------------------------------------------------------
def _to_dev(a, dev):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(a).to(dev)


class L2Flush:
    """Between timed steps: write a buffer twice the L2 size, then read another one, so the timed
    kernels start with none of their inputs (and no dirty lines) in L2."""

    def __init__(self, dev, active: bool = True):
        import torch
        self.w = self.r = None
        if active:
            l2 = torch.cuda.get_device_properties(dev).L2_cache_size
            self.w = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
            self.r = torch.zeros(2 * l2 // 4, dtype=torch.float32, device=dev)

    @property
    def active(self) -> bool:
        return self.w is not None

    def __call__(self):
        if self.w is not None:
            self.w.zero_()
            self.r.max()


def decode_measure(args, wl, dev, steps: int, warmup: int, world: int, sampler, with_e2e: bool,
                   step_kind: str = "fused", graph_mode: str = "auto", overlap_mode: str = "auto", ctas_arg: int = 0):
    """Times ``steps`` decode steps of ``wl`` (append + attention per layer) on ``dev``; returns a record."""
    import torch

    import paged_kv_cache_180_gb300 as pkv
    from workloads import torch_gen

    L = wl.num_layers
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
    dec = [tuple(_to_dev(a, dev) for a in wl.decode_tokens(layer)) for layer in range(L)]
    out = torch.empty(wl.num_seqs, 32, 64, dtype=torch.float32, device=dev)
    ws = pkv.decode_workspace(wl.num_seqs, device=dev)
    blocks = wl.max_blocks
    stride = L * blocks
    stream = torch.cuda.current_stream(dev)
    ctas, attn_launches = pkv.decode_plan(wl.num_seqs, wl.max_context)
    if ctas_arg:
        ctas = ctas_arg
    flush = L2Flush(dev, active=wl.num_pages * 32768 < 2 * torch.cuda.get_device_properties(dev).L2_cache_size)

    fused = step_kind == "fused"
    # the layers' steps read disjoint pages, so each may start while the previous one finishes
    overlap = fused and (overlap_mode == "on" or (overlap_mode == "auto" and L > 1))

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
                                           status, num_ctas=ctas_arg)
            if e_marks is not None:
                e_marks[2].record(stream)
                e_marks = e_marks[3:]

    use_graph = graph_mode == "on" or (graph_mode == "auto" and wl.name != "bandwidth")
    graphs = None
    if use_graph:
        for _ in range(2):
            step()
        torch.cuda.synchronize()
        # whole step, and attention only (for the per-kernel roofline), each one graph
        graphs = []
        for attention_only in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(attention_only=attention_only)
            graphs.append(g)
        stream = torch.cuda.current_stream(dev)
    # ---- W warm-up steps, then the timed region at once (no idle gap between them) ----
    with nvtx("warmup"):
        for _ in range(warmup):
            if graphs is None:
                step()
            else:
                graphs[0].replay()
                graphs[1].replay()
        torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # A short spin kernel ahead of the first timed step keeps the GPU busy while the host queues
    # that step, so its start event is not reached before its kernel has been launched.
    torch.cuda._sleep(LEAD_SPIN_CYCLES)
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
                attn_ms.append(b_)
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
        import torch.distributed as dist
        dist.barrier()
    clocks = sampler.summary(t_wall0, t_wall1)
    ms = sum(step_ms) / steps
    ms_max = max_over_ranks(ms, dev)

    attn_b, app_b = step_bytes(wl)
    bytes_step = (attn_b + app_b) * L
    attn_avg_s = (sum(attn_ms) / len(attn_ms)) * 1e-3
    # dominant kernel: the fused step kernel (attention + append bytes) or the attention kernel
    kernel_b = attn_b + app_b if (fused and graphs is None) else attn_b
    rec = dict(wl=wl, L=L, steps=steps, warmup=warmup, step_ms=step_ms, attn_ms=attn_ms, append_ms=append_ms,
               ms=ms, ms_max=ms_max, bytes_step=bytes_step, attn_b=attn_b, app_b=app_b, kernel_b=kernel_b,
               achieved=kernel_b / attn_avg_s / 1e9, attn_avg_s=attn_avg_s, graphs=graphs is not None,
               fused=fused, overlap=overlap, ctas=ctas, attn_launches=attn_launches, clocks=clocks,
               flush=flush.active, e2e=None)

    # ---- end to end through the public calls with host buffers ----
    if with_e2e:
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
                                               wl.scale, ws, status, num_ctas=ctas_arg)

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
                if flush.active:
                    flush()
                    torch.cuda.synchronize()
                t0 = time.perf_counter()
                e2e_step()
                ts.append(time.perf_counter() - t0)
        t_e2e = max_over_ranks(sum(ts) / len(ts), dev)
        # the last layer's output through host memory equals the device-resident run's, bit for bit
        e2e_same = bool(torch.equal(h_out[L - 1], out.cpu()))
        rec["e2e"] = {"value": round(whole_job_gbs(bytes_step, world, t_e2e * 1e3), 3), "unit": "GB/s",
                      "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": round(t_e2e * 1e3, 4), "matches_device_run": e2e_same,
                      "how": "host wall clock per step, one CUDA graph replay + stream synchronize: H2D copy of the "
                             "tables and lengths from pinned memory; q, new K/V rows and slots read by the kernel "
                             "from mapped pinned host memory; every layer's output written to pinned host memory"}
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    rec["gpu_launches"] = steps * L * ((0 if fused else 1) + attn_launches) + (
        steps * L * attn_launches if graphs is not None else 0)
    del pool, ws
    return rec


def _step_stats(step_ms):
    return {"min": round(min(step_ms), 5), "median": round(statistics.median(step_ms), 5),
            "max": round(max(step_ms), 5), "first": round(step_ms[0], 5), "last": round(step_ms[-1], 5)}


def decode_summary(rec, peak: float) -> dict:
    """A compact per-workload entry: kernel time, GB/s, roofline fraction, step time."""
    wl, L = rec["wl"], rec["L"]
    step_gbs = rec["bytes_step"] / (rec["ms"] * 1e-3) / 1e9
    ent = {"workload": wl.name, "num_seqs": wl.num_seqs, "layers": L, "pool_pages": wl.num_pages,
           "steps": rec["steps"], "warmup": rec["warmup"],
           "l2": "flushed between steps" if rec["flush"] else "inputs larger than L2",
           "timing": ("CUDA graph replay per step; attention-only graph for the kernel figure" if rec["graphs"]
                      else "CUDA events around each kernel"),
           "kernel": ("paged_decode_attention" if (rec["graphs"] or not rec["fused"]) else "pkv_decode_step"),
           "kernel_us": round(rec["attn_avg_s"] * 1e6, 3),
           "kernel_algorithmic_bytes": rec["kernel_b"],
           "kernel_gbs": round(rec["achieved"], 2),
           "roofline": {"bound": "hbm", "achieved": round(rec["achieved"], 2), "peak": peak, "unit": "GB/s",
                        "frac": round(rec["achieved"] / peak, 4)},
           "step_us": round(rec["ms"] * 1e3, 3), "step_bytes": rec["bytes_step"], "step_gbs": round(step_gbs, 2),
           "step_frac": round(step_gbs / peak, 4),
           "seq_layers_per_s": round(wl.num_seqs * L / (rec["ms"] * 1e-3), 1),
           "split_ctas": rec["ctas"], "overlap_previous": rec["overlap"], "clocks": rec["clocks"]}
    if L > 1:
        ent["per_layer_step_us"] = round(rec["ms"] * 1e3 / L, 3)
    return ent


def trace_host_steps(tr, steps: int) -> dict:
    """The library's scheduler plans ``steps`` steps of the trace; returns each step's host inputs
    (new K/V rows and slots, queries, tables, lengths), its algorithmic bytes, and totals."""
    import paged_kv_cache_180_gb300 as pkv
    sched = pkv.Scheduler(tr.num_pages, 1, 16, tr.max_context, tr.num_slots, tr.free_order)
    for rid in range(tr.num_requests):
        sched.submit(rid, int(tr.prompt_lens[rid]), int(tr.new_budgets[rid]))
    t0 = time.perf_counter()
    plans = [sched.step() for _ in range(steps)]
    host_plan_us = (time.perf_counter() - t0) / steps * 1e6
    # the same plans from a second scheduler through the bare C call (no copies into numpy
    # arrays): the native scheduler's own cost per step
    native = pkv.Scheduler(tr.num_pages, 1, 16, tr.max_context, tr.num_slots, tr.free_order)
    for rid in range(tr.num_requests):
        native.submit(rid, int(tr.prompt_lens[rid]), int(tr.new_budgets[rid]))
    raw = pkv.binding.PkvStepPlan()
    step_fn, handle = pkv.binding._lib.pkv_sched_step, native._h
    t0 = time.perf_counter()
    for _ in range(steps):
        step_fn(handle, ctypes.byref(raw))
    native_plan_us = (time.perf_counter() - t0) / steps * 1e6
    host_steps, bytes_per_step = [], []
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
        n_app = len(reqs)
        k_all = np.concatenate(ks) if n_app else None
        v_all = np.concatenate(vs) if n_app else None
        slots_all = np.ascontiguousarray(pl["append_slot_mapping"][0]) if n_app else None
        # the plan lists the admitted prompts' tokens first, then one decode token per decoding
        # slot (ascending): the prompts go through kv_append, the decode tokens through the
        # fused decode step (one row per slot, slot -1 where a slot does not decode)
        dec = pl["decode_slot"]
        n_pr = n_app - len(dec)
        k_new = np.zeros((tr.num_slots, 8, 64), np.uint16)
        v_new = np.zeros((tr.num_slots, 8, 64), np.uint16)
        slot_new = np.full(tr.num_slots, -1, np.int32)
        if len(dec):
            k_new[dec], v_new[dec], slot_new[dec] = k_all[n_pr:], v_all[n_pr:], slots_all[n_pr:]
        host_steps.append(dict(k=k_all, v=v_all, slots=slots_all, q=q,
                               bt=np.ascontiguousarray(pl["block_tables"][:, 0, :]), lens=np.ascontiguousarray(lens),
                               k_prompt=k_all[:n_pr] if n_pr else None, v_prompt=v_all[:n_pr] if n_pr else None,
                               slots_prompt=slots_all[:n_pr] if n_pr else None, k_new=k_new, v_new=v_new,
                               slot_new=slot_new))
        live = lens > 0
        ab = int(lens.sum()) * 2048 + int(live.sum()) * 4096 + 4 * int(np.ceil(lens[live] / 16).sum()) \
            + 4 * tr.num_slots
        attn_bytes += ab
        app_bytes += n_app * APPEND_BYTES_PER_TOKEN
        bytes_per_step.append(ab + n_app * APPEND_BYTES_PER_TOKEN)
        seq_layers += int(live.sum())
    return {"host_steps": host_steps, "bytes_per_step": bytes_per_step, "attn_bytes": attn_bytes,
            "app_bytes": app_bytes, "seq_layers": seq_layers, "host_plan_us": round(host_plan_us, 2),
            "native_plan_us": round(native_plan_us, 2),
            "stats": sched.stats()}


def trace_measure(args, dev, steps: int, warmup: int, world: int, sampler, with_cpu: bool):
    """Continuous-batching trace: 32 slots, 1 layer, 1000 steps planned by the library's
    scheduler (prompts U[16, 512], new-token budgets U[1, 512], 4096-page pool).  Each step
    appends its tokens (admitted prompts + one per decoding slot) and attends over every slot.
    Plans and inputs are prepared before timing; each step's device time is taken with CUDA
    events after an L2 flush (write of a 2x L2 buffer, then read of another)."""
    import torch

    import paged_kv_cache_180_gb300 as pkv
    from workloads import configs

    tr = configs.trace()
    steps = min(steps, tr.num_steps)
    plan = trace_host_steps(tr, steps)
    host_steps, bytes_per_step = plan["host_steps"], plan["bytes_per_step"]
    attn_bytes, app_bytes, seq_layers = plan["attn_bytes"], plan["app_bytes"], plan["seq_layers"]
    gpu_keys = ("k_prompt", "v_prompt", "slots_prompt", "k_new", "v_new", "slot_new", "q", "bt", "lens")
    per_step = [{key: (None if hx[key] is None else _to_dev(hx[key], dev)) for key in gpu_keys} for hx in host_steps]
    pool = pkv.KVPool(tr.num_pages, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = pkv.decode_workspace(tr.num_slots, device=dev)
    out = torch.empty(tr.num_slots, 32, 64, dtype=torch.float32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)

    def run_step(x):
        # admitted prompts are appended first; each decoding slot's new token is appended by the
        # attention launch itself (pkv_decode_step)
        if x["k_prompt"] is not None:
            pkv.kv_append(pool, x["k_prompt"], x["v_prompt"], x["slots_prompt"], status)
        pkv.decode_step(pool, x["k_new"], x["v_new"], x["slot_new"], out, x["q"], x["bt"], x["bt"].shape[1],
                        x["lens"], tr.max_context, 0.125, ws, status)

    for x in per_step[:warmup]:       # warm-up on the first steps (replayed again below)
        run_step(x)
    pool.buffer.zero_()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in per_step]
    tw0 = time.time()
    for x, (e0, e1) in zip(per_step, ev):
        flush()
        e0.record(stream)
        run_step(x)
        e1.record(stream)
    torch.cuda.synchronize()
    tw1 = time.time()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dev)
    peak, _ = measured_peak()
    gbs = whole_job_gbs(attn_bytes + app_bytes, world, total_ms)
    rec = {"workload": "trace", "slots": tr.num_slots, "layers": 1, "pool_pages": tr.num_pages,
           "requests": tr.num_requests, "prompt": "U[16, 512]", "new_tokens": "U[1, 512]", "steps": steps,
           "warmup": warmup, "l2": "flushed before every step",
           "timing": "CUDA events around each step: kv_append of admitted prompts (when any), then one fused "
                     "append + attention launch (pkv_decode_step)",
           "step_us": round(total_ms / steps * 1e3, 3), "step_gbs": round(gbs, 3),
           "step_frac": round(gbs / world / peak, 4),
           "roofline": {"bound": "hbm", "achieved": round(gbs / world, 3), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / world / peak, 4),
                        "note": "whole step (prompt append + fused decode step) over its algorithmic bytes: "
                                "launch-bound"},
           "algorithmic_bytes": attn_bytes + app_bytes,
           "seq_layers_per_s": round(world * seq_layers / (total_ms * 1e-3), 1),
           "host_plan_us_per_step": plan["host_plan_us"], "native_plan_us_per_step": plan["native_plan_us"],
           "scheduler_stats": plan["stats"],
           "clocks": sampler.summary(tw0, tw1),
           "gpu_launches": sum((1 if x["k_prompt"] is not None else 0) + 1 for x in per_step),
           "_total_ms": total_ms, "_gbs": gbs}
    del pool, per_step
    if with_cpu:
        with nvtx("cpu_baseline trace"):
            rec["cpu_baseline"] = cpu_baseline_trace(tr, host_steps, bytes_per_step)
    return rec


def prefill_shape(args) -> tuple[int, int, str]:
    """(sequences, prompt tokens, workload name) of the prefill workload: 16 x 512 is "prefill"."""
    nseq, plen = (int(x) for x in str(getattr(args, "prefill_shape", "16,512")).split(","))
    if not (nseq >= 1 and 1 <= plen <= 2048):
        raise SystemExit("--prefill-shape wants SEQS >= 1 and 1 <= TOKENS <= 2048")
    return nseq, plen, "prefill" if (nseq, plen) == (16, 512) else f"prefill_{nseq}x{plen}"


def prefill_measure(args, dev, steps: int, warmup: int, world: int, sampler, with_cpu: bool):
    """Paged prefill: 16 sequences x 512-token prompts (the pages' longest prompt) by default, 1 layer.
    A step appends every prompt token (kv_append) and runs causal paged prefill attention.
    Tensor-bound: the roofline counts the causal flops, 4 * head_dim * q_heads * sum_i (p_i + 1)
    (QK^T and PV, 2 flops per multiply-add), against the measured bf16 tensor peak."""
    import torch

    import paged_kv_cache_180_gb300 as pkv
    from workloads import configs, rng, torch_gen

    nseq, plen, label = prefill_shape(args)
    wl = configs.custom(187, [plen] * nseq, name="prefill")
    pool = pkv.KVPool(wl.num_pages, device=dev)
    k, v, slots = torch_gen.workload_kv(wl, 0, dev)
    n = wl.num_seqs * wl.num_q_heads * wl.head_dim * plen
    qkey = rng.stream_key(187, "prefill-q")
    q = torch_gen.normal_bf16(qkey, 0, n, dev).view(nseq * plen, 32, 64)
    qs = torch.arange(0, (nseq + 1) * plen, plen, dtype=torch.int32, device=dev)
    bt = torch.from_numpy(np.ascontiguousarray(wl.block_tables[:, 0, :])).to(dev)
    lens = torch.from_numpy(wl.context_lens).to(dev)
    out = torch.empty(nseq * plen, 32, 64, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
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

    for _ in range(2):
        step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # Each step replays as a CUDA graph (whole step, and attention alone for the per-kernel
    # figure), so host-side call overhead never shows up as device idle time.
    graphs = None
    if args.graph != "off":
        graphs = []
        for attention_only in (False, True):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(attention_only=attention_only)
            graphs.append(g)
        stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        if graphs is None:
            step()
        else:
            graphs[0].replay()
            graphs[1].replay()
    torch.cuda.synchronize()
    tw0 = time.time()
    if graphs is None:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
        for e in ev:
            flush()
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
            flush()
            ev[i][0].record(stream)
            graphs[0 if i < steps else 1].replay()
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        all_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(steps)]
        att_ms = [ev[steps + i][0].elapsed_time(ev[steps + i][1]) for i in range(steps)]
        app_ms = [max(0.0, a - b) for a, b in zip(all_ms, att_ms)]
    tw1 = time.time()
    assert int(status.item()) == 0
    step_ms = max_over_ranks(sum(all_ms) / steps, dev)
    flops = 4 * 64 * 32 * nseq * (plen * (plen + 1) // 2)
    att_s = sum(att_ms) / steps * 1e-3
    tflops = flops / att_s / 1e12
    peak, peak_kind = measured_tensor_peak()
    rec = {"workload": label, "num_seqs": nseq, "prompt_tokens": plen, "layers": 1, "steps": steps,
           "warmup": warmup, "overlap_previous": bool(overlap), "l2": "flushed between steps",
           "timing": ("CUDA graph replay per step (whole step; attention-only graph for the per-kernel figure)"
                      if graphs is not None else "CUDA events around each kernel"),
           "kernel": "paged_prefill_kernel (tcgen05.mma, TMEM accumulators)",
           "kernel_us": round(att_s * 1e6, 3), "kernel_tflops": round(tflops, 2),
           "roofline": {"bound": "tensor", "achieved": round(tflops, 2), "peak": peak, "unit": "TFLOP/s",
                        "frac": round(tflops / peak, 4),
                        "traffic": committed_traffic("prefill_attention_traffic.json", "prefill_attention.cu",
                                                     label),
                        "algorithmic_flops_per_launch": flops, "avg_launch_us": round(att_s * 1e6, 3),
                        "peak_source": (f"{peak_kind} bf16_tflops (MEASURED_PEAKS.json, cuBLAS burst)"
                                        if peak_kind == "measured" else "fallback 1.9 PFLOP/s")},
           "step_us": round(step_ms * 1e3, 3),
           "step_tflops": round(world * flops / (step_ms * 1e-3) / 1e12, 3),
           "kernel_us_by_part": {("kv_append (all prompt tokens)" if graphs is None else
                                  "kv_append (step minus attention)"): round(1e3 * sum(app_ms) / steps, 3),
                                 "paged_prefill_attention": round(att_s * 1e6, 3)},
           "clocks": sampler.summary(tw0, tw1),
           "gpu_launches": 2 * steps + (steps if graphs is not None else 0),
           "_step_ms": step_ms, "_flops": flops}
    del pool
    if with_cpu:
        with nvtx("cpu_baseline prefill"):
            q_host = rng.normal_bf16(qkey, 0, n).reshape(nseq * plen, 32, 64)
            rec["cpu_baseline"] = cpu_baseline_prefill(wl, q_host, plen, flops)
    return rec


def _public(rec: dict) -> dict:
    return {k: v for k, v in rec.items() if not k.startswith("_")}


def other_configs(args, dev, sampler) -> dict:
    """The other workloads, measured in the same run at one GPU: kernel time, roofline fraction,
    step time and the oracle on the host cores for each."""
    import torch
    peak, _ = measured_peak()
    res = {}
    for name, steps in (("tiny", 200), ("llama_step", 200), ("ragged", 200)):
        wl = make_workload(name)
        with nvtx(f"other {name}"):
            rec = decode_measure(args, wl, dev, steps, 10, 1, sampler, with_e2e=False)
        ent = decode_summary(rec, peak)
        if not args.no_cpu_baseline:
            with nvtx(f"cpu_baseline {name}"):
                ent["cpu_baseline"] = cpu_baseline(wl)
        res[name] = ent
        torch.cuda.empty_cache()
    with nvtx("other trace"):
        res["trace"] = _public(trace_measure(args, dev, 1000, 3, 1, sampler, with_cpu=not args.no_cpu_baseline))
    torch.cuda.empty_cache()
    with nvtx("other prefill"):
        res["prefill"] = _public(prefill_measure(args, dev, 200, 10, 1, sampler,
                                                 with_cpu=not args.no_cpu_baseline))
    return res


# ---------------------------------------------------------------------------
def _dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    return world, rank, local, torch.device("cuda", local)


def _dist_teardown(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


def run_native(args):
    world, rank, local, dev = _dist_setup()
    wl = make_workload(args.config)
    L = wl.num_layers
    steps = args.steps if args.steps is not None else (10000 if wl.name == "bandwidth" else 2000)
    warmup = args.warmup if args.warmup is not None else 20
    sampler = ClockSampler(local)
    sampler.start()
    rec = decode_measure(args, wl, dev, steps, warmup, world, sampler, with_e2e=not args.no_e2e,
                         step_kind=args.step, graph_mode=args.graph, overlap_mode=args.overlap, ctas_arg=args.ctas)
    ms_max = rec["ms_max"]
    value = whole_job_gbs(rec["bytes_step"], world, ms_max)
    peak, peak_kind = measured_peak()
    fused, graphs = rec["fused"], rec["graphs"]
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
                       "l2": ("inputs larger than L2 (1 GiB pool)" if not rec["flush"] else
                              "L2 flushed between steps (write of a 2x L2 buffer, then read of another)"),
                       "timing": ("CUDA graph replay per step (whole step; attention-only graph for the "
                                  "per-kernel figure)" if graphs else "CUDA events around each kernel"),
                       "split_ctas": rec["ctas"],
                       "lead": "a ~2 ms spin kernel is queued before the first timed step (outside its events) so "
                               "that the step's launch is queued before its start event is reached"},
            "seq_layers_per_s": round(world * wl.num_seqs * L / (ms_max * 1e-3), 1),
            "pct_of_peak": {"measured": round(100 * value / world / peak, 2),
                            "nominal_8TBps": round(100 * value / world / NOMINAL_HBM_GBS, 2)},
            "roofline": {"bound": "hbm", "achieved": round(rec["achieved"], 2), "peak": peak, "unit": "GB/s",
                         "frac": round(rec["achieved"] / peak, 4),
                         "traffic": committed_traffic("decode_attention_traffic.json", "decode_attention.cu",
                                                      wl.name),
                         "kernel": ("pkv_decode_step (append + split-context attention + merge, one launch)"
                                    if (fused and not graphs) else
                                    "paged_decode_attention (split-context attention + merge, one launch)"),
                         "algorithmic_bytes_per_launch": rec["kernel_b"],
                         "avg_launch_us": round(rec["attn_avg_s"] * 1e6, 3),
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)" if peak_kind == "measured"
                         else "fallback 6.8 TB/s"},
            "kernel_us": ({"decode_step": round(1e3 * sum(rec["attn_ms"]) / len(rec["attn_ms"]), 3)}
                          if (fused and not graphs) else
                          {("kv_append" if not graphs else "append (step minus attention)"):
                           round(1e3 * sum(rec["append_ms"]) / len(rec["append_ms"]), 3),
                           "paged_decode_attention": round(1e3 * sum(rec["attn_ms"]) / len(rec["attn_ms"]), 3)}),
            "step_ms_stats": _step_stats(rec["step_ms"]),
            "step_kind": args.step, "overlap_previous": bool(rec["overlap"]),
            "clocks": rec["clocks"],
            "gpu_launches": rec["gpu_launches"],
            "e2e": rec["e2e"],
        }
    # CPU baseline (the oracle as it stands), rank 0 at N=1 only, on the machine's host cores; the
    # other workloads likewise at one GPU only.
    if rank == 0 and world == 1:
        if not args.no_cpu_baseline:
            with nvtx("cpu_baseline"):
                line["cpu_baseline"] = cpu_baseline(wl)
        if wl.name == "bandwidth" and not args.no_other_configs:
            line["other_configs"] = other_configs(args, dev, sampler)
    sampler.stop()
    _dist_teardown(world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_trace(args):
    world, rank, local, dev = _dist_setup()
    sampler = ClockSampler(local)
    sampler.start()
    steps = args.steps if args.steps is not None else 1000
    warmup = args.warmup if args.warmup is not None else 3
    rec = trace_measure(args, dev, steps, warmup, world, sampler, with_cpu=(rank == 0 and world == 1
                                                                            and not args.no_cpu_baseline))
    sampler.stop()
    if rank == 0:
        line = {"metric": METRIC, "value": round(rec["_gbs"], 3), "unit": "GB/s", "n_gpus": world,
                "steps": rec["steps"], "warmup": warmup, "ms_per_step": round(rec["_total_ms"] / rec["steps"], 5),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "bf16 in, f32 accumulate/out", "data": "synthetic (seeded N(0,1) bf16; seeded request trace)",
                "config": {k: rec[k] for k in ("workload", "slots", "layers", "pool_pages", "requests", "prompt",
                                               "new_tokens", "l2", "timing")} | {"parallelism": f"replicas x{world}"},
                **{k: rec[k] for k in ("roofline", "seq_layers_per_s", "host_plan_us_per_step",
                                       "native_plan_us_per_step", "scheduler_stats",
                                       "clocks", "gpu_launches") if k in rec}}
        if "cpu_baseline" in rec:
            line["cpu_baseline"] = rec["cpu_baseline"]
        print(json.dumps(line), flush=True)
    _dist_teardown(world)
    return 0


def run_prefill(args):
    world, rank, local, dev = _dist_setup()
    sampler = ClockSampler(local)
    sampler.start()
    steps = args.steps if args.steps is not None else 500
    warmup = args.warmup if args.warmup is not None else 10
    rec = prefill_measure(args, dev, steps, warmup, world, sampler, with_cpu=(rank == 0 and world == 1
                                                                              and not args.no_cpu_baseline))
    sampler.stop()
    if rank == 0:
        line = {"metric": "paged prefill attention TFLOP/s (causal) and % of the bf16 tensor peak",
                "value": rec["step_tflops"], "unit": "TFLOP/s", "n_gpus": world, "steps": steps, "warmup": warmup,
                "ms_per_step": round(rec["_step_ms"], 5), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16 in, f32 accumulate/out", "data": "synthetic (seeded N(0,1) bf16)",
                "config": {k: rec[k] for k in ("workload", "num_seqs", "prompt_tokens", "layers", "overlap_previous",
                                               "l2", "timing")} | {"q_heads": 32, "kv_heads": 8, "head_dim": 64,
                                                                   "page_tokens": 16},
                "roofline": rec["roofline"], "kernel_us": rec["kernel_us_by_part"], "clocks": rec["clocks"],
                "gpu_launches": rec["gpu_launches"]}
        if "cpu_baseline" in rec:
            line["cpu_baseline"] = rec["cpu_baseline"]
        print(json.dumps(line), flush=True)
    _dist_teardown(world)
    return 0


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
