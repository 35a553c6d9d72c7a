"""Benchmark: paged decode attention (and chunked prefill) on GB300.

One step = one decode step of the E2B-like workload through every layer:
the KV store of the new token on the 7 owning layers and paged decode
attention on all 12 layers (7 owning + 5 KV-shared), batch 64, contexts
U[512, 4096], 8 query heads / 1 KV head, sliding D 256 W 512 / full D 512.
An owning layer's store runs inside its decode launch
(fa_paged_decode_store_attn), so the step is 12 launches of decode_kernel.

Prints one JSON line.  `value` is the achieved HBM bandwidth of the step:
algorithmic bytes (KV the layers must read + q + out + the store's rows)
divided by the device time of the step.  L2 is flushed (256 MiB write)
before every timed step.  Inputs are seeded synthetic N(0,1) bf16.

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload (the only other place this file runs the oracle).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------
# algorithmic bytes
# ----------------------------------------------------------------------------

def visible(L, d):
    return min(int(L), d["window"]) if d["kind"] == W.SLIDING else int(L)


def decode_bytes(d, lens, kv_dtype):
    """Bytes a decode launch must move: K and V rows of every visible key
    (plus the fp32 scales in int8), the queries, the bf16 outputs and lse."""
    q8 = kv_dtype != W.KV_BF16   # int8 / fp8: one byte per element plus an fp32 scale per row
    per_tok = d["num_kv_heads"] * 2 * (d["head_dim"] * (1 if q8 else 2) + (4 if q8 else 0))
    kv = sum(visible(L, d) for L in lens) * per_tok
    B = len(lens)
    qo = B * d["num_q_heads"] * (2 * d["head_dim"] * 2 + 4)
    return kv + qo


def store_bytes(d, B, kv_dtype):
    row_in = d["num_kv_heads"] * d["head_dim"] * 2
    q8 = kv_dtype != W.KV_BF16
    row_out = d["num_kv_heads"] * (d["head_dim"] * (1 if q8 else 2) + (4 if q8 else 0))
    return B * 2 * (row_in + row_out) + B * 4


# ----------------------------------------------------------------------------
# environment helpers
# ----------------------------------------------------------------------------

def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", 0)), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200", "-i", str(self.gpu)], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() in ("active", "1", "yes"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def source_digest(*names):
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "full_attention_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(kernel_tag, digest):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel source that is built now (else None)."""
    p = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.split(":", 1)[0].strip() in ("source_digest", "dram_bytes_per_launch"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_digest") != digest or "dram_bytes_per_launch" not in vals:
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except ValueError:
        return None


# ----------------------------------------------------------------------------
# the decode step on the GPU
# ----------------------------------------------------------------------------

class DecodeStep:
    def __init__(self, w: W.DecodeWorkload, device, seed_offset=0):
        import torch
        import full_attention_gb300 as fa
        self.torch, self.fa = torch, fa
        self.w = w
        self.layers = w.layers
        self.lens = W.seq_lens(w)
        self.B = len(self.lens)
        self.max_len = int(self.lens.max())
        self.device = device
        full = W.plan_pages(self.lens, w.page_size, w.seed)
        self.tables = {}
        num_pages = full.num_pages
        for i, d in enumerate(self.layers):
            if d["kind"] == W.SLIDING and w.sliding_window_table:
                p = W.plan_pages(self.lens, w.page_size, w.seed + 1000, window=d["window"],
                                 max_pages=full.block_table.shape[1])
            else:
                p = full
            self.tables[i] = p.block_table
            num_pages = max(num_pages, p.num_pages)
        self.cache = fa.Cache(self.layers, num_pages, w.page_size, w.kv_dtype)
        # block tables, lengths and slots are written once, before any step
        self.cache.set_flags(fa.FLAG_EARLY_METADATA)
        self.src = [self.cache.source(i) for i in range(len(self.layers))]
        self.slabs = self.cache.allocate(device)
        s0 = 1000 * (seed_offset + 1) + w.seed
        for i, (k, v, ks, vs) in self.slabs.items():
            if w.kv_dtype == W.KV_BF16:
                k.copy_(W.randn_bf16(tuple(k.shape), s0 + 2 * i, device))
                v.copy_(W.randn_bf16(tuple(v.shape), s0 + 2 * i + 1, device))
            else:
                self._fill_8bit(i, s0)
        self.bt = {i: torch.from_numpy(t).to(device) for i, t in self.tables.items()}
        self.lens_dev = torch.from_numpy(self.lens).to(device)
        self.q, self.out, self.lse, self.ws = {}, {}, {}, {}
        for i, d in enumerate(self.layers):
            self.q[i] = W.randn_bf16((self.B, d["num_q_heads"], d["head_dim"]), s0 + 100 + i, device)
            self.out[i] = torch.empty((self.B, d["num_q_heads"], d["head_dim"]), dtype=torch.bfloat16, device=device)
            self.lse[i] = torch.empty((self.B, d["num_q_heads"]), dtype=torch.float32, device=device)
            n = self.cache.decode_workspace_bytes(i, self.B, self.max_len)
            self.ws[i] = fa.workspace(n, device) if n else None
        self.new = {}
        for i in self.slabs:
            d = self.layers[i]
            sl = torch.from_numpy(W.decode_slot_mapping(self.lens, self.tables[i], w.page_size)).to(device)
            self.new[i] = (W.randn_bf16((self.B, d["num_kv_heads"], d["head_dim"]), s0 + 200 + i, device),
                           W.randn_bf16((self.B, d["num_kv_heads"], d["head_dim"]), s0 + 300 + i, device), sl)
        # the multi-layer variant of the step: one store launch for the owning
        # layers, then one decode launch per head_dim group
        self.groups = [g for g in ([i for i, d in enumerate(self.layers) if d["head_dim"] == D] for D in (256, 512)) if g]
        self.ws_group = []
        for g in self.groups:
            n = self.cache.decode_layers_workspace_bytes(g, self.B, self.max_len)
            self.ws_group.append(fa.workspace(n, device) if n else None)
        self.decode_bytes = [decode_bytes(d, self.lens, w.kv_dtype) for d in self.layers]
        self.store_bytes = sum(store_bytes(self.layers[i], self.B, w.kv_dtype) for i in self.slabs)
        self.step_bytes = sum(self.decode_bytes) + self.store_bytes
        # the same step with each slab's K/V counted once (a KV-shared layer
        # reads its source's pages again; what DRAM must serve at least)
        qo = [self.B * d["num_q_heads"] * (2 * d["head_dim"] * 2 + 4) for d in self.layers]
        self.unique_bytes = sum(self.decode_bytes[i] for i in self.slabs) + \
            sum(qo[i] for i in range(len(self.layers)) if self.src[i] != i) + self.store_bytes
        torch.cuda.synchronize()

    def _fill_8bit(self, i, s0):
        torch = self.torch
        d = self.layers[i]
        slots = []
        for b, L in enumerate(self.lens):
            lo = max(0, int(L) - d["window"]) if d["kind"] == W.SLIDING else 0
            slots.append(W.slots_for_positions(self.tables[i][b], np.arange(lo, int(L)), self.w.page_size))
        sl = torch.from_numpy(np.concatenate(slots)).to(self.device)
        for c0 in range(0, sl.numel(), 1 << 18):
            part = sl[c0:c0 + (1 << 18)]
            k = W.randn_bf16((part.numel(), d["num_kv_heads"], d["head_dim"]), s0 + 7 * i + c0, self.device)
            v = W.randn_bf16((part.numel(), d["num_kv_heads"], d["head_dim"]), s0 + 7 * i + c0 + 1, self.device)
            self.cache.store(i, k, v, part)

    def launches_per_step(self):
        return len(self.layers)   # one launch per layer: owning layers store their rows in it

    def run_layers(self):
        """The same step through the multi-layer calls: the owning layers'
        stores in one launch, then one decode launch per head_dim group."""
        own = sorted(self.slabs)
        self.cache.store_layers(own, [self.new[i][0] for i in own], [self.new[i][1] for i in own],
                                [self.new[i][2] for i in own])
        for g, ws in zip(self.groups, self.ws_group):
            self.cache.decode_layers(g, [self.q[i] for i in g], [self.bt[i] for i in g], self.lens_dev,
                                     self.max_len, [self.out[i] for i in g], [self.lse[i] for i in g], ws)

    def run(self, events=None):
        for i in range(len(self.layers)):
            if events is not None:
                events[i][0].record()
            if self.src[i] == i:
                k, v, sl = self.new[i]
                self.cache.decode_store(i, self.q[i], k, v, sl, self.bt[i], self.lens_dev, self.max_len,
                                        self.out[i], self.lse[i], self.ws[i])
            else:
                self.cache.decode(i, self.q[i], self.bt[i], self.lens_dev, self.max_len, self.out[i],
                                  self.lse[i], self.ws[i])
            if events is not None:
                events[i][1].record()


def reduce_over_ranks(value: float, op: str, world: int, device="cpu") -> float:
    """max or sum of one float over the ranks of the process group (every rank
    gets the result); the value itself when running alone.  Replicas are
    independent: this is the only cross-rank exchange, outside the timed
    region."""
    if world <= 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX if op == "max" else torch.distributed.ReduceOp.SUM)
    return float(t.item())


def gpu_arm(args, rank, world):
    import torch
    import full_attention_gb300 as fa
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = W.ALL[args.workload]()
    step = DecodeStep(w, dev, seed_offset=rank)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    nl = len(step.layers)
    events = [(torch.cuda.Event(enable_timing=True, external=True),
               torch.cuda.Event(enable_timing=True, external=True)) for _ in range(nl)]

    def capture(ev):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                step.run(ev)
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step.run(ev)
            torch.cuda.synchronize()
            return g
        except Exception as e:   # capture unsupported: time eager launches
            print(f"# graph capture failed ({e}); timing eager launches", file=sys.stderr)
            torch.cuda.synchronize()
            return None

    # the step itself is timed from a graph with no event nodes between its
    # kernels; a second graph with an event pair around every decode launch
    # gives the per-launch durations of the roofline
    graph = capture(None)
    graph_ev = capture(events)
    st0, st1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ms, dec_ms = [], [0.0] * nl
    gpu_idx = getattr(torch.cuda.get_device_properties(dev), "pci_bus_id", None) or dev.index
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    n_ev = max(1, min(args.steps, 500))
    with ClockSampler(gpu_idx) as clk:
        for _ in range(args.steps):
            flush.zero_()
            st0.record()
            if graph is not None:
                graph.replay()
            else:
                step.run()
            st1.record()
            st1.synchronize()
            step_ms.append(st0.elapsed_time(st1))
        wall = time.perf_counter() - wall0
        for _ in range(n_ev):
            flush.zero_()
            if graph_ev is not None:
                graph_ev.replay()
            else:
                step.run(events)
            torch.cuda.synchronize()
            for i in range(nl):
                dec_ms[i] += events[i][0].elapsed_time(events[i][1])
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    assert fa.device_error() == 0
    t_step = sum(step_ms) / len(step_ms) / 1e3       # seconds per step (device time)
    # the slowest rank's time; the bytes every rank's replica moved (replicas
    # are seeded per rank, so their lengths differ)
    t_max = reduce_over_ranks(sum(step_ms), "max", world, dev) / 1e3 / args.steps
    job_bytes = reduce_over_ranks(step.step_bytes, "sum", world, dev)
    job_unique = reduce_over_ranks(step.unique_bytes, "sum", world, dev)
    hbm, bf16, bf16s, peak_src = measured_peaks()
    dec_bytes = sum(step.decode_bytes)
    dec_time = sum(dec_ms) / 1e3 / n_ev               # seconds of decode launches per step
    per_kind = {}
    for kind, name in ((W.FULL, "full"), (W.SLIDING, "sliding")):
        idx = [i for i, d in enumerate(step.layers) if d["kind"] == kind]
        b = sum(step.decode_bytes[i] for i in idx)
        t = sum(dec_ms[i] for i in idx) / 1e3 / n_ev
        per_kind[name] = {"launches_per_step": len(idx), "gb_per_s": round(b / t / 1e9, 1) if t else None,
                          "us_per_launch": round(t / len(idx) * 1e6, 2) if idx else None}
    # Every launch of the step is decode_kernel (stores run inside it), so
    # its average launch duration in the step is the step time / launches;
    # the event-bracketed graph above gives each layer's time run alone.
    launch_bytes = step.step_bytes / nl
    achieved = step.step_bytes / t_step / 1e9
    digest = source_digest("fa_decode.cu", "fa_ptx.cuh")
    traffic = profiled_traffic(f"decode_{args.workload}", digest)
    clocks = clk.summary()
    res = {
        "metric": "paged decode-attn achieved HBM GB/s (% of peak); chunked-prefill TFLOP/s",
        "value": round(job_bytes / t_max / 1e9, 1),
        "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(t_max * 1e3, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {W.KV_BF16: "bf16", W.KV_INT8: "int8", W.KV_FP8: "fp8"}[w.kv_dtype],
        "data": "synthetic (seeded N(0,1) bf16)",
        "config": {"workload": w.name, "batch": step.B, "layers": nl, "page_size": w.page_size,
                   "max_ctx": step.max_len, "l2": "flushed before every step (256 MiB write)",
                   "graph": graph is not None, "early_metadata": True,
                   "parallelism": f"replicas x{world}"},
        "tokens_per_s": round(step.B * world / t_max, 1),
        "pct_of_peak": round(100 * job_bytes / world / t_max / 1e9 / hbm, 1),
        "unique_bytes_per_step": int(step.unique_bytes),
        "unique_gb_per_s": round(job_unique / t_max / 1e9, 1),
        "roofline": {"kernel": "decode_kernel (paged decode attention, split-K merged in-kernel)",
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 3), "peak_source": peak_src,
                     "traffic": traffic, "algorithmic_bytes_per_launch": round(launch_bytes),
                     "avg_launch_us_in_step": round(t_step / nl * 1e6, 2),
                     "per_kind_alone": per_kind,
                     "alone_gb_per_s": round(dec_bytes / dec_time / 1e9, 1)},
        "gpu_launches": step.launches_per_step() * args.steps,
        "clocks": clocks,
        "wall_s_timed": round(wall, 3),
    }
    res["multi_layer_step"] = multi_layer_measure(step, args, torch, flush, hbm)
    res["decode_store"] = decode_store_measure(step, torch)
    # end to end on every rank; the job's bytes over the slowest rank's time
    if world > 1:
        torch.distributed.barrier()
    e2 = e2e_decode(step, args, torch)
    t_e2e = reduce_over_ranks(e2["ms_per_step"], "max", world, dev) / 1e3
    e2["value"] = round(job_bytes / t_e2e / 1e9, 1)
    e2["ms_per_step"] = round(t_e2e * 1e3, 4)
    e2["h2d_bytes_per_step"] = int(reduce_over_ranks(e2["h2d_bytes_per_step"], "sum", world, dev))
    e2["d2h_bytes_per_step"] = int(reduce_over_ranks(e2["d2h_bytes_per_step"], "sum", world, dev))
    res["e2e"] = e2
    if args.workload == "tiny_decode":
        res["config"]["role"] = "parity only: latency-bound (about 26 KB per step); GB/s is not a roofline figure"
        res["roofline"]["frac"] = None
    if rank == 0:
        if args.workload == "e2b_decode" and not args.no_prefill:
            res["prefill"] = prefill_measure(args, dev)
        if args.workload == "e2b_decode" and not args.no_subrecords:
            # the other decode workloads, driver-observed: long context, int8,
            # fp8 (configs 4 and 5, and 5 in the fp8 format) and the tiny one
            del step
            torch.cuda.empty_cache()
            res["workloads"] = {n: decode_subrecord(n, args, dev, flush)
                                for n in ("long_decode", "int8_decode", "fp8_decode", "tiny_decode")}
        if not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
        print(json.dumps(res), flush=True)


def time_graph(torch, fn, flush, n):
    """Capture fn() in a CUDA graph (eager if capture fails) and return its
    mean device time in seconds over n replays, L2 flushed before each."""
    g = None
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
    except Exception as e:
        print(f"# graph capture failed ({e}); timing eager launches", file=sys.stderr)
        torch.cuda.synchronize()
        g = None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tot = 0.0
    for _ in range(n):
        flush.zero_()
        e0.record()
        g.replay() if g is not None else fn()
        e1.record()
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    return tot / n / 1e3, g is not None


def decode_subrecord(name, args, dev, flush):
    """A compact record of another decode workload (the same 12-layer step,
    per-layer launches in a graph, L2 flushed before every step): GB/s against
    the measured HBM peak, and the oracle on a sample of it.  The tiny
    workload moves 26 KB per step: it is a parity case, so it gets its
    latency only."""
    import torch
    import full_attention_gb300 as fa
    w = W.ALL[name]()
    step = DecodeStep(w, dev)
    for _ in range(max(3, args.warmup)):
        step.run()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    n = max(5, min(args.steps, 100))
    t, graphed = time_graph(torch, step.run, flush, n)
    tm, _ = time_graph(torch, step.run_layers, flush, n)
    assert fa.device_error() == 0
    hbm = measured_peaks()[0]
    rec = {"workload": w.name, "ms_per_step": round(t * 1e3, 4), "tokens_per_s": round(step.B / t, 1),
           "dtype": {W.KV_BF16: "bf16", W.KV_INT8: "int8", W.KV_FP8: "fp8"}[w.kv_dtype],
           "steps": n, "graph": graphed, "l2": "flushed before every step (256 MiB write)"}
    if name == "tiny_decode":
        rec.update({"role": "parity only: latency-bound (about 26 KB per step), no bandwidth figure",
                    "unit": "ms per step", "value": rec["ms_per_step"]})
    else:
        gbs = step.step_bytes / t / 1e9
        rec.update({"value": round(gbs, 1), "unit": "GB/s", "pct_of_peak": round(100 * gbs / hbm, 1),
                    "roofline": {"kernel": "decode_kernel", "bound": "hbm", "achieved": round(gbs, 1),
                                 "peak": hbm, "unit": "GB/s", "frac": round(gbs / hbm, 3),
                                 "algorithmic_bytes_per_launch": round(step.step_bytes / len(step.layers)),
                                 "traffic": profiled_traffic(f"decode_{name}", source_digest("fa_decode.cu",
                                                                                            "fa_ptx.cuh"))},
                    "multi_layer_step": {"ms_per_step": round(tm * 1e3, 4),
                                         "unique_gb_per_s": round(step.unique_bytes / tm / 1e9, 1),
                                         "frac_unique_of_peak": round(step.unique_bytes / tm / 1e9 / hbm, 3)}})
    if not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(name, min(args.cpu_seconds, 6.0))
    del step
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def decode_store_measure(step, torch):
    """The per-token store of a decode step on its own (fa_kv_store of the B
    current rows of one owning layer per head_dim; in the timed step these
    stores are fused into the decode launches).  They are latency-bound, so
    the figure is microseconds per call: 50 back-to-back calls in a graph,
    and a single call between two events inside a graph."""
    out = {}
    for D in (256, 512):
        owners = [i for i in sorted(step.slabs) if step.layers[i]["head_dim"] == D]
        if not owners:
            continue
        i = owners[0]
        k, v, sl = step.new[i]
        call = lambda: step.cache.store(i, k, v, sl)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        g = None
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                call()
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                for _ in range(50):
                    call()
            torch.cuda.synchronize()
        except Exception as e:
            print(f"# decode store graph capture failed ({e})", file=sys.stderr)
            torch.cuda.synchronize()
            g = None
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        back = None
        if g is not None:
            g.replay()
            torch.cuda.synchronize()
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            back = e0.elapsed_time(e1) * 1e3 / 50
        # one call between two events, all three captured in a graph, so the
        # interval is the device's (the host's launch latency stays outside)
        single = []
        a, b = torch.cuda.Event(enable_timing=True, external=True), torch.cuda.Event(enable_timing=True, external=True)
        try:
            g1 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1):
                a.record()
                call()
                b.record()
            torch.cuda.synchronize()
            for _ in range(20):
                g1.replay()
                torch.cuda.synchronize()
                single.append(a.elapsed_time(b) * 1e3)
        except Exception as e:
            print(f"# decode store single-call graph failed ({e})", file=sys.stderr)
            torch.cuda.synchronize()
            single = [float("nan")]
        nb = store_bytes(step.layers[i], step.B, step.w.kv_dtype)
        out[f"D{D}"] = {"layer": i, "rows": step.B * step.layers[i]["num_kv_heads"] * 2, "bytes_per_call": nb,
                        "us_per_call_back_to_back": None if back is None else round(back, 2),
                        "us_per_call_single_median": round(float(np.median(single)), 2)}
    return out


def multi_layer_measure(step, args, torch, flush, hbm):
    """The step through fa_kv_store_layers + fa_paged_decode_attn_layers (one
    store launch, one decode launch per head_dim group): same bytes, same
    outputs, fewer launch ramps and tails.  A separate figure: in a model each
    layer's queries come from the previous layer, so the per-layer step is the
    headline."""
    import full_attention_gb300 as fa
    for _ in range(3):
        step.run_layers()
    torch.cuda.synchronize()
    g = None
    try:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step.run_layers()
        torch.cuda.current_stream().wait_stream(s)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step.run_layers()
        torch.cuda.synchronize()
    except Exception as e:
        print(f"# multi-layer graph capture failed ({e})", file=sys.stderr)
        torch.cuda.synchronize()
        g = None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(args.steps, 400))
    tot = 0.0
    for _ in range(n):
        flush.zero_()
        e0.record()
        if g is not None:
            g.replay()
        else:
            step.run_layers()
        e1.record()
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    t = tot / n / 1e3
    gbs = step.step_bytes / t / 1e9
    ub = step.unique_bytes / t / 1e9
    # the shared layers read their source's slab in the same launch, so those
    # repeated reads come from L2: the step's algorithmic bytes per second can
    # exceed the HBM peak.  The figure against HBM is therefore the unique
    # bytes (each slab once) per second; the algorithmic rate is kept apart
    return {"value": round(ub, 1), "unit": "GB/s (unique bytes)", "frac_of_peak": round(ub / hbm, 3),
            "ms_per_step": round(t * 1e3, 4), "tokens_per_s": round(step.B / t, 1),
            "unique_bytes_per_step": int(step.unique_bytes), "unique_gb_per_s": round(ub, 1),
            "frac_unique_of_peak": round(ub / hbm, 3),
            "algorithmic_gb_per_s_l2_included": round(gbs, 1),
            "launches_per_step": 1 + len(step.groups), "graph": g is not None}


def _arena_offsets(tensors):
    """Byte offsets of `tensors` laid end to end in 256-byte aligned pieces, and the total."""
    offs, n = [], 0
    for t in tensors:
        offs.append(n)
        n += (t.numel() * t.element_size() + 255) // 256 * 256
    return offs, n


def _arena(torch, tensors, device, pinned):
    """One byte buffer holding `tensors` end to end (256-byte aligned pieces);
    returns (buffer, views with the tensors' shapes and dtypes)."""
    offs, n = _arena_offsets(tensors)
    buf = torch.empty(max(n, 1), dtype=torch.uint8, device=device)
    if pinned:
        buf = buf.pin_memory()
    views = [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape) for o, t in zip(offs, tensors)]
    return buf, views


def e2e_decode(step, args, torch):
    """Same metric through the public API with host buffers: every step copies
    all of its inputs (queries, new k/v rows, slots, lengths, tables) from a
    pinned host buffer into a device buffer the calls read (one copy), runs
    the step, and reads every layer's output back into a pinned host buffer
    (one copy).  Two device buffers alternate between steps, and the copies
    run on two copy streams ordered by events, so a step's copies overlap the
    neighbouring steps' compute; every step's copies lie inside the timed
    region, which spans all steps."""
    dev = step.device
    keys = [("q", i) for i in sorted(step.q)] + [("new", i, j) for i in sorted(step.new) for j in range(3)] + \
        [("bt", i) for i in sorted(step.bt)] + [("lens",)]

    def get(k):
        if k[0] == "q":
            return step.q[k[1]]
        if k[0] == "new":
            return step.new[k[1]][k[2]]
        if k[0] == "bt":
            return step.bt[k[1]]
        return step.lens_dev

    saved = (dict(step.q), dict(step.new), dict(step.bt), step.lens_dev, dict(step.out))
    srcs = [get(k) for k in keys]
    outs = [step.out[i] for i in sorted(step.out)]
    h_in, h_views = _arena(torch, [t.cpu() for t in srcs], "cpu", True)
    for hv, t in zip(h_views, srcs):
        hv.copy_(t.cpu())
    bufs = []
    for _ in range(2):
        d_in, d_views = _arena(torch, srcs, dev, False)
        d_out, d_oviews = _arena(torch, outs, dev, False)
        h_out, _ = _arena(torch, [t.cpu() for t in outs], "cpu", True)
        views = {"q": {}, "new": {}, "bt": {}, "lens": None}
        for k, v in zip(keys, d_views):
            if k[0] == "q":
                views["q"][k[1]] = v
            elif k[0] == "new":
                views["new"].setdefault(k[1], [None] * 3)[k[2]] = v
            elif k[0] == "bt":
                views["bt"][k[1]] = v
            else:
                views["lens"] = v
        views["new"] = {i: tuple(v) for i, v in views["new"].items()}
        views["out"] = {i: v for i, v in zip(sorted(saved[4]), d_oviews)}
        bufs.append((d_in, d_out, h_out, views, d_oviews))
    bi = int(h_in.numel())
    bo = int(bufs[0][2].numel())
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cs = torch.cuda.current_stream()
    xs_in, xs_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("in", "done", "out")}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(args.steps, 200))

    def one_step(i):
        b = i % 2
        d_in, d_out, h_out, views, _ = bufs[b]
        with torch.cuda.stream(xs_in):   # this step's inputs, once buffer b's last user is done
            xs_in.wait_event(ev["done"][b])
            d_in.copy_(h_in, non_blocking=True)
            ev["in"][b].record(xs_in)
        cs.wait_event(ev["in"][b])
        cs.wait_event(ev["out"][b])      # buffer b's previous outputs have been read back
        step.q, step.new, step.bt, step.lens_dev, step.out = (views["q"], views["new"], views["bt"], views["lens"],
                                                              views["out"])
        step.run()
        ev["done"][b].record(cs)
        with torch.cuda.stream(xs_out):
            xs_out.wait_event(ev["done"][b])
            h_out.copy_(d_out, non_blocking=True)
            ev["out"][b].record(xs_out)

    try:
        for i in range(4):               # warm-up of the pipeline
            one_step(i)
        torch.cuda.synchronize()
        flush.zero_()
        e0.record(cs)
        xs_in.wait_stream(cs)
        xs_out.wait_stream(cs)
        for i in range(n):
            one_step(i)
        cs.wait_stream(xs_out)
        e1.record(cs)
        e1.synchronize()
        tot = e0.elapsed_time(e1)
        last = bufs[(n - 1) % 2]
        got = [last[2][o.data_ptr() - last[1].data_ptr():][: t.numel() * t.element_size()].clone()
               for o, t in zip(last[4], outs)]
    finally:
        step.q, step.new, step.bt, step.lens_dev, step.out = saved
    # the outputs read back are the step's: compare with the device-resident path
    step.run()
    torch.cuda.synchronize()
    for g, t in zip(got, outs):
        assert torch.equal(g, t.contiguous().view(torch.uint8).view(-1).cpu()), "end-to-end output differs"
    t = tot / n / 1e3
    return {"value": round(step.step_bytes / t / 1e9, 1), "unit": "GB/s", "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "ms_per_step": t * 1e3,
            "path": "C-ABI calls; per step one host-to-device and one device-to-host copy (pinned buffers), "
                    "double-buffered on two copy streams so copies overlap the neighbouring steps"}


def visible_pairs(kind, window, P, n):
    """(query, key) pairs a chunk of n tokens over a prefix of P sees."""
    tot = 0
    for i in range(n):
        q = P + i
        tot += min(window, q + 1) if kind == W.SLIDING else q + 1
    return tot


class PrefillStep:
    """The chunked-prefill workload: B prompts of S tokens in chunks of C; per
    chunk and owning layer, the KV store of the chunk rows then extend."""

    def __init__(self, w: W.ExtendWorkload, device):
        import torch
        import full_attention_gb300 as fa
        self.torch, self.fa, self.w, self.device = torch, fa, w, device
        B, S, C = w.batch, w.prompt_len, w.chunk
        self.nchunks = S // C
        lens = np.full(B, S, np.int32)
        plan = W.plan_pages(lens, w.page_size, w.seed)
        self.cache = fa.Cache(w.layers, plan.num_pages, w.page_size, w.kv_dtype)
        self.cache.set_flags(fa.FLAG_EARLY_METADATA)
        # the extend split workspace: a launch whose last wave would leave
        # more than half of the SMs idle runs that wave's jobs as two CTAs each
        self.split_ws = fa.workspace(fa.extend_workspace_bytes(), device)
        self.cache.bind_extend_workspace(self.split_ws)
        self.slabs = self.cache.allocate(device)
        for k, v, _, _ in self.slabs.values():
            k.zero_()
            v.zero_()
        self.bt = torch.from_numpy(plan.block_table).to(device)
        self.indptr = torch.arange(0, B * C + 1, C, dtype=torch.int32, device=device)
        self.inputs = []      # [chunk][layer] -> (q, k, v, slots)
        self.prefix = []
        self.flops = []       # [chunk][layer]
        for c in range(self.nchunks):
            P = c * C
            self.prefix.append(torch.full((B,), P, dtype=torch.int32, device=device))
            pos = np.arange(P, P + C)
            slots = np.concatenate([W.slots_for_positions(plan.block_table[b], pos, w.page_size) for b in range(B)])
            row, fl = [], []
            for li, d in enumerate(w.layers):
                s0 = w.seed * 1000 + 10 * c + 3 * li
                q = W.randn_bf16((B * C, d["num_q_heads"], d["head_dim"]), s0, device)
                k = W.randn_bf16((B * C, d["num_kv_heads"], d["head_dim"]), s0 + 1, device)
                v = W.randn_bf16((B * C, d["num_kv_heads"], d["head_dim"]), s0 + 2, device)
                row.append((q, k, v, torch.from_numpy(slots).to(device), self.prefix[c], self.indptr))
                fl.append(4.0 * d["head_dim"] * d["num_q_heads"] * B *
                          visible_pairs(d["kind"], d["window"], P, C))
            self.inputs.append(row)
            self.flops.append(fl)
        self.out = [torch.empty((B * C, d["num_q_heads"], d["head_dim"]), dtype=torch.bfloat16, device=device)
                    for d in w.layers]
        self.total_flops = sum(sum(f) for f in self.flops)
        self.tokens = B * S
        torch.cuda.synchronize()

    def launches(self):
        return self.nchunks * len(self.w.layers) * 2

    def store_bytes(self, li):
        """Bytes one chunk store of layer li must move: the chunk's bf16 k, v
        rows read, their slab rows (and 8-bit scales) written."""
        d = self.w.layers[li]
        q8 = self.w.kv_dtype != W.KV_BF16
        rows = self.w.batch * self.w.chunk * d["num_kv_heads"] * 2
        return rows * (d["head_dim"] * 2 + d["head_dim"] * (1 if q8 else 2) + (4 if q8 else 0)) + \
            self.w.batch * self.w.chunk * 4

    def run(self, events=None, store_events=None, inputs=None, outs=None, per_chunk=None):
        """One prefill: per chunk and layer the store of the chunk rows, then
        extend.  `inputs`/`outs` replace the device-resident tensors (the
        end-to-end path); per_chunk(c, phase) runs before ("in") and after
        ("out") each chunk's calls."""
        C = self.w.chunk
        inputs = self.inputs if inputs is None else inputs
        for c in range(self.nchunks):
            if per_chunk is not None:
                per_chunk(c, "in")
            for li in range(len(self.w.layers)):
                q, k, v, slots, prefix, indptr = inputs[c][li]
                if store_events is not None:
                    store_events[c][li][0].record()
                self.cache.store(li, k, v, slots)
                if store_events is not None:
                    store_events[c][li][1].record()
                if events is not None:
                    events[c][li][0].record()
                out = self.out[li] if outs is None else outs[c][li]
                self.cache.extend(li, q, k, v, indptr, prefix, self.bt, C, c * C, out)
                if events is not None:
                    events[c][li][1].record()
            if per_chunk is not None:
                per_chunk(c, "out")


def prefill_measure(args, dev):
    """Chunked prefill TFLOP/s on the chunked-prefill workload (extend kernel),
    its slabs in the format --prefill-kv names (bf16 by default); the chunk
    stores' GB/s; the same prefill end to end from host buffers; the oracle's
    rate on a sample of the same workload."""
    import dataclasses
    import torch
    import full_attention_gb300 as fa
    w = W.chunked_prefill()
    kv = {"bf16": W.KV_BF16, "int8": W.KV_INT8, "fp8": W.KV_FP8}[getattr(args, "prefill_kv", "bf16")]
    if kv != w.kv_dtype:
        w = dataclasses.replace(w, kv_dtype=kv)
    step = PrefillStep(w, dev)
    for _ in range(3):
        step.run()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    nl = len(w.layers)

    def ev_grid():
        return [[(torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) for _ in range(nl)] for _ in range(step.nchunks)]
    events, store_events = ev_grid(), ev_grid()

    def capture(ev, sev):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s):
                step.run(ev, sev)
            torch.cuda.current_stream().wait_stream(s)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step.run(ev, sev)
            torch.cuda.synchronize()
            return g
        except Exception as e:
            print(f"# prefill graph capture failed ({e})", file=sys.stderr)
            torch.cuda.synchronize()
            return None

    g_plain, g_ev = capture(None, None), capture(events, store_events)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = max(3, min(args.prefill_steps, 50))
    tot = 0.0
    for _ in range(reps):
        flush.zero_()
        e0.record()
        g_plain.replay() if g_plain is not None else step.run()
        e1.record()
        e1.synchronize()
        tot += e0.elapsed_time(e1)
    t = tot / reps / 1e3
    ext_ms = [[0.0] * nl for _ in range(step.nchunks)]
    st_ms = [[0.0] * nl for _ in range(step.nchunks)]
    for _ in range(reps):
        flush.zero_()
        g_ev.replay() if g_ev is not None else step.run(events, store_events)
        torch.cuda.synchronize()
        for c in range(step.nchunks):
            for li in range(nl):
                ext_ms[c][li] += events[c][li][0].elapsed_time(events[c][li][1]) / reps
                st_ms[c][li] += store_events[c][li][0].elapsed_time(store_events[c][li][1]) / reps
    assert fa.device_error() == 0
    hbm, bf16, bf16s, src = measured_peaks()
    ext_t = sum(sum(r) for r in ext_ms) / 1e3
    per_layer = {}
    for li, d in enumerate(w.layers):
        fl = sum(step.flops[c][li] for c in range(step.nchunks))
        tl = sum(ext_ms[c][li] for c in range(step.nchunks)) / 1e3
        per_layer["sliding D256" if d["kind"] == W.SLIDING else "full D512"] = {
            "tflops": round(fl / tl / 1e12, 1), "ms": round(tl * 1e3, 4),
            "executed_flop_factor": 1.5 if d["head_dim"] == 512 else 1.0}
    achieved = step.total_flops / ext_t / 1e12
    # the chunk stores (store_kernel), each event-bracketed: algorithmic bytes / time
    st_bytes = sum(step.store_bytes(li) for li in range(nl)) * step.nchunks
    st_t = sum(sum(r) for r in st_ms) / 1e3
    store = {"kernel": "store_kernel (chunk rows into the paged slab)", "bound": "hbm",
             "achieved": round(st_bytes / st_t / 1e9, 1), "peak": hbm, "unit": "GB/s",
             "frac": round(st_bytes / st_t / 1e9 / hbm, 3), "peak_source": src,
             "bytes_per_call": {("sliding D256" if d["kind"] == W.SLIDING else "full D512"): step.store_bytes(li)
                                for li, d in enumerate(w.layers)},
             "us_per_call": round(st_t / (step.nchunks * nl) * 1e6, 2),
             "traffic": profiled_traffic("store_chunked_prefill", source_digest("fa_store.cu", "fa_row.cuh"))}
    res = {"workload": w.name, "kv_format": getattr(args, "prefill_kv", "bf16"),
           "value": round(step.total_flops / t / 1e12, 1), "unit": "TFLOP/s",
           "ms_per_prefill": round(t * 1e3, 4), "tokens_per_s": round(step.tokens / t, 1),
           "algorithmic_tflop": round(step.total_flops / 1e12, 4),
           "roofline": {"kernel": "extend_kernel (tcgen05 chunked prefill)", "bound": "tensor",
                        "achieved": round(achieved, 1), "peak": bf16, "unit": "TFLOP/s",
                        "frac": round(achieved / bf16, 3), "peak_source": src + " (dense bf16 burst)",
                        "traffic": profiled_traffic("extend_chunked_prefill" + ("" if kv == W.KV_BF16 else
                                                                                  "_" + args.prefill_kv),
                                                    source_digest("fa_extend.cu", "fa_ptx.cuh")),
                        "algorithmic_flop_per_launch": round(step.total_flops / (step.nchunks * nl)),
                        "per_layer": per_layer},
           "store": store,
           "gpu_launches_per_prefill": step.launches(), "graph": g_plain is not None,
           "extend_split": "workspace bound: a launch whose last wave would fill at most half of the SMs "
                           "runs that wave's jobs as two CTAs each (head_dim 512: 56 of 512 jobs on 152 SMs)"}
    res["e2e"] = e2e_prefill(step, args, torch, flush)
    if not args.no_cpu_baseline:
        res["cpu_baseline"] = prefill_cpu_baseline(w, args.cpu_seconds)
    return res


def e2e_prefill(step, args, torch, flush):
    """The prefill through the public API from host buffers: per chunk one
    host-to-device copy of that chunk's inputs (q, k, v and slots of both
    layers, the prefix lengths, the chunk offsets) from one pinned host
    buffer, the stores and extends reading the copied views, and one
    device-to-host copy of the chunk's outputs into one pinned host buffer.
    The copies run on two copy streams, ordered by events, so chunk c + 1's
    inputs and chunk c - 1's outputs move while chunk c computes; all of a
    prefill's copies lie inside the timed region."""
    import full_attention_gb300 as fa
    nl = len(step.w.layers)
    nc = step.nchunks
    order = [(c, li, j) for c in range(nc) for li in range(nl) for j in range(6)]
    srcs = [step.inputs[c][li][j] for c, li, j in order]
    offs, n_in = _arena_offsets(srcs)
    d_in, d_views = _arena(torch, srcs, step.device, False)
    h_in, h_views = _arena(torch, [x.cpu() for x in srcs], "cpu", True)
    for hv, x in zip(h_views, srcs):
        hv.copy_(x.cpu())
    views = {k: v for k, v in zip(order, d_views)}
    inputs = [[tuple(views[(c, li, j)] for j in range(6)) for li in range(nl)] for c in range(nc)]
    outs_t = [step.out[li] for c in range(nc) for li in range(nl)]
    ooffs, n_out = _arena_offsets(outs_t)
    d_out, d_oviews = _arena(torch, outs_t, step.device, False)
    h_out, _ = _arena(torch, [x.cpu() for x in outs_t], "cpu", True)
    outs = [[d_oviews[c * nl + li] for li in range(nl)] for c in range(nc)]
    # byte range of each chunk in the two arenas
    in_rng = [(offs[c * nl * 6], offs[(c + 1) * nl * 6] if c + 1 < nc else n_in) for c in range(nc)]
    out_rng = [(ooffs[c * nl], ooffs[(c + 1) * nl] if c + 1 < nc else n_out) for c in range(nc)]
    cs = torch.cuda.current_stream()
    xs_in, xs_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev = {k: [torch.cuda.Event() for _ in range(nc)] for k in ("in", "done", "out")}

    def one_prefill():
        with torch.cuda.stream(xs_in):   # every chunk's inputs, each once its last reader is done
            for c in range(nc):
                a, b = in_rng[c]
                xs_in.wait_event(ev["done"][c])
                d_in[a:b].copy_(h_in[a:b], non_blocking=True)
                ev["in"][c].record(xs_in)

        def per_chunk(c, phase):
            if phase == "in":
                cs.wait_event(ev["in"][c])
                cs.wait_event(ev["out"][c])   # the previous prefill's chunk-c outputs were read back
            else:
                ev["done"][c].record(cs)
                with torch.cuda.stream(xs_out):
                    xs_out.wait_event(ev["done"][c])
                    a, b = out_rng[c]
                    h_out[a:b].copy_(d_out[a:b], non_blocking=True)
                    ev["out"][c].record(xs_out)

        step.run(inputs=inputs, outs=outs, per_chunk=per_chunk)

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(3, min(args.prefill_steps, 20))
    for _ in range(2):
        one_prefill()
    torch.cuda.synchronize()
    flush.zero_()
    e0.record(cs)
    xs_in.wait_stream(cs)
    xs_out.wait_stream(cs)
    for _ in range(n):
        one_prefill()
    cs.wait_stream(xs_out)
    e1.record(cs)
    e1.synchronize()
    tot = e0.elapsed_time(e1)
    # the last chunk's outputs read back equal the device-resident prefill's
    step.run()
    torch.cuda.synchronize()
    assert fa.device_error() == 0
    for li in range(nl):
        o = step.out[li]
        nb = o.numel() * o.element_size()
        got = h_out[ooffs[(nc - 1) * nl + li]:][:nb]
        assert torch.equal(got, o.contiguous().view(torch.uint8).view(-1).cpu()), "end-to-end prefill output differs"
    t = tot / n / 1e3
    return {"value": round(step.total_flops / t / 1e12, 1), "unit": "TFLOP/s", "h2d_bytes_per_step": int(n_in),
            "d2h_bytes_per_step": int(n_out), "ms_per_step": round(t * 1e3, 4),
            "path": "C-ABI store + extend calls; per chunk one host-to-device and one device-to-host copy "
                    "(pinned buffers) on two copy streams overlapping the compute; a step is one whole prefill"}


# ----------------------------------------------------------------------------
# oracle (CPU baseline and the reference arm)
# ----------------------------------------------------------------------------

def _bf16_normal(r, shape):
    """Seeded N(0,1) values as bf16 bit patterns (input generation, CPU)."""
    x = r.standard_normal(shape, dtype=np.float32).view(np.uint32)
    return ((x + 0x7FFF + ((x >> 16) & 1)) >> 16).astype(np.uint16)


def _oracle_worker(conn, name, units, seed):
    """A spawned process that holds seeded inputs for its (sequence, layer)
    units and, on each request, runs the oracle on the next n of them; only
    the oracle calls are timed."""
    import oracle
    w = W.ALL[name]()
    lens = W.seq_lens(w)
    ps = w.page_size
    r = W.rng(seed)
    data = []
    for b, li in units:
        d = dict(w.layers[li], kv_source=W.KV_OWN)
        L = int(lens[b])
        npg = (L + ps - 1) // ps
        shape = (npg, d["num_kv_heads"], ps, d["head_dim"])
        if w.kv_dtype == W.KV_BF16:
            slab = (_bf16_normal(r, shape), _bf16_normal(r, shape))
        elif w.kv_dtype == W.KV_INT8:
            sc = (r.random(shape[:3], dtype=np.float32) * 0.03).astype(np.float32)
            slab = (r.integers(-127, 128, size=shape, dtype=np.int8), r.integers(-127, 128, size=shape, dtype=np.int8),
                    sc, sc.copy())
        else:
            # e4m3 codes: any byte but the two NaN patterns
            sc = (r.random(shape[:3], dtype=np.float32) * 0.01).astype(np.float32)
            codes = [r.integers(0, 254, size=shape, dtype=np.uint8) for _ in range(2)]
            slab = tuple(np.where(c >= 0x7F, c + 1, c).astype(np.uint8) for c in codes) + (sc, sc.copy())
        q = _bf16_normal(r, (1, d["num_q_heads"], d["head_dim"]))
        data.append((d, slab, q, np.arange(npg, dtype=np.int32)[None], np.array([L], np.int32),
                     decode_bytes(d, [L], w.kv_dtype)))
    conn.send("ready")
    k = 0
    while True:
        n = conn.recv()
        if n is None:
            break
        t = 0.0
        nb = 0
        for _ in range(n):
            d, slab, q, bt, L, by = data[k % len(data)]
            k += 1
            t0 = time.perf_counter()
            oracle.paged_decode([d], 0, {0: slab}, q, bt, L, ps)
            t += time.perf_counter() - t0
            nb += by
        conn.send((t, nb))


def _extend_oracle_worker(conn, kv_dtype, units, seed):
    """A spawned process for the chunked-prefill workload: it holds seeded
    inputs for its (chunk, layer) units (one sequence each, prefix c * chunk,
    a whole chunk of new tokens) and on each request runs the extend oracle on
    the next n of them, for 4 random tokens of the chunk and every query head;
    only the oracle calls are timed.  Replies (seconds, flops)."""
    import oracle
    w = W.chunked_prefill()
    C, ps = w.chunk, w.page_size
    r = W.rng(seed)
    data = []
    for c, li in units:
        d = dict(w.layers[li], kv_source=W.KV_OWN)
        P = c * C
        npg = max(1, (P + ps - 1) // ps)
        shape = (npg, d["num_kv_heads"], ps, d["head_dim"])
        if kv_dtype == W.KV_BF16:
            slab = (_bf16_normal(r, shape), _bf16_normal(r, shape))
        elif kv_dtype == W.KV_INT8:
            sc = (r.random(shape[:3], dtype=np.float32) * 0.03).astype(np.float32)
            slab = (r.integers(-127, 128, size=shape, dtype=np.int8), r.integers(-127, 128, size=shape, dtype=np.int8),
                    sc, sc.copy())
        else:
            sc = (r.random(shape[:3], dtype=np.float32) * 0.01).astype(np.float32)
            codes = [r.integers(0, 254, size=shape, dtype=np.uint8) for _ in range(2)]
            slab = tuple(np.where(x >= 0x7F, x + 1, x).astype(np.uint8) for x in codes) + (sc, sc.copy())
        q = _bf16_normal(r, (C, d["num_q_heads"], d["head_dim"]))
        kx = _bf16_normal(r, (C, d["num_kv_heads"], d["head_dim"]))
        vx = _bf16_normal(r, (C, d["num_kv_heads"], d["head_dim"]))
        data.append((d, slab, q, kx, vx, P, np.arange(npg, dtype=np.int32)[None]))
    conn.send("ready")
    k = 0
    while True:
        n = conn.recv()
        if n is None:
            break
        t = fl = 0.0
        for _ in range(n):
            d, slab, q, kx, vx, P, bt = data[k % len(data)]
            k += 1
            toks = sorted(r.choice(C, size=4, replace=False).tolist())
            rows = [(tt, j) for tt in toks for j in range(d["num_q_heads"])]
            t0 = time.perf_counter()
            oracle.paged_extend([d], 0, {0: slab}, q, kx, vx, np.array([0, C], np.int32), np.array([P], np.int32),
                                bt, ps, rows=rows)
            t += time.perf_counter() - t0
            for tt in toks:
                vis = min(d["window"], P + tt + 1) if d["kind"] == W.SLIDING else P + tt + 1
                fl += 4.0 * d["head_dim"] * d["num_q_heads"] * vis
        conn.send((t, fl))


class OraclePool:
    """One spawned oracle process per host core, each owning a share of the
    workload's units: (sequence, layer) pairs of a decode workload, or
    (chunk, layer) pairs of the chunked-prefill workload.  Spawned, never
    forked, so it is safe after CUDA is initialised."""

    def __init__(self, name, procs=None, seed=0, prefill_kv=None):
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"   # one thread per process: `cores` counts processes
        if prefill_kv is None:
            w = W.ALL[name]()
            B = len(W.seq_lens(w))
            units = [(b, li) for b in range(B) for li in range(len(w.layers))]
        else:
            w = W.chunked_prefill()
            units = [(c, li) for c in range(w.prompt_len // w.chunk) for li in range(len(w.layers))]
        self.procs = max(1, min(procs or os.cpu_count() or 1, len(units) if prefill_kv is None else 10 ** 6))
        self.units = len(units)
        ctx = mp.get_context("spawn")
        self.conns, self.ps = [], []
        for i in range(self.procs):
            a, b = ctx.Pipe()
            if prefill_kv is None:
                target, pargs = _oracle_worker, (b, name, units[i::self.procs], seed + i)
            else:
                # every process holds two of the (chunk, layer) units, spread over all chunks
                mine = [units[(2 * i + j) % len(units)] for j in range(2)]
                target, pargs = _extend_oracle_worker, (b, prefill_kv, mine, seed + i)
            p = ctx.Process(target=target, args=pargs, daemon=True)
            p.start()
            self.conns.append(a)
            self.ps.append(p)
        for c in self.conns:
            assert c.recv() == "ready"

    def run(self, n_per_proc):
        """Every process runs n units; returns (bytes, busy seconds = max over processes)."""
        for c in self.conns:
            c.send(int(n_per_proc))
        res = [c.recv() for c in self.conns]
        return sum(b for _, b in res), max(t for t, _ in res)

    def close(self):
        for c in self.conns:
            c.send(None)
        for p in self.ps:
            p.join(timeout=10)


def cpu_baseline(name, seconds):
    """The oracle on the whole decode step (every sequence, every layer), one
    process per core, repeated until about `seconds` of oracle time."""
    pool = OraclePool(name)
    try:
        per = -(-pool.units // pool.procs)
        nb, t = pool.run(per)
        reps = 1
        while t < seconds * 2 / 3 and reps < 64:
            b2, t2 = pool.run(per)
            nb, t, reps = nb + b2, t + t2, reps + 1
    finally:
        pool.close()
    w = W.ALL[name]()
    return {"value": round(nb / t / 1e9, 4), "unit": "GB/s", "cores": pool.procs, "kind": "oracle",
            "sample": f"the whole step ({len(W.seq_lens(w))} sequences x {len(w.layers)} layers) x {reps}, "
                      f"fp64 numpy oracle, {pool.procs} processes, {t:.2f} s of oracle wall time"}


def prefill_cpu_baseline(w, seconds):
    """The extend oracle on a seeded sample of the chunked-prefill workload:
    every process takes (chunk, layer) units spread over all chunks and both
    layers and computes 4 random tokens x every query head per unit, until
    about `seconds` of oracle time; the rate (algorithmic flops of the rows
    computed / the busiest process's time) extrapolates linearly to the whole
    prefill."""
    pool = OraclePool(w.name, prefill_kv=w.kv_dtype)
    try:
        fl, t = pool.run(2)
        reps = 1
        while t < seconds * 2 / 3 and reps < 64:
            f2, t2 = pool.run(2)
            fl, t, reps = fl + f2, t + t2, reps + 1
    finally:
        pool.close()
    step_flops = 0.0
    for d in w.layers:
        for c in range(w.prompt_len // w.chunk):
            step_flops += 4.0 * d["head_dim"] * d["num_q_heads"] * w.batch * visible_pairs(d["kind"], d["window"],
                                                                                          c * w.chunk, w.chunk)
    rate = fl / t
    return {"value": round(rate / 1e12, 6), "unit": "TFLOP/s", "cores": pool.procs, "kind": "oracle",
            "sample": f"{2 * reps} (chunk, layer) units per process x 4 random tokens x every query head, spread "
                      f"over all 8 chunks and both layers, fp64 numpy oracle, {pool.procs} processes, "
                      f"{t:.2f} s of oracle wall time; the whole prefill ({step_flops / 1e12:.3f} TFLOP) would "
                      f"take about {step_flops / rate:.0f} s at this rate (linear extrapolation by flops)"}


def reference_arm(args, rank, world):
    if rank != 0:
        return
    w = W.ALL[args.workload]()
    pool = OraclePool(args.workload)
    try:
        _, t1 = pool.run(1)                       # one unit per process: sizes the step
        budget = 150.0                            # seconds for the whole run
        n = max(1, int(min(1.0, budget / (args.steps + args.warmup)) / max(t1, 1e-4)))
        for _ in range(args.warmup):
            pool.run(n)
        nb = t = 0.0
        for _ in range(args.steps):
            b, dt = pool.run(n)
            nb += b
            t += dt
    finally:
        pool.close()
    value = round(nb / t / 1e9, 4)
    sample = f"{n} (sequence, layer) units per process per step, {pool.procs} processes, fp64 numpy oracle"
    res = {"impl": "reference", "metric": "paged decode-attn achieved HBM GB/s (% of peak); chunked-prefill TFLOP/s",
           "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(t / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
           "config": {"workload": w.name, "sample_per_step": sample},
           "cpu_baseline": {"value": value, "unit": "GB/s", "cores": pool.procs, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="e2b_decode", choices=["e2b_decode", "long_decode", "int8_decode",
                                                                  "fp8_decode", "tiny_decode"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="skip the long-context, int8, fp8 and tiny decode records of the default run")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--prefill-steps", type=int, default=20)
    ap.add_argument("--prefill-kv", default="bf16", choices=["bf16", "int8", "fp8"],
                    help="slab format of the chunked-prefill measurement")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        torch.distributed.init_process_group("nccl")
    try:
        gpu_arm(args, rank, world)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
