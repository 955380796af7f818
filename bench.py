#!/usr/bin/env python
"""Benchmark of one DeepSeek-V4 sparse-MLA decode step on GB300.

A step is one call of dsv4_sparse_mla_decode (index combine + gather/dequant +
attention + split merge) over the mid-size decode workload: 32 query tokens,
64 heads, 8192-token histories in 64-token pages, top-k 512, window 128, FP8
E4M3 + UE8M0 latent and BF16 rope in the cache, BF16 queries.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

ours: inputs resident in HBM; K steps replayed from CUDA graphs, each step on
one of R replicas of the whole workload (cache pages, block tables, queries,
outputs) so the bytes the timed steps gather exceed 4x the L2; CUDA events on
the launching stream, barrier + synchronize on both sides, max over ranks.
The roofline divides the algorithmic bytes (or FLOPs) of a step by the CUDA-event
time of the whole decode call; per-kernel shares come from the committed ncu launch
list (CUPTI kernel records are not available on the GPU machines).  e2e repeats the step through
the same C ABI with every step's host<->device copies inside the timed region: one packed upload
of the inputs from pinned memory and one read-back of the output and LSE per step, on copy
streams double-buffered against the calls (as a serving loop overlaps them), 64 steps a graph.

Other ops, timed the same way on their own workloads: --op topk-select (top-k selection from
indexer scores), --op combine-compressed (the compressed-region combine), --op
qnorm-rope-insert (fused query norm/RoPE and FP8 KV insert).
N > 1: every rank decodes its own batch on its own GPU (no data-path
collective; weak scaling).

reference: the fp64 CPU oracle on the host cores, K + W steps of a bounded
sample (some tokens x some heads) of the same workload, rank 0 only.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode query-tokens/s; gathered-KV GB/s & TFLOP/s as % of roofline"
UNIT = "tokens/s"
WORKLOAD = 2
KV_BYTES_PER_KEY = 644          # 512 E4M3 + 64 x BF16 + 4 UE8M0 (padding not counted)
FLOPS_PER_KEY_HEAD = 2 * (576 + 512)
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=WORKLOAD, help="decode workload 1..5 (default: 2, mid decode)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU-baseline sample length")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="time only --workload (the default line also times all five decode workloads)")
    ap.add_argument("--op", choices=["decode", "combine-compressed", "topk-select", "qnorm-rope-insert", "mtp-union"],
                    default="decode", help="decode (the headline), or one of the steps around it on its own")
    ap.add_argument("--topk-workload", choices=["long-batch", "long-decode"], default="long-batch",
                    help="top-k selection workload (synth.topk_config)")
    ap.add_argument("--replicas", type=int, default=0,
                    help="workload replicas to rotate through (default: enough for 4x the L2)")
    return ap.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def workload_config(w, extra=None):
    cfg = {"workload": w.name, "tokens_per_step": w.num_tokens, "heads": w.num_heads,
           "seq_len": int(w.seq_lens.max()), "topk": w.topk_width, "window": w.window, "page_block": w.page,
           "kv_entry": "512 x E4M3 + 4 x UE8M0 (per 128) latent, 64 x BF16 rope, 656 B",
           "sink": w.sink is not None}
    if extra:
        cfg.update(extra)
    return cfg


def combined_lengths(w):
    """Per-token number of keys (distinct valid top-k outside the window + window length)."""
    lens = np.zeros(w.num_tokens, dtype=np.int64)
    for t in range(w.num_tokens):
        pos = int(w.seq_lens[t]) - 1
        n = w.topk_width if w.topk_lens is None else int(min(max(w.topk_lens[t], 0), w.topk_width))
        lo = max(0, pos - w.window + 1)
        v = w.topk_idx[t, :n]
        lens[t] = np.unique(v[(v >= 0) & (v < lo)]).size + (pos - lo + 1 if pos >= 0 else 0)
    return lens


# ----------------------------------------------------------------------------
# clocks during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str):
        self.uuid = uuid.lower()
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            self.samples.append((time.time(), parts[0].lower(), parts[1:]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        uids = {u for (_, u, _) in self.samples}
        mine = {u for u in uids if self.uuid and (self.uuid in u or u in self.uuid)}
        if not mine and len(uids) == 1:
            mine = uids
        samples = [(ts, s) for (ts, u, s) in self.samples if u in mine]
        inside = [s for (ts, s) in samples if t0 <= ts <= t1]
        if not inside and samples:   # timed region shorter than the sampling period: nearest sample
            mid = 0.5 * (t0 + t1)
            inside = [min(samples, key=lambda x: abs(x[0] - mid))[1]]
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(s[0]) for s in inside]
        mx = [num(s[1]) for s in inside]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in inside for i in range(4) if s[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": reasons, "samples": len(inside),
                "power_w_max": max(num(s[2]) for s in inside)}


# ----------------------------------------------------------------------------
# oracle CPU baseline / reference arm
# ----------------------------------------------------------------------------
def cpu_baseline(w, seconds: float):
    import oracle
    cores = os.cpu_count() or 1
    oracle.sparse_mla_decode(w, tokens=[0], n_threads=1)     # load + warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.sparse_mla_decode(w, n_threads=cores)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": reps * w.num_tokens / el, "unit": UNIT, "cores": min(cores, w.num_tokens), "kind": "oracle",
            "sample": f"all {w.num_tokens} tokens x {w.num_heads} heads of the workload, repeated {reps}x "
                      f"({el:.1f} s, fp64, one thread per token)"}


def max_over_ranks(x: float, device=None) -> float:
    """The largest of every rank's value: the whole job's time is its slowest rank's (one rank:
    the value itself)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput under weak scaling: every rank processes its own units_per_rank,
    all of them within the slowest rank's ms."""
    return world * units_per_rank / (ms / 1e3)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    import synth
    w = synth.config(args.workload)
    cores = os.cpu_count() or 1
    H, T = w.num_heads, w.num_tokens
    ntok = min(T, cores)
    # size one step so that warmup + steps end within ~2 minutes
    budget = 120.0 / max(1, args.steps + args.warmup)
    oracle.sparse_mla_decode(w, tokens=list(range(ntok)), n_threads=ntok, heads=(0, 1))
    t0 = time.perf_counter()
    oracle.sparse_mla_decode(w, tokens=list(range(ntok)), n_threads=ntok, heads=(0, 1))
    t1 = time.perf_counter() - t0
    hs = 1
    while hs * 2 <= H and t1 * hs * 2 <= budget:
        hs *= 2
    while ntok > 1 and t1 * hs > budget:
        ntok //= 2
    toks = [list(range(ntok))]

    def step(i):
        h0 = (i * hs) % H
        sel = [(i * ntok + j) % T for j in range(ntok)]
        oracle.sparse_mla_decode(w, tokens=sel, n_threads=ntok, heads=(h0, h0 + hs))

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(i)
    el = time.perf_counter() - t0
    tokens = args.steps * ntok * hs / H
    value = tokens / el
    sample = f"{ntok} tokens x {hs} of {H} heads per step (fp64 oracle, {ntok} threads)"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, {"reference": "CPU fp64 oracle (no GPU)"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": ntok, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    del toks
    return 0


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def ncu_shares():
    """Per-kernel time shares of one decode step from the committed ncu launch-list summary."""
    try:
        with open(os.path.join(ROOT, "profiles", "launch_shares.json")) as f:
            return json.load(f)
    except Exception:
        return None


# workload names of the single-step benchmarks (the JSON line's config.workload; the key of their
# committed DRAM-traffic records)
TOPK_WORKLOADS = {"long-batch": "top-k selection: 128 tokens x 32768 candidate scores, top-k 2048",
                  "long-decode": "top-k selection: 16 tokens x 1024..131071 candidate scores, top-k 2048"}
COMBINE_COMPRESSED_WORKLOAD = ("compressed combine: 64 requests x 4 tokens, top-k 2048 of a 4x-compressed region, "
                               "window 128, rows of 2304")
INSERT_WORKLOAD = "q RMSNorm + GPT-J RoPE + FP8 KV insert: 128 tokens x 128 heads, 65536-slot cache"


def decode_launches(w, sms: int) -> int:
    """Kernels one decode call enqueues: the decode, plus the one-CTA ordering kernel when the
    tokens' list lengths are given and the (token, 64-head group) units outnumber the
    multiprocessors (the rule of the C ABI's decode call)."""
    units = w.num_tokens * ((w.num_heads + 63) // 64)
    return 2 if (w.topk_lens is not None and units > sms) else 1


def traffic_record(kernel_key: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the current kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            recs = json.load(f)
    except Exception:
        return None
    for r in recs:
        if r.get("kernel") != kernel_key or r.get("workload") != workload:
            continue
        src = os.path.join(ROOT, r["source"])
        try:
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()
        except OSError:
            return None
        return r["dram_bytes_per_launch"] if h == r.get("source_sha256") else None
    return None


class DecodeBench:
    """One decode workload resident on the device as R replicas at distinct addresses (cache pages,
    block tables, queries, outputs), so that the bytes gathered over one rotation exceed 4x the
    L2; steps replayed from CUDA graphs, CUDA events on the launching stream."""

    def __init__(self, pkg, w, dev, replicas=0, mtp_union=False):
        import torch
        self.pkg, self.w, self.dev = pkg, w, dev
        self.mtp_union = mtp_union
        self.base = synth_to_device(w, dev)
        self.T, self.H, self.K, self.W = w.num_tokens, w.num_heads, w.topk_width, w.window
        lens = combined_lengths(w)
        self.keys_per_step = int(lens.sum())
        self.bytes_per_step = self.keys_per_step * KV_BYTES_PER_KEY
        self.flops_per_step = self.keys_per_step * self.H * FLOPS_PER_KEY_HEAD
        props = torch.cuda.get_device_properties(dev)
        self.l2 = int(getattr(props, "L2_cache_size", 128 << 20))
        cache_bytes = self.base["kv_cache"].numel()
        R = max(2, math.ceil(4 * self.l2 / max(1, self.bytes_per_step)))
        R = int(min(R, max(2, (24 << 30) // max(1, cache_bytes))))
        if replicas > 0:
            R = replicas
        self.R = R
        nb = self.nb = w.num_blocks
        T, H = self.T, self.H
        self.pool = torch.empty((R * nb, w.page, 656), dtype=torch.uint8, device=dev)
        self.bts, self.qs, self.outs, self.lses = [], [], [], []
        for r in range(R):
            self.pool[r * nb:(r + 1) * nb].copy_(self.base["kv_cache"])
            bt = self.base["block_table"]
            self.bts.append(torch.where(bt >= 0, bt + r * nb, bt).contiguous())
            self.qs.append(self.base["q"].clone())
            self.outs.append(torch.empty((T, H, 512), dtype=torch.bfloat16, device=dev))
            self.lses.append(torch.empty((T, H), dtype=torch.float32, device=dev))
        del self.base["kv_cache"]
        self.ws = (pkg.workspace_for_mtp_union if mtp_union else pkg.workspace_for)(T, H, self.K, self.W, dev)
        self.stream = torch.cuda.Stream(device=dev)

    def step(self, i, stream=None):
        r = i % self.R
        b = self.base
        call = self.pkg.dsv4_sparse_mla_decode_mtp_union if self.mtp_union else self.pkg.dsv4_sparse_mla_decode
        return call(self.qs[r], self.pool, self.bts[r], b["req_idx"], b["topk_idx"], b["topk_lens"], b["seq_lens"],
                    self.W, b["sink"], b["softmax_scale"], self.outs[r], self.lses[r], self.ws, stream=stream)

    def time(self, steps, warmup, world=1, sampler=None):
        """Milliseconds for exactly `steps` steps (max over ranks) and the host times around them."""
        import torch
        import torch.distributed as dist
        pkg = self.pkg
        # first calls outside capture: library set-up, kernel attributes, the status word
        for i in range(self.R):
            pkg.check(self.step(i), "decode")
        torch.cuda.synchronize()
        pkg.check(pkg.dsv4_get_device_status(), "device status")
        stream = self.stream

        def capture(n_steps):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(n_steps):
                    rc = self.step(i, stream)
                    if rc != 0:
                        raise RuntimeError(f"decode failed during capture: {rc}")
            return g

        G = self.R * max(1, math.ceil(64 / self.R))   # steps per graph: whole rotations
        g_full = capture(G)
        nrep, rem = divmod(steps, G)
        g_rem = capture(rem) if rem else None
        wrep, wrem = divmod(warmup, G)
        g_wrem = capture(wrem) if wrem else None
        with torch.cuda.stream(stream):
            for _ in range(wrep):
                g_full.replay()
            if g_wrem is not None:
                g_wrem.replay()
        torch.cuda.synchronize()
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        h0 = time.time()
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(nrep):
                g_full.replay()
            if g_rem is not None:
                g_rem.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
        h1 = time.time()
        if world > 1:
            dist.barrier()
        ms = max_over_ranks(ev0.elapsed_time(ev1), self.dev)
        pkg.check(pkg.dsv4_get_device_status(), "device status")
        return ms, h0, h1

    def isolated(self, calls=40):
        """Latency of one call on its own: L2 flushed (a write larger than L2) before each call, the
        call issued directly (no graph, no neighbouring call to overlap its prologue with), CUDA
        events around it on its stream after a GPU-side pause that lets the host queue the call
        first. Median and minimum in microseconds."""
        import torch
        pkg = self.pkg
        stream = self.stream
        flush = torch.empty(2 * self.l2, dtype=torch.uint8, device=self.dev)
        times = []
        for i in range(calls):
            ev0 = torch.cuda.Event(enable_timing=True)
            ev1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                flush.fill_(i & 0xFF)
                # the GPU idles ~0.5 ms before the first event, so that the call is already queued
                # when it starts: the events time the GPU, not the host's launch
                torch.cuda._sleep(1_000_000)
                ev0.record(stream)
                pkg.check(self.step(i % self.R, stream), "decode")
                ev1.record(stream)
            torch.cuda.synchronize()
            times.append(ev0.elapsed_time(ev1) * 1e3)
        del flush
        pkg.check(pkg.dsv4_get_device_status(), "device status")
        times.sort()
        return {"median_us": times[len(times) // 2], "min_us": times[0], "calls": calls,
                "method": "one C-ABI call at a time, L2 flushed before each, CUDA events around the call on its "
                          "stream (queued behind a GPU-side pause so that the host's launch is not timed)"}

    def roofline(self, call_s):
        """The decode call against max(gathered KV bytes / HBM peak, FLOPs / BF16 tensor peak)."""
        hbm_peak, bf16_peak, _, peak_src = peaks()
        t_hbm = self.bytes_per_step / (hbm_peak * 1e9)
        t_tc = self.flops_per_step / (bf16_peak * 1e12)
        if t_hbm >= t_tc:
            ach = self.bytes_per_step / call_s / 1e9
            r = {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak}
        else:
            ach = self.flops_per_step / call_s / 1e12
            r = {"bound": "tensor", "achieved": ach, "peak": bf16_peak, "unit": "TFLOP/s", "frac": ach / bf16_peak}
        r.update({"peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                  "call_us": call_s * 1e6, "roofline_us": max(t_hbm, t_tc) * 1e6,
                  "algorithmic_bytes_per_launch": self.bytes_per_step, "flops_per_launch": self.flops_per_step,
                  "kv_gbs": self.bytes_per_step / call_s / 1e9, "tflops": self.flops_per_step / call_s / 1e12})
        return r

    def l2_note(self):
        return (f"inputs larger than L2: {self.R} rotating replicas ({self.R * self.bytes_per_step / 1e6:.0f} MB "
                f"gathered per rotation, L2 {self.l2 / 1e6:.0f} MB)")

    def e2e(self, steps, world=1):
        """The same step end to end through the C ABI: every step uploads its inputs (q, top-k rows,
        lengths, block table: one packed pinned buffer per replica, one H2D copy) and reads its output
        and LSE back (one D2H copy), decoding against the replica's cache pages, so the gathered KV
        rotates through more than 4x the L2 as in the device-timed loop.  As in a serving loop the
        copies run on their own streams, double-buffered, so that step i's kernel overlaps step i+1's
        upload and step i-1's read-back; 64 steps a CUDA graph."""
        import torch
        import torch.distributed as dist
        import numpy as np
        pkg, w, dev, T, H, R = self.pkg, self.w, self.dev, self.T, self.H, self.R
        arrays0 = {"q": np.ascontiguousarray(w.q.view(np.int16)), "topk_idx": w.topk_idx, "seq_lens": w.seq_lens}
        if w.topk_lens is not None:
            arrays0["topk_lens"] = w.topk_lens
        if w.req_idx is not None:
            arrays0["req_idx"] = w.req_idx
        bt0 = w.block_table
        shapes = {**{k: a.shape for k, a in arrays0.items()}, "block_table": bt0.shape}
        nbytes = {**{k: a.nbytes for k, a in arrays0.items()}, "block_table": bt0.nbytes}
        offs, total = {}, 0
        for k in shapes:
            offs[k] = total
            total += -(-nbytes[k] // 256) * 256
        out_bytes = T * H * 512 * 2
        res_total = out_bytes + T * H * 4
        h_in = []
        for r in range(R):
            hb = torch.zeros(total, dtype=torch.uint8).pin_memory()
            bt = np.where(bt0 >= 0, bt0 + r * self.nb, bt0).astype(np.int32)
            for k in shapes:
                a = bt if k == "block_table" else arrays0[k]
                hb[offs[k]:offs[k] + nbytes[k]].copy_(torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).reshape(-1)))
            h_in.append(hb)
        d_in = [torch.empty(total, dtype=torch.uint8, device=dev) for _ in range(2)]
        d_res = [torch.empty(res_total, dtype=torch.uint8, device=dev) for _ in range(2)]
        h_res = [torch.empty(res_total, dtype=torch.uint8).pin_memory() for _ in range(2)]

        def views(j):
            v = {}
            for k in shapes:
                x = d_in[j][offs[k]:offs[k] + nbytes[k]]
                v[k] = (x.view(torch.bfloat16) if k == "q" else x.view(torch.int32)).view(shapes[k])
            return v, d_res[j][:out_bytes].view(torch.bfloat16).view(T, H, 512), \
                d_res[j][out_bytes:].view(torch.float32).view(T, H)
        bufs = [views(0), views(1)]
        stream = self.stream
        s_up, s_down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev_in = [torch.cuda.Event() for _ in range(2)]     # inputs of buffer j uploaded
        ev_done = [torch.cuda.Event() for _ in range(2)]   # the call on buffer j finished
        ev_read = [torch.cuda.Event() for _ in range(2)]   # results of buffer j read back
        G = 64

        def e2e_step(i, first):
            j = i & 1
            if not first:
                s_up.wait_event(ev_done[j])
            with torch.cuda.stream(s_up):
                d_in[j].copy_(h_in[i % R], non_blocking=True)
                ev_in[j].record(s_up)
            stream.wait_event(ev_in[j])
            if not first:
                stream.wait_event(ev_read[j])
            v, d_out, d_lse = bufs[j]
            rc = pkg.dsv4_sparse_mla_decode(v["q"], self.pool, v["block_table"], v.get("req_idx"), v["topk_idx"],
                                            v.get("topk_lens"), v["seq_lens"], self.W, self.base["sink"],
                                            self.base["softmax_scale"], d_out, d_lse, self.ws, stream=stream)
            ev_done[j].record(stream)
            s_down.wait_event(ev_done[j])
            with torch.cuda.stream(s_down):
                h_res[j].copy_(d_res[j], non_blocking=True)
                ev_read[j].record(s_down)
            if rc != 0:
                raise RuntimeError(f"decode failed: {rc}")

        def capture_e2e(n):
            """n steps as one CUDA graph: the copy streams fork from and join back into `stream`."""
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                s_up.wait_stream(stream)
                s_down.wait_stream(stream)
                for i in range(n):
                    e2e_step(i, i < 2)
                stream.wait_stream(s_up)
                stream.wait_stream(s_down)
            return g
        g_e2e = capture_e2e(G)
        e_rep, e_rem = divmod(steps, G)
        g_e2e_rem = capture_e2e(e_rem) if e_rem else None
        with torch.cuda.stream(stream):
            for _ in range(2):
                g_e2e.replay()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(e_rep):
                g_e2e.replay()
            if g_e2e_rem is not None:
                g_e2e_rem.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        ems = max_over_ranks(e0.elapsed_time(e1), dev)
        # the last step read back replica (n - 1) % R's result: it equals the device-timed run's output there
        n_last = e_rem if e_rem else G
        last_buf = (n_last - 1) & 1
        r_last = (n_last - 1) % R
        if not torch.equal(h_res[last_buf][:out_bytes].view(torch.int16),
                           self.outs[r_last].view(torch.int16).reshape(-1).cpu()):
            raise RuntimeError("end-to-end output differs from the device-timed output")
        return {"value": job_rate(T * steps, world, ems), "unit": UNIT, "h2d_bytes_per_step": total,
                "d2h_bytes_per_step": res_total, "steps": steps,
                "method": "per step: one pinned H2D copy of q/topk/seq_lens/block_table (packed, one buffer per cache "
                          f"replica), the C-ABI call on that replica's pages ({R} replicas, as the device-timed loop), "
                          "one D2H copy of out+lse; copies on their own streams, double-buffered, overlapping the "
                          "neighbouring steps' calls; 64 steps a CUDA graph"}


def synth_to_device(w, dev):
    import synth
    return synth.to_device(w, dev)


def cpu_baseline_sample(w, seconds: float, max_tokens: int = 16):
    """The oracle as it stands on a bounded sample of the workload: up to max_tokens tokens (all
    heads), repeated for about `seconds`, one thread per token."""
    import oracle
    cores = os.cpu_count() or 1
    toks = list(range(min(w.num_tokens, max_tokens, cores)))
    oracle.sparse_mla_decode(w, tokens=[0], n_threads=1)     # load + warm
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.sparse_mla_decode(w, tokens=toks, n_threads=len(toks))
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": reps * len(toks) / el, "unit": UNIT, "cores": len(toks), "kind": "oracle",
            "sample": f"{len(toks)} of {w.num_tokens} tokens x all {w.num_heads} heads, repeated {reps}x "
                      f"({el:.1f} s, fp64, one thread per token)"}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import synth
    import sparse_mla_decode_combine_gb300 as pkg
    from sparse_mla_decode_combine_gb300 import build as pkg_build

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    if rank == 0 or world == 1:
        pkg_build.build()
    if world > 1:
        dist.barrier()
    pkg.load_library()
    props = torch.cuda.get_device_properties(dev)

    w = synth.config(args.workload)
    bench = DecodeBench(pkg, w, dev, args.replicas)
    T = w.num_tokens
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    if rank == 0:
        sampler.start()
        time.sleep(0.5)
    ms, h0, h1 = bench.time(args.steps, args.warmup, world)
    clocks = sampler.summary(h0, h1) if rank == 0 else None
    value = job_rate(T * args.steps, world, ms)

    # roofline of the decode call (the kernel that combines, decodes and merges its splits; for varying
    # list lengths over many units, an ordering kernel ahead of it), timed with CUDA events over the
    # timed region
    launches_per_step = decode_launches(w, props.multi_processor_count)
    call_s = ms / 1e3 / args.steps
    roofline = bench.roofline(call_s)
    decode_kernel = "decode_tc_kernel"
    roofline.update({
        "traffic": traffic_record(decode_kernel, w.name), "kernel": decode_kernel,
        "timed": ("whole decode call per step (the kernel that combines, decodes and merges its splits, after "
                  "the one-CTA ordering kernel when the call enqueues one), "
                  "CUDA events on the launching stream over the timed region; per-kernel shares of the step are "
                  "in ncu_shares (committed ncu launch list)"),
        "ncu_shares": ncu_shares()})

    e2e = None
    if not args.no_e2e:
        e2e = bench.e2e(args.steps, world)
    isolated = bench.isolated() if rank == 0 else None
    config = workload_config(w, {"l2": bench.l2_note(), "replicas": bench.R, "keys_per_step": bench.keys_per_step})
    del bench
    torch.cuda.empty_cache()

    # every decode workload, each timed the same way (rotating replicas larger than L2), with its own
    # roofline and a bounded oracle sample; the headline above is the mid-size decode
    per_workload = None
    if world == 1 and not args.no_per_workload:
        per_workload = []
        for n in range(1, 6):
            wn = w if n == args.workload else synth.config(n)
            bn = DecodeBench(pkg, wn, dev)
            msn, a0, a1 = bn.time(args.steps, args.warmup)
            rl = bn.roofline(msn / 1e3 / args.steps)
            rl["traffic"] = traffic_record(decode_kernel, wn.name)
            entry = {"workload": wn.name, "ms_per_step": msn / args.steps, "value": wn.num_tokens * args.steps / (msn / 1e3),
                     "unit": UNIT, "steps": args.steps, "replicas": bn.R, "keys_per_step": bn.keys_per_step,
                     "launches_per_step": decode_launches(wn, props.multi_processor_count),
                     "roofline": {k: rl[k] for k in ("bound", "achieved", "peak", "unit", "frac", "call_us",
                                                     "roofline_us", "kv_gbs", "tflops", "traffic")},
                     "clocks": sampler.summary(a0, a1) if rank == 0 else None}
            del bn
            torch.cuda.empty_cache()
            if not args.no_cpu_baseline:
                entry["cpu_baseline"] = cpu_baseline_sample(wn, 2.0)
            per_workload.append(entry)
    if rank == 0:
        time.sleep(0.2)
        sampler.stop()

    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(w, args.cpu_seconds)
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config, "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
                "gpu_launches": launches_per_step * args.steps, "launches_per_step": launches_per_step,
                "clocks": clocks, "isolated_call": isolated, "per_workload": per_workload}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_mtp_union(args):
    """The MTP union decode on the spec-verify workload (64 requests x 2 tokens x 128 heads), against
    the plain decode on the same inputs, as synthesised (each token's top-k row drawn on its own) and
    with 90 % of each draft token's picks shared with its partner. A step is one call; the union
    call enqueues the combine, the union kernel, the ordering kernel and the decode."""
    import torch
    import synth
    import sparse_mla_decode_combine_gb300 as pkg
    from sparse_mla_decode_combine_gb300 import build as pkg_build
    pkg_build.build()
    pkg.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    time.sleep(0.5)
    w0 = synth.config(4)
    rows = {}
    for label, w in (("independent picks", w0), ("90% shared picks", synth.with_shared_picks(w0, 17, 0.9))):
        for mode in ("union", "plain"):
            bn = DecodeBench(pkg, w, dev, mtp_union=(mode == "union"))
            msn, a0, a1 = bn.time(args.steps, args.warmup)
            rl = bn.roofline(msn / 1e3 / args.steps)
            rows[(label, mode)] = {"ms_per_step": msn / args.steps, "value": w.num_tokens * args.steps / (msn / 1e3),
                                   "frac": rl["frac"], "clocks": sampler.summary(a0, a1), "bench": bn}
            if not (label == "independent picks" and mode == "union"):
                del bn
                rows[(label, mode)].pop("bench")
                torch.cuda.empty_cache()
    # combine, union lists, (ordering when the units outnumber the multiprocessors), decode
    launches = 3 + (1 if (w0.num_tokens // 2) * (w0.num_heads // 32) > props.multi_processor_count else 0)
    head = rows[("independent picks", "union")]
    bn = head.pop("bench")
    rl = bn.roofline(head["ms_per_step"] / 1e3)
    rl.update({"kernel": "decode_tc_kernel", "traffic": None,
               "timed": "whole MTP union call per step (combine, union kernel, ordering kernel, decode), CUDA events on the launching stream"})
    config = workload_config(w0, {"l2": bn.l2_note(), "replicas": bn.R, "keys_per_step": bn.keys_per_step,
                                  "call": "dsv4_sparse_mla_decode_mtp_union"})
    del bn
    torch.cuda.empty_cache()
    sampler.stop()
    line = {"op": "mtp-union", "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": config, "roofline": rl,
            "gpu_launches": launches * args.steps, "launches_per_step": launches, "clocks": head["clocks"],
            "comparison": {f"{label}, {mode}": {k: v for k, v in r.items() if k != "clocks"}
                           for (label, mode), r in rows.items()}}
    print(json.dumps(line), flush=True)
    return 0


def run_combine_compressed(args):
    """The compressed-region combine on its own: 64 requests x 4 tokens (speculative verify
    shape), top-k 2048 of a 4x-compressed region, window 128, rows of 2304 entries. Bytes per
    token: the top-k entries read (4 * topk_len) plus the row and length written (4 * width + 4)."""
    import torch
    import sparse_mla_decode_combine_gb300 as pkg
    from sparse_mla_decode_combine_gb300 import build as pkg_build
    pkg_build.build()
    pkg.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(1)
    R, qlen, top_k, C, W, width = 64, 4, 2048, 4, 128, 2304
    seqs = rng.integers(8192, 65536, size=R).astype(np.int32)
    gls = np.full(R, W + qlen, dtype=np.int32)
    N = 65536 // C
    M = N + int(gls.max())
    T = R * qlen
    # replicas of the batch so that one rotation moves more than 4x the L2
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    pos = np.repeat(seqs, qlen) - qlen + np.tile(np.arange(qlen), R)
    tk = np.minimum((pos + 1) // C, top_k)
    sw = np.minimum(pos + 1, W)
    bytes_per_step = int((4 * tk).sum() + T * (4 * width + 4))
    reps = max(2, math.ceil(4 * l2 / bytes_per_step))
    qsl = torch.from_numpy((np.arange(R + 1) * qlen).astype(np.int32)).to(dev)
    s_d = torch.from_numpy(seqs).to(dev)
    g_d = torch.from_numpy(gls).to(dev)
    ins = [torch.from_numpy(rng.integers(-1, N, size=(T, top_k)).astype(np.int32)).to(dev) for _ in range(reps)]
    outs = [torch.empty((T, width), dtype=torch.int32, device=dev) for _ in range(reps)]
    lens = [torch.empty((T,), dtype=torch.int32, device=dev) for _ in range(reps)]
    stream = torch.cuda.Stream(dev)

    def step(i):
        pkg.check(pkg.dsv4_combine_topk_swa_indices_compressed(ins[i % reps], qsl, s_d, g_d, M, N, top_k, C, W,
                                                               outs[i % reps], lens[i % reps], stream=stream))
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize()
    # one rotation over the replicas as a CUDA graph, replayed (the host does not pace the GPU),
    # then a shorter graph for the last K mod replicas steps, so that exactly K steps are timed
    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        return g
    graph = capture(reps)
    replays, rem = divmod(max(args.steps, 1), reps)
    tail = capture(rem) if rem else None
    torch.cuda.synchronize()
    steps = replays * reps + rem
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        if tail is not None:
            tail.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    args.steps = steps
    ms = ev0.elapsed_time(ev1)
    step_s = ms / 1e3 / args.steps
    hbm_peak, _, _, peak_src = peaks()
    ach = bytes_per_step / step_s / 1e9
    line = {"metric": "compressed-region combine query-tokens/s (bytes moved vs HBM roofline)",
            "value": T / step_s, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int32", "data": "synthetic",
            "config": {"workload": COMBINE_COMPRESSED_WORKLOAD, "tokens_per_step": T, "replicas": reps,
                       "l2": f"inputs larger than L2: {reps} rotating replicas"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                         "traffic": traffic_record("combine_compressed_kernel", COMBINE_COMPRESSED_WORKLOAD),
                         "kernel": "combine_compressed_kernel",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                         "algorithmic_bytes_per_launch": bytes_per_step,
                         "timed": "one call (one launch) per step, CUDA events on the launching stream"},
            "gpu_launches": args.steps, "launches_per_step": 1, "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line), flush=True)
    return 0


def run_topk_select(args):
    """Top-k selection on its own (synth.topk_config): bytes per step are the candidate scores
    read once (4 * sum n_t) plus the rows and lengths written (T * (4 * K + 4))."""
    import torch
    import synth
    import sparse_mla_decode_combine_gb300 as pkg
    from sparse_mla_decode_combine_gb300 import build as pkg_build
    pkg_build.build()
    pkg.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    w = synth.topk_config(args.topk_workload)
    T, K = w.num_tokens, w.top_k
    nc = np.clip(w.num_cand, 0, w.width).astype(np.int64)
    bytes_per_step = int(4 * nc.sum() + T * (4 * K + 4))
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    reps = args.replicas if args.replicas > 0 else max(2, math.ceil(4 * l2 / (4 * int(nc.sum()))))
    base = torch.from_numpy(w.scores).to(dev)
    scs = [base.clone() for _ in range(reps)]
    del base
    nc_d = torch.from_numpy(w.num_cand).to(dev)
    outs = [torch.empty((T, K), dtype=torch.int32, device=dev) for _ in range(reps)]
    lens = [torch.empty((T,), dtype=torch.int32, device=dev) for _ in range(reps)]
    stream = torch.cuda.Stream(dev)

    def step(i):
        pkg.check(pkg.dsv4_topk_select(scs[i % reps], nc_d, K, outs[i % reps], lens[i % reps], stream=stream))
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        return g
    graph = capture(reps)
    replays, rem = divmod(max(args.steps, 1), reps)
    tail = capture(rem) if rem else None
    torch.cuda.synchronize()
    steps = replays * reps + rem
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        if tail is not None:
            tail.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    step_s = ms / 1e3 / steps
    hbm_peak, _, _, peak_src = peaks()
    ach = bytes_per_step / step_s / 1e9
    desc = TOPK_WORKLOADS[w.name]
    line = {"metric": "top-k selection query-tokens/s (bytes moved vs HBM roofline)",
            "value": T / step_s, "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic",
            "config": {"workload": desc, "tokens_per_step": T, "candidates_per_step": int(nc.sum()), "top_k": K,
                       "replicas": reps, "l2": f"inputs larger than L2: {reps} rotating replicas"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                         "traffic": traffic_record("topk_select_kernel", desc), "kernel": "topk_select_kernel",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                         "algorithmic_bytes_per_launch": bytes_per_step,
                         "timed": "one call (one launch) per step, CUDA events on the launching stream"},
            "gpu_launches": steps, "launches_per_step": 1, "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line), flush=True)
    return 0


def run_qnorm_rope_insert(args):
    """The fused query RMSNorm + GPT-J RoPE + FP8 KV insert on its own: 128 tokens x 128 heads
    (the long-context decode's shape), positions below 32768, distinct slots in a 65536-slot
    cache. Bytes per step: queries read and written (2 * T * H * 1152), keys read (T * 1152),
    entries written (T * 656), cos/sin rows, positions and slots read (T * 272)."""
    import torch
    import synth
    import sparse_mla_decode_combine_gb300 as pkg
    from sparse_mla_decode_combine_gb300 import build as pkg_build
    pkg_build.build()
    pkg.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rng = np.random.default_rng(7)
    T, H, P, S = 128, 128, 32768, 65536
    bytes_per_step = 2 * T * H * 1152 + T * 1152 + T * 656 + T * 272
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    reps = args.replicas if args.replicas > 0 else max(2, math.ceil(4 * l2 / bytes_per_step))
    q0 = torch.from_numpy(synth.bf16_bits(rng.standard_normal((T, H, 576))).view(np.int16)).view(torch.bfloat16).to(dev)
    kv0 = torch.from_numpy(synth.bf16_bits(rng.standard_normal((T, 576))).view(np.int16)).view(torch.bfloat16).to(dev)
    qs = [q0.clone() for _ in range(reps)]
    qo = [torch.empty_like(q0) for _ in range(reps)]
    kvs = [kv0.clone() for _ in range(reps)]
    ang = rng.uniform(0, 2 * np.pi, (P, 32))
    table = torch.from_numpy(np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)).to(dev)
    pos = torch.from_numpy(rng.integers(0, P, T).astype(np.int64)).to(dev)
    slots = torch.from_numpy(rng.permutation(S)[:T].astype(np.int64)).to(dev)
    cache = torch.zeros((S, 656), dtype=torch.uint8, device=dev)
    w = torch.from_numpy(rng.uniform(0.5, 1.5, 576).astype(np.float32)).to(dev)
    stream = torch.cuda.Stream(dev)

    def step(i):
        r = i % reps
        pkg.check(pkg.dsv4_qnorm_rope_kv_insert(qs[r], qo[r], kvs[r], pos, slots, table, cache, w, 1e-6,
                                                stream=stream))
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 1)):
            step(i)
    torch.cuda.synchronize()

    def capture(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                step(i)
        return g
    graph = capture(reps)
    replays, rem = divmod(max(args.steps, 1), reps)
    tail = capture(rem) if rem else None
    torch.cuda.synchronize()
    steps = replays * reps + rem
    sampler = ClockSampler(str(getattr(props, "uuid", "")))
    sampler.start()
    time.sleep(0.2)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(replays):
            graph.replay()
        if tail is not None:
            tail.replay()
        ev1.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    time.sleep(0.2)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)
    step_s = ms / 1e3 / steps
    hbm_peak, _, _, peak_src = peaks()
    ach = bytes_per_step / step_s / 1e9
    line = {"metric": "fused q-norm/RoPE/KV-insert query-tokens/s (bytes moved vs HBM roofline)",
            "value": T / step_s, "unit": "tokens/s", "n_gpus": 1, "steps": steps, "warmup": args.warmup,
            "ms_per_step": ms / steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": INSERT_WORKLOAD,
                       "tokens_per_step": T, "heads": H, "replicas": reps,
                       "l2": f"inputs larger than L2: {reps} rotating replicas"},
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm_peak, "unit": "GB/s", "frac": ach / hbm_peak,
                         "traffic": traffic_record("qnorm_rope_kv_insert_kernel", INSERT_WORKLOAD),
                         "kernel": "qnorm_rope_kv_insert_kernel",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json)" if peak_src == "measured" else "fallback",
                         "algorithmic_bytes_per_launch": bytes_per_step,
                         "timed": "one call (one launch) per step, CUDA events on the launching stream"},
            "gpu_launches": steps, "launches_per_step": 1, "clocks": sampler.summary(t0, t1)}
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    if args.op == "qnorm-rope-insert":
        if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
            return 0
        return run_qnorm_rope_insert(args)
    if args.op == "topk-select":
        if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
            return 0
        return run_topk_select(args)
    if args.op == "combine-compressed":
        if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
            return 0
        return run_combine_compressed(args)
    if args.op == "mtp-union":
        if args.impl == "reference" or int(os.environ.get("RANK", "0")) != 0:
            return 0
        return run_mtp_union(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
