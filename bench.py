#!/usr/bin/env python
"""Throughput of cached incremental attention on GB300 through libkvc's C ABI.

The default run prints one JSON line: the headline workload (mha_decode) and,
under "workloads", the three other configurations measured the same way
(gqa_decode, mqa_decode, suffix), each with its own value, roofline, CPU
baseline, end-to-end number and clocks.

Workloads (seeded, synthetic; sizes as the pages' workloads are stated):

* mha_decode (headline): B = 32, H = 32, d_h = 128, bf16, C = 8192,
  old lengths uniform in [1, 8128], 64 decode steps.  One bench step =
  kvc_truncate back to the old lengths + 64 kvc_append_attend calls.  Metric:
  K/V bytes the attention must read (every retained row of every lane at every
  decode step) per second.
* gqa_decode / mqa_decode: B = 64, H_q = 32, H_kv = 8 / 1, C = 32768, old
  lengths uniform in [16384, 32736], 32 decode steps.
* suffix: B = 8, H = 32, d_h = 128, 16384 cached tokens with one edited id
  each + 512 appended: one bench step = kvc_lcp per sequence + kvc_truncate +
  kvc_prefill_suffix of the suffix chunk.  Metric: TFLOP/s of the unmasked
  QK^T and PV work.

Every step reads far more than the 129 MB L2 (2.2 GB of K/V per MHA decode
step), so no L2 flush is inserted.  `value` is device-timed with inputs
resident in HBM; `e2e` repeats the measurement through the same C-ABI calls
with the per-step inputs copied from pinned host memory and the outputs
copied back inside the timed region (suffix: kvc_prefill_suffix_host, which
takes the pinned host buffers and overlaps each stage of sequences' copies
with another stage's work).  `roofline` times the dominant kernel
with CUDA events recorded by the library around each launch on its stream,
in a second pass over the same number of steps (so that the event records do
not weigh on `value`); per-launch events break the overlap of consecutive
dependent launches, so `roofline.step_frac` also divides the same algorithmic
work by the whole step's time (`ms_per_step`).
`cpu_baseline` times the float64 oracle on a bounded sample, one oracle process
per host core side by side (`cores`), plus `one_core` (one process alone).
`--impl reference` times that oracle as the reference arm; it builds the same
seeded inputs with torch and never loads libkvc.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attention KV GB/s & %HBM peak; suffix-chunk TFLOP/s; steps/s"

# DRAM traffic of the dominant kernel from ncu captures of smaller cases of the
# same kernel build (dram__bytes_read.sum + dram__bytes_write.sum per launch),
# scaled to a full launch: decode traffic grows with the K/V bytes streamed
# (ratio to the algorithmic bytes), the tile kernel's with the number of
# sequences (each sequence's K/V comes from DRAM about once, then from L2).
TRAFFIC = {
    "mha_decode": ("ratio", 1.0126),
    "gqa_decode": ("ratio", 1.0062),
    "mqa_decode": ("ratio", 1.012),
    "mha_decode_short": ("ratio", 1.0579),
    "suffix": ("per_sequence", 375510016.0 + 175409664.0),
}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="default",
                   choices=["default", "mha_decode", "mha_decode_short", "gqa_decode", "mqa_decode", "suffix", "all"],
                   help="default: one line, mha_decode with gqa_decode, mqa_decode and suffix under "
                        "'workloads'; all: one line per workload")
    p.add_argument("--block-rows", type=int, default=0,
                   help="paged storage with blocks of this many rows (a multiple of 64); 0 = contiguous")
    p.add_argument("--split-rows", type=int, default=0,
                   help="decode: key rows per split (a multiple of 64); 0 = the library's choice")
    p.add_argument("--graph", action="store_true",
                   help="decode workloads: lengths kept on the device, each bench step's decode calls "
                        "captured once in a CUDA graph and replayed")
    p.add_argument("--suffix-kernel", type=int, default=0, choices=[0, 1, 2, 3, 4, 5],
                   help="suffix: 0 = the library's choice, 1 = generic, 2 = one-SM tile kernel, 3 = pair-of-SMs "
                        "tile kernel, 4 = persistent tile kernel, 5 = tile kernel with two softmax threads per query row")
    p.add_argument("--host-chunk", type=int, default=0,
                   help="suffix e2e: sequences per stage of the host-buffer call; 0 = the library's choice")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--batch", type=int, default=0,
                   help="override B of a workload (a smaller case for ncu captures; not a bench line)")
    return p.parse_args()


# GB300 datasheet figures (dense): HBM3e bandwidth and bf16 tensor throughput
NOMINAL_HBM_GBS, NOMINAL_BF16_TFLOPS = 7900.0, 2250.0
# sub-workloads of the default line
SUB_WORKLOADS = ("gqa_decode", "mqa_decode", "suffix")


def peaks():
    """Roofline denominators: the measured copy rate (read + write GB/s of a device copy)
    and the measured cuBLAS bf16 burst rate, else the fallback figures."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sustained_bf16():
    """The measured cuBLAS bf16 rate of a seconds-long back-to-back loop under the power
    cap (None when not measured)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except Exception:
        return None


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.lines and time.time() - t0 < 5.0:   # first sample before timing starts
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_index(local_rank):
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        ids = [x for x in vis.split(",") if x.strip()]
        if local_rank < len(ids) and ids[local_rank].strip().isdigit():
            return int(ids[local_rank])
    return local_rank


# ----------------------------------------------------------------- decode workloads

class DecodeBench:
    """A decode workload.  ``with_cache`` False (the reference arm) draws the same seeded
    inputs and builds no libkvc cache (the library is never loaded)."""

    def __init__(self, name, device, batch=0, graph=False, block_rows=0, with_cache=True):
        from kv_cache_append_rope_gb300 import workloads as W
        cfg = dict(W.CONFIGS[name])
        if batch:
            cfg["B"] = batch
        self.name, self.cfg, self.device, self.block_rows = name, cfg, device, block_rows
        B, Hq, Hkv, D, C, steps = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["D"], cfg["C"], cfg["steps"]
        self.L0 = W.old_lengths(cfg["seed"], B, cfg["lo"], cfg["hi"], C, steps)
        self.cache = None
        if with_cache:
            from kv_cache_append_rope_gb300.kvc import KVCache
            self.cache = KVCache(B, Hq, C, D, heads_kv=Hkv, dtype="bf16", rope_base=10000.0,
                                 device=device.index or 0, block_rows=block_rows)
        S = int(self.L0.max())
        seed = cfg["seed"] * 1000
        # unrotated prefix rows (kept for the oracle sample), appended without attending
        self.k_prefix = W.normal((B, Hkv, S, D), seed + 1, device=device)
        self.v_prefix = W.normal((B, Hkv, S, D), seed + 2, device=device)
        if with_cache:
            self.cache.prefill_suffix(0, None, self.k_prefix, self.v_prefix, seqlen=self.L0.tolist(), out=False)
        self.q = W.normal((steps, B, Hq, 1, D), seed + 3, device=device)
        self.k = W.normal((steps, B, Hkv, 1, D), seed + 4, device=device)
        self.v = W.normal((steps, B, Hkv, 1, D), seed + 5, device=device)
        self.out = torch.empty((steps, B, Hq, 1, D), dtype=torch.float32, device=device) if with_cache else None
        if device.type == "cuda":
            torch.cuda.synchronize(device)
        # algorithmic K/V bytes read by attention over the 64 steps: every lane reads t rows of K and V
        t = self.L0[None, :] + 1 + np.arange(steps)[:, None]          # [steps, B]
        self.kv_bytes_per_call = (t.sum(axis=1) * Hkv * D * 2 * 2).astype(np.float64)
        self.kv_bytes = float(self.kv_bytes_per_call.sum())
        # everything else the step must move: q/k/v rows in, new K/V rows written, outputs out
        self.io_bytes = float(steps * B * (Hq * D * 2 + 2 * Hkv * D * 2 + 2 * Hkv * D * 2 + Hq * D * 4))
        self.steps = steps
        self.graph, self.graph_launches, self.replays = None, 0, 0
        # the step's calls, their arguments marshalled once (the same buffers every step)
        self.calls = ([self.cache.bind_append_attend(0, self.q[i], self.k[i], self.v[i], self.out[i])
                       for i in range(steps)] if with_cache else [])
        if graph and with_cache:
            self.capture()

    def step(self):
        self.cache.truncate(self.L0.tolist())
        if self.graph is not None:
            self.graph.replay()
            self.replays += 1
            return
        for call in self.calls:
            call()

    def capture(self):
        """Device-held lengths, then the step's decode calls recorded once in a CUDA graph."""
        from kv_cache_append_rope_gb300 import _lib as L
        self.cache.set_option(L.OPT_DEVICE_LENGTHS, 1)
        self.step()                                   # uncaptured: allocates the split scratch
        torch.cuda.synchronize(self.device)
        self.cache.truncate(self.L0.tolist())
        _, before = self.cache.kernel_stats(-1)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(self.steps):
                self.cache.append_attend(0, self.q[i], self.k[i], self.v[i], out=self.out[i])
        _, after = self.cache.kernel_stats(-1)
        self.graph_launches = after - before
        self.graph = g

    def timing_pass(self):
        """The step with per-launch events: a captured graph holds none, so replay it eagerly."""
        g, self.graph = self.graph, None
        self.step()
        self.graph = g

    def graph_kernel_launches(self):
        return self.graph_launches * self.replays

    def e2e_setup(self):
        # each step's q, k and v rows packed in one pinned host row, so that a step's inputs
        # go up in one copy
        n_q, n_k = self.q[0].numel(), self.k[0].numel()
        self.hin = torch.cat([self.q.reshape(self.steps, -1), self.k.reshape(self.steps, -1),
                              self.v.reshape(self.steps, -1)], dim=1).cpu().pin_memory()
        if self.graph is not None:
            # the graph reads the fixed input tensors: whole-tensor uploads
            self.hq, self.hk, self.hv = (x.cpu().pin_memory() for x in (self.q, self.k, self.v))
        self.hout = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        # two device input rows: step i+1 uploads while step i computes
        self.din = [torch.empty_like(self.hin[0], device=self.device) for _ in range(2)]
        views = [(d[:n_q].view(self.q[0].shape), d[n_q:n_q + n_k].view(self.k[0].shape),
                  d[n_q + n_k:].view(self.v[0].shape)) for d in self.din]
        self.copy_stream = torch.cuda.Stream(self.device)
        compute = torch.cuda.current_stream(self.device)
        self.e2e_calls = [self.cache.bind_append_attend(0, *views[i % 2], self.out[i], stream=compute)
                          for i in range(self.steps)]
        self.h2d = self.hin.nbytes
        self.d2h = self.hout.nbytes

    def _upload(self, i):
        self.din[i % 2].copy_(self.hin[i], non_blocking=True)

    def e2e_step(self):
        """Every step: its q/k/v uploaded from pinned host memory and its output read
        back, on a copy stream overlapping the neighbouring steps' compute."""
        if self.graph is not None:
            # the graph reads the step's fixed input buffers: upload all, replay, read back
            self.q.copy_(self.hq, non_blocking=True)
            self.k.copy_(self.hk, non_blocking=True)
            self.v.copy_(self.hv, non_blocking=True)
            self.step()
            self.hout.copy_(self.out, non_blocking=True)
            return
        compute, copy = torch.cuda.current_stream(self.device), self.copy_stream
        self.cache.truncate(self.L0.tolist())
        uploaded = [torch.cuda.Event(), torch.cuda.Event()]
        consumed = [torch.cuda.Event(), torch.cuda.Event()]
        copy.wait_stream(compute)
        with torch.cuda.stream(copy):
            self._upload(0)
            uploaded[0].record(copy)
        for i in range(self.steps):
            s = i % 2
            compute.wait_event(uploaded[s])
            self.e2e_calls[i]()
            consumed[s].record(compute)
            with torch.cuda.stream(copy):
                if i + 1 < self.steps:
                    copy.wait_event(consumed[(i + 1) % 2]) if i >= 1 else None
                    self._upload(i + 1)
                    uploaded[(i + 1) % 2].record(copy)
                copy.wait_event(consumed[s])
                self.hout[i].copy_(self.out[i], non_blocking=True)
        compute.wait_stream(copy)

    def dominant(self):
        return "decode"

    def kernel_name(self):
        """The decode kernel the library picks for this workload's fused steps."""
        c = self.cfg
        G = c["Hq"] // c["Hkv"]
        if 16 < G <= 32 and not self.block_rows and self.graph is None:
            return "decode_tck_kernel" if c["B"] * c["Hkv"] <= 256 else "decode_tc_kernel"
        if G <= 4 and c["B"] * c["Hkv"] >= 4 * 2 * 152 and c["hi"] + c["steps"] <= 512 and self.graph is None:
            return "decode_lanes_kernel"
        return "decode_bf16_kernel"

    def dominant_algorithmic(self, launches):
        """Algorithmic bytes of `launches` decode-kernel launches (cycling through the 64 steps)."""
        reps, rem = divmod(launches, self.steps)
        return reps * self.kv_bytes + float(self.kv_bytes_per_call[:rem].sum())

    def units(self, n_steps):
        return n_steps * self.kv_bytes / 1e9, "GB/s"

    def config(self):
        c = self.cfg
        return {"workload": self.name, "B": c["B"], "H_q": c["Hq"], "H_kv": c["Hkv"], "d_h": c["D"], "C": c["C"],
                "decode_steps_per_step": c["steps"], "old_length_range": [int(self.L0.min()), int(self.L0.max())],
                "old_length_rule": f"uniform integers in [{c['lo']}, min({c['hi']}, C - steps)] from seed {c['seed']}",
                "l2": ("inputs larger than L2: each decode step streams "
                       f"{self.kv_bytes / self.steps / 1e9:.2f} GB of K/V (L2 is 0.129 GB)")
                if self.kv_bytes / self.steps > 0.129e9 else
                ("K/V of a decode step fits in L2 "
                 f"({self.kv_bytes / self.steps / 1e9:.3f} GB); the 64 steps stream "
                 f"{self.kv_bytes / 1e9:.2f} GB; L2 not flushed between bench steps"),
                "launch": f"CUDA graph of the {self.steps} decode calls, lengths on the device" if self.graph is not None
                else "one kvc_append_attend call per decode step",
                "storage": (f"paged, {self.block_rows}-row blocks" if self.block_rows else "contiguous")}

    def cpu_tasks(self, n, steps=None):
        """``n`` oracle tasks (one (sequence, key/value head) lane each, lanes of old length
        nearest the median, the first ``steps`` decode steps -- all by default) for the host
        cores: (tasks, attention bytes of each, description)."""
        c = self.cfg
        G = c["Hq"] // c["Hkv"]
        steps = min(self.steps, steps or self.steps)
        order = np.argsort(np.abs(self.L0 - np.median(self.L0)), kind="stable")
        tasks, work = [], []
        for i in range(n):
            b = int(order[i % len(order)])
            hk = (i // len(order)) % c["Hkv"]
            L0 = int(self.L0[b])
            k = np.concatenate([self.k_prefix[b, hk, :L0].double().cpu().numpy(),
                                self.k[:steps, b, hk, 0].double().cpu().numpy()])[None]
            v = np.concatenate([self.v_prefix[b, hk, :L0].double().cpu().numpy(),
                                self.v[:steps, b, hk, 0].double().cpu().numpy()])[None]
            q = self.q[:steps, b, hk * G:(hk + 1) * G, 0].double().cpu().numpy()
            tasks.append({"kind": "decode", "q": q, "k": k, "v": v, "L0": np.int64(L0)})
            work.append(float(((L0 + 1 + np.arange(steps)) * c["D"] * 2 * 2).sum()))
        desc = (f"(b, kv-head) lanes of old length near the median ({int(np.median(self.L0))}) x {steps} "
                f"decode steps (all {G} query heads each)")
        return tasks, work, desc


# ----------------------------------------------------------------- suffix workload

class SuffixBench:
    """The suffix-chunk workload.  ``with_cache`` False (the reference arm) draws the same
    seeded inputs, takes the cuts from the oracle and never loads libkvc."""

    def __init__(self, device, batch=0, block_rows=0, with_cache=True):
        from kv_cache_append_rope_gb300 import workloads as W
        c = dict(W.CONFIGS["suffix"])
        if batch:
            c["B"] = batch
        self.cfg, self.device, self.name, self.block_rows = c, device, "suffix", block_rows
        B, H, D = c["B"], c["Hq"], c["D"]
        self.T = c["prefix"] + c["appended"]
        self.cached, self.query, self.edit = W.edited_histories(c["seed"], B, c["prefix"], c["appended"], c["vocab"])
        self.cache = None
        seed = c["seed"] * 1000
        self.k_prefix = W.normal((B, H, c["prefix"], D), seed + 1, device=device)
        self.v_prefix = W.normal((B, H, c["prefix"], D), seed + 2, device=device)
        if with_cache:
            from kv_cache_append_rope_gb300 import kvc
            from kv_cache_append_rope_gb300.kvc import KVCache
            self.cache = KVCache(B, H, self.T, D, dtype="bf16", rope_base=10000.0, device=device.index or 0,
                                 block_rows=block_rows)
            self.cache.prefill_suffix(0, None, self.k_prefix, self.v_prefix, out=False)
            self.cuts = [kvc.lcp(self.cached[b].tolist(), self.query[b].tolist()) for b in range(B)]
        else:
            from oracle import prefix as P
            self.cuts = [P.lcp_cut(self.cached[b].tolist(), self.query[b].tolist()) for b in range(B)]
        self.S = self.T - min(self.cuts)
        self.q = W.normal((B, H, self.S, D), seed + 3, device=device)
        self.k = W.normal((B, H, self.S, D), seed + 4, device=device)
        self.v = W.normal((B, H, self.S, D), seed + 5, device=device)
        self.out = torch.empty((B, H, self.S, D), dtype=torch.float32, device=device) if with_cache else None
        self.seqlen = [self.T - cu for cu in self.cuts]
        self.flops = float(sum(H * 4 * D * (s * cu + s * (s + 1) / 2) for s, cu in zip(self.seqlen, self.cuts)))
        self.host_chunk = 0
        if device.type == "cuda":
            torch.cuda.synchronize(device)

    def step(self):
        from kv_cache_append_rope_gb300 import kvc
        cuts = [kvc.lcp(self.cached[b], self.query[b]) for b in range(self.cfg["B"])]
        self.cache.truncate(cuts)
        self.cache.prefill_suffix(0, self.q, self.k, self.v, seqlen=self.seqlen, out=self.out)

    def e2e_setup(self):
        self.hq, self.hk, self.hv = (x.cpu().pin_memory() for x in (self.q, self.k, self.v))
        self.hout = torch.empty(self.out.shape, dtype=torch.float32).pin_memory()
        # the host-buffer call copies rows 0 .. seqlen[b]-1 of every head, in and out
        c = self.cfg
        rows = sum(self.seqlen)
        self.h2d = rows * (c["Hq"] + 2 * c["Hq"]) * c["D"] * 2
        self.d2h = rows * c["Hq"] * c["D"] * 4

    def e2e_step(self):
        """The cut search on the host, truncate, then kvc_prefill_suffix_host on pinned host
        buffers: each stage of sequences is uploaded, attended and read back while the next
        stage's rows are on their way in."""
        from kv_cache_append_rope_gb300 import kvc
        cuts = [kvc.lcp(self.cached[b], self.query[b]) for b in range(self.cfg["B"])]
        self.cache.truncate(cuts)
        self.cache.prefill_suffix_host(0, self.hq, self.hk, self.hv, seqlen=self.seqlen, out=self.hout,
                                       chunk_sequences=self.host_chunk, sync=False)

    def dominant(self):
        return "suffix" if self.cache.kernel_stats("suffix")[1] else "generic_attend"

    def dominant_algorithmic(self, launches):
        return launches * self.flops

    def units(self, n_steps):
        return n_steps * self.flops / 1e12, "TFLOP/s"

    def config(self):
        c = self.cfg
        return {"workload": "suffix", "B": c["B"], "H": c["Hq"], "d_h": c["D"], "prefix_tokens": c["prefix"],
                "appended_tokens": c["appended"], "C": self.T, "cuts": self.cuts,
                "flops_per_step": self.flops,
                "l2": "inputs larger than L2: the K/V prefix alone is "
                      f"{self.k_prefix.nbytes * 2 / 1e9:.1f} GB",
                "storage": (f"paged, {self.block_rows}-row blocks" if self.block_rows else "contiguous")}

    def cpu_tasks(self, n, rows=384):
        """``n`` oracle tasks for the host cores, each ``rows`` suffix rows (spread over the
        suffix) of one (sequence, head) lane against its full masked prefix:
        (tasks, flops of each, description)."""
        c = self.cfg
        B, H = c["B"], c["Hq"]
        tasks, work = [], []
        for i in range(n):
            b, h = i % B, (i // B) % H
            cut, S = self.cuts[b], self.seqlen[b]
            sel = np.linspace(0, S - 1, min(rows, S)).astype(np.int64)
            k = np.concatenate([self.k_prefix[b, h, :cut].double().cpu().numpy(),
                                self.k[b, h, :S].double().cpu().numpy()])
            v = np.concatenate([self.v_prefix[b, h, :cut].double().cpu().numpy(),
                                self.v[b, h, :S].double().cpu().numpy()])
            q = self.q[b, h:h + 1, :S].double().cpu().numpy()
            tasks.append({"kind": "suffix", "q": q, "k": k[None], "v": v[None], "T": np.int64(self.T),
                          "cut": np.int64(cut), "rows": sel})
            work.append(float(sum(4 * c["D"] * (cut + int(r) + 1) for r in sel)))
        desc = f"{rows} suffix rows per (b, h) lane, spread over the suffix, against the full masked prefix"
        return tasks, work, desc


# ----------------------------------------------------------------- main

def make_bench(name, device, batch=0, graph=False, block_rows=0, with_cache=True):
    if name == "suffix":
        return SuffixBench(device, batch, block_rows, with_cache)
    return DecodeBench(name, device, batch, graph, block_rows, with_cache)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    return world, rank, local


def max_over_ranks(x, world):
    """The largest of every rank's value (NCCL: through the GPU; gloo: on the host)."""
    if world == 1:
        return x
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# Oracle task sizes: the CPU baseline (one task per host core, each a few seconds of
# float64 work) and the reference arm (smaller tasks, one batch per bench step).
CPU_TASK = {"mha_decode": dict(steps=64), "mha_decode_short": dict(steps=64), "gqa_decode": dict(steps=32),
            "mqa_decode": dict(steps=8), "suffix": dict(rows=384)}
REF_TASK = {"mha_decode": dict(steps=16), "mha_decode_short": dict(steps=64), "gqa_decode": dict(steps=8),
            "mqa_decode": dict(steps=2), "suffix": dict(rows=96)}


def start_workers(n=None):
    """One one-thread oracle process per host core (exec'd interpreters, started before
    this process touches the GPU)."""
    from oracle.timing import Workers
    return Workers(n or os.cpu_count() or 1)


CPU_BASELINE_SECONDS = 10.0     # timed oracle wall time per workload (rounds of one task per core)


def cpu_baseline(bench, workers, unit, seconds=CPU_BASELINE_SECONDS):
    """The oracle on the host cores, warm (a first untimed round): rounds of one task per
    core side by side until about `seconds` of wall time (value = the rounds' work / the sum
    of each round's slowest task), and one task alone (`one_core`, at least a fifth as long)."""
    scale = 1e9 if unit == "GB/s" else 1e12
    tasks, work, desc = bench.cpu_tasks(workers.n, **CPU_TASK[bench.name])
    workers.run(tasks)                    # untimed: each process builds its cos/sin table once
    wall = cpu = 0.0
    rounds = 0
    while rounds == 0 or (wall < seconds and rounds < 10000):
        secs = workers.run(tasks)
        wall += max(secs)
        cpu += sum(secs)
        rounds += 1
    line = {"value": round(rounds * sum(work) / scale / wall, 6), "unit": unit, "cores": workers.n, "kind": "oracle",
            "sample": f"{rounds} rounds of {workers.n} {desc}, one oracle process per core side by side",
            "seconds": round(wall, 2), "cpu_seconds": round(cpu, 2)}
    one, n1 = 0.0, 0
    while n1 == 0 or (one < seconds / 5 and n1 < 10000):
        one += workers.run(tasks[:1])[0]
        n1 += 1
    line["one_core"] = {"value": round(n1 * work[0] / scale / one, 6), "unit": unit, "cores": 1,
                        "sample": f"{n1} rounds of 1 {desc}, alone", "seconds": round(one, 2)}
    return line


def run_ours(args, name, world, rank, local, workers=None):
    from kv_cache_append_rope_gb300 import _lib as L
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    hbm, tflops, peak_kind = peaks()
    bench = make_bench(name, device, args.batch, args.graph, args.block_rows)
    if hasattr(bench, "host_chunk"):
        bench.host_chunk = args.host_chunk
    cache = bench.cache
    if args.split_rows:
        cache.set_option(L.OPT_DECODE_SPLIT_ROWS, args.split_rows)
    if args.suffix_kernel:
        cache.set_option(L.OPT_SUFFIX_KERNEL, args.suffix_kernel)
    for _ in range(args.warmup):
        bench.step()
    torch.cuda.synchronize(device)
    cache.reset_stats()
    if hasattr(bench, "replays"):
        bench.replays = 0
    stream = torch.cuda.current_stream(device)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # pass 1: the whole step, device-timed, no per-kernel events
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(gpu_index(local)) as clocks:
        start.record(stream)
        for _ in range(args.steps):
            bench.step()
        stop.record(stream)
        torch.cuda.synchronize(device)
    barrier(world)
    ms = max_over_ranks(start.elapsed_time(stop), world)
    _, launches = cache.kernel_stats(-1)
    if getattr(bench, "graph", None) is not None:
        launches += bench.graph_kernel_launches()     # kernels the replayed graphs launched
    # pass 2: the same steps again with a CUDA event pair recorded by the library
    # around every launch on its stream, for the dominant kernel's duration
    cache.reset_stats()
    cache.set_option(L.OPT_TIMING, 1)
    for _ in range(args.steps):
        getattr(bench, "timing_pass", bench.step)()
    torch.cuda.synchronize(device)
    dom = bench.dominant()
    dom_ms, dom_launches = cache.kernel_stats(dom)
    cache.set_option(L.OPT_TIMING, 0)
    units, unit = bench.units(args.steps)
    value = units * world / (ms / 1e3)
    per_step_ms = ms / args.steps

    # roofline of the dominant kernel: algorithmic bytes (or flops) per launch / event-timed
    # duration; and the same work per bench step / the whole step's time (no per-launch events)
    alg = bench.dominant_algorithmic(dom_launches)
    alg_step = alg / args.steps
    traffic = None
    kind = TRAFFIC.get(bench.config()["workload"])
    if kind and kind[0] == "ratio":
        traffic = round(kind[1] * alg / dom_launches)
    elif kind and kind[0] == "per_sequence":
        traffic = round(kind[1] * bench.cfg["B"])
    if unit == "GB/s":
        achieved = alg / 1e9 / (dom_ms / 1e3)
        achieved_step = alg_step / 1e9 / (per_step_ms / 1e3)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic, "kernel": bench.kernel_name(),
                "peak_source": f"{peak_kind} hbm_gbs (a device copy's read + write rate, not a datasheet peak)",
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "nominal_peak": NOMINAL_HBM_GBS,
                "kernel_ms_per_launch": round(dom_ms / dom_launches, 5),
                "algorithmic_bytes_per_launch": round(alg / dom_launches),
                "step_achieved": round(achieved_step, 1), "step_frac": round(achieved_step / hbm, 4)}
    else:
        achieved = alg / 1e12 / (dom_ms / 1e3)
        achieved_step = alg_step / 1e12 / (per_step_ms / 1e3)
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tflops, "unit": "TFLOP/s",
                "frac": round(achieved / tflops, 4), "traffic": traffic, "kernel": dom,
                "peak_source": f"{peak_kind} bf16_tflops (burst)",
                "frac_of_nominal": round(achieved / NOMINAL_BF16_TFLOPS, 4), "nominal_peak": NOMINAL_BF16_TFLOPS,
                "frac_of_sustained": (round(achieved / sustained_bf16(), 4) if sustained_bf16() else None),
                "kernel_ms_per_launch": round(dom_ms / dom_launches, 3),
                "algorithmic_flops_per_launch": round(alg / dom_launches),
                "step_achieved": round(achieved_step, 1), "step_frac": round(achieved_step / tflops, 4)}
    roof["launch_modes"] = ("achieved/frac: per-launch CUDA events (a second pass; the events serialise "
                            "dependent launches); step_achieved/step_frac: the same algorithmic work per "
                            "bench step / ms_per_step of the event-free pass")

    e2e = None
    if not args.no_e2e:
        # five runs of the timed steps (on a shared machine a host-buffer step now and then
        # takes several times as long as the others); the median is reported, every run listed
        bench.e2e_setup()
        for _ in range(max(1, args.warmup)):
            bench.e2e_step()
        torch.cuda.synchronize(device)
        runs = []
        for _ in range(5):
            barrier(world)
            t0 = time.perf_counter()
            for _ in range(args.steps):
                bench.e2e_step()
            torch.cuda.synchronize(device)
            barrier(world)
            e2e_s = max_over_ranks(time.perf_counter() - t0, world)
            runs.append(units * world / e2e_s)
        e2e = {"value": round(sorted(runs)[2], 2), "unit": unit, "h2d_bytes_per_step": int(bench.h2d),
               "d2h_bytes_per_step": int(bench.d2h), "runs": [round(r, 2) for r in runs],
               "statistic": "median of 5 runs of the timed steps"}

    cpu = None
    if rank == 0 and world == 1 and workers is not None:
        cpu = cpu_baseline(bench, workers, unit)

    cache.check()
    line = {"metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(per_step_ms, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": bench.config(), "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(launches), "clocks": clocks.summary()}
    if unit == "GB/s":
        line["hbm_peak_frac"] = round(value / world / hbm, 4)
        line["decode_steps_per_s"] = round(bench.steps * args.steps * world / (ms / 1e3), 1)
    else:
        line["tensor_peak_frac"] = round(value / world / tflops, 4)
        line["steps_per_s"] = round(args.steps / (ms / 1e3), 3)
    release(bench)
    return line


def release(bench):
    """Frees a workload's device memory before the next one is built."""
    import gc
    if getattr(bench, "cache", None) is not None:
        bench.cache.destroy()
    bench.__dict__.clear()
    gc.collect()
    torch.cuda.empty_cache()


def run_reference(args, name, workers):
    """The oracle as the reference arm: each bench step one batch of oracle tasks, one per
    host core side by side, on the same seeded inputs (built with torch; libkvc is not
    loaded)."""
    device = torch.device("cuda", 0) if torch.cuda.is_available() else None
    if device is None:
        return {"impl": "reference", "unavailable": "the workload inputs are generated on a CUDA device"}
    bench = make_bench(name, device, with_cache=False)
    _, unit = bench.units(1)
    scale = 1e9 if unit == "GB/s" else 1e12
    tasks, work, desc = bench.cpu_tasks(workers.n, **REF_TASK[name])
    config = bench.config()
    release(bench)
    for _ in range(args.warmup):
        workers.run(tasks)
    secs = 0.0
    for _ in range(args.steps):
        secs += max(workers.run(tasks))
    value = sum(work) * args.steps / scale / secs
    sample = f"{workers.n} {desc}, one oracle process per core side by side, per step"
    cpu = {"value": round(value, 6), "unit": unit, "cores": workers.n, "kind": "oracle", "sample": sample}
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": unit, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(secs / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config, "cpu_baseline": cpu,
            "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


SUB_KEYS = ("value", "unit", "ms_per_step", "roofline", "cpu_baseline", "e2e", "clocks", "config", "gpu_launches",
            "hbm_peak_frac", "decode_steps_per_s", "tensor_peak_frac", "steps_per_s")


def main():
    args = parse()
    rank_env = int(os.environ.get("RANK", "0"))
    world_env = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference" and rank_env != 0:
        return                                   # the oracle arm runs on rank 0 only
    # the oracle processes start before this process touches the GPU
    workers = None
    if rank_env == 0 and (args.impl == "reference" or (world_env == 1 and not args.no_cpu_baseline)):
        workers = start_workers()
    try:
        world, rank, local = dist_setup(args) if args.impl == "ours" else (1, 0, 0)
        if args.workload == "default":
            groups = [("mha_decode", SUB_WORKLOADS)]
        elif args.workload == "all":
            groups = [(n, ()) for n in ("mha_decode", "mha_decode_short", "gqa_decode", "mqa_decode", "suffix")]
        else:
            groups = [(args.workload, ())]
        for head, subs in groups:
            if args.impl == "reference":
                line = run_reference(args, head, workers)
                if subs:
                    line["workloads"] = {}
                    for n in subs:
                        sub = run_reference(args, n, workers)
                        line["workloads"][n] = {k: sub[k] for k in SUB_KEYS if k in sub}
                print(json.dumps(line), flush=True)
                continue
            line = run_ours(args, head, world, rank, local, workers)
            if subs:
                line["workloads"] = {}
                for n in subs:
                    sub = run_ours(args, n, world, rank, local, workers)
                    line["workloads"][n] = {k: sub[k] for k in SUB_KEYS if k in sub}
            if rank == 0:
                print(json.dumps(line), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    finally:
        if workers is not None:
            workers.close()


if __name__ == "__main__":
    main()
