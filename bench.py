"""Benchmark of the EAGLE tree-verify hot path on GB300.

One step = one pass of every hot-path call over one batch:
  draft round  depth x (LM-head top-k over the expanded parents' drafter rows
               + one EAGLE-2 expansion step), then rerank/flatten
  verify       tree attention (one target-layer-shaped call), fused EAGLE-3
               projection of the verify rows, LM-head top-k of the verify
               rows (k = 1: the target argmax), tree verification
Metric: tree nodes verified per second (B * budget / step time); the step
time in microseconds is reported beside it.

Default workload: the LLaMA-3.1-8B-shaped batch-1 case (d 4096, 32/8 heads x
128, V 128256, ctx 2048, depth 6, top-k 10, width 10, budget 60, greedy).
Inputs are seeded synthetic tensors resident in HBM; weights ~ N(0, 0.02^2).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl reference]
Under torchrun each rank runs an independent replica (weak scaling, no
collective on the data path); rank 0 prints one JSON line.
"""
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

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from eagle_speculative_decoding_gb300 import binding as eb  # noqa: E402
from eagle_speculative_decoding_gb300 import synth  # noqa: E402

METRIC = "tree-verify step: tree nodes/s (B*budget / step time)"
UNIT = "nodes/s"
PROFILE = os.path.join(ROOT, "profiles", "lmhead_topk_llama8b.md")


# --------------------------------------------------------------- workload
class Workload:
    """Device-resident inputs of one step plus pinned host copies of the
    per-step inputs for the end-to-end measurement."""

    def __init__(self, name, device, seed=0):
        c = synth.CONFIGS[name]
        self.name, self.c, self.dev = name, c, device
        self.B, self.d, self.V = c["B"], c["d"], c["V"]
        self.Hq, self.Hkv, self.D = c["Hq"], c["Hkv"], c["D"]
        self.k, self.width, self.depth, self.N = c["topk"], c["width"], c["depth"], c["N"]
        self.R = self.N + 1
        self.T = c["temps"][0]
        self.dt = synth.torch_dtype(c["dtype"])
        B, d, V, R = self.B, self.d, self.V, self.R
        g = synth.generator(seed, device)
        gc = synth.generator(seed + 1)
        nrm = lambda shape, std=1.0: synth.normal(shape, std, self.dt, g, device)
        # model state (resident)
        self.w_lm = nrm((V, d), synth.WEIGHT_STD)
        self.w_proj = nrm((d, 3 * d), synth.WEIGHT_STD)
        ctx = synth.ctx_lengths(c, gc)
        kc, vc, table = synth.paged_kv(ctx.tolist(), self.Hkv, self.D, c["page"], self.dt, gc)
        self.k_cache, self.v_cache = kc.to(device), vc.to(device)
        self.block_table, self.ctx_lens = table.to(device), ctx.to(device)
        # per-step inputs: drafter rows per depth, verify-row activations
        self.P = [1 if s == 0 else self.width for s in range(self.depth)]
        host = {}
        host["draft_x"] = [synth.normal((B * p, d), 1.0, self.dt, gc) for p in self.P]
        host["root"] = synth.random_tokens((B,), V, gc)
        host["q"] = synth.normal((B, R, self.Hq, self.D), 1.0, self.dt, gc)
        host["k_tree"] = synth.normal((B, R, self.Hkv, self.D), 1.0, self.dt, gc)
        host["v_tree"] = synth.normal((B, R, self.Hkv, self.D), 1.0, self.dt, gc)
        host["h"] = [synth.normal((B * R, d), 1.0, self.dt, gc) for _ in range(3)]
        host["x_v"] = synth.normal((B * R, d), 1.0, self.dt, gc)
        # the per-step inputs live in one pinned host buffer and one device
        # buffer (256-byte aligned slots), so a step's upload is one copy
        flat = [t for v in host.values() for t in (v if isinstance(v, list) else [v])]
        offs, n = [], 0
        for t in flat:
            offs.append(n)
            n += -(-t.numel() * t.element_size() // 256) * 256
        self.host_buf = torch.empty(n, dtype=torch.uint8).pin_memory()
        # two device copies: the end-to-end loop uploads step k + 1's inputs
        # into one while step k reads the other
        self.dev_bufs = [torch.empty(n, dtype=torch.uint8, device=device) for _ in range(2)]
        self.dev_buf = self.dev_bufs[0]

        def slot(buf, t, off):
            nb = t.numel() * t.element_size()
            return buf[off:off + nb].view(t.dtype).view(t.shape)

        it = iter(range(len(flat)))
        self.host, self.dev_sets = {}, [{}, {}]
        for k, v in host.items():
            ts = v if isinstance(v, list) else [v]
            hs, ds = [], [[], []]
            for t in ts:
                i = next(it)
                h = slot(self.host_buf, t, offs[i])
                h.copy_(t)
                hs.append(h)
                for b in range(2):
                    ds[b].append(slot(self.dev_bufs[b], t, offs[i]))
            self.host[k] = hs if isinstance(v, list) else hs[0]
            for b in range(2):
                self.dev_sets[b][k] = ds[b] if isinstance(v, list) else ds[b][0]
        for b in range(2):
            self.dev_bufs[b].copy_(self.host_buf)
        self.dev_in = self.dev_sets[0]
        # outputs / state
        z = lambda *s, t=torch.int32: torch.zeros(s, dtype=t, device=device)
        self.max_nodes = 1 + synth.n_candidates(c)
        self.cand = [(z(B * p, self.k), z(B * p, self.k, t=torch.float32)) for p in self.P]
        self.tree = dict(parent=z(B, self.max_nodes), token=z(B, self.max_nodes),
                         logv=z(B, self.max_nodes, t=torch.float32), depth=z(B, self.max_nodes),
                         count=z(B), frontier=z(B, self.width), nf=z(B))
        self.flat = {n: z(B, R) for n in ("token", "parent_row", "depth", "node_id", "position")}
        self.flat["mask"] = z(B, R, t=torch.int64)
        self.flat["n_rows"] = z(B)
        self.attn_out = torch.empty((B, R, self.Hq, self.D), dtype=self.dt, device=device)
        self.g = torch.empty((B * R, d), dtype=self.dt, device=device)
        self.amax = z(B * R, 1)
        self.amax_lp = z(B * R, 1, t=torch.float32)
        # stochastic verification reads statistics of the verification LM head
        # (race candidates, row log-sum-exp, child logits), never [B, R, V] logits
        self.race_k = self.k + 1  # > children of any node of a top-k tree
        self.race_ids = z(B * R, self.race_k)
        self.race_keys = z(B * R, self.race_k, t=torch.float32)
        self.row_max = z(B * R, t=torch.float32)
        self.row_sumexp = z(B * R, t=torch.float32)
        self.child_logit = z(B * R, t=torch.float32)
        self.acc, self.path, self.out_tok = z(B), z(B, self.depth + 1), z(B, self.depth + 1)
        self.status = z(1)
        # workspaces (caller-owned scratch)
        dt_code = eb.EAGLE_BF16 if self.dt == torch.bfloat16 else eb.EAGLE_FP32
        self.dt_code = dt_code
        lm_ws = max(eb.eagle_lmhead_topk_workspace_size(B * p, d, V, self.k, dt_code) for p in self.P)
        lm_ws = max(lm_ws, eb.eagle_lmhead_topk_workspace_size(B * R, d, V, self.race_k, dt_code))
        self.ws_lm = eb.workspace(lm_ws, device)
        self.ws_fp = eb.workspace(eb.eagle_fuse_proj_workspace_size(B * R, d, dt_code), device)
        self.ws_attn = eb.workspace(eb.eagle_tree_attn_workspace_size(
            B, R, self.Hq, self.Hkv, self.D, table.shape[1], c["page"], 0, dt_code), device)
        self.ws_ver = eb.workspace(eb.eagle_tree_verify_workspace_size(B, R, V), device)

    # ------------------------------------------------------------- step
    def step(self, lm_events=None, row_events=None):
        """Launch one step on the current stream.  ``lm_events``: list that
        receives (start, end) CUDA events around each LM-head GEMM launch;
        ``row_events``: dict name -> list of (start, end) around every other
        call of the step."""
        t, f, x = self.tree, self.flat, self.dev_in

        def rt(name, call):
            if row_events is None:
                call()
                return
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            call()
            e1.record()
            row_events.setdefault(name, []).append((e0, e1))

        def timed(call, M, k):
            if lm_events is not None:
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record()
            call()
            if lm_events is not None:
                e1.record()
                lm_events.append((e0, e1, M, k))

        def lm(xr, k, ids, lps):
            if lm_events is None:
                eb.eagle_lmhead_topk(xr, self.w_lm, k, ids, lps, temperature=1.0, ws=self.ws_lm,
                                     status=self.status)
                return
            # the same kernels as eagle_lmhead_topk, with events around the GEMM alone
            timed(lambda: eb.eagle_lmhead_topk_partial(xr, self.w_lm, k, self.ws_lm, temperature=1.0,
                                                       status=self.status), xr.shape[0], k)
            eb.eagle_lmhead_topk_merge(xr.shape[0], self.d, self.V, ids, lps, self.ws_lm, dtype=self.dt_code,
                                       temperature=1.0, status=self.status)

        for s in range(self.depth):
            ids, lps = self.cand[s]
            lm(x["draft_x"][s], self.k, ids, lps)
            rt("tree_expand", lambda: eb.eagle_tree_expand(
                s, self.width, ids, lps, x["root"], t["parent"], t["token"], t["logv"], t["depth"],
                t["count"], t["frontier"], t["nf"], status=self.status))
        rt("tree_expand_finalize", lambda: eb.eagle_tree_expand_finalize(
            self.N, t["parent"], t["token"], t["logv"], t["depth"], t["count"], self.ctx_lens, f["token"],
            f["parent_row"], f["depth"], f["mask"], f["node_id"], f["position"], f["n_rows"], status=self.status))
        rt("tree_attn", lambda: eb.eagle_tree_attn(
            x["q"], x["k_tree"], x["v_tree"], self.k_cache, self.v_cache, self.block_table, self.ctx_lens,
            f["mask"], self.attn_out, ws=self.ws_attn, status=self.status))
        rt("fuse_proj", lambda: eb.eagle_fuse_proj(x["h"][0], x["h"][1], x["h"][2], self.w_proj, self.g,
                                                   ws=self.ws_fp, status=self.status))
        if self.T == 0:
            lm(x["x_v"], 1, self.amax, self.amax_lp)
            rt("tree_verify", lambda: eb.eagle_tree_verify(
                f["parent_row"], f["token"], 0.0, self.depth, self.acc, self.path, self.out_tok,
                n_rows=f["n_rows"], target_argmax=self.amax.view(self.B, self.R), V=self.V, ws=self.ws_ver,
                status=self.status))
        else:
            rt("lmhead_verify_stats", lambda: eb.eagle_lmhead_verify_stats(
                x["x_v"], self.w_lm, f["parent_row"], f["token"], self.T, self.race_k,
                self.race_ids, self.race_keys, self.row_max, self.row_sumexp, self.child_logit,
                n_rows=f["n_rows"], seed=1234, ws=self.ws_lm, status=self.status))
            rt("tree_verify_stats", lambda: eb.eagle_tree_verify_stats(
                f["parent_row"], f["token"], self.T, self.depth, self.row_max, self.row_sumexp,
                self.child_logit, self.race_ids, self.acc, self.path, self.out_tok, self.V, n_rows=f["n_rows"],
                seed=1234, status=self.status))

    def h2d(self, b=0):
        """Copy this step's inputs from pinned host memory into device input
        buffer b (one copy of the packed input buffer) on the current stream;
        returns the bytes copied."""
        self.dev_bufs[b].copy_(self.host_buf, non_blocking=True)
        return self.host_buf.numel()

    def use(self, b):
        """Make the next step() read device input buffer b."""
        self.dev_in = self.dev_sets[b]

    def d2h(self, host_out):
        n = 0
        for src, dst in zip((self.acc, self.path, self.out_tok), host_out):
            dst.copy_(src, non_blocking=True)
            n += src.numel() * src.element_size()
        return n

    def lm_bytes(self, M, k):
        es = self.w_lm.element_size()
        return self.V * self.d * es + M * self.d * es + M * k * 8


# ------------------------------------------------------------ measurement
class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling, running from before the
    first warm-up step to after the last GPU measurement.  Each sample is
    stamped with the host clock, so the samples of one window (a timed
    region) can be picked out; a window too short to hold a sample (20 steps
    of about 1 ms) falls back to the samples taken under load during the
    whole GPU run, and the summary says which."""
    Q = ("clocks.sm,clocks.max.sm,utilization.gpu,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.samples = index, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.perf_counter()  # let the sampler start before any GPU work
            while not self.samples and time.perf_counter() - t0 < 3.0:
                time.sleep(0.01)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.perf_counter(), line.strip()))

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.1)  # one more sample after the last measurement
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    @classmethod
    def parse(cls, line):
        """(sm_mhz, max_mhz, util %, set of active reasons) or None."""
        f = [x.strip() for x in line.split(",")]
        if len(f) < 7:
            return None
        try:
            sm, mx = float(f[0]), float(f[1])
        except ValueError:
            return None
        try:
            util = float(f[2])
        except ValueError:
            util = None
        reasons = {nm for nm, v in zip(cls.REASONS, f[3:7]) if v.lower() == "active"}
        return sm, mx, util, reasons

    def summary(self, t0=None, t1=None):
        """Clock record of the window [t0, t1] (host perf_counter times), or
        of every sample taken under load when the window holds none."""
        rows = [(t, self.parse(ln)) for t, ln in self.samples]
        rows = [(t, r) for t, r in rows if r is not None]
        window = [r for t, r in rows if t0 is not None and t0 <= t <= t1]
        kind = "timed region"
        if not window:
            window = [r for _, r in rows if r[2] is None or r[2] >= 50.0]
            kind = "whole GPU run, samples at >= 50 % utilisation (the timed region is shorter " \
                   "than the sampling period)"
        if not window:
            window = [r for _, r in rows]
            kind = "whole GPU run, all samples"
        if not window:
            return None
        reasons = sorted(set().union(*(r[3] for r in window)))
        return {"sm_mhz": statistics.median(r[0] for r in window),
                "sm_max_mhz": max(r[1] for r in window), "reasons": reasons,
                "samples": len(window), "window": kind}


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def bound_row(byts, flops, us, peaks):
    """Roofline of one call: the higher of its byte floor (HBM copy peak) and
    its flop floor.  Calls are timed inside a pass of whole steps, so a
    tensor-bound call is held to the sustained bf16 peak (the GEMM rate under
    the power cap), not the burst."""
    tc = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
    if byts / (peaks["hbm_gbs"] * 1e9) >= flops / (tc * 1e12):
        gbs = byts / us / 1e3
        return dict(bound="hbm", bytes_per_call=byts, flops_per_call=flops, achieved=round(gbs, 1),
                    unit="GB/s", peak=peaks["hbm_gbs"], frac=round(gbs / peaks["hbm_gbs"], 4))
    tfs = flops / us / 1e6
    return dict(bound="tensor", bytes_per_call=byts, flops_per_call=flops, achieved=round(tfs, 1),
                unit="TFLOP/s", peak=tc, peak_kind="sustained", frac=round(tfs / tc, 4))


def profile_traffic():
    """Per-launch DRAM bytes of the LM-head kernel from the committed ncu
    summary, valid only while the kernel source hash matches the capture."""
    src = os.path.join(ROOT, "eagle_speculative_decoding_gb300", "csrc", "gemm_tc.cu")
    cur = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    if not os.path.exists(PROFILE):
        return None
    vals = {}
    for line in open(PROFILE):
        if ": " in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].rsplit(": ", 1)  # keys may hold ':' themselves
            vals[k.strip()] = v.strip()
    if vals.get("gemm_tc.cu sha256[:16]") != cur:
        return None
    try:
        return float(vals["dram bytes per launch (verify-row call, M=61)"])
    except (KeyError, ValueError):
        return None


def call_work(wl, name):
    """Algorithmic (bytes, flops) of one call of the step, or None for the
    latency-bound calls."""
    es = wl.w_lm.element_size()
    M = wl.B * wl.R
    if name == "fuse_proj":
        return 3 * wl.d * wl.d * es + 4 * M * wl.d * es, 2 * M * 3 * wl.d * wl.d
    if name == "tree_attn":
        # prefix K/V, tree K/V, Q and O; Q K^T and P V over every key of each row
        ctx_sum = int(wl.ctx_lens.sum().item())
        return ((ctx_sum + M) * wl.Hkv * wl.D * 2 * es + 2 * M * wl.Hq * wl.D * es,
                4 * wl.R * wl.Hq * wl.D * (ctx_sum + wl.B * wl.R))
    if name == "lmhead_verify_stats":
        # W_U once plus the activation rows; 2 M d V flops
        return wl.V * wl.d * es + M * wl.d * es, 2 * M * wl.d * wl.V
    return None


def graph_call_us(call, dev, reps=10):
    """GPU time of one call replayed from a CUDA graph of `reps` x (256 MB
    write, call), less a graph of the writes alone: no host launch in the
    time and every call starts with a cold L2, as a call inside the step
    graph does (the step streams W_U, 8x the L2, between two such calls)."""
    flush = torch.zeros(64 * 1024 * 1024, device=dev)
    def gtime(fn):
        s = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(s):
            fn()
            fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                fn()
        g.replay()
        torch.cuda.synchronize()
        ts = []
        for _ in range(5):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / reps)
        del g
        return statistics.median(ts)
    base = gtime(lambda: flush.add_(1.0))
    t = gtime(lambda: (flush.add_(1.0), call()))
    del flush
    return max(t - base, 1e-3)


def graph_rows(wl, rows, peaks, dev):
    """Add to the rows of the calls that stream or contract their time from
    CUDA-graph replays (graph_us) and its roofline fraction (graph_frac)."""
    t, f, x = wl.tree, wl.flat, wl.dev_in
    calls = {
        "tree_attn": lambda: eb.eagle_tree_attn(
            x["q"], x["k_tree"], x["v_tree"], wl.k_cache, wl.v_cache, wl.block_table, wl.ctx_lens, f["mask"],
            wl.attn_out, ws=wl.ws_attn, status=wl.status),
        "fuse_proj": lambda: eb.eagle_fuse_proj(x["h"][0], x["h"][1], x["h"][2], wl.w_proj, wl.g, ws=wl.ws_fp,
                                                status=wl.status),
    }
    if wl.T != 0:
        calls["lmhead_verify_stats"] = lambda: eb.eagle_lmhead_verify_stats(
            x["x_v"], wl.w_lm, f["parent_row"], f["token"], wl.T, wl.race_k, wl.race_ids, wl.race_keys,
            wl.row_max, wl.row_sumexp, wl.child_logit, n_rows=f["n_rows"], seed=1234, ws=wl.ws_lm,
            status=wl.status)
    for name, call in calls.items():
        if name not in rows:
            continue
        us = graph_call_us(call, dev)
        byts, flops = call_work(wl, name)
        b = bound_row(byts, flops, us, peaks)
        rows[name].update({"graph_us": round(us, 2), "graph_frac": b["frac"],
                           "graph_timing": "CUDA-graph replays of 10 x (256 MB write, call), the writes' "
                                           "own graph subtracted: no host launch, cold L2"})


def row_rooflines(wl, steps, peaks):
    """Per-call timing of every other call of the step (CUDA events around
    each call in a separate pass; events between kernels stop the next
    kernel's early launch, so these are per-call upper bounds), with the
    roofline of the calls that stream or contract: algorithmic bytes for
    the fused projection and the attention, flops for the statistics-mode
    verification LM head; the expansion, finalize and verification walks are
    latency-bound and report their time only."""
    ev = {}
    torch.cuda.synchronize()
    torch.cuda._sleep(4_000_000)  # the host stays ahead of the GPU
    for _ in range(steps):
        wl.step(row_events=ev)
    torch.cuda.synchronize()
    out = {}
    for name, lst in ev.items():
        us = sum(a.elapsed_time(b) for a, b in lst) / len(lst) * 1e3
        row = {"avg_call_us": round(us, 2), "calls_per_step": len(lst) // steps}
        work = call_work(wl, name)
        if work is not None:
            row.update(bound_row(work[0], work[1], us, peaks))
        else:
            row.update(bound="latency")
        out[name] = row
    return out


def measure_draft_input(wl, calls, peak_gbs):
    """The drafter input FC u = W_I [r; e(x)] at this workload's draft-row
    shape (B * width rows), timed per call with CUDA events.  Its weights
    (2 d^2 bf16) are smaller than L2, so the calls rotate over copies of W_I
    that together exceed it: every call streams its weights from HBM."""
    M, d, dev = wl.B * wl.width, wl.d, wl.dev
    g = synth.generator(7, dev)
    es = wl.w_lm.element_size()
    n_copies = max(2, -(-(256 << 20) // (2 * d * d * es)))
    w_in = [synth.normal((d, 2 * d), synth.WEIGHT_STD, wl.dt, g, dev) for _ in range(n_copies)]
    r = synth.normal((M, d), 1.0, wl.dt, g, dev)
    ids = torch.randint(0, wl.V, (M,), dtype=torch.int32, device=dev, generator=g)
    u = torch.empty((M, d), dtype=wl.dt, device=dev)
    dt_code = eb.EAGLE_BF16 if wl.dt == torch.bfloat16 else eb.EAGLE_FP32
    ws = eb.workspace(eb.eagle_draft_input_workspace_size(M, d, dt_code), dev)
    for i in range(3):  # warm-up
        eb.eagle_draft_input(r, ids, wl.w_lm, w_in[i % n_copies], u, ws=ws, status=wl.status)
    torch.cuda.synchronize()
    evs = []
    torch.cuda._sleep(4_000_000)  # ~2 ms of GPU spin: the host queues every call meanwhile
    for i in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        eb.eagle_draft_input(r, ids, wl.w_lm, w_in[i % n_copies], u, ws=ws, status=wl.status)
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    st = eb.read_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {eb.STATUS.get(st, st)} in the drafter input FC")
    us = sum(a.elapsed_time(b) for a, b in evs) / calls * 1e3
    # weights + feature rows + looked-up embedding rows + output
    byts = 2 * d * d * es + 3 * M * d * es
    gbs = byts / us / 1e3
    return {"call": "eagle_draft_input", "rows": M, "hidden": d, "avg_call_us": round(us, 2),
            "bytes_per_call": byts, "achieved": round(gbs, 1), "unit": "GB/s",
            "frac": round(gbs / peak_gbs, 4), "bound": "hbm",
            "timing": f"CUDA events per call, {calls} calls rotating over {n_copies} copies of W_I "
                      "(together larger than L2); the embedding table is W_U's shape"}


def measure_draft_layer(wl, calls, peak_gbs):
    """The drafter's decoder layer at this workload's draft-row shape (B
    requests x width new nodes, the middle depth of a round), timed per call
    with CUDA events.  Its weights (>= 416 MB) exceed L2, so back-to-back
    calls stream them from HBM each time."""
    B, W, d, dev, dt = wl.B, wl.width, wl.d, wl.dev, wl.dt
    Hq, Hkv, D, I, R = wl.Hq, wl.Hkv, wl.D, synth.FFN_WIDTH[d], wl.R
    g = synth.generator(11, dev)
    nrm = lambda shape, std: synth.normal(shape, std, dt, g, dev)
    wts = dict(norm1=nrm((d,), 1.0), qkv=nrm(((Hq + 2 * Hkv) * D, d), synth.WEIGHT_STD),
               o=nrm((d, Hq * D), synth.WEIGHT_STD), norm2=nrm((d,), 1.0),
               gu=nrm((2 * I, d), synth.WEIGHT_STD), down=nrm((d, I), synth.WEIGHT_STD))
    x = nrm((B * W, d), 1.0)
    r0 = min(1 + (wl.depth // 2) * W, R - W)
    q_tree = torch.zeros((B, R, Hq, D), dtype=dt, device=dev)
    k_tree, v_tree = nrm((B, R, Hkv, D), 1.0), nrm((B, R, Hkv, D), 1.0)
    rows = torch.arange(R, device=dev)
    masks = ((torch.ones(R, dtype=torch.int64, device=dev) << rows) | 1).repeat(B, 1)  # root + self
    pos = (wl.ctx_lens[:, None] + wl.depth // 2 + 1).to(torch.int32).repeat(1, W).contiguous()
    out = torch.empty_like(x)
    dt_code = eb.EAGLE_BF16 if dt == torch.bfloat16 else eb.EAGLE_FP32
    ws = eb.workspace(eb.eagle_draft_layer_workspace_size(B, W, d, Hq, Hkv, D, I, R, wl.block_table.shape[1],
                                                          dt_code), dev)
    call = lambda: eb.eagle_draft_layer(x, wts, pos, wl.k_cache, wl.v_cache, wl.block_table, wl.ctx_lens,
                                        q_tree, k_tree, v_tree, masks, r0, out, ws=ws, status=wl.status)
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    evs = []
    torch.cuda._sleep(4_000_000)  # the host queues every call meanwhile
    for _ in range(calls):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        call()
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    st = eb.read_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {eb.STATUS.get(st, st)} in the drafter layer")
    us = sum(a.elapsed_time(b) for a, b in evs) / calls * 1e3
    es = x.element_size()
    w_bytes = sum(t.numel() for t in wts.values()) * es
    kv_bytes = int(wl.ctx_lens.sum().item()) * Hkv * D * 2 * es
    byts = w_bytes + kv_bytes + 2 * B * W * d * es
    gbs = byts / us / 1e3
    return {"call": "eagle_draft_layer", "rows": B * W, "hidden": d, "ffn": I, "avg_call_us": round(us, 2),
            "bytes_per_call": byts, "achieved": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak_gbs, 4),
            "bound": "hbm", "timing": f"CUDA events per call, {calls} calls; weights "
                                      f"{w_bytes / 1e6:.0f} MB + drafter prefix K/V {kv_bytes / 1e6:.0f} MB"}


def measure_draft_round(wl, rounds, peak_gbs):
    """A whole EAGLE draft round at this workload's shape, timed with CUDA
    events around each round: per depth, eagle_draft_rows -> eagle_draft_input
    -> eagle_draft_layer -> eagle_lmhead_topk -> eagle_tree_expand, the root
    pass first, then depth - 1 passes over width nodes per request (the last
    expansion's nodes are not drafted from).  The drafter's prefix is the
    workload's KV cache; its embedding table is W_U's shape."""
    B, d, dev, dt = wl.B, wl.d, wl.dev, wl.dt
    Hq, Hkv, D, I, W, k, depth = wl.Hq, wl.Hkv, wl.D, synth.FFN_WIDTH[d], wl.width, wl.k, wl.depth
    Rmax = 1 + (depth - 1) * W
    if Rmax > 64:
        return None
    g = synth.generator(13, dev)
    nrm = lambda shape, std: synth.normal(shape, std, dt, g, dev)
    wts = dict(norm1=nrm((d,), 1.0), qkv=nrm(((Hq + 2 * Hkv) * D, d), synth.WEIGHT_STD),
               o=nrm((d, Hq * D), synth.WEIGHT_STD), norm2=nrm((d,), 1.0),
               gu=nrm((2 * I, d), synth.WEIGHT_STD), down=nrm((d, I), synth.WEIGHT_STD))
    w_in = nrm((d, 2 * d), synth.WEIGHT_STD)
    g_root = nrm((B, d), 1.0)
    z = lambda *s_, t=torch.int32: torch.zeros(s_, dtype=t, device=dev)
    max_nodes = 1 + synth.n_candidates(wl.c)
    tree = dict(parent=z(B, max_nodes), token=z(B, max_nodes), logv=z(B, max_nodes, t=torch.float32),
                depth=z(B, max_nodes), count=z(B), frontier=z(B, W), nf=z(B))
    node_row, row_mask = z(B, max_nodes), z(B, Rmax, t=torch.int64)
    q_tree = torch.zeros((B, Rmax, Hq, D), dtype=dt, device=dev)
    k_tree, v_tree = torch.zeros((B, Rmax, Hkv, D), dtype=dt, device=dev), torch.zeros((B, Rmax, Hkv, D), dtype=dt, device=dev)
    bufs = {}
    for Wp in {1, W}:
        bufs[Wp] = dict(r=torch.empty((B * Wp, d), dtype=dt, device=dev), tok=z(B * Wp), pos=z(B, Wp),
                        u=torch.empty((B * Wp, d), dtype=dt, device=dev), ids=z(B * Wp, k),
                        lps=z(B * Wp, k, t=torch.float32))
    a_out = [torch.empty((B * (1 if s == 0 else W), d), dtype=dt, device=dev) for s in range(depth)]
    dt_code = eb.EAGLE_BF16 if dt == torch.bfloat16 else eb.EAGLE_FP32
    ws_in = eb.workspace(eb.eagle_draft_input_workspace_size(B * W, d, dt_code), dev)
    ws_layer = eb.workspace(max(eb.eagle_draft_layer_workspace_size(B, Wp, d, Hq, Hkv, D, I, Rmax,
                                                                     wl.block_table.shape[1], dt_code)
                                for Wp in (1, W)), dev)
    root = wl.dev_in["root"]

    def one_round():
        prev = g_root
        for s in range(depth):
            Wp = 1 if s == 0 else W
            bf = bufs[Wp]
            eb.eagle_draft_rows(s, W, wl.ctx_lens, node_row, row_mask, prev, bf["r"], bf["tok"], bf["pos"],
                                root_token=root, frontier=tree["frontier"], n_frontier=tree["nf"],
                                node_parent=tree["parent"], node_token=tree["token"], node_depth=tree["depth"],
                                status=wl.status)
            eb.eagle_draft_input(bf["r"], bf["tok"], wl.w_lm, w_in, bf["u"], ws=ws_in, status=wl.status)
            eb.eagle_draft_layer(bf["u"], wts, bf["pos"], wl.k_cache, wl.v_cache, wl.block_table, wl.ctx_lens,
                                 q_tree, k_tree, v_tree, row_mask, 0 if s == 0 else 1 + (s - 1) * W, a_out[s],
                                 ws=ws_layer, status=wl.status)
            eb.eagle_lmhead_topk(a_out[s], wl.w_lm, k, bf["ids"], bf["lps"], temperature=1.0, ws=wl.ws_lm,
                                 status=wl.status)
            eb.eagle_tree_expand(s, W, bf["ids"].view(B, Wp, k), bf["lps"].view(B, Wp, k), root, tree["parent"],
                                 tree["token"], tree["logv"], tree["depth"], tree["count"], tree["frontier"],
                                 tree["nf"], status=wl.status)
            prev = a_out[s]

    for _ in range(2):
        one_round()
    torch.cuda.synchronize()
    evs = []
    torch.cuda._sleep(20_000_000)  # the host queues the rounds meanwhile
    for _ in range(rounds):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        one_round()
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    st = eb.read_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {eb.STATUS.get(st, st)} in the draft round")
    us = sum(a.elapsed_time(b) for a, b in evs) / rounds * 1e3
    es = wl.w_lm.element_size()
    w_bytes = (sum(t.numel() for t in wts.values()) + w_in.numel() + wl.w_lm.numel()) * es
    kv_bytes = int(wl.ctx_lens.sum().item()) * Hkv * D * 2 * es
    byts = depth * (w_bytes + kv_bytes)
    gbs = byts / us / 1e3
    nodes = B * (k + (depth - 1) * W * k)
    return {"call": "draft round (rows, input FC, decoder layer, LM head, expansion per depth)",
            "depth": depth, "avg_round_us": round(us, 1), "draft_nodes_per_round": nodes,
            "bytes_per_round": byts, "achieved": round(gbs, 1), "unit": "GB/s", "frac": round(gbs / peak_gbs, 4),
            "bound": "hbm", "timing": f"CUDA events per round, {rounds} rounds; per depth the drafter's weights, "
                                      "W_U and the drafter prefix K/V stream once"}


def workload_config(name, world):
    """The ``config`` object of both arms' JSON lines for one workload."""
    c = synth.CONFIGS[name]
    es = 2 if c["dtype"] == "bf16" else 4
    return {"workload": name, "batch": c["B"], "hidden": c["d"],
            "heads": f"{c['Hq']}/{c['Hkv']}x{c['D']}", "vocab": c["V"], "ctx": list(c["ctx"]),
            "tree": f"depth {c['depth']}, top-k {c['topk']}, width {c['width']}, budget {c['N']}",
            "temperature": c["temps"][0], "parallelism": f"replicas x{world}",
            "l2": "not flushed: inputs larger than L2 (each step streams W_U, "
                  f"{c['V'] * c['d'] * es / 1e9:.2f} GB, {c['depth'] + 1} times)"}


def graphs_of(wl, stream, dev):
    """The step's public calls captured once into a CUDA graph per device
    input buffer (the calls never synchronise or allocate, and dependent
    launches are kept as graph edges).  The library's launches per step are
    counted on the eager step that precedes each capture."""
    graphs, per_step = [], 0
    for b in range(2):
        wl.use(b)
        side = torch.cuda.Stream(device=dev)
        side.wait_stream(stream)
        c0 = eb.launch_count()
        with torch.cuda.stream(side):
            wl.step()
        per_step = eb.launch_count() - c0
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            wl.step()
        graphs.append(g)
    wl.use(0)
    torch.cuda.synchronize()
    return graphs, per_step


def measure_workload(name, args, rank, world, clk, peaks, peak_kind, detail=True):
    """Every GPU measurement of one workload: the timed steps (device
    resident), the LM-head launches, the end-to-end loop, the per-call rows
    and (``detail``) the drafter calls."""
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    wl = Workload(name, dev, seed=args.seed + 1000 * rank)
    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        wl.step()
    torch.cuda.synchronize()
    st = eb.read_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {eb.STATUS.get(st, st)} after warm-up ({name})")
    graphs, per_step = graphs_of(wl, stream, dev)

    # ---- device-resident timing (per-step events).  No L2 flush: every step
    # streams the LM-head weights (>= 1 GB, 8x the L2) once per draft depth and
    # once more for verification, so nothing a step reads survives in L2 from
    # the previous step.
    step_events = []
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graphs[0].replay()
        e1.record(stream)
        step_events.append((e0, e1))
    torch.cuda.synchronize()
    t_wall1 = time.perf_counter()
    launches = per_step * args.steps

    # ---- the LM-head GEMM launches: a second pass of the same steps with
    # CUDA events around every LM-head GEMM launch (events between kernels
    # stop the next kernel's early launch, so this pass is not the one timed)
    lm_events = []
    barrier(world)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        wl.step(lm_events)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in step_events]
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    nodes = wl.B * wl.N * world
    value = nodes / (ms_per_step / 1e3)
    lm_ms = [a.elapsed_time(b) for a, b, _, _ in lm_events]
    lm_bytes = [wl.lm_bytes(M, k) for _, _, M, k in lm_events]
    lm_avg_ms = sum(lm_ms) / len(lm_ms)
    achieved = (sum(lm_bytes) / len(lm_bytes)) / (lm_avg_ms / 1e3) / 1e9

    # ---- end to end through the public API: every step uploads its inputs
    # from pinned host memory, runs, and the host reads its result (accepted
    # lengths, path rows, tokens) back before the next step is issued; the
    # upload of step k + 1 (a copy stream, into the other device buffer)
    # overlaps step k, as a serving loop would do it.  Timed from the first
    # upload to the last read-back.
    host_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (wl.acc, wl.path, wl.out_tok)]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event(), torch.cuda.Event()]
    barrier(world)
    torch.cuda.synchronize()
    e_start = torch.cuda.Event(enable_timing=True)
    e_start.record(copy_stream)
    with torch.cuda.stream(copy_stream):
        hb = wl.h2d(0)
    copied[0].record(copy_stream)
    db, done = 0, None
    for k in range(args.steps):
        cur = k & 1
        stream.wait_event(copied[cur])
        graphs[cur].replay()
        db = wl.d2h(host_out)
        done = torch.cuda.Event(enable_timing=True)
        done.record(stream)
        if k + 1 < args.steps:
            # the other buffer was last read by step k - 1, complete at the
            # previous read-back
            with torch.cuda.stream(copy_stream):
                wl.h2d(1 - cur)
            copied[1 - cur].record(copy_stream)
        done.synchronize()
    e2e_total = max_over_ranks(e_start.elapsed_time(done), world)
    e2e_value = nodes / (e2e_total / args.steps / 1e3)
    st = eb.read_status(wl.status)
    if st != 0:
        raise RuntimeError(f"device status {eb.STATUS.get(st, st)} ({name})")

    rows = row_rooflines(wl, max(min(args.steps, 50), 3), peaks)
    graph_rows(wl, rows, peaks, dev)
    rows["lmhead_topk"] = {"avg_call_us": round(lm_avg_ms * 1e3, 2), "calls_per_step": len(lm_events) // args.steps,
                           "bound": "hbm", "achieved": round(achieved, 1), "unit": "GB/s",
                           "frac": round(achieved / peaks["hbm_gbs"], 4),
                           "timing": "CUDA events around each launch of the LM-head GEMM kernel"}
    if detail:
        rows.update({"draft_input": measure_draft_input(wl, max(args.steps, 10), peaks["hbm_gbs"]),
                     "draft_layer": measure_draft_layer(wl, max(min(args.steps, 50), 10), peaks["hbm_gbs"]),
                     "draft_round": measure_draft_round(wl, max(min(args.steps // 10, 10), 3),
                                                        peaks["hbm_gbs"])})
    lm_roof = {"kernel": "lmhead_topk_kernel (tcgen05 LM head + top-k)", "bound": "hbm",
               "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
               "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_kind": peak_kind,
               "traffic": profile_traffic() if name == "llama8b" else None,
               "avg_launch_us": round(lm_avg_ms * 1e3, 2),
               "launches_per_step": len(lm_events) // args.steps,
               "timing": "CUDA events around each launch of the LM-head GEMM kernel "
                         "(eagle_lmhead_topk_partial; its partial merge follows outside the "
                         "events) in a second pass of the timed steps; the statistics-mode "
                         "verification call of T > 0 workloads is not among them"}
    res = {"value": round(value, 1), "unit": UNIT, "ms_per_step": round(ms_per_step, 4),
           "step_us": round(ms_per_step * 1e3, 1),
           "median_step_us": round(statistics.median(step_ms) * 1e3, 1),
           "dtype": "bf16" if wl.dt == torch.bfloat16 else "f32",
           "config": workload_config(name, world), "gpu_launches": launches, "roofline": lm_roof,
           "e2e": {"value": round(e2e_value, 1), "unit": UNIT, "h2d_bytes_per_step": hb,
                   "d2h_bytes_per_step": db,
                   "timing": "first upload to last read-back; each step's result is read on the host "
                             "before the next step is issued, and step k+1's upload (copy stream, second "
                             "device buffer) overlaps step k; the step's public calls are captured once "
                             "into a CUDA graph per input buffer and replayed"},
           "clocks": clk.summary(t_wall0, t_wall1), "rows": rows,
           "launch": "each timed step replays a CUDA graph of the step's public calls",
           "wall_s": round(t_wall1 - t_wall0, 3)}
    # the other calls that bound the step (per-call rows above)
    others = {k: rows[k] for k in ("lmhead_verify_stats", "tree_attn", "fuse_proj") if k in rows}
    res["rooflines"] = {k: {kk: v[kk] for kk in ("bound", "achieved", "peak", "unit", "frac", "avg_call_us",
                                                 "graph_us", "graph_frac")
                            if kk in v} for k, v in others.items()}
    del graphs
    return res, wl


def run_ours(args, rank, world):
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    peaks, peak_kind = measured_peaks()
    names = [args.workload] + [n for n in args.also if n != args.workload]
    out = {}
    with ClockSampler(dev.index) as clk:
        for i, name in enumerate(names):
            r, wl = measure_workload(name, args, rank, world, clk, peaks, peak_kind)
            out[name] = r
            del wl
            torch.cuda.empty_cache()
    head = out[names[0]]
    res = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
           "step_us": head["step_us"], "median_step_us": head["median_step_us"],
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
           "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights)",
           "config": head["config"], "gpu_launches": head["gpu_launches"], "roofline": head["roofline"],
           "rooflines": head["rooflines"], "e2e": head["e2e"], "clocks": head["clocks"],
           "rows": head["rows"], "launch": head["launch"], "wall_s": head["wall_s"]}
    if len(names) > 1:
        res["workloads"] = {n: out[n] for n in names[1:]}
    return res


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle
class OracleStep:
    """The CPU oracle running one full step of the workload (test
    infrastructure, used only for the CPU baseline and the reference arm).
    ``requests`` < B runs the step on the first ``requests`` requests of the
    batch only (a bounded sample of a large workload: apart from the weight
    reads, the oracle's work is per request)."""

    def __init__(self, name, seed=0, requests=None):
        import numpy as np
        import oracle
        self.np, self.oracle = np, oracle
        c = synth.CONFIGS[name]
        self.c = c
        B, d, V, width, depth, N = c["B"], c["d"], c["V"], c["width"], c["depth"], c["N"]
        R = N + 1
        b = B if requests is None else max(1, min(int(requests), B))
        self.B = b
        gen = synth.generator(seed)
        dt = synth.torch_dtype(c["dtype"])
        f64 = lambda t: t.double().numpy()
        self.w_lm = f64(synth.normal((V, d), synth.WEIGHT_STD, dt, gen))
        self.w_proj = f64(synth.normal((d, 3 * d), synth.WEIGHT_STD, dt, gen))
        self.ctx = synth.ctx_lengths(c, gen)[:b]
        kc, vc, table = synth.paged_kv(self.ctx.tolist(), c["Hkv"], c["D"], c["page"], dt, gen)
        self.kc, self.vc, self.table = f64(kc), f64(vc), table.numpy()
        self.rows = [f64(synth.normal((b * (1 if s == 0 else width), d), 1.0, dt, gen))
                     for s in range(depth)]
        self.q = f64(synth.normal((b, R, c["Hq"], c["D"]), 1.0, dt, gen))
        self.kt = f64(synth.normal((b, R, c["Hkv"], c["D"]), 1.0, dt, gen))
        self.vt = f64(synth.normal((b, R, c["Hkv"], c["D"]), 1.0, dt, gen))
        self.hs = [f64(synth.normal((b * R, d), 1.0, dt, gen)) for _ in range(3)]
        self.xv = f64(synth.normal((b * R, d), 1.0, dt, gen))
        self.T = c["temps"][0]
        self.nodes = b * N

    def run(self):
        """One step; returns its wall seconds."""
        np, oracle, c = self.np, self.oracle, self.c
        B, k, width, depth, N = self.B, c["topk"], c["width"], c["depth"], c["N"]
        R = N + 1
        t0 = time.perf_counter()
        sts = [oracle.tree_expand_init(7) for _ in range(B)]
        for s in range(depth):
            P = 1 if s == 0 else width
            res = oracle.lmhead_topk(self.rows[s], self.w_lm, k)
            for b in range(B):
                n = len(sts[b]["frontier"])
                oracle.tree_expand_step(sts[b], res["ids"][b * P:b * P + n],
                                        res["logprobs"][b * P:b * P + n], width)
        flats = [oracle.tree_expand_finalize(sts[b], N, int(self.ctx[b]), R_out=R) for b in range(B)]
        mask = np.stack([f["mask"] for f in flats])
        oracle.tree_attn(self.q, self.kt, self.vt, self.kc, self.vc, self.table, self.ctx.numpy(), mask)
        oracle.fuse_proj(*self.hs, self.w_proj)
        parent = np.stack([f["parent_row"] for f in flats])
        tok = np.stack([f["token"] for f in flats])
        nr = [f["n_rows"] for f in flats]
        if self.T == 0:
            am = oracle.lmhead_topk(self.xv, self.w_lm, 1)["ids"].reshape(B, R)
            oracle.tree_verify(parent, tok, 0.0, depth, n_rows=nr, target_argmax=am)
        else:
            st = oracle.verify_stats(self.xv, self.w_lm, parent, tok, self.T, k + 1, seed=1234,
                                     n_rows=nr)
            oracle.tree_verify_stats(parent, tok, self.T, depth, st["row_max"], st["row_sumexp"],
                                     st["child_logit"], st["race_ids"], n_rows=nr, seed=1234)
        return time.perf_counter() - t0


# bounded samples of each workload for the CPU figures: (requests, seconds of
# timed oracle work to aim for), on all cores and on one core
CPU_SAMPLE = {"serve64": (8, 4), "chain3": (8, 4), "long4": (1, 1)}


def sample_requests(name, one_core):
    c = synth.CONFIGS[name]
    req = CPU_SAMPLE.get(name, (c["B"], c["B"]))[1 if one_core else 0]
    return min(req, c["B"])


def time_oracle(name, requests, budget_s, max_steps=50):
    """Whole oracle steps on ``requests`` requests until about ``budget_s``
    seconds of CPU work (at least one step); returns (nodes per step, step
    seconds)."""
    o = OracleStep(name, requests=requests)
    secs = [o.run()]
    while sum(secs) < budget_s and len(secs) < max_steps:
        secs.append(o.run())
    return o.nodes, secs


def oracle_figure(name, nodes, secs, cores, requests, where):
    mean = sum(secs) / len(secs)
    B = synth.CONFIGS[name]["B"]
    part = f" on {requests} of its {B} requests" if requests < B else ""
    return {"value": round(nodes / mean, 3), "median_value": round(nodes / statistics.median(secs), 3),
            "unit": UNIT, "cores": cores,
            "sample": f"{len(secs)} {name} step(s){part} {where}, {sum(secs):.1f} s of CPU time, "
                      f"{mean * 1e3:.0f} ms per step (mean; nodes/s = nodes of the sample / step time)"}


def one_core_figure(name):
    """The oracle on one core: a child process with one BLAS thread, pinned
    to one CPU before its timed steps."""
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    env.pop("RANK", None)
    env.pop("WORLD_SIZE", None)
    try:
        out = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-one-core", name],
                             env=env, capture_output=True, text=True, timeout=600)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except (subprocess.SubprocessError, ValueError, IndexError, OSError) as e:
        return {"error": f"one-core oracle run failed: {type(e).__name__}"}


def one_core_child(name):
    """Body of the child process of one_core_figure."""
    req = sample_requests(name, one_core=True)
    o = OracleStep(name, requests=req)  # set-up on the process's threads
    cpu = sorted(os.sched_getaffinity(0))[0]
    os.sched_setaffinity(0, {cpu})
    torch.set_num_threads(1)
    secs = [o.run()]
    while sum(secs) < 10.0 and len(secs) < 20:
        secs.append(o.run())
    print(json.dumps(oracle_figure(name, o.nodes, secs, 1, req, "on one core (one BLAS thread)")))


def cpu_baseline(name):
    """The oracle on the host cores: a bounded sample of the workload on all
    cores (the headline ``value``), and the same on one core."""
    req = sample_requests(name, one_core=False)
    nodes, secs = time_oracle(name, req, 12.0)
    res = oracle_figure(name, nodes, secs, cpu_cores(), req, "on all cores")
    res["kind"] = "oracle"
    res["one_core"] = one_core_figure(name)
    return res


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def run_reference(args, rank, world):
    """The CPU oracle timed as the reference arm (rank 0 only): each step is
    one oracle step of the workload on the host cores (a bounded sample of
    the requests where a whole step would take minutes)."""
    if rank != 0:
        return None
    req = sample_requests(args.workload, one_core=False)
    o = OracleStep(args.workload, requests=req)
    for _ in range(args.warmup):
        o.run()
    secs = [o.run() for _ in range(args.steps)]
    fig = oracle_figure(args.workload, o.nodes, secs, cpu_cores(), req, "on all cores")
    ms = 1e3 * sum(secs) / len(secs)
    value = fig["value"]
    fig["kind"] = "oracle"
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
           "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 1), "median_step_us": round(statistics.median(secs) * 1e6, 1),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded N(0,1) activations, N(0,0.02^2) weights)",
           "config": workload_config(args.workload, world), "cpu_baseline": fig,
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    extra = [n for n in args.also if n != args.workload]
    if extra:
        res["workloads"] = {}
        for n in extra:
            req = sample_requests(n, one_core=False)
            nodes, secs = time_oracle(n, req, 8.0, max_steps=args.steps)
            f = oracle_figure(n, nodes, secs, cpu_cores(), req, "on all cores")
            res["workloads"][n] = {"value": f["value"], "unit": UNIT, "config": workload_config(n, world),
                                   "cpu_baseline": dict(f, kind="oracle")}
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 1000; 20 for --impl reference, whose steps run the CPU oracle)")
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default="llama8b", choices=sorted(synth.CONFIGS),
                    help="the headline workload (value, roofline, e2e of the line)")
    ap.add_argument("--also", default="serve64",
                    help="comma-separated further workloads measured in the same run and reported "
                         "under 'workloads' ('none' for none); default: serve64, the batch-64 half "
                         "of the metric")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-one-core", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_one_core:
        one_core_child(args.oracle_one_core)
        return
    args.also = [] if args.also in ("", "none") else args.also.split(",")
    for n in args.also:
        if n not in synth.CONFIGS:
            ap.error(f"unknown workload {n}")
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 1000
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        torch.distributed.init_process_group("nccl" if args.impl == "ours" else "gloo")
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            torch.cuda.empty_cache()
            res["cpu_baseline"] = cpu_baseline(args.workload)
            for n, w in res.get("workloads", {}).items():
                req = sample_requests(n, one_core=False)
                nodes, secs = time_oracle(n, req, 8.0)
                w["cpu_baseline"] = dict(oracle_figure(n, nodes, secs, cpu_cores(), req, "on all cores"),
                                         kind="oracle")
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
