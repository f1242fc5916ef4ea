#!/usr/bin/env python
"""Benchmark of the split-residency MoE layer-step on GB300.

One step = one layer-step of every layer of the workload over one batch of
synthetic input: route + split + count, the MXFP4 expert FFN over both
residency banks (one call over both banks; ``--banks streams``: two calls on
two streams), and the finalize.

By default (``--config all``) one run measures every workload, with one
context holding the 16-stream decode's four layers (layers 0 and 2 split
295 hot / 89 cold, layers 1 and 3 all in HBM):
  - headline: the 16-stream decode step (4 layers, 112 tokens);
  - ``configs.decode1``: the one-user decode step on layer 0 (7 tokens);
  - ``configs.prefill_shift``: an 8192-token chunk on split layer 0 right
    after a domain shift, with the cold staging pool off and on;
  - ``configs.adaptive``: 128 one-user steps on layer 0 with a domain shift
    at step 64, counts read every 16 steps and the policy's swaps applied
    between steps (up to 8 per step), timing steps and swaps;
  - ``configs.prefill``: an 8192-token prefill chunk on layer 1 (all 384
    experts in HBM, near-uniform routing).
``--config NAME`` measures one workload alone in a context of its own.

Prints one JSON line.  ``value`` = tokens/s of the whole job with inputs
resident in HBM (each step CUDA-graph replayed, timed with CUDA events on the
launching stream, L2 flushed before every timed step); ``e2e`` = the same
metric with the inputs copied from pinned host memory and the outputs copied
back inside the timed region.  ``bytes_roofline`` = the step's bytes
roofline against its time: the distinct hot experts' bytes at the HBM peak
and the distinct cold experts' bytes at the measured host-link bandwidth,
taken as the larger of the two per layer (``frac_max``, a bound: the banks
stream at the same time) and as their sum (``frac_sum``, the metric's literal
form, which bank overlap lets exceed 1).

``--impl reference`` times the CPU oracle on the host cores instead (a
bounded sample of the same workload).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer-step µs & tokens/s; fraction of HBM+host-link bytes roofline"
WORKLOADS = {
    "decode1": "one-user decode step, 1 MoE layer: 384 experts, top-6, H=4096, I=2880, 7 tokens, "
               "Zipf(1.1) skew, 295 hot (HBM) / 89 cold (pinned host)",
    "decode16": "16-stream decode step, 4 MoE layers (layers 0,2 split 295/89, layers 1,3 all-HBM), "
                "112 tokens, 384 experts, top-6, H=4096, I=2880, Zipf(1.1) skew per layer",
    "adaptive": "adaptive residency under a domain shift: 1 layer of the one-user shape, 128 decode steps of "
                "7 tokens, Zipf ranking redrawn at step 64, counts read every 16 steps, up to 8 swaps per step",
    "prefill": "prefill chunk, 1 MoE layer, 384 experts all in HBM, top-6, 8192 tokens, near-uniform routing",
}
HEADLINE = "decode16"


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="all", choices=sorted(WORKLOADS) + ["all"])
    ap.add_argument("--pool", type=int, default=16, help="distinct input batches cycled through")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--banks", default="fused", choices=["streams", "fused"],
                    help="the two banks' FFN calls on two streams at once, or one call over both banks")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of CPU-oracle work")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling-size variant: this many experts per layer (same expert geometry)")
    ap.add_argument("--hot", type=int, default=0, help="hot-bank experts for --experts")
    ap.add_argument("--tokens", type=int, default=0, help="profiling-size variant: tokens per step")
    ap.add_argument("--skip", default="", help="comma-separated sub-configs of --config all to leave out")
    ap.add_argument("--act", default="e4m3x2", choices=["e4m3x2", "mxfp8"],
                    help="activation format of prefill-sized steps for --config prefill")
    return ap.parse_args(argv)


def bench_config(args, name=None):
    """The workload of a run: the named config, optionally narrowed to fewer
    experts (``--experts``/``--hot``) or another token count (``--tokens``).
    Both arms use it."""
    name = name or (HEADLINE if args.config == "all" else args.config)
    cfg = synth.get_config(name)
    if args.experts:
        cfg = synth.get_config(name, E=args.experts, n_hot=args.hot or cfg.n_hot * args.experts // cfg.E)
    if args.tokens:
        cfg = dataclasses.replace(cfg, T=args.tokens)
    return cfg


def slowest_rank_ms(total_ms, dist=None, device="cpu"):
    """The job's time: the largest of the ranks' own totals (one process per
    GPU, each timing its steps with CUDA events)."""
    if dist is None:
        return float(total_ms)
    import torch
    t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world, tokens_per_step, steps, total_ms):
    """Whole-job throughput: the tokens all ranks processed over the slowest
    rank's time."""
    return world * tokens_per_step * steps / (total_ms * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def distinct_experts(ids, mask):
    u = np.unique(ids)
    return int((mask[u] == 1).sum()), int((mask[u] == 0).sum())


def bytes_roofline(dh, dc, step_ms, eb, hbm_gbs, link_gbs):
    """Per step, per layer: t_sum = hot bytes / HBM + cold bytes / link and
    t_max = the larger of the two; summed over layers and steps, over the
    steps' measured time.  dh, dc: [steps][layers] distinct hot / cold
    experts."""
    dh = np.asarray(dh, np.float64)
    dc = np.asarray(dc, np.float64)
    th = dh * eb / (hbm_gbs * 1e9)
    tc = dc * eb / (link_gbs * 1e9)
    t_meas = float(np.sum(step_ms)) * 1e-3
    return {"frac_max": float(np.sum(np.maximum(th, tc)) / t_meas),
            "frac_sum": float(np.sum(th + tc) / t_meas),
            "t_roof_max_us": float(np.mean(np.sum(np.maximum(th, tc), axis=1))) * 1e6,
            "t_roof_sum_us": float(np.mean(np.sum(th + tc, axis=1))) * 1e6,
            "t_step_us": t_meas / len(step_ms) * 1e6,
            "distinct_hot": float(np.mean(dh.sum(axis=1))), "distinct_cold": float(np.mean(dc.sum(axis=1))),
            "note": "frac_max counts each layer's slower bank (the banks stream at the same time, so this is "
                    "the bound); frac_sum adds the two banks' times and can exceed 1 when they overlap"}


class ClockSampler:
    """nvidia-smi samples during the timed region (read only)."""

    def __init__(self, dev):
        self.dev = dev
        self.lines = []
        self.proc = None

    def __enter__(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def wait_first(self, timeout=10.0):
        """Wait until nvidia-smi has produced a sample: its start-up takes driver
        locks that would otherwise stall the timed launches."""
        t0 = time.time()
        while self.proc and not self.lines and time.time() - t0 < timeout:
            time.sleep(0.02)

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------- CPU oracle

def cpu_oracle_steps(cfg, layer_weights, pool, budget_s):
    """Time the CPU oracle on whole layer-steps until the budget is spent.
    layer_weights: {layer: stacked logical weights}; pool: list of
    (layer, logits, x) layer-steps, taken in order.  Returns (tokens/s of the
    workload -- a step of cfg.L layer-steps processes cfg.T tokens --,
    layer-steps done, seconds, threads)."""
    import oracle
    t_used, done = 0.0, 0
    while t_used < budget_s and done < len(pool):
        layer, lg, x = pool[done]
        t0 = time.perf_counter()
        oracle.layer_step(layer_weights[layer], lg, x, cfg.k)
        t_used += time.perf_counter() - t0
        done += 1
    tokens = done * pool[0][1].shape[0] / cfg.L
    return tokens / t_used, done, t_used, oracle.num_threads()


def single_core_oracle(cfg, layer_weights, pool, budget_s):
    """The same oracle layer-steps on one host thread, at least one whole
    layer-step (one-user decode sizes only: larger steps need every core).
    Returns the cpu_baseline sub-entry."""
    import oracle
    if pool[0][1].shape[0] > 16:
        return None
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        tps, n, used, _ = cpu_oracle_steps(cfg, layer_weights, pool, budget_s)
    finally:
        oracle.set_num_threads(cores)
    return {"value": tps, "unit": "tokens/s", "cores": 1, "sample": f"{n} whole layer-steps, {used:.1f} s"}


def oracle_pool(cfg, layers, n, T):
    """Layer-steps for the oracle's sample: step s of layer layers[s % len]."""
    out = []
    for s in range(n):
        l = layers[s % len(layers)]
        out.append((l, synth.router_logits(cfg, l, s, T=T), synth.activations(cfg, l, s, T=T)))
    return out


def cpu_sample_layers(cfg):
    """Layers the CPU sample walks through: all of them up to two."""
    return list(range(min(cfg.L, 2)))


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    cfg = bench_config(args)
    layers = cpu_sample_layers(cfg)
    weights = {l: synth.layer_weights(cfg, l) for l in layers}
    n = max(1, min(args.steps + args.warmup, 64))
    T = cfg.T if cfg.T <= 256 else 64
    pool = oracle_pool(cfg, layers, n, T)
    budget = min(120.0, max(10.0, args.cpu_budget))
    tps, done, used, cores = cpu_oracle_steps(cfg, weights, pool, budget)
    sample = (f"{done} whole layer-steps of {T} tokens (layers {layers} of the {cfg.name} workload), {used:.1f} s; "
              f"tokens/s counts a {cfg.L}-layer step of {T} tokens as {cfg.L} layer-steps")
    name = HEADLINE if args.config == "all" else args.config
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": done, "warmup": 0, "ms_per_step": used / done * 1e3 * cfg.L, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOADS[name] + ("" if T == cfg.T else f"; sampled at {T} tokens")},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "single_core": single_core_oracle(cfg, weights, pool, max(1.0, budget / 4))},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- profiles

def code_only(text):
    """C++/CUDA source without its comments, all white space collapsed to
    single blanks: what the compiler reads of it (string and character
    literals are kept whole)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_sha():
    """Hash of the FFN kernels' code, comments and layout aside (a stored
    profile is used only while the code is unchanged)."""
    h = hashlib.sha256()
    for name in ("ffn_tc.cu", "ffn_tc_decode.cuh"):
        with open(os.path.join(ROOT, "cold_expert_residency_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(config, key="bytes_per_hot_expert"):
    """DRAM bytes of an FFN call per unit of work (per distinct hot expert for
    the decode calls, per routed pick for the prefill calls) from a committed
    ncu summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(config)
        if e and e.get("source_sha") == source_sha():
            return e.get(key)
    except Exception:
        pass
    return None


# ------------------------------------------------------------- GPU session

class Session:
    """One process on one GPU: the library, the peaks, the host-link probe, an
    L2 flush buffer and the launching stream."""

    def __init__(self, args):
        import torch
        import cold_expert_residency_gb300 as moe
        self.torch, self.moe, self.args = torch, moe, args
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        torch.cuda.set_device(self.local)
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl", device_id=torch.device("cuda", self.local))
            self.dist = dist
        moe.build()
        self.dev = torch.device("cuda", self.local)
        self.hbm_peak, self.tf_burst, self.tf_sust, self.peak_src = load_peaks()
        self.main = torch.cuda.Stream(device=self.dev)
        self.flush = torch.empty(512 << 20, dtype=torch.uint8, device=self.dev)
        try:   # external events become timing nodes inside a captured graph
            torch.cuda.Event(enable_timing=True, external=True)
            self.in_graph_events = True
        except TypeError:
            self.in_graph_events = False
        self.link_gbs = self.hbm_probe_gbs = None

    def event(self):
        if self.in_graph_events:
            return self.torch.cuda.Event(enable_timing=True, external=True)
        return self.torch.cuda.Event(enable_timing=True)

    def place(self, cfg, T_max, layer_masks):
        """A context of len(layer_masks) layers of cfg's geometry; layer l is
        placed with layer_masks[l] and the weights of synthetic layer l.
        Returns (ctx, weights kept for the CPU sample's layers)."""
        moe = self.moe
        ctx = moe.moe_create(len(layer_masks), cfg.E, cfg.k, cfg.H, cfg.I, T_max, device=self.local)
        keep = {}
        for l, m in enumerate(layer_masks):
            w = synth.layer_weights(cfg, l)
            moe.moe_init_banks(ctx, l, *w, m)
            if l in cpu_sample_layers(cfg) and self.rank == 0:
                keep[l] = w
            del w
        if self.link_gbs is None:
            self.link_gbs, self.hbm_probe_gbs = moe.moe_probe_link(ctx, 1 << 30, 5)
        return ctx, keep

    def barrier(self):
        if self.dist:
            self.dist.barrier()
        self.torch.cuda.synchronize()


class StepRunner:
    """Graph-replayed layer-steps of `layers` of a context (one step = one
    layer-step of each, in order) over a pool of synthetic inputs."""

    def __init__(self, S, ctx, cfg, layers, T, npool, count_on, input_layers=None, step_offset=0):
        torch, moe = S.torch, S.moe
        from cold_expert_residency_gb300.runtime import LayerStep
        self.S, self.ctx, self.cfg, self.layers, self.T = S, ctx, cfg, list(layers), T
        self.count_on = count_on
        self.npool = npool
        src = list(input_layers) if input_layers is not None else self.layers
        # synthetic inputs: step s of input layer src[i] feeds context layer layers[i]
        self.pool_lg = [[synth.router_logits(cfg, l, step_offset + s, T=T) for l in src] for s in range(npool)]
        self.pool_x = [[synth.activations(cfg, l, step_offset + s, T=T) for l in src] for s in range(npool)]
        dev = S.dev
        self.d_lg = torch.stack([torch.from_numpy(np.stack(p)) for p in self.pool_lg]).to(dev)
        self.d_x = torch.stack([torch.from_numpy(np.stack(p).view(np.int16)) for p in self.pool_x]).to(dev)
        self.steps = [LayerStep(ctx, cfg.E, cfg.k, cfg.H, T, device=dev) for _ in self.layers]
        self.ffn_ev = {l: (S.event(), S.event()) for l in self.layers}
        self.graph = None

    def load_inputs(self, i, stream):
        with self.S.torch.cuda.stream(stream):
            for n, st in enumerate(self.steps):
                st.buf.logits[:self.T].copy_(self.d_lg[i % self.npool, n], non_blocking=True)
                st.buf.x[:self.T].copy_(self.d_x[i % self.npool, n], non_blocking=True)

    def enqueue(self, count=None, ffn_events=False):
        S, moe, T = self.S, self.S.moe, self.T
        cnt = self.count_on if count is None else count
        for l, st in zip(self.layers, self.steps):
            b = st.buf
            moe.moe_route_split_count(self.ctx, l, b.logits, T, cnt, b.ids, b.w, b.ws_ptr, S.main)
            if ffn_events:
                self.ffn_ev[l][0].record(S.main)
            if S.args.banks == "fused":   # both banks' FFN, one launch per GEMM
                moe.moe_expert_ffn_bank(self.ctx, l, moe.MOE_BANK_BOTH, b.x, T, b.ws_ptr, b.Y, S.main)
            else:                         # the two banks' calls on two streams at once
                st.ev_routed.record(S.main)
                st.cold_stream.wait_event(st.ev_routed)
                moe.moe_expert_ffn_bank(self.ctx, l, moe.MOE_BANK_COLD, b.x, T, b.ws_ptr, b.Y, st.cold_stream)
                st.ev_cold.record(st.cold_stream)
                moe.moe_expert_ffn_bank(self.ctx, l, moe.MOE_BANK_HOT, b.x, T, b.ws_ptr, b.Y, S.main)
                S.main.wait_event(st.ev_cold)
            if ffn_events:
                self.ffn_ev[l][1].record(S.main)
            moe.moe_finalize(b.Y, b.w, T, self.cfg.k, self.cfg.H, b.out, S.main)

    def capture(self):
        """One eager step (counting this library's launches), then the graph."""
        S, torch = self.S, self.S.torch
        self.load_inputs(0, S.main)
        n0 = S.moe.moe_kernel_launches()
        with torch.cuda.stream(S.main):
            self.enqueue()
        S.main.synchronize()
        self.launches_per_step = S.moe.moe_kernel_launches() - n0
        if S.args.no_graph:
            return
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=S.main):
            self.enqueue(ffn_events=S.in_graph_events)

    def run_step(self):
        if self.graph is not None:
            self.graph.replay()
        else:
            with self.S.torch.cuda.stream(self.S.main):
                self.enqueue(ffn_events=True)

    def settle(self, warmup):
        """Every pooled batch once, untimed (the first read of a weight page
        sets up its address translation and runs far slower), then `warmup`
        flushed steps."""
        S, torch = self.S, self.S.torch
        for i in range(self.npool):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                self.run_step()
        S.main.synchronize()
        for i in range(warmup):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                self.run_step()
        S.main.synchronize()

    def timed(self, steps, first, clocks=True):
        """`steps` flushed steps enqueued back to back and synchronized once
        (so a host stall cannot open a gap inside a step's events); returns
        (step ms list, clock summary or None)."""
        S, torch = self.S, self.S.torch
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        S.barrier()
        clk = ClockSampler(S.local) if clocks else None
        if clk:
            clk.__enter__()
            clk.wait_first()
        try:
            S.barrier()
            for i in range(steps):
                self.load_inputs(first + i, S.main)
                with torch.cuda.stream(S.main):
                    S.flush.zero_()
                    evs[i][0].record(S.main)
                    self.run_step()
                    evs[i][1].record(S.main)
            S.main.synchronize()
        finally:
            if clk:
                clk.__exit__(None, None, None)
        return [a.elapsed_time(b) for a, b in evs], (clk.summary() if clk else None)

    def ffn_in_step_ms(self, n, first=0):
        """Each layer's FFN call inside the replayed step (eager steps where
        events cannot be graph nodes), one step at a time."""
        S, torch = self.S, self.S.torch
        out = {l: [] for l in self.layers}
        for i in range(n):
            self.load_inputs(first + i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                if self.graph is not None and S.in_graph_events:
                    self.graph.replay()
                else:
                    self.enqueue(ffn_events=True)
            S.main.synchronize()
            for l in self.layers:
                out[l].append(self.ffn_ev[l][0].elapsed_time(self.ffn_ev[l][1]))
        return out

    def distinct(self, i, masks):
        """[layers] distinct hot and cold experts of pooled step i, and hot picks."""
        dh, dc, hp = [], [], []
        k = self.cfg.k
        for n, l in enumerate(self.layers):
            ids = np.argsort(-self.pool_lg[i % self.npool][n], axis=1, kind="stable")[:, :k]
            a, c = distinct_experts(ids, masks[l])
            dh.append(a)
            dc.append(c)
            hp.append(int((masks[l][ids] == 1).sum()))
        return dh, dc, hp

    def e2e_ms(self, n):
        """Host inputs -> step -> host outputs through the library's host-buffer
        call (moe_layer_step_host: copies in, route, both banks' FFN, finalize,
        copy out), one call per layer, all inside the events."""
        S, torch, moe = self.S, self.S.torch, self.S.moe
        T, L = self.T, len(self.layers)
        h_lg = self.d_lg.cpu().pin_memory()
        h_x = self.d_x.cpu().pin_memory()
        h_out = torch.zeros((L, T, self.cfg.H), dtype=torch.int16).pin_memory()
        scratch = torch.empty(moe.moe_step_scratch_bytes(self.ctx, T) + 256, dtype=torch.uint8, device=S.dev)
        sp = (scratch.data_ptr() + 255) // 256 * 256
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for i in range(n):
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                ev0.record(S.main)
                for m, l in enumerate(self.layers):
                    moe.moe_layer_step_host(self.ctx, l, h_lg[i % self.npool, m], h_x[i % self.npool, m], T,
                                            self.count_on, h_out[m], sp, S.main)
                ev1.record(S.main)
            S.main.synchronize()
            ts.append(ev0.elapsed_time(ev1))
        h2d = L * T * (self.cfg.E * 4 + self.cfg.H * 2)
        d2h = L * T * self.cfg.H * 2
        return ts, h2d, d2h

    def replay_graph_us(self, build, n):
        """Mean µs of a graph built by build() (enqueueing on the main stream),
        replayed after an L2 flush with events around it."""
        S, torch = self.S, self.S.torch
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=S.main):
            build()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ts = []
        for i in range(n):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                ev0.record(S.main)
                g.replay()
                ev1.record(S.main)
            S.main.synchronize()
            ts.append(ev0.elapsed_time(ev1) * 1e3)
        return ts

    def call_alone_us(self, call, n):
        """µs of one call alone: events captured inside a replayed graph just
        around it (so the graph's launch is outside the timed span), after an
        L2 flush; plain stream events when graphs cannot hold events."""
        S, torch = self.S, self.S.torch
        ea = (S.event(), S.event())
        g = None
        if self.graph is not None and S.in_graph_events:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=S.main):
                ea[0].record(S.main)
                call()
                ea[1].record(S.main)
        ts = []
        for i in range(n):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                if g is not None:
                    g.replay()
                else:
                    ea[0].record(S.main)
                    call()
                    ea[1].record(S.main)
            S.main.synchronize()
            ts.append(ea[0].elapsed_time(ea[1]) * 1e3)
        return ts

    def call_repeated_us(self, call, reps, n):
        """µs per call of `reps` calls back to back inside one replayed graph
        (events around the whole run, after an L2 flush): the first call reads
        its inputs from DRAM, the rest from L2, as a call right after the
        kernel that wrote them would.  Eager calls between plain stream events
        when graphs cannot hold events."""
        S, torch = self.S, self.S.torch
        ea = (S.event(), S.event())
        g = None
        if self.graph is not None and S.in_graph_events:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=S.main):
                ea[0].record(S.main)
                for _ in range(reps):
                    call()
                ea[1].record(S.main)
        ts = []
        for i in range(n):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                if g is not None:
                    g.replay()
                else:
                    ea[0].record(S.main)
                    for _ in range(reps):
                        call()
                    ea[1].record(S.main)
            S.main.synchronize()
            ts.append(ea[0].elapsed_time(ea[1]) * 1e3 / reps)
        return ts

    def bank_alone_ms(self, layer_idx, bank, n):
        """One FFN call over `bank` of one layer after its routing, with events
        around the call inside a replayed graph; returns (ms list, distinct
        experts of that bank per step)."""
        S, moe, torch = self.S, self.S.moe, self.S.torch
        l = self.layers[layer_idx]
        b = self.steps[layer_idx].buf
        ea = (S.event(), S.event())
        T = self.T
        g = None
        if self.graph is not None and S.in_graph_events:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=S.main):
                moe.moe_route_split_count(self.ctx, l, b.logits, T, self.count_on, b.ids, b.w, b.ws_ptr, S.main)
                ea[0].record(S.main)
                moe.moe_expert_ffn_bank(self.ctx, l, bank, b.x, T, b.ws_ptr, b.Y, S.main)
                ea[1].record(S.main)
        ts = []
        for i in range(n):
            self.load_inputs(i, S.main)
            with torch.cuda.stream(S.main):
                S.flush.zero_()
                if g is not None:
                    g.replay()
                else:
                    moe.moe_route_split_count(self.ctx, l, b.logits, T, self.count_on, b.ids, b.w, b.ws_ptr, S.main)
                    ea[0].record(S.main)
                    moe.moe_expert_ffn_bank(self.ctx, l, bank, b.x, T, b.ws_ptr, b.Y, S.main)
                    ea[1].record(S.main)
            S.main.synchronize()
            ts.append(ea[0].elapsed_time(ea[1]))
        return ts


def pct(ms):
    return {q: float(np.percentile(ms, p)) * 1e3 for q, p in (("p10", 10), ("median", 50), ("p90", 90))}


def ffn_roofline(S, kernel, hot_experts, ms, eb, traffic_per_expert=None, timing=""):
    """HBM roofline of an FFN call that reads `hot_experts` distinct experts
    from the hot bank (mean over the timed calls)."""
    gbs = float(np.mean(hot_experts)) * eb / (float(np.mean(ms)) * 1e-3) / 1e9
    return {"kernel": kernel, "bound": "hbm", "achieved": gbs, "peak": S.hbm_peak, "unit": "GB/s",
            "frac": gbs / S.hbm_peak, "peak_source": f"{S.peak_src} (burst copy; 'of measured')",
            "traffic": (traffic_per_expert * float(np.mean(hot_experts)) if traffic_per_expert else None),
            "algorithmic_bytes": float(np.mean(hot_experts)) * eb, "us_per_launch": float(np.mean(ms)) * 1e3,
            "timing": timing}


# ------------------------------------------------------------- workloads

def measure_decode16(S, ctx, cfg, masks, args):
    """The 16-stream decode step over all four layers: the headline."""
    T = cfg.T
    run = StepRunner(S, ctx, cfg, range(cfg.L), T, max(2, min(args.pool, args.steps + args.warmup)),
                     cfg.count_on and T <= 256)
    run.capture()
    run.settle(args.warmup)
    step_ms, clocks = run.timed(args.steps, args.warmup)
    dh, dc, hp = zip(*[run.distinct(args.warmup + i, masks) for i in range(args.steps)])
    eb = S.moe.moe_expert_bytes(cfg.H, cfg.I)
    br = bytes_roofline(dh, dc, step_ms, eb, S.hbm_peak, S.link_gbs)
    nffn = min(args.steps, 20)
    ffn = run.ffn_in_step_ms(nffn, args.warmup)
    hbm_layer = next((l for l in range(cfg.L) if masks[l].all()), 0)
    split_layer = next((l for l in range(cfg.L) if not masks[l].all()), 0)
    hot_hbm = [run.distinct(args.warmup + i, masks)[0][hbm_layer] for i in range(nffn)]
    roof = ffn_roofline(S, f"FFN call over layer {hbm_layer} (all 384 experts in HBM), inside the step: "
                           "ffn_tc_decode_kernel<32,1,hot> + <32,2,hot> with prep_x / prep_h / round_y",
                        hot_hbm, ffn[hbm_layer], eb, profiled_traffic("decode16"),
                        "in-graph events around the layer's FFN call" if S.in_graph_events else "eager events")
    cold_split = [run.distinct(args.warmup + i, masks)[1][split_layer] for i in range(nffn)]
    hot_split = [run.distinct(args.warmup + i, masks)[0][split_layer] for i in range(nffn)]
    t_split = float(np.mean(ffn[split_layer])) * 1e-3
    link_gbs = float(np.mean(cold_split)) * eb / t_split / 1e9
    roof_link = {"kernel": f"FFN call over both banks of split layer {split_layer}, inside the step",
                 "bound": "host-link", "achieved": link_gbs, "peak": S.link_gbs, "unit": "GB/s",
                 "frac": link_gbs / S.link_gbs, "peak_source": "measured on this GPU by moe_probe_link",
                 "distinct_cold": float(np.mean(cold_split)), "distinct_hot": float(np.mean(hot_split)),
                 "frac_max": float(np.mean([max(h * eb / (S.hbm_peak * 1e9), c * eb / (S.link_gbs * 1e9))
                                            for h, c in zip(hot_split, cold_split)]) / t_split),
                 "us_per_launch": t_split * 1e6}
    e2e, h2d, d2h = run.e2e_ms(min(args.steps, 20))
    counter_ab = None
    if run.count_on and run.graph is not None:
        t_on = run.replay_graph_us(lambda: run.enqueue(count=True), min(args.steps, 10))
        t_off = run.replay_graph_us(lambda: run.enqueue(count=False), min(args.steps, 10))
        counter_ab = {"step_on_us": float(np.median(t_on)), "step_off_us": float(np.median(t_off)),
                      "note": "whole step graph-replayed with the usage count on and off, same inputs"}
    out = {
        "step_ms": step_ms, "clocks": clocks, "bytes_roofline": br, "roofline": roof, "roofline_link": roof_link,
        "ffn_in_step_us": {str(l): float(np.mean(v)) * 1e3 for l, v in ffn.items()},
        "e2e_ms": e2e, "h2d": h2d, "d2h": d2h, "launches_per_step": run.launches_per_step,
        "graph": run.graph is not None, "counter_ab": counter_ab,
    }
    del run
    return out


def measure_decode1(S, ctx, cfg, masks, args, layer=0, want_breakdown=True):
    """The one-user decode step on context layer `layer` (7 tokens)."""
    T = cfg.T
    run = StepRunner(S, ctx, cfg, [layer], T, max(2, min(32, args.steps + args.warmup)), cfg.count_on,
                     input_layers=[0])
    run.capture()
    run.settle(args.warmup)
    step_ms, clocks = run.timed(args.steps, args.warmup)
    m = {layer: masks[layer]}
    dist = [run.distinct(args.warmup + i, m) for i in range(args.steps)]
    dh = [d[0] for d in dist]
    dc = [d[1] for d in dist]
    eb = S.moe.moe_expert_bytes(cfg.H, cfg.I)
    br = bytes_roofline(dh, dc, step_ms, eb, S.hbm_peak, S.link_gbs)
    n = min(args.steps, 20)
    hot_ms = run.bank_alone_ms(0, S.moe.MOE_BANK_HOT, n)
    hot_exp = [run.distinct(i, m)[0][0] for i in range(n)]
    roof = ffn_roofline(S, "hot-bank expert FFN call alone after routing (ffn_tc_decode_kernel<8,1,hot> + <8,2,hot>)",
                        hot_exp, hot_ms, eb, profiled_traffic("decode1"),
                        "in-graph events, hot-bank call alone after routing")
    out = {"step_ms": step_ms, "clocks": clocks, "bytes_roofline": br, "roofline": roof,
           "launches_per_step": run.launches_per_step}
    if want_breakdown and run.graph is not None:
        b = run.steps[0].buf
        moe = S.moe
        route_us = run.call_alone_us(lambda: moe.moe_route_split_count(
            ctx, layer, b.logits, T, run.count_on, b.ids, b.w, b.ws_ptr, S.main), n)
        wr = S.torch.from_numpy(synth.router_weights(cfg, 0).view(np.int16)).to(S.dev)
        bias = S.torch.from_numpy(synth.router_bias(cfg, 0)).to(S.dev)
        lo = S.torch.empty((T, cfg.E), dtype=S.torch.float32, device=S.dev)
        router_us = run.call_alone_us(lambda: moe.moe_router_logits(ctx, b.x, wr, bias, T, cfg.E, cfg.H, lo, S.main), n)
        route_rep = run.call_repeated_us(lambda: moe.moe_route_split_count(
            ctx, layer, b.logits, T, run.count_on, b.ids, b.w, b.ws_ptr, S.main), 32, 5)
        router_rep = run.call_repeated_us(
            lambda: moe.moe_router_logits(ctx, b.x, wr, bias, T, cfg.E, cfg.H, lo, S.main), 32, 5)
        cold_ms = run.bank_alone_ms(0, moe.MOE_BANK_COLD, n)
        out["breakdown"] = {"route_us": float(np.mean(route_us)), "router_gemm_us": float(np.mean(router_us)),
                            "hot_alone_us": float(np.mean(hot_ms)) * 1e3, "cold_alone_us": float(np.mean(cold_ms)) * 1e3,
                            "note": "in-graph events after an L2 flush: the routing call alone, the router GEMM "
                                    "(hidden states -> logits, outside the step) alone, each bank's FFN call "
                                    "alone after routing",
                            "back_to_back": {
                                "route_us": float(np.median(route_rep)),
                                "router_gemm_us": float(np.median(router_rep)),
                                "note": "per call of 32 calls back to back in one replayed graph after an L2 flush "
                                        "(median of 5): inputs come from L2 after the first call, as right after "
                                        "the kernel that wrote them, and one event pair spans all 32"}}
        if run.count_on:
            t_on = run.replay_graph_us(lambda: run.enqueue(count=True), n)
            t_off = run.replay_graph_us(lambda: run.enqueue(count=False), n)
            out["breakdown"]["counter_ab"] = {"step_on_us": float(np.median(t_on)), "step_off_us": float(np.median(t_off))}
    e2e, h2d, d2h = run.e2e_ms(min(args.steps, 20))
    out.update(e2e_ms=e2e, h2d=h2d, d2h=d2h)
    return out


def measure_adaptive(S, ctx, n_layers, acfg, args, layer=0):
    """128 one-user steps on context layer `layer` with the domain shift: the
    policy reads the counts every 16 steps and its swaps go in between steps,
    at most 8 per step.  Times every step (graph replay after an L2 flush)
    and every swap batch (events around moe_swap_rows on the launching
    stream)."""
    torch, moe = S.torch, S.moe
    ex = acfg.extra
    T = acfg.T
    run = StepRunner(S, ctx, acfg, [layer], T, 1, True, input_layers=[0])
    run.capture()
    run.settle(3)
    counts0 = moe.moe_read_counts(ctx, n_layers, acfg.E)[layer]
    pol = moe.moe_policy(acfg.E, read_every=ex["read_every"], half_life=ex["half_life"],
                         hysteresis=ex["hysteresis"], min_avg=ex["min_avg"], max_pairs=ex["max_per_read"],
                         counts_now=counts0)
    step_us, swap_us, swaps, queue = [], [], 0, []
    cold_picks = []
    b = run.steps[0].buf
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sw0, sw1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(S.local)
    clk.__enter__()
    clk.wait_first()
    try:
        for s in range(acfg.steps):
            lg = synth.router_logits(acfg, 0, s)
            x = synth.activations(acfg, 0, s)
            rm = moe.moe_get_rowmap(ctx, layer, acfg.E)
            ids = np.argsort(-lg, axis=1, kind="stable")[:, :acfg.k]
            cold_picks.append(int((rm[ids] < 0).sum()))
            with torch.cuda.stream(S.main):
                b.logits[:T].copy_(torch.from_numpy(lg).pin_memory(), non_blocking=True)
                b.x[:T].copy_(torch.from_numpy(x.view(np.int16)).pin_memory(), non_blocking=True)
                S.flush.zero_()
                ev0.record(S.main)
                run.run_step()
                ev1.record(S.main)
            S.main.synchronize()
            step_us.append(ev0.elapsed_time(ev1) * 1e3)
            if (s + 1) % ex["read_every"] == 0:
                counts = moe.moe_read_counts(ctx, n_layers, acfg.E, S.main)[layer]
                pro, dem = pol.read(counts, moe.moe_get_rowmap(ctx, layer, acfg.E))
                queue.extend(zip(pro.tolist(), dem.tolist()))
            if queue:   # between this step and the next: at most max_per_step swaps
                batch, queue = queue[:ex["max_per_step"]], queue[ex["max_per_step"]:]
                with torch.cuda.stream(S.main):
                    sw0.record(S.main)
                    n, _ = moe.moe_swap_rows(ctx, layer, [p for p, _ in batch], [d for _, d in batch], S.main)
                    sw1.record(S.main)
                S.main.synchronize()
                if n:
                    swap_us.append(sw0.elapsed_time(sw1) * 1e3 / n)
                    swaps += n
    finally:
        clk.__exit__(None, None, None)
    sa = acfg.shift_at
    return {
        "workload": WORKLOADS["adaptive"], "tokens_per_step": T, "steps": acfg.steps,
        "step_us_mean": float(np.mean(step_us)),
        "step_us_before_shift": float(np.mean(step_us[16:sa])),
        "step_us_after_shift_first16": float(np.mean(step_us[sa:sa + 16])),
        "step_us_last16": float(np.mean(step_us[-16:])),
        "cold_picks_before_shift": float(np.mean(cold_picks[16:sa])),
        "cold_picks_after_shift_first16": float(np.mean(cold_picks[sa:sa + 16])),
        "cold_picks_last16": float(np.mean(cold_picks[-16:])),
        "swaps_applied": swaps, "us_per_swap": float(np.mean(swap_us)) if swap_us else None,
        "swap_batches": len(swap_us),
        "swap_note": "a swap = hot row -> HBM staging, cold row -> hot slot, staging -> cold slot (three copies "
                     "of 18.8 MB, two over the host link) and the 2-element row-map write, on the step stream",
        "policy": {k: ex[k] for k in ("read_every", "half_life", "hysteresis", "min_avg", "max_per_read",
                                      "max_per_step")},
        "timing": "each step graph-replayed after an L2 flush, events around it; swaps between steps",
        "clocks": clk.summary(),
    }


def measure_prefill(S, ctx, pcfg, args, layer, fmt=0):
    """The 8192-token prefill chunk on context layer `layer` (all experts in
    HBM), with the token rows as two e4m3 pieces (fmt 0, the default) or in
    the MXFP8 format (fmt 1: one MMA per product)."""
    T = pcfg.T
    steps = max(3, min(args.steps, 20))
    S.moe.moe_set_act_format(ctx, fmt)
    try:
        run = StepRunner(S, ctx, pcfg, [layer], T, 2, False, input_layers=[0])
        run.capture()
        run.settle(max(3, min(args.warmup, 5)))
        step_ms, clocks = run.timed(steps, 0)
        ffn = run.ffn_in_step_ms(min(steps, 10))[layer]
    finally:
        S.moe.moe_set_act_format(ctx, 0)
    eb = S.moe.moe_expert_bytes(pcfg.H, pcfg.I)
    picks = T * pcfg.k
    flops = picks * 2.0 * 3.0 * pcfg.I * pcfg.H
    tf = flops / (float(np.mean(ffn)) * 1e-3) / 1e12
    if fmt == 0:
        peak, src = S.tf_burst, (f"{S.peak_src} bf16 dense burst ('of measured'): rows carry bf16-class precision "
                                 "as two e4m3 pieces, two fp8-rate MMAs per product = the bf16 rate")
        kern = f"ffn_tc_kernel<{kPrefillTile},1,hot,false> + <{kPrefillTile},2,hot,false> with prep_x, prep_h"
    else:
        peak, src = 2.0 * S.tf_burst, (f"{S.peak_src} bf16 dense burst x 2 (the nominal fp8 : bf16 dense ratio, "
                                       "4.5 : 2.25 PFLOP/s; 'of measured'): one fp8-rate MMA per product")
        kern = (f"ffn_tc_kernel<{kPrefillTileMx},1,hot,true> + <{kPrefillTileMx},2,hot,true> with tile_scan, "
                "prep_x_mx8, prep_h_mx8")
    # DRAM bytes of the FFN call (prep kernels and both GEMMs), captured on the
    # 64-expert profiling case (about 128 picks per expert, as here) and scaled
    # by the routed picks: weights and token rows both grow with them
    per_pick = profiled_traffic("prefill_mxfp8" if fmt else "prefill", "bytes_per_pick")
    traffic = per_pick * picks if per_pick is not None else None
    traffic_src = ("ncu dram__bytes_read.sum + dram__bytes_write.sum of the FFN call's launches on the 64-expert "
                   f"profiling case, per routed pick x {picks} picks") if per_pick is not None else None
    return {
        "workload": WORKLOADS["prefill"], "tokens_per_step": T, "steps": steps,
        "activations": "two e4m3 pieces per value (bf16-class)" if fmt == 0 else "MXFP8 (e4m3, e8m0 per 32)",
        "us_per_layer_step": float(np.mean(step_ms)) * 1e3, "tokens_per_s": T / (float(np.mean(step_ms)) * 1e-3),
        "step_us_pct": pct(step_ms),
        "roofline": {"kernel": f"FFN call inside the step ({kern})", "bound": "tensor", "achieved": tf, "peak": peak,
                     "unit": "TFLOP/s", "frac": tf / peak, "flops_per_launch": flops, "peak_source": src,
                     "hbm_gbs_achieved": pcfg.E * eb / (float(np.mean(ffn)) * 1e-3) / 1e9,
                     "traffic": traffic, "traffic_source": traffic_src, "us_per_launch": float(np.mean(ffn)) * 1e3},
        "clocks": clocks, "launches_per_step": run.launches_per_step,
    }


def measure_prefill_shift(S, ctx, args, layer=0, slots=16):
    """An 8192-token prefill chunk on split context layer `layer` (295 hot /
    89 cold by the first ranking) right after the domain shift: the logits
    follow the redrawn ranking, so the new domain's popular experts are
    still cold and draw several 144-token tiles each.  Timed with the cold
    staging pool off and on (`slots` rows)."""
    acfg = synth.get_config("adaptive")
    scfg = dataclasses.replace(acfg, name="prefill_shift", T=8192, shift_at=0, steps=1)
    T, eb = scfg.T, S.moe.moe_expert_bytes(scfg.H, scfg.I)
    mask = synth.hot_mask(acfg, 0)
    out = {"workload": "prefill chunk right after a domain shift: 8192 tokens on a split layer (295 hot / 89 cold by "
                       "the first ranking), logits from the redrawn ranking (Spearman 0.15), top-6, Zipf(1.1) skew",
           "tokens_per_step": T}
    for mode, n_slots in (("unstaged", 0), ("staged", slots)):
        S.moe.moe_set_cold_staging(ctx, n_slots)
        try:
            steps = max(3, min(args.steps, 8))
            run = StepRunner(S, ctx, scfg, [layer], T, 2, False, input_layers=[0])
            run.capture()
            run.settle(3)
            step_ms, clocks = run.timed(steps, 0)
            rows = S.moe.moe_read_stage(ctx, run.steps[0].buf.ws_ptr, T) if n_slots else None
        finally:
            S.moe.moe_set_cold_staging(ctx, 0)
        out[mode] = {"us_per_layer_step": float(np.mean(step_ms)) * 1e3, "step_us_pct": pct(step_ms),
                     "tokens_per_s": T / (float(np.mean(step_ms)) * 1e-3), "clocks": clocks}
        if rows is not None:
            out[mode]["staged_experts"] = int((rows >= 0).sum())
    # host-link reads per step: one per cold (expert, token tile) unstaged; one
    # per distinct cold expert when every multi-tile expert is staged
    ids = np.argsort(-run.pool_lg[0][0], axis=1, kind="stable")[:, :scfg.k]
    u, n = np.unique(ids, return_counts=True)
    cold = mask[u] == 0
    tiles = np.ceil(n[cold] / kPrefillTile)
    multi = np.sort(n[cold][tiles > 1])[::-1][:slots]
    saved = float(np.sum(np.ceil(multi / kPrefillTile) - 1))
    out["cold_tiles_unstaged"] = int(tiles.sum())
    out["cold_link_bytes_unstaged"] = float(tiles.sum() * eb)
    out["cold_link_bytes_staged"] = float((tiles.sum() - saved) * eb)
    out["link_gbs"] = S.link_gbs
    out["speedup"] = out["unstaged"]["us_per_layer_step"] / out["staged"]["us_per_layer_step"]
    out["note"] = ("staged: the FFN call first copies each cold expert with more picks than one token tile into an "
                   "HBM pool (once per step) and its units read it there; rows bit-identical to unstaged")
    return out


# Token rows per tile of the prefill FFN on steps of more than 256 tokens:
# two-piece rows (the default format), MXFP8 rows.  The library's own widths;
# the link-byte accounting of the shifted prefill chunk counts tiles with them.
kPrefillTile = 144
kPrefillTileMx = 160


def line_for(S, name, cfg, m, args, cpu):
    """The JSON line of a decode workload measured by measure_decode16/1."""
    world = S.world
    total_ms = slowest_rank_ms(sum(m["step_ms"]), S.dist, S.dev)
    e2e_total = slowest_rank_ms(sum(m["e2e_ms"]), S.dist, S.dev)
    L = cfg.L
    return {
        "metric": METRIC, "value": job_tokens_per_s(world, cfg.T, len(m["step_ms"]), total_ms), "unit": "tokens/s",
        "n_gpus": world, "steps": len(m["step_ms"]), "warmup": args.warmup,
        "ms_per_step": total_ms / len(m["step_ms"]), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1 weights (e8m0 scales) x e4m3 rows (two pieces), block-scaled tensor cores, f32 accumulate, bf16 rows",
        "data": "synthetic (seeded SplitMix64; Zipf-skewed routing)",
        "config": {"workload": WORKLOADS[name] + (f" [profiling variant: {cfg.E} experts, {cfg.n_hot} hot, {cfg.T} tokens]"
                                                  if (args.experts or args.tokens) else ""),
                   "layers": L, "tokens_per_step": cfg.T,
                   "l2": "flushed (512 MiB write) before every timed step", "cuda_graph": m["graph"] if "graph" in m else True,
                   "ffn_calls": "one call over both banks" if args.banks == "fused" else "hot and cold bank calls on two streams",
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "us_per_layer_step": total_ms / len(m["step_ms"]) * 1e3 / L,
        "step_us_pct": pct(m["step_ms"]),
        "bytes_roofline": dict(m["bytes_roofline"], expert_bytes=S.moe.moe_expert_bytes(cfg.H, cfg.I),
                               hbm_gbs=S.hbm_peak, hbm_peak_source=S.peak_src, link_gbs=S.link_gbs,
                               hbm_probe_gbs=S.hbm_probe_gbs),
        "roofline": m["roofline"],
        "cpu_baseline": cpu,
        "e2e": {"value": job_tokens_per_s(world, cfg.T, len(m["e2e_ms"]), e2e_total), "unit": "tokens/s",
                "h2d_bytes_per_step": m["h2d"], "d2h_bytes_per_step": m["d2h"],
                "path": "moe_layer_step_host per layer: pinned host inputs copied in, route, both banks' FFN, finalize, output rows copied back, all in the C ABI call"},
        "gpu_launches": m["launches_per_step"] * len(m["step_ms"]),
        "clocks": m["clocks"],
    }


def cpu_baseline(S, cfg, weights, args, T=None):
    if S.rank != 0 or not weights:
        return None
    layers = sorted(weights)
    T = T or (cfg.T if cfg.T <= 256 else 64)
    pool = oracle_pool(cfg, layers, 64, T)
    tps, done, used, cores = cpu_oracle_steps(cfg, weights, pool, args.cpu_budget)
    return {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} whole layer-steps of {T} tokens (layers {layers} of this workload), {used:.1f} s; "
                      f"a {cfg.L}-layer step of {cfg.T} tokens counts as {cfg.L} layer-steps"}


def run_all(S, args):
    """One context with the 16-stream decode's four layers; every workload."""
    cfg = bench_config(args, "decode16")
    masks = [synth.hot_mask(cfg, l) for l in range(cfg.L)]
    skip = set(filter(None, args.skip.split(",")))
    ctx, keep = S.place(cfg, synth.get_config("prefill").T if "prefill" not in skip else cfg.T, masks)
    try:
        m16 = measure_decode16(S, ctx, cfg, masks, args)
        cpu = cpu_baseline(S, cfg, keep, args)
        line = line_for(S, "decode16", cfg, m16, args, cpu)
        line["roofline_link"] = m16["roofline_link"]
        line["ffn_in_step_us"] = m16["ffn_in_step_us"]
        if m16["counter_ab"]:
            line["counter_ab"] = m16["counter_ab"]
        subs = {}
        if "decode1" not in skip:
            c1 = dataclasses.replace(bench_config(args, "decode1"), E=cfg.E, n_hot=cfg.n_hot)
            m1 = measure_decode1(S, ctx, c1, masks, args, layer=0)
            t1 = slowest_rank_ms(sum(m1["step_ms"]), S.dist, S.dev)
            subs["decode1"] = {
                "workload": WORKLOADS["decode1"] + " (layer 0 of this context: the same weights and placement)",
                "value": job_tokens_per_s(S.world, c1.T, len(m1["step_ms"]), t1), "unit": "tokens/s",
                "us_per_layer_step": t1 / len(m1["step_ms"]) * 1e3, "step_us_pct": pct(m1["step_ms"]),
                "bytes_roofline": m1["bytes_roofline"], "roofline": m1["roofline"],
                "breakdown": m1.get("breakdown"),
                "e2e": {"value": job_tokens_per_s(S.world, c1.T, len(m1["e2e_ms"]),
                                                  slowest_rank_ms(sum(m1["e2e_ms"]), S.dist, S.dev)),
                        "unit": "tokens/s", "h2d_bytes_per_step": m1["h2d"], "d2h_bytes_per_step": m1["d2h"]},
                "clocks": m1["clocks"]}
        if "prefill_shift" not in skip:   # before the adaptive run moves layer 0's rows
            subs["prefill_shift"] = measure_prefill_shift(S, ctx, args, layer=0)
        if "adaptive" not in skip:
            acfg = synth.get_config("adaptive")
            subs["adaptive"] = measure_adaptive(S, ctx, cfg.L, acfg, args, layer=0)
        if "prefill" not in skip:
            pcfg = synth.get_config("prefill")
            hbm_layer = next(l for l in range(cfg.L) if masks[l].all())
            p = measure_prefill(S, ctx, pcfg, args, hbm_layer)
            p["workload"] += f" (layer {hbm_layer} of this context)"
            p["mxfp8"] = measure_prefill(S, ctx, pcfg, args, hbm_layer, fmt=1)
            p["mxfp8"].pop("workload")
            subs["prefill"] = p
        line["configs"] = subs
    finally:
        S.moe.moe_destroy(ctx)
    return line


def run_single(S, args):
    name = args.config
    cfg = bench_config(args)
    masks = [synth.hot_mask(cfg, l) for l in range(cfg.L)]
    ctx, keep = S.place(cfg, cfg.T, masks)
    try:
        if name == "decode16":
            m = measure_decode16(S, ctx, cfg, masks, args)
            line = line_for(S, name, cfg, m, args, cpu_baseline(S, cfg, keep, args))
            line["roofline_link"] = m["roofline_link"]
            line["ffn_in_step_us"] = m["ffn_in_step_us"]
        elif name == "decode1":
            m = measure_decode1(S, ctx, cfg, masks, args)
            m["graph"] = not args.no_graph
            line = line_for(S, name, cfg, m, args, cpu_baseline(S, cfg, keep, args))
            line["breakdown"] = m.get("breakdown")
        elif name == "adaptive":
            a = measure_adaptive(S, ctx, cfg.L, cfg, args)
            line = {"metric": METRIC, "value": a["tokens_per_step"] / (a["step_us_mean"] * 1e-6), "unit": "tokens/s",
                    "n_gpus": S.world, "steps": a["steps"], "warmup": 3, "ms_per_step": a["step_us_mean"] * 1e-3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "config": {"workload": WORKLOADS[name]}, "adaptive": a, "clocks": a["clocks"],
                    "cpu_baseline": cpu_baseline(S, cfg, keep, args)}
        else:
            p = measure_prefill(S, ctx, cfg, args, 0, fmt=1 if args.act == "mxfp8" else 0)
            line = {"metric": METRIC, "value": p["tokens_per_s"], "unit": "tokens/s", "n_gpus": S.world,
                    "steps": p["steps"], "warmup": 3, "ms_per_step": p["us_per_layer_step"] * 1e-3,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                    "config": {"workload": WORKLOADS[name] + (f" [profiling variant: {cfg.E} experts, {cfg.T} tokens]"
                                                              if (args.experts or args.tokens) else "")},
                    "roofline": p["roofline"], "clocks": p["clocks"],
                    "gpu_launches": p["launches_per_step"] * p["steps"],
                    "cpu_baseline": cpu_baseline(S, cfg, keep, args, T=64)}
    finally:
        S.moe.moe_destroy(ctx)
    return line


def main(argv=None):
    args = parse(argv)
    if args.impl == "reference":
        return run_reference(args)
    S = Session(args)
    line = run_all(S, args) if args.config == "all" else run_single(S, args)
    if S.rank == 0:
        print(json.dumps(line), flush=True)
    if S.dist:
        S.dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
