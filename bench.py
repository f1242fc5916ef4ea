#!/usr/bin/env python
"""Benchmark of the split-residency MoE layer-step on GB300.

One step = one layer-step of the whole hot path over one batch of synthetic
inputs: route + split + count, the hot-bank and cold-bank MXFP4 expert FFN
(one call over both banks; ``--banks streams``: two calls on two streams),
and the finalize.  Default workload: the one-user decode step
(1 layer, 384 experts, top-6, H=4096, I=2880, 7 tokens, Zipf-skewed routing,
295 experts in HBM and 89 in pinned host memory).

Prints one JSON line.  ``value`` = tokens/s of the whole job with inputs
resident in HBM (each step CUDA-graph replayed, timed with CUDA events on the
launching stream, L2 flushed between steps); ``e2e`` = the same metric with
the inputs copied from pinned host memory and the output copied back inside
the timed region.  ``bytes_roofline`` = the metric's fraction of the bytes
roofline: distinct hot experts' bytes / HBM peak + distinct cold experts'
bytes / measured host-link bandwidth, over the measured step time.

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
                "112 tokens",
    "prefill": "prefill chunk, 1 MoE layer, 384 experts all in HBM, top-6, 8192 tokens, near-uniform routing",
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="decode1", choices=sorted(WORKLOADS))
    ap.add_argument("--pool", type=int, default=32, help="distinct input batches cycled through")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--banks", default="fused", choices=["streams", "fused"],
                    help="the two banks' FFN calls on two streams at once, or one call over both banks")
    ap.add_argument("--cpu-budget", type=float, default=20.0, help="seconds of CPU-oracle work")
    ap.add_argument("--experts", type=int, default=0,
                    help="profiling-size variant: this many experts per layer (same expert geometry)")
    ap.add_argument("--hot", type=int, default=0, help="hot-bank experts for --experts")
    ap.add_argument("--tokens", type=int, default=0, help="profiling-size variant: tokens per step")
    return ap.parse_args()


def bench_config(args):
    """The workload of a run: the named config, optionally narrowed to fewer
    experts (``--experts``/``--hot``) or another token count (``--tokens``).
    Both arms use it."""
    cfg = synth.get_config(args.config)
    if args.experts:
        cfg = synth.get_config(args.config, E=args.experts, n_hot=args.hot or cfg.n_hot * args.experts // cfg.E)
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


def cpu_oracle_steps(cfg, weights, mask, pool_lg, pool_x, budget_s):
    """Time the CPU oracle on whole layer-steps until the budget is spent."""
    import oracle
    t_used, steps, tokens = 0.0, 0, 0
    while t_used < budget_s and steps < len(pool_lg):
        lg, x = pool_lg[steps], pool_x[steps]
        t0 = time.perf_counter()
        oracle.layer_step(weights, lg, x, cfg.k)
        t_used += time.perf_counter() - t0
        steps += 1
        tokens += lg.shape[0]
    return tokens / t_used, steps, t_used, oracle.num_threads()


def single_core_oracle(cfg, weights, mask, pool_lg, pool_x, budget_s):
    """The same oracle layer-steps on one host thread, at least one whole
    step (decode-sized workloads only; prefill needs every core).  Returns
    the cpu_baseline sub-entry."""
    import oracle
    if pool_lg[0].shape[0] > 256:
        return None
    cores = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        tps, n, used, _ = cpu_oracle_steps(cfg, weights, mask, pool_lg, pool_x, budget_s)
    finally:
        oracle.set_num_threads(cores)
    return {"value": tps, "unit": "tokens/s", "cores": 1, "sample": f"{n} whole layer-steps, {used:.1f} s"}


def make_pool(cfg, n, layers):
    lg = [[synth.router_logits(cfg, l, s) for l in range(layers)] for s in range(n)]
    xs = [[synth.activations(cfg, l, s) for l in range(layers)] for s in range(n)]
    return lg, xs


def source_sha():
    """Hash of the FFN kernels' sources (a stored profile is used only while
    they are unchanged)."""
    h = hashlib.sha256()
    for name in ("ffn_tc.cu", "ffn_tc_decode.cuh"):
        with open(os.path.join(ROOT, "cold_expert_residency_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic(config):
    """DRAM bytes per launch of the hot-bank FFN from a committed ncu summary,
    if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d.get(config)
        if e and e.get("source_sha") == source_sha():
            return e.get("bytes_per_hot_expert")
    except Exception:
        pass
    return None


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import oracle
    cfg = bench_config(args)
    if cfg.L != 1:
        cfg = dataclasses.replace(cfg, L=1)
    weights = synth.layer_weights(cfg, 0)
    mask = synth.hot_mask(cfg, 0)
    n = max(1, min(args.steps + args.warmup, 64))
    T = cfg.T if args.config != "prefill" else 64
    lg = [synth.router_logits(cfg, 0, s, T=T) for s in range(n)]
    xs = [synth.activations(cfg, 0, s, T=T) for s in range(n)]
    budget = min(120.0, max(10.0, args.cpu_budget))
    tps, steps, used, cores = cpu_oracle_steps(cfg, weights, mask, lg, xs, budget)
    sample = f"{steps} whole layer-steps of {T} tokens ({args.config} geometry), {used:.1f} s"
    line = {
        "impl": "reference", "metric": METRIC, "value": tps, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": 0, "ms_per_step": used / steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": WORKLOADS[args.config] + ("" if T == cfg.T else f"; sampled at {T} tokens")},
        "cpu_baseline": {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
                         "single_core": single_core_oracle(cfg, weights, mask, lg, xs, max(1.0, budget / 4))},
        "e2e": {"value": tps, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import cold_expert_residency_gb300 as moe
    from cold_expert_residency_gb300.runtime import LayerStep

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    moe.build()

    cfg = bench_config(args)
    hbm_peak, tf_burst, tf_sust, peak_src = load_peaks()
    L = cfg.L
    ctx = moe.moe_create(L, cfg.E, cfg.k, cfg.H, cfg.I, cfg.T, device=local)
    masks, weights0 = [], None
    for l in range(L):
        w = synth.layer_weights(cfg, l)
        m = synth.hot_mask(cfg, l)
        moe.moe_init_banks(ctx, l, *w, m)
        masks.append(m)
        if l == 0:
            weights0 = w
        else:
            del w
    link_gbs, hbm_probe_gbs = moe.moe_probe_link(ctx, 1 << 30, 5)

    T, E, k, H = cfg.T, cfg.E, cfg.k, cfg.H
    npool = max(2, min(args.pool, args.steps + args.warmup))
    if T > 256:
        npool = min(npool, 4)     # large batches: a few distinct inputs suffice
    pool_lg, pool_x = make_pool(cfg, npool, L)
    dev = torch.device("cuda", local)
    d_lg = torch.stack([torch.from_numpy(np.stack(p)) for p in pool_lg]).to(dev)            # [n][L][T][E]
    d_x = torch.stack([torch.from_numpy(np.stack(p).view(np.int16)) for p in pool_x]).to(dev)  # [n][L][T][H]
    h_lg = d_lg.cpu().pin_memory()
    h_x = d_x.cpu().pin_memory()
    h_out = torch.zeros((L, T, H), dtype=torch.int16).pin_memory()

    steps = [LayerStep(ctx, E, k, H, T, device=dev) for _ in range(L)]
    main = torch.cuda.Stream(device=dev)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    count_on = cfg.count_on and T <= 256

    use_graph = not args.no_graph
    try:   # external events become timing nodes inside a captured graph
        ev_hot = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)]
        in_graph_events = True
    except TypeError:
        ev_hot = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        in_graph_events = False

    def enqueue(timed_hot=False, count=None):
        cnt = count_on if count is None else count
        for l in range(L):
            st = steps[l]
            b = st.buf
            moe.moe_route_split_count(ctx, l, b.logits, T, cnt, b.ids, b.w, b.ws_ptr, main)
            if timed_hot and l == 0:
                ev_hot[0].record(main)
            if args.banks == "fused":   # both banks' FFN, one launch per GEMM
                moe.moe_expert_ffn_bank(ctx, l, moe.MOE_BANK_BOTH, b.x, T, b.ws_ptr, b.Y, main)
            else:                       # the two banks' calls on two streams at once
                st.ev_routed.record(main)
                st.cold_stream.wait_event(st.ev_routed)
                moe.moe_expert_ffn_bank(ctx, l, moe.MOE_BANK_COLD, b.x, T, b.ws_ptr, b.Y, st.cold_stream)
                st.ev_cold.record(st.cold_stream)
                moe.moe_expert_ffn_bank(ctx, l, moe.MOE_BANK_HOT, b.x, T, b.ws_ptr, b.Y, main)
                main.wait_event(st.ev_cold)
            if timed_hot and l == 0:
                ev_hot[1].record(main)
            moe.moe_finalize(b.Y, b.w, T, k, H, b.out, main)

    def load_inputs(i, stream):
        with torch.cuda.stream(stream):
            for l in range(L):
                steps[l].buf.logits[:T].copy_(d_lg[i % npool, l], non_blocking=True)
                steps[l].buf.x[:T].copy_(d_x[i % npool, l], non_blocking=True)

    # one eager step (also counts this library's launches per step)
    load_inputs(0, main)
    n0 = moe.moe_kernel_launches()
    with torch.cuda.stream(main):
        enqueue()
    main.synchronize()
    launches_per_step = moe.moe_kernel_launches() - n0
    graph = None
    hot_timing = "in-graph events" if use_graph else "eager events"
    if use_graph:
        graph = torch.cuda.CUDAGraph()
        if not in_graph_events:
            hot_timing = "eager pass (no external events)"
        try:
            with torch.cuda.graph(graph, stream=main):
                enqueue(timed_hot=in_graph_events)
        except Exception as ex:   # event record nodes unavailable: time the hot FFN eagerly
            hot_timing = f"eager pass ({type(ex).__name__})"
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=main):
                enqueue(timed_hot=False)

    def run_step():
        if graph is not None:
            graph.replay()
        else:
            with torch.cuda.stream(main):
                enqueue(timed_hot=True)

    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # steady state: every pooled input batch once, untimed, so each expert a
    # timed step routes to has been read before (the first read of a weight
    # page sets up its address translation and runs far slower); every timed
    # step still computes everything, after an L2 flush
    for i in range(npool):
        load_inputs(i, main)
        with torch.cuda.stream(main):
            run_step()
    main.synchronize()
    for i in range(args.warmup):
        load_inputs(i, main)
        with torch.cuda.stream(main):
            flush.zero_()
        with torch.cuda.stream(main):
            run_step()
    main.synchronize()

    step_ms, hot_ms, hot_bytes, cold_bytes, dh, dc, hot_picks = [], [], [], [], [], [], []
    eb = moe.moe_expert_bytes(cfg.H, cfg.I)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev_steps = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        clk.wait_first()
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        # every timed step is enqueued back to back and the host synchronizes
        # once, so a host-side stall cannot open a gap inside a step's events
        for i in range(args.steps):
            j = args.warmup + i
            load_inputs(j, main)
            with torch.cuda.stream(main):
                flush.zero_()
                ev_steps[i][0].record(main)
                run_step()
                ev_steps[i][1].record(main)
        main.synchronize()
    for i in range(args.steps):
        j = args.warmup + i
        step_ms.append(ev_steps[i][0].elapsed_time(ev_steps[i][1]))
        nh = nc = 0
        for l in range(L):
            lg = pool_lg[j % npool][l]
            ids = np.argsort(-lg, axis=1, kind="stable")[:, :k]
            a, c = distinct_experts(ids, masks[l])
            nh += a
            nc += c
            if l == 0:
                hot_bytes.append(a * eb)
                hot_picks.append(int((masks[l][ids] == 1).sum()))
        dh.append(nh)
        dc.append(nc)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    total_ms = slowest_rank_ms(sum(step_ms), dist, dev)

    # the step's FFN call (layer 0), one step at a time
    if hot_timing in ("in-graph events", "eager events"):
        for i in range(min(args.steps, 20)):
            load_inputs(args.warmup + i, main)
            with torch.cuda.stream(main):
                flush.zero_()
                run_step()
            main.synchronize()
            hot_ms.append(ev_hot[0].elapsed_time(ev_hot[1]))
    if not hot_ms:   # eager timing of the FFN call
        for i in range(min(args.steps, 20)):
            load_inputs(i, main)
            with torch.cuda.stream(main):
                flush.zero_()
                enqueue(timed_hot=True)
            main.synchronize()
            hot_ms.append(ev_hot[0].elapsed_time(ev_hot[1]))
    ffn_ms = hot_ms   # layer 0's FFN call over both banks, inside the step

    def ffn_alone(bank):
        """One FFN call over `bank` of layer 0 after routing, graph-replayed with
        events around the call (in the graph when possible); returns the
        times (ms) and the inputs' distinct hot-expert bytes."""
        st = steps[0]
        b = st.buf
        ea = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(2)] if in_graph_events else ev_hot
        g2 = None
        if use_graph and in_graph_events:
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=main):
                moe.moe_route_split_count(ctx, 0, b.logits, T, count_on, b.ids, b.w, b.ws_ptr, main)
                ea[0].record(main)
                moe.moe_expert_ffn_bank(ctx, 0, bank, b.x, T, b.ws_ptr, b.Y, main)
                ea[1].record(main)
        ts, by = [], []
        for i in range(min(args.steps, 20)):
            load_inputs(i, main)
            with torch.cuda.stream(main):
                flush.zero_()
                if g2 is not None:
                    g2.replay()
                else:
                    moe.moe_route_split_count(ctx, 0, b.logits, T, count_on, b.ids, b.w, b.ws_ptr, main)
                    ea[0].record(main)
                    moe.moe_expert_ffn_bank(ctx, 0, bank, b.x, T, b.ws_ptr, b.Y, main)
                    ea[1].record(main)
            main.synchronize()
            ts.append(ea[0].elapsed_time(ea[1]))
            ids = np.argsort(-pool_lg[i % npool][0], axis=1, kind="stable")[:, :k]
            by.append(distinct_experts(ids, masks[0])[0] * eb)
        return ts, by

    # the roofline's kernel: the hot-bank FFN call on its own (inside the step
    # it shares its launches with the cold bank)
    hot_ms, hot_bytes_alone = ffn_alone(moe.MOE_BANK_HOT)
    hot_timing = ("in-graph events" if (use_graph and in_graph_events) else "eager events") + \
        ", hot-bank call alone after routing"

    # e2e: host inputs -> device -> step -> host output, all inside the events
    e2e_ms = []
    h2d = L * T * (E * 4 + H * 2)
    d2h = L * T * H * 2
    for i in range(min(args.steps, 20)):
        with torch.cuda.stream(main):
            flush.zero_()
            ev0.record(main)
            for l in range(L):
                steps[l].buf.logits[:T].copy_(h_lg[i % npool, l], non_blocking=True)
                steps[l].buf.x[:T].copy_(h_x[i % npool, l], non_blocking=True)
            run_step()
            for l in range(L):
                h_out[l].copy_(steps[l].buf.out[:T], non_blocking=True)
            ev1.record(main)
        main.synchronize()
        e2e_ms.append(ev0.elapsed_time(ev1))

    # breakdown: each bank alone (layer 0), graph-replayed like the step
    breakdown = None
    if graph is not None:
        def part(hot, cold, count=None):
            st = steps[0]
            b = st.buf
            g2 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g2, stream=main):
                moe.moe_route_split_count(ctx, 0, b.logits, T, count_on if count is None else count, b.ids, b.w,
                                          b.ws_ptr, main)
                if hot:
                    moe.moe_expert_ffn_bank(ctx, 0, moe.MOE_BANK_HOT, b.x, T, b.ws_ptr, b.Y, main)
                if cold:
                    moe.moe_expert_ffn_bank(ctx, 0, moe.MOE_BANK_COLD, b.x, T, b.ws_ptr, b.Y, main)
            ts = []
            for i in range(min(args.steps, 20)):
                load_inputs(i, main)
                with torch.cuda.stream(main):
                    flush.zero_()
                    ev0.record(main)
                    g2.replay()
                    ev1.record(main)
                main.synchronize()
                ts.append(ev0.elapsed_time(ev1) * 1e3)
            return float(np.mean(ts))
        r_us = part(False, False)

        def router_alone():
            """The router GEMM that would produce layer 0's logits from its
            hidden states (the workload supplies logits, so it is outside the
            step), graph-replayed after an L2 flush."""
            wr = torch.from_numpy(synth.router_weights(cfg, 0).view(np.int16)).to(dev)
            br = torch.from_numpy(synth.router_bias(cfg, 0)).to(dev)
            rl = torch.empty((T, E), dtype=torch.float32, device=dev)
            g3 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g3, stream=main):
                moe.moe_router_logits(ctx, steps[0].buf.x, wr, br, T, E, H, rl, main)
            ts = []
            for i in range(min(args.steps, 20)):
                load_inputs(i, main)
                with torch.cuda.stream(main):
                    flush.zero_()
                    ev0.record(main)
                    g3.replay()
                    ev1.record(main)
                main.synchronize()
                ts.append(ev0.elapsed_time(ev1) * 1e3)
            return float(np.mean(ts))
        def whole_step(count):
            """The whole step (all layers) with counting on or off, graph-replayed
            after an L2 flush, alternating with the other setting."""
            g4 = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g4, stream=main):
                enqueue(count=count)
            return g4

        counter_ab = None
        if count_on:
            g_on, g_off = whole_step(True), whole_step(False)
            t_on, t_off = [], []
            for i in range(min(args.steps, 20)):
                for g4, ts in ((g_on, t_on), (g_off, t_off)):
                    load_inputs(i, main)
                    with torch.cuda.stream(main):
                        flush.zero_()
                        ev0.record(main)
                        g4.replay()
                        ev1.record(main)
                    main.synchronize()
                    ts.append(ev0.elapsed_time(ev1) * 1e3)
            counter_ab = {"step_on_us": float(np.median(t_on)), "step_off_us": float(np.median(t_off)),
                          "route_on_us": r_us, "route_off_us": part(False, False, count=False),
                          "note": "medians over the same inputs, on and off alternating; the usage count is "
                                  "also incremented by the on runs"}
        breakdown = {"route_us": r_us, "router_gemm_us": router_alone(), "counter_ab": counter_ab, "hot_alone_us": float(np.mean(hot_ms)) * 1e3,
                     "cold_alone_us": float(np.mean(ffn_alone(moe.MOE_BANK_COLD)[0])) * 1e3,
                     "ffn_in_step_us": float(np.mean(ffn_ms)) * 1e3, "banks": args.banks,
                     "note": "layer 0: each bank's FFN call alone after routing, and the step's both-bank FFN call; "
                             "the router GEMM (hidden states -> logits) alone, outside the step"}

    ms = total_ms / args.steps
    tokens_per_step = T   # one layer-step of T tokens (all layers of the config)
    value = job_tokens_per_s(world, tokens_per_step, args.steps, total_ms)
    e2e_total_ms = slowest_rank_ms(sum(e2e_ms), dist, dev)
    hot_avg_ms = float(np.mean(hot_ms))
    hot_gbs = float(np.mean(hot_bytes_alone)) / (hot_avg_ms * 1e-3) / 1e9
    roofline = {"kernel": "hot-bank expert FFN (moe_expert_ffn_bank, layer 0)", "bound": "hbm",
                "achieved": hot_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": hot_gbs / hbm_peak,
                "peak_source": f"{peak_src} (burst copy)",
                # ncu DRAM bytes per hot expert (profiles/traffic.json) x this run's mean hot experts
                "traffic": (profiled_traffic(args.config) * float(np.mean(hot_bytes_alone)) / eb
                            if profiled_traffic(args.config) else None),
                "timing": hot_timing, "us_per_launch": hot_avg_ms * 1e3}
    if T > 256:
        # large batches are a dense contraction: 2 flops per weight element per pick
        flops = float(np.mean(hot_picks)) * 2.0 * (3.0 * cfg.I * cfg.H)
        tf = flops / (hot_avg_ms * 1e-3) / 1e12
        roofline.update({"bound": "tensor", "achieved": tf, "peak": tf_burst, "unit": "TFLOP/s",
                         "frac": tf / tf_burst, "flops_per_launch": flops,
                         # rows carry bf16-class precision as two e4m3 pieces: two fp8-rate
                         # MMAs per product, i.e. the tensor pipe's bf16 rate
                         "peak_source": f"{peak_src} bf16 dense burst (two e4m3 pieces per row at the fp8 rate)",
                         "hbm_gbs_achieved": hot_gbs})
    # bytes roofline of the step (the metric's definition)
    t_roof = [(a * eb) / (hbm_peak * 1e9) + (c * eb) / (link_gbs * 1e9) for a, c in zip(dh, dc)]
    t_roof_max = [max((a * eb) / (hbm_peak * 1e9), (c * eb) / (link_gbs * 1e9)) for a, c in zip(dh, dc)]
    frac = float(np.sum(t_roof) / (np.sum(step_ms) * 1e-3))
    frac_max = float(np.sum(t_roof_max) / (np.sum(step_ms) * 1e-3))

    cpu = None
    if rank == 0:
        cfg1 = cfg if cfg.L == 1 else dataclasses.replace(cfg, L=1)
        if args.config == "prefill":
            lgs = [synth.router_logits(cfg1, 0, s, T=64) for s in range(8)]
            xss = [synth.activations(cfg1, 0, s, T=64) for s in range(8)]
            sample_T = 64
        else:
            lgs = [pool_lg[s][0] for s in range(npool)]
            xss = [pool_x[s][0] for s in range(npool)]
            sample_T = T
        tps, n, used, cores = cpu_oracle_steps(cfg1, weights0, masks[0], lgs, xss, args.cpu_budget)
        cpu = {"value": tps, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} single-layer steps of {sample_T} tokens of this workload's layer 0, {used:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e2m1 weights (e8m0 scales) x e4m3 rows (two pieces), block-scaled tensor cores, f32 accumulate, bf16 rows",
            "data": "synthetic (seeded SplitMix64; Zipf-skewed routing)",
            "config": {"workload": WORKLOADS[args.config] + (
                           f" [profiling variant: {cfg.E} experts, {cfg.n_hot} hot, {cfg.T} tokens]"
                           if (args.experts or args.tokens) else ""),
                       "layers": L, "tokens_per_step": T,
                       "l2": "flushed (512 MiB write) before every timed step", "cuda_graph": graph is not None,
                       "ffn_calls": "one call over both banks" if args.banks == "fused" else "hot and cold bank calls on two streams",
                       "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
            "us_per_layer_step": ms * 1e3 / L,
            "step_us_pct": {q: float(np.percentile(step_ms, p)) * 1e3 for q, p in (("p10", 10), ("median", 50),
                                                                               ("p90", 90))},
            "bytes_roofline": {"frac_sum": frac, "frac_max": frac_max,
                               "t_roof_us": float(np.mean(t_roof)) * 1e6, "t_step_us": ms * 1e3,
                               "distinct_hot": float(np.mean(dh)), "distinct_cold": float(np.mean(dc)),
                               "expert_bytes": eb, "hbm_gbs": hbm_peak, "hbm_peak_source": peak_src,
                               "link_gbs": link_gbs, "hbm_probe_gbs": hbm_probe_gbs},
            "roofline": roofline,
            "breakdown": breakdown,
            "cpu_baseline": cpu,
            "e2e": {"value": job_tokens_per_s(world, T, len(e2e_ms), e2e_total_ms), "unit": "tokens/s",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk.summary(),
        }
        print(json.dumps(line), flush=True)
    moe.moe_destroy(ctx)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
