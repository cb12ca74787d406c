#!/usr/bin/env python3
"""Benchmark of the sparse MoE FFN layer forward pass on GB300.

One step = one whole moe_ffn_forward call (router -> grouping -> experts ->
combine) over one batch of seeded synthetic tokens, weights resident in HBM.
Prints ONE JSON line (rank 0).  By default every workload of moe_inputs.WORKLOADS
is measured in turn: the headline keys describe the Qwen3.5-mini decode batch of
64 tokens, and `per_workload` holds one record per workload (step time, tokens/s,
roofline of each expert kernel, phase split, end-to-end rate, clocks, routing
load, near ties and the CPU oracle baseline with its parity on the sample).
Multi-GPU runs are independent replicas (the layer has no exchange step on one
node): value = all ranks' tokens / the slowest rank's time.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME|all]
  python bench.py --impl reference ...   # the fp64 CPU oracle on this host's cores
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; decode HBM GB/s and prefill TFLOP/s vs roofline (1×GB300)"
HEADLINE_WORKLOAD = "qwen35_mini_moe_decode_t64"
FLUSH_BYTES = 256 << 20          # > 2x the 129 MB L2


def flush_l2(buf, sink):
    """Evict L2: write a buffer larger than L2, then read another one, so that no
    dirty lines of the write remain to be written back inside the next timed step."""
    import torch
    buf[0].fill_(1)
    sink.add_(buf[1].view(torch.int64).sum())      # int64 view: a read sweep, no copy


PHASES = ("router_logits", "router_select", "permute", "gate_up", "down", "combine")


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="all",
                    help="one workload name, or 'all' (headline: the Qwen3.5-mini T=64 decode batch)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU oracle baseline budget of the headline workload (0 disables); "
                         "the other workloads take half of it each")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--path", choices=["auto", "decode", "prefill", "decode-registers"], default="auto",
                    help="the expert path (cfg.path); auto picks by tokens per expert")
    return ap.parse_args(argv)


def workload_names(arg):
    import moe_inputs as mi
    if arg == "all":
        return list(mi.WORKLOAD_ORDER)
    if arg not in mi.WORKLOADS:
        raise SystemExit(f"unknown workload {arg!r}; one of {', '.join(mi.WORKLOAD_ORDER)} or 'all'")
    return [arg]


def headline_of(names):
    return HEADLINE_WORKLOAD if HEADLINE_WORKLOAD in names else names[0]


def peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, source)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_hash(fname):
    path = os.path.join(ROOT, "sparse_moe_ffn_route_gb300", "csrc", fname)
    if not os.path.exists(path):
        return None
    return hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]


def ncu_traffic(workload, phase):
    """Per-launch DRAM bytes of `phase` from the committed ncu summary, if the kernel
    source is unchanged since the capture (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    rec = json.load(open(p)).get(workload, {}).get(phase)
    if not rec or rec.get("source_sha256_16") != kernel_hash(rec.get("kernel_file", "")):
        return None
    return rec.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._t = None

    def _run(self):
        try:
            proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                     "--format=csv,noheader,nounits", "-lms", "50"],
                                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        try:
            for line in proc.stdout:
                self.samples.append((time.perf_counter(), line.strip()))
                if self._stop.is_set():
                    break
        finally:
            proc.terminate()
            proc.wait()

    def start(self):
        self._t = threading.Thread(target=self._run, daemon=True)
        self._t.start()
        time.sleep(0.3)

    def stop(self):
        self._stop.set()
        if self._t:
            self._t.join(timeout=5)

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.samples:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                rows.append((ts, float(f[0]), float(f[1]), f))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        note = "samples inside the timed region"
        if not inside and rows:
            mid = 0.5 * (t0 + t1)
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:3]
            note = "timed region shorter than the sampling period: nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i in range(4)
                          if r[3][4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside),
                "sm_max_mhz": max(r[2] for r in inside), "reasons": reasons,
                "samples": len(inside), "note": note}


# ----------------------------------------------------------------------------- work counting
def expert_bytes(spec):
    """(gate+up bytes, down bytes) of one routed expert and of the shared expert."""
    d, ff, sff = spec.d_model, spec.expert_ff, spec.shared_ff
    if spec.mxfp4:
        gu = 2 * ff * (d // 32) * 17 + 2 * ff * 2          # blocks + scales + bias
        dn = d * (ff // 32) * 17 + d * 2
    else:
        gu = 2 * ff * d * 2
        dn = d * ff * 2
    return gu, dn, 2 * sff * d * 2, d * sff * 2


def launches_per_step(plan, mxfp4, spec_slots, tokens=0, n_experts=0):
    """Kernels of this library one moe_ffn_forward enqueues, by kernel plan."""
    router = 2                                            # logits, select
    permute = 3 if spec_slots > 2048 else 1               # count, scan, scatter (or one CTA)
    if plan in (1, 2, 5):                                 # decode: gate_up, down (5: one launch), combine
        # up to 32 tokens, 256 experts, 2048 slots: the select kernel also permutes
        fused = tokens <= 32 and n_experts <= 256 and spec_slots <= 2048
        return router + (0 if fused else permute) + (2 if plan == 5 else 3)
    if plan == 3:                                         # 2 GEMMs, combine (MXFP4: 2 scale transposes, gather)
        return router + permute + 3 + (3 if mxfp4 else 0)
    return router + permute + 6   # scale prep, gather, gate_up, h fix-up, down, combine


def work(spec, ids, accumulate=False):
    """Algorithmic bytes and flops per phase for one step with routing `ids` [T, k].
    accumulate: the prefill down projection adds the weighted expert outputs into
    per-token fp32 sums [T, d] (cleared by the select kernel, read once by the finish
    kernel) instead of writing Y [T*K, d] for the combine."""
    import numpy as np
    T, d, ff, sff, E, k = (spec.tokens, spec.d_model, spec.expert_ff, spec.shared_ff,
                           spec.n_experts, spec.top_k)
    distinct = int(len(np.unique(ids)))
    gu, dn, sgu, sdn = expert_bytes(spec)
    has_sh = sff > 0
    S = T * (k + has_sh)
    rows = T * k
    x_bytes = T * d * 2
    h_bytes = (rows * ff + T * sff) * 2
    Y_bytes = S * d * 4
    acc_bytes = T * d * 4
    by = {
        "router_logits": (E + has_sh) * d * 2 + x_bytes + T * (E + has_sh) * 4,
        "router_select": T * (E + has_sh) * 4 + S * 8,
        "permute": S * 4 * 3,
        "gate_up": distinct * gu + (sgu if has_sh else 0) + x_bytes + h_bytes + (acc_bytes if accumulate else 0),
        "down": distinct * dn + (sdn if has_sh else 0) + h_bytes + (acc_bytes if accumulate else Y_bytes),
        "combine": (acc_bytes if accumulate else Y_bytes + S * 8) + T * d * 2,
    }
    fl = {
        "router_logits": 2 * T * (E + has_sh) * d,
        "gate_up": 2 * rows * 2 * ff * d + 2 * T * 2 * sff * d,
        "down": 2 * rows * ff * d + 2 * T * sff * d,
    }
    per_unit = {"gate_up": gu, "down": dn}
    return by, fl, distinct, per_unit


def plan_dtype(plan, mxfp4):
    """The arithmetic type the expert kernels of a plan multiply in."""
    if mxfp4 and plan in (2, 4):
        return "f16 operands (MXFP4 weights decoded exactly), fp32 accumulation"
    if mxfp4:
        return "bf16 operands (MXFP4 weights decoded exactly), fp32 accumulation"
    return "bf16"


def kernel_roofline(name, by, fl, ms, hbm, tf_burst):
    """Roofline of one expert kernel timed between L2 flushes: HBM when its arithmetic
    intensity is below the ridge of the measured peaks, else tensor (against the burst
    bf16 peak; f16 operands run at the bf16 rate, a nominal ratio of 1)."""
    secs = ms / 1e3
    gbs = by / secs / 1e9
    tfs = fl / secs / 1e12
    tensor = fl / by > (tf_burst * 1e12) / (hbm * 1e9)
    return {"bound": "tensor" if tensor else "hbm", "kernel": name,
            "achieved": tfs if tensor else gbs, "peak": tf_burst if tensor else hbm,
            "unit": "TFLOP/s" if tensor else "GB/s",
            "frac": (tfs / tf_burst) if tensor else (gbs / hbm),
            "ms": ms, "hbm_gbs": gbs, "hbm_frac": gbs / hbm,
            "tensor_tflops": tfs, "tensor_frac": tfs / tf_burst,
            "algorithmic_bytes_per_launch": by, "algorithmic_flops_per_launch": fl}


def routing_load(ids, n_experts):
    """Tokens per routed expert for this step's routing."""
    import numpy as np
    cnt = np.bincount(ids.ravel().astype(np.int64), minlength=n_experts)
    srt = np.sort(cnt)[::-1]
    rec = {"min": int(cnt.min()), "max": int(cnt.max()), "mean": float(cnt.mean()),
           "cv": float(cnt.std() / cnt.mean()) if cnt.mean() > 0 else 0.0,
           "idle_experts": int((cnt == 0).sum()),
           "top4_share": float(srt[:4].sum() / max(cnt.sum(), 1))}
    if n_experts <= 64:
        rec["tokens_per_expert"] = [int(c) for c in cnt]
    else:
        rec["top8"] = [int(c) for c in srt[:8]]
    return rec


def near_tie_count(logits, k, eps=1e-5):
    """Tokens whose k-th/(k+1)-th largest fp32 logit, or two adjacent selected ones,
    lie within eps (their selection may legitimately differ from exact arithmetic)."""
    import numpy as np
    s = -np.sort(-logits.astype(np.float64), axis=1)
    gap_k = s[:, k - 1] - s[:, k] if logits.shape[1] > k else np.full(len(s), np.inf)
    gap_adj = np.min(np.diff(-s[:, :k], axis=1), axis=1) if k > 1 else np.full(len(s), np.inf)
    return int(((gap_k < eps) | (gap_adj < eps)).sum())


# ----------------------------------------------------------------------------- arms
def cpu_oracle_rate(spec, lay, seconds, tokens=None):
    """tokens/s of the fp64 oracle over repeated passes on `tokens` (default: all);
    also returns the last pass's result."""
    import numpy as np
    import oracle
    g = oracle.gating_for(spec)
    tok = np.arange(spec.tokens, dtype=np.int32) if tokens is None else tokens
    n, t0 = 0, time.perf_counter()
    while True:
        res = oracle.forward(g, lay, tokens=tok)
        n += len(tok)
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return n / el, n, el, oracle.num_threads(), res


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle timed on this host's cores, rank 0 only."""
    if rank != 0:
        return
    import numpy as np
    import moe_inputs as mi
    import oracle
    spec = mi.WORKLOADS[headline_of(workload_names(args.workload))]
    lay = mi.make_layer(spec)
    g = oracle.gating_for(spec)
    n_tok = min(spec.tokens, 16)
    rng = np.random.default_rng(0)

    def step():
        tok = np.sort(rng.choice(spec.tokens, size=n_tok, replace=False)).astype(np.int32)
        t0 = time.perf_counter()
        oracle.forward(g, lay, tokens=tok)
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step()
    times = [step() for _ in range(args.steps)]
    ms = 1e3 * statistics.mean(times)
    value = n_tok / (ms / 1e3)
    cores = oracle.num_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(spec),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_tok} random tokens of the {spec.tokens}-token batch per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def max_over_ranks(x, world, dev):
    """The largest x over the ranks (the slowest replica's time); x itself alone."""
    if world <= 1:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens, ms, world):
    """Whole-job tokens/s: every replica's T tokens over the slowest replica's step time."""
    return world * tokens / (ms / 1e3)


def config_of(spec):
    return {"workload": spec.name, "tokens": spec.tokens, "d_model": spec.d_model,
            "n_experts": spec.n_experts, "top_k": spec.top_k, "expert_ff": spec.expert_ff,
            "shared_ff": spec.shared_ff, "weights": "mxfp4" if spec.mxfp4 else "bf16",
            "router_bias": spec.bias[0] if spec.bias else None,
            "l2": "flushed between timed steps (256 MiB write + 256 MiB read, outside the step events)",
            "parallelism": "replicas"}


class LayerCache:
    """Host layers and their device copies, shared by workloads of one layer: the three
    Qwen3.5-mini workloads differ only in x and the router bias (the weights come from
    the same seeded streams), so their 1.6 GB of experts are generated and uploaded once."""

    def __init__(self, dev):
        self.dev = dev
        self.key = None
        self.host = None
        self.device = None

    def get(self, spec):
        import moe_inputs as mi
        from sparse_moe_ffn_route_gb300 import hostio
        key = (spec.family, spec.d_model, spec.n_experts, spec.expert_ff, spec.shared_ff, spec.seed,
               spec.scale_lo, spec.scale_hi)
        if key != self.key:
            self.key, self.host, self.device = key, None, None
            import torch
            torch.cuda.empty_cache()
            self.host = mi.make_layer(spec)
            self.device = hostio.upload(self.host, self.dev)
            return self.host, self.device
        lay = dataclasses.replace(self.host, spec=spec, x=mi.make_x(spec),
                                  router_b=mi.make_router_bias(spec))
        _, router, experts, shared = self.device
        router = dataclasses.replace(router, bias=hostio.bf16_tensor(lay.router_b, self.dev))
        return lay, (hostio.bf16_tensor(lay.x, self.dev), router, experts, shared)


def measure(spec, lay, dev_layer, args, rank, world, local_rank, dev, flush, sink, cpu_seconds):
    """Every number of one workload: timed steps, phase split, graph replay, the host
    entry point end to end, rooflines, routing load, near ties, the CPU baseline."""
    import numpy as np
    import torch
    import sparse_moe_ffn_route_gb300 as moe

    x, router, experts, shared = dev_layer
    if spec.family == "qwen":
        cfg = moe.qwen_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff, spec.shared_ff)
    else:
        cfg = moe.gptoss_cfg(spec.d_model, spec.n_experts, spec.top_k, spec.expert_ff)
    cfg = cfg.replace(path={"auto": moe.PATH_AUTO, "decode": moe.PATH_DECODE, "prefill": moe.PATH_PREFILL,
                            "decode-registers": moe.PATH_DECODE_REGISTERS}[args.path])
    T = spec.tokens
    ws = moe.workspace(cfg, T, dev)
    y = torch.empty_like(x)
    ids = torch.empty((T, spec.top_k), dtype=torch.int32, device=dev)

    plan = moe.moe_kernel_plan(cfg, T)
    moe.moe_ffn_forward(cfg, x, router, experts, shared, y=y, topk_ids=ids, ws=ws)
    torch.cuda.synchronize()
    st, bits = moe.moe_device_status(ws)
    if st != 0:
        raise RuntimeError(f"{spec.name}: device status {st} bits {bits:#x}")
    ids_np = ids.cpu().numpy()
    accumulate = plan in (moe.PLAN_PREFILL_BF16, moe.PLAN_PREFILL_F16) and not cfg.deterministic
    by, fl, distinct, per_unit = work(spec, ids_np, accumulate)

    for _ in range(args.warmup):
        flush_l2(flush, sink)
        moe.moe_ffn_forward(cfg, x, router, experts, shared, y=y, ws=ws)
    torch.cuda.synchronize()

    # Timed steps record only start/end events (so the kernels may overlap their
    # launches); a separate pass with all seven phase events gives the phase split.
    n_ph = max(10, min(args.steps, 50))
    ph_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(n_ph)]
    for i in range(n_ph):
        flush_l2(flush, sink)
        moe.moe_set_phase_events(ph_evs[i])
        moe.moe_ffn_forward(cfg, x, router, experts, shared, y=y, ws=ws)
    moe.moe_set_phase_events(None)
    torch.cuda.synchronize()
    phase_ms = {p: statistics.mean(e[i].elapsed_time(e[i + 1]) for e in ph_evs)
                for i, p in enumerate(PHASES)}

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    for e in evs:           # create the event handles outside the timed region
        for ev in e:
            ev.record()
    torch.cuda.synchronize()
    sampler = ClockSampler(local_rank)
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2(flush, sink)
        moe.moe_set_phase_events(evs[i])
        moe.moe_ffn_forward(cfg, x, router, experts, shared, y=y, ws=ws)
    moe.moe_set_phase_events(None)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.perf_counter()
    sampler.stop()

    step_ms = [e[0].elapsed_time(e[1]) for e in evs]
    ms = max_over_ranks(statistics.mean(step_ms), world, dev)
    value = job_rate(T, ms, world)

    # The same step captured once in a CUDA graph and replayed (how a serving loop
    # would drive it): launch work leaves the critical path.
    graph_rec = None
    if not args.no_graph:
        gs = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                moe.moe_ffn_forward(cfg, x, router, experts, shared, y=y, ws=ws, stream=gs)
        torch.cuda.synchronize()
        for _ in range(3):
            graph.replay()
        g_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for i in range(args.steps):
            flush_l2(flush, sink)
            g_evs[i][0].record()
            graph.replay()
            g_evs[i][1].record()
        torch.cuda.synchronize()
        g_ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[1]) for e in g_evs), world, dev)
        graph_rec = {"ms_per_step": g_ms, "value": job_rate(T, g_ms, world), "unit": "tokens/s",
                     "note": "one captured moe_ffn_forward replayed per step, L2 flushed between"}
        del graph

    # end to end through the host-buffer entry point: pinned x in, pinned y out; the
    # call bound once (arguments marshalled once), as a decode loop would use it
    e2e = None
    if not args.no_e2e:
        x_host = x.cpu().pin_memory()
        y_host = torch.empty_like(x_host).pin_memory()
        step = moe.BoundForwardHost(cfg, x_host, router, experts, shared, y_host=y_host, ws=ws)
        for _ in range(3):
            step()
        n_e2e = max(10, min(args.steps, 200))
        if world > 1:
            torch.distributed.barrier()
        te = []
        for _ in range(n_e2e):
            flush_l2(flush, sink)
            torch.cuda.synchronize()
            a = time.perf_counter()
            step()
            te.append(time.perf_counter() - a)
        e_ms = max_over_ranks(1e3 * statistics.mean(te), world, dev)
        e2e = {"value": job_rate(T, e_ms, world), "unit": "tokens/s",
               "h2d_bytes_per_step": x_host.numel() * 2, "d2h_bytes_per_step": y_host.numel() * 2,
               "ms_per_step": e_ms}
        del step

    # routing statistics from the library's own router: per-expert load, near ties
    logits = torch.empty((T, spec.n_experts), dtype=torch.float32, device=dev)
    moe.moe_route(cfg, x, router, shared, logits=logits, ws=ws)
    # fp32 output for the parity figure of the CPU baseline's sample
    y32 = moe.moe_ffn_forward(cfg.replace(y_fp32=1), x, router, experts, shared, ws=ws)
    torch.cuda.synchronize()
    load = routing_load(ids_np, spec.n_experts)
    ties = near_tie_count(logits.cpu().numpy(), spec.top_k)
    n_sample = min(T, 64)
    y32_sample = y32[:n_sample].cpu().numpy().astype(np.float64)
    del ws, y, y32, logits

    if rank != 0:
        return None
    hbm, tf, tf_sus, src = peaks()
    step_bytes = sum(by.values())
    if plan == moe.PLAN_DECODE_FUSED:
        # gate_up and down are one kernel: the phase between their marks holds all of it
        # (the next mark follows it at once); its algorithmic bytes are both projections'
        GD = "gate_up+down"
        phase_ms = {(GD if p == "gate_up" else p): t for p, t in phase_ms.items() if p != "down"}
        by[GD], fl[GD], per_unit[GD] = by["gate_up"] + by["down"], fl["gate_up"] + fl["down"], \
            per_unit["gate_up"] + per_unit["down"]
        expert_phases = (GD,)
    else:
        expert_phases = ("gate_up", "down")
    kernels = {p: kernel_roofline(p, by[p], fl.get(p, 0), phase_ms[p], hbm, tf) for p in expert_phases}
    dom = max(expert_phases, key=lambda p: phase_ms[p])
    roof = dict(kernels[dom])
    roof.update({"peak_source": src + (" (bf16 burst, L2 flushed between steps)" if roof["bound"] == "tensor"
                                       else " (HBM copy)"),
                 "traffic": ncu_traffic(spec.name, dom),
                 "per_unit_bytes": per_unit[dom], "units_per_launch": distinct,
                 "path": moe.PLAN_NAMES[plan]})
    cpu = None
    if cpu_seconds > 0:
        tok = np.arange(n_sample, dtype=np.int32)
        rate, n, el, cores, res = cpu_oracle_rate(spec, lay, cpu_seconds, tokens=tok)
        rms = float(np.sqrt(np.mean(res.y ** 2)))
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n} token-evaluations (first {n_sample} tokens, repeated) in {el:.1f} s",
               "parity_on_sample": {"tokens": n_sample,
                                    "max_abs_err_over_rms": float(np.max(np.abs(y32_sample - res.y))) / rms,
                                    "ids_equal": int(np.sum(np.all(res.ids == ids_np[:n_sample], axis=1))),
                                    "bar": 2e-2}}
    return {
        "spec": spec, "plan": plan, "ms": ms, "value": value, "step_ms": step_ms,
        "roofline": roof, "kernels": kernels, "cpu_baseline": cpu, "e2e": e2e, "graph": graph_rec,
        "gpu_launches": launches_per_step(plan, spec.mxfp4, T * (spec.top_k + (spec.shared_ff > 0)), T,
                                          spec.n_experts) * args.steps,
        "clocks": sampler.summary(t0, t1), "phases_ms": phase_ms,
        "step_hbm_gbs": step_bytes / (ms / 1e3) / 1e9, "step_algorithmic_bytes": step_bytes,
        "distinct_experts": distinct, "load": load, "near_ties": ties,
        "dtype": plan_dtype(plan, spec.mxfp4), "accumulate": accumulate,
    }


def compact(rec):
    """The per-workload record of the JSON line (rounded, without the raw step list)."""
    def r(v, n=4):
        if isinstance(v, float):
            return float(f"{v:.{n}g}")
        if isinstance(v, dict):
            return {k: r(w, n) for k, w in v.items()}
        if isinstance(v, list):
            return [r(w, n) for w in v]
        return v
    spec = rec["spec"]
    kern = {p: {k: r(v) for k, v in kr.items()
                if k in ("bound", "ms", "achieved", "unit", "frac", "hbm_frac", "tensor_frac")}
            for p, kr in rec["kernels"].items()}
    roof = {k: r(v) for k, v in rec["roofline"].items()
            if k in ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic",
                     "algorithmic_bytes_per_launch", "algorithmic_flops_per_launch",
                     "per_unit_bytes", "units_per_launch")}
    out = {"tokens": spec.tokens, "ms_per_step": r(rec["ms"]), "value": r(rec["value"]),
           "unit": "tokens/s", "dtype": rec["dtype"], "plan": rec["plan"], "roofline": roof,
           "kernels": kern, "phases_ms": r(rec["phases_ms"], 3),
           "graph_ms_per_step": r(rec["graph"]["ms_per_step"]) if rec["graph"] else None,
           "e2e": r(rec["e2e"]) if rec["e2e"] else None,
           "clocks": {k: rec["clocks"].get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")},
           "step_algorithmic_bytes": rec["step_algorithmic_bytes"],
           "step_hbm_gbs": r(rec["step_hbm_gbs"]), "distinct_experts": rec["distinct_experts"],
           "load": r(rec["load"], 3), "near_ties": rec["near_ties"],
           "gpu_launches": rec["gpu_launches"], "accumulated_prefill": rec["accumulate"],
           "cpu_baseline": r(rec["cpu_baseline"]) if rec["cpu_baseline"] else None}
    return out


def run_ours(args, rank, world, local_rank):
    import torch
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    import moe_inputs as mi
    import sparse_moe_ffn_route_gb300  # noqa: F401  (fails loudly without libmoe.so)

    names = workload_names(args.workload)
    head = headline_of(names)
    flush = (torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev),
             torch.zeros(FLUSH_BYTES, dtype=torch.uint8, device=dev))
    sink = torch.zeros((), dtype=torch.int64, device=dev)
    cache = LayerCache(dev)
    # same-layer workloads next to each other, so each layer is generated once
    order = sorted(names, key=lambda n: (mi.WORKLOADS[n].family != mi.WORKLOADS[head].family,
                                         mi.WORKLOADS[n].family, names.index(n)))
    recs = {}
    for name in order:
        spec = mi.WORKLOADS[name]
        if args.path != "auto" and spec.name != head:
            continue
        lay, dev_layer = cache.get(spec)
        budget = args.cpu_seconds if name == head else 0.5 * args.cpu_seconds
        recs[name] = measure(spec, lay, dev_layer, args, rank, world, local_rank, dev, flush, sink, budget)
        torch.cuda.synchronize()
    if rank != 0:
        return
    h = recs[head]
    spec = h["spec"]
    out = {
        "metric": METRIC, "value": h["value"], "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": h["ms"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": h["dtype"], "data": "synthetic",
        "config": dict(config_of(spec), **({} if args.path == "auto" else {"path": args.path})),
        "ms_per_step_median": statistics.median(h["step_ms"]), "ms_per_step_min": min(h["step_ms"]),
        "roofline": h["roofline"],
        "cpu_baseline": h["cpu_baseline"],
        "e2e": h["e2e"],
        "graph": h["graph"],
        "gpu_launches": h["gpu_launches"],
        "clocks": h["clocks"],
        "phases_ms": h["phases_ms"],
        "step_hbm_gbs": h["step_hbm_gbs"],
        "step_algorithmic_bytes": h["step_algorithmic_bytes"],
        "distinct_experts": h["distinct_experts"],
        "per_workload": {n: compact(recs[n]) for n in names if n in recs},
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
