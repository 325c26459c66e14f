"""Benchmark of the FastMTP verify step on GB300.

One step = the whole hot path over one batch: the MoE FFN layer at 32
sequences x (K=3)+1 = 128 tokens (route, permute, grouped SwiGLU experts,
shared experts, combine) followed by greedy acceptance over the verifier's
[32, 4, 129280] bf16 logits.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is verified tokens/s with all inputs
resident in HBM; `e2e` is the same through the public API with host buffers
(pinned host -> device copies and the read-back inside the timed region).
Between timed steps L2 is flushed by writing a 256 MB buffer (outside the
timed events).  The `--impl reference` arm times the CPU oracle on a bounded
sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "decode"
METRIC = "MoE verify-step tokens/s at 32x(K+1) tokens; % of HBM / tensor-core roofline"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 256 << 20


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        hbm = d.get("hbm_gbs")
        if hbm:
            return float(hbm), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def wait_first_sample(self, timeout=3.0):
        """Block until nvidia-smi has printed its first sample (it takes a moment to start)."""
        self._first = None
        if self.proc is None:
            return
        import select
        r, _, _ = select.select([self.proc.stdout], [], [], timeout)
        if r:
            self._first = self.proc.stdout.readline()

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            first = [self._first] if getattr(self, "_first", None) else []
            self.lines = [l for l in first + out.splitlines() if l.strip()]
        else:
            self.lines = []

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            parts = [p.strip() for p in l.split(",")]
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def layer_source_hash():
    h = hashlib.sha256()
    for f in ("ffn.cu", "ptx.cuh", "prefetch.cu", "route.cu", "permute.cu", "combine.cu", "ffn_plan.cuh", "api.cu"):
        with open(os.path.join(ROOT, "lossless_speculative_verification_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_hash):
    """DRAM bytes of one layer (sum over its launches) from the committed ncu summary, if it was
    taken on this source."""
    path = os.path.join(ROOT, "profiles", "layer_decode_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_layer")


# ----------------------------------------------------------------------------- reference arm (CPU oracle)
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from lossless_speculative_verification_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[WORKLOAD]
    d = w.dims
    prob = synth.moe_problem(w, seed=args.seed)
    logits, planted, drafts = synth.verify_problem(w, seed=args.seed)
    tok_per_step = 2          # tokens of the 128-token batch the oracle takes per step

    def step(i):
        toks = np.array([(2 * i) % d.T, (2 * i + 1) % d.T], np.int32)
        oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up, prob.ws_down,
                         d.k, d.S, tokens=toks)
        b = (i % w.B)
        oracle.accept(logits[b:b + 1], drafts[b:b + 1])

    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = tok_per_step * args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode verify step: MoE layer T=128 (B=32,K=3), H=1280, E=64 top-6, S=2, I=896, "
                               "then acceptance over [32,4,129280] bf16", "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": "%d tokens of the 128-token layer + 1 sequence's acceptance per step" % tok_per_step},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline_sample(seconds=12.0, seed=0):
    """The oracle as it stands, single-threaded, on a bounded sample of the same workload."""
    import oracle
    from lossless_speculative_verification_gb300 import synth
    oracle.build()
    w = synth.WORKLOADS[WORKLOAD]
    d = w.dims
    prob = synth.moe_problem(w, seed=seed)
    logits, planted, drafts = synth.verify_problem(w, seed=seed)
    n = 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        t = n % d.T
        oracle.moe_layer(prob.x, prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up, prob.ws_down,
                         d.k, d.S, tokens=np.array([t], np.int32))
        b = t // (w.K + 1)
        if t % (w.K + 1) == 0:
            oracle.accept(logits[b:b + 1], drafts[b:b + 1])
        n += 1
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": "%d token passes (cycling over the 128 tokens) through the oracle layer (route, 6 routed "
                      "+ 2 shared experts, combine) plus the acceptance of their sequences, %.1f s" % (n, dt)}


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch
    from lossless_speculative_verification_gb300 import _build, api, synth

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if world > 1:
        dist.barrier()

    w = synth.WORKLOADS[WORKLOAD]
    d = w.dims
    prob = synth.moe_problem(w, seed=args.seed + 1000 * rank)
    logits_np, planted, drafts_np = synth.verify_problem(w, seed=args.seed + 1000 * rank)

    def tdev(a):
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)

    x = tdev(prob.x)
    W = [tdev(a) for a in (prob.w_router, prob.w_gate_up, prob.w_down, prob.ws_gate_up, prob.ws_down)]
    del prob.w_gate_up, prob.w_down
    sh = api.shape(d.T, d.H, d.E, d.k, d.S, d.I)
    wts = api.weights(*W)
    ws = api.workspace(sh, dev)
    logits = tdev(logits_np)
    drafts = torch.from_numpy(drafts_np).to(dev)
    aws = api.spec_verify_workspace(w.B, w.K, w.V, dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    T, k = d.T, d.k
    idx = torch.empty((T, k), dtype=torch.int32, device=dev)
    counts = torch.empty(d.E, dtype=torch.int32, device=dev)
    out = torch.empty((T, d.H), dtype=torch.bfloat16, device=dev)
    alen = torch.empty(w.B, dtype=torch.int32, device=dev)
    comm = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    # launches per step: route, permute+gather, grouped experts, combine | argmax partials, accept
    launches_per_step = 6

    def layer():
        api.moe_verify_layer(x, wts, sh, ws, out=out, topk_idx=idx, counts=counts)

    def accept():
        api.spec_verify_accept(logits, drafts, aws, accept_len=alen, committed=comm)

    for _ in range(max(args.warmup, 0)):
        layer(); accept()
    torch.cuda.synchronize()
    assert api.get_device_error() == 0

    # eager launches, for context
    eager_ms = []
    for i in range(min(args.steps, 10)):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        layer(); accept()
        b.record(stream)
        b.synchronize()
        eager_ms.append(a.elapsed_time(b))

    # the step as two CUDA graphs: the MoE layer (one PDL chain) and the acceptance
    graphs = [torch.cuda.CUDAGraph() for _ in range(2)]
    for g, fn in zip(graphs, (layer, accept)):
        with torch.cuda.graph(g):
            fn()
    for _ in range(max(args.warmup, 0)):
        for g in graphs:
            g.replay()
    torch.cuda.synchronize()
    assert api.get_device_error() == 0

    n_touched = int((counts > 0).sum().item())
    H, I, S, E = d.H, d.I, d.S, d.E
    # algorithmic bytes of the layer: router + touched routed + shared expert weights, x in, out
    layer_bytes = E * H * 2 + (n_touched + S) * 3 * H * I * 2 + 2 * T * H * 2
    accept_bytes = w.B * (w.K + 1) * w.V * 2

    # timed region: per step, flush L2 (untimed), then events around the two graphs
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the sampler polls every 100 ms: keep the GPU in the same back-to-back load for a
        # moment before and after the timed steps so that its samples describe them
        clk.wait_first_sample()
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            flush.fill_(0)
            for g in graphs:
                g.replay()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            graphs[0].replay()
            evs[i][1].record(stream)
            graphs[1].replay()
            evs[i][2].record(stream)
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            flush.fill_(0)
            for g in graphs:
                g.replay()
        torch.cuda.synchronize()
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    layer_ms = [e[0].elapsed_time(e[1]) for e in evs]
    accept_ms = [e[1].elapsed_time(e[2]) for e in evs]
    total_ms = sum(step_ms)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        dist.barrier()
    assert api.get_device_error() == 0

    # end to end through the public API: pinned host inputs in, results back to the host
    hx = x.cpu().pin_memory()
    hl = logits.cpu().pin_memory()
    hd = drafts.cpu().pin_memory()
    h_out = torch.empty_like(out, device="cpu").pin_memory()
    h_len = torch.empty_like(alen, device="cpu").pin_memory()
    h_comm = torch.empty_like(comm, device="cpu").pin_memory()
    dx, dl, dd = torch.empty_like(x), torch.empty_like(logits), torch.empty_like(drafts)

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        dl.copy_(hl, non_blocking=True)
        dd.copy_(hd, non_blocking=True)
        api.moe_verify_layer(dx, wts, sh, ws, out=out)
        api.spec_verify_accept(dl, dd, aws, accept_len=alen, committed=comm)
        h_out.copy_(out, non_blocking=True)
        h_len.copy_(alen, non_blocking=True)
        h_comm.copy_(comm, non_blocking=True)

    for _ in range(max(args.warmup, 1)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = []
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        e2e_step()
        b.record(stream)
        b.synchronize()
        e2e_ms.append(a.elapsed_time(b))
    e2e_total = sum(e2e_ms)
    if world > 1:
        t = torch.tensor([e2e_total], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_total = float(t.item())
    assert api.get_device_error() == 0
    h2d = hx.numel() * 2 + hl.numel() * 2 + hd.numel() * 4
    d2h = h_out.numel() * 2 + h_len.numel() * 4 + h_comm.numel() * 4

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    ms_per_step = total_ms / args.steps
    tokens = T * world * args.steps
    value = tokens / (total_ms / 1e3)
    peak, peak_kind = peaks()
    layer_avg = sum(layer_ms) / len(layer_ms)
    accept_avg = sum(accept_ms) / len(accept_ms)
    achieved = layer_bytes / (layer_avg / 1e3) / 1e9
    khash = layer_source_hash()
    traffic = ncu_traffic(khash)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "decode verify step: MoE layer T=128 (B=32,K=3), H=1280, E=64 top-6, S=2, I=896, "
                               "then greedy acceptance over [32,4,129280] bf16 logits",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "flushed between timed steps (256 MB write, outside the events)",
                   "timing": "step replayed as 2 CUDA graphs (layer, acceptance), CUDA events per step",
                   "clocks_window": "nvidia-smi every 100 ms over back-to-back steps around the timed ones",
                   "eager_ms_per_step": sum(eager_ms) / len(eager_ms)},
        "roofline": {"bound": "hbm",
                     "kernel": "moe_verify_layer: router, permute+gather, grouped SwiGLU experts (tcgen05), "
                               "combine; one PDL-chained launch sequence (the experts kernel carries the HBM stream)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_source": peak_kind, "traffic": traffic, "algorithmic_bytes": layer_bytes,
                     "touched_experts": n_touched, "layer_ms": layer_avg, "kernel_source_hash": khash,
                     "accept": {"ms": accept_avg, "algorithmic_bytes": accept_bytes,
                                "achieved_gbs": accept_bytes / (accept_avg / 1e3) / 1e9}},
        "e2e": {"value": T * world * args.steps / (e2e_total / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if world == 1:
        line["cpu_baseline"] = cpu_baseline_sample()
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    rank, world, local = dist_env()
    if args.warmup < 0 or args.steps <= 0:
        raise SystemExit("steps must be positive")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
