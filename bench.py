"""Benchmark of the FastMTP verify step on GB300.

Default workload ("decode"): one step = the whole hot path over one batch,
i.e. the MoE FFN layer at 32 sequences x (K=3)+1 = 128 tokens (route, permute,
grouped SwiGLU experts, shared experts, combine) followed by greedy
acceptance over the verifier's [32, 4, 129280] bf16 logits.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|prefill|sweep|stack|lmhead|attention|draft]

Prints one JSON line per measured configuration (rank 0; the default run
prints exactly one).  `value` is tokens/s with all inputs resident in HBM;
`e2e` is the same through the public API with host buffers (pinned host ->
device copies and the read-back inside the timed region).  Before every
timed step L2 is flushed by writing a 256 MB buffer and reading it back (outside the
events), so that no dirty line of the flush is written back inside the step.
The `--impl reference` arm times the CPU oracle on a bounded sample of the
same workload.

Other workloads (not the default line):
  prefill  8 pages x (1,156 visual + 64 prompt) = 9,760 tokens through the layer
  sweep    B in {1,4,8,16,32,64} x K in {0,1,2,3}: layer + acceptance, one line each, then one
           "k_policy" line: per B, the K that maximises tau(K) * t(K=0) / t(K) with the pages'
           conditional acceptances and the measured step times t (spec_k_policy)
  stack    11 layers (Zipf-skewed routing, residual + RMSNorm) at 64 x 4 tokens + acceptance
  lmhead   the verifier's output layer fused with greedy verification at 32 x 4 positions
  attention  causal attention of 32 x 4 verified positions over page-shaped caches
  draft    3 recursive FastMTP draft-block steps for 32 sequences
  spec     one speculative step per batch size B in {1,4,8,16,32,64} and K in {0,1,2,3}: K draft-block
           steps, then the verify pass of an 11-layer decoder (attention over page-shaped caches + the
           MoE layer per layer, the output layer fused with the acceptance rule) over K+1 positions;
           one line each, then the "k_policy" line from these step costs
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
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "sweep", "stack", "lmhead", "attention", "draft", "spec"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the timed oracle sample (for profiler runs; the line then has no cpu_baseline)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="no benchmark: read an ncu CSV of this workload's run (metrics dram__bytes_read.sum, "
                         "dram__bytes_write.sum, gpu__time_duration.sum) and write profiles/layer_<workload>"
                         "_traffic.json, the DRAM bytes of one layer that the roofline's `traffic` reports")
    ap.add_argument("--ncu-command", default="", help="with --record-traffic: the command that made the CSV")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def peaks():
    """(hbm GB/s, bf16 TFLOP/s, source) from MEASURED_PEAKS.json, else the fallback figures."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), float(d.get("bf16_tflops") or FALLBACK_BF16_TFLOPS), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms around the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []
        self._first = None

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
            first = [self._first] if self._first else []
            self.lines = [l for l in first + out.splitlines() if l.strip()]

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


# per workload: the sources its kernels come from, and the first and last kernel of one step
STEP_SOURCES = {
    "draft": ("draft.cu", "skinny.cu", "attention.cu", "lmhead.cu", "accept.cu", "combine.cu", "ptx.cuh", "api.cu",
              "tmap.h"),
    "layer": ("ffn.cu", "ptx.cuh", "route.cu", "permute.cu", "combine.cu", "ffn_plan.cuh", "api.cu", "tmap.h"),
    "lmhead": ("lmhead.cu", "accept.cu", "ptx.cuh", "api.cu", "tmap.h"),
    "attention": ("attention.cu", "ptx.cuh", "api.cu"),
}
STEP_BOUNDS = {"layer": ("route", "combine_kernel"), "lmhead": ("lmhead_argmax_kernel", "accept_finalize_kernel"),
               "attention": ("attn_split_kernel", "attn_combine_kernel"),
               "draft": ("draft_norm_kernel", "accept_finalize_kernel")}   # one recursion step


def step_kind(workload):
    return workload if workload in STEP_SOURCES else "layer"


def layer_source_hash(workload="decode"):
    h = hashlib.sha256()
    for f in STEP_SOURCES[step_kind(workload)]:
        with open(os.path.join(ROOT, "lossless_speculative_verification_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel_hash):
    """DRAM bytes of one layer (sum over its launches) from the committed ncu summary, if it was
    taken on this source."""
    path = os.path.join(ROOT, "profiles", "layer_%s_traffic.json" % workload)
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    if d.get("kernel_source_hash") != kernel_hash:
        return None
    return d.get("dram_bytes_per_layer")


def record_traffic(args):
    """Sum DRAM bytes over each layer's launches (a layer: from a router launch to the next combine)
    in an ncu CSV, and store the mean per layer beside the source hash it was taken on."""
    import csv
    launches = {}
    with open(args.record_traffic, newline="") as f:
        hdr = None
        for row in csv.reader(f):
            if row and row[0] == "ID":
                hdr = row
                continue
            if not hdr or len(row) != len(hdr):
                continue
            r = dict(zip(hdr, row))
            e = launches.setdefault(int(r["ID"]), {"name": r["Kernel Name"].split("(")[0].split("::")[-1].strip()})
            scale = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "nsecond": 1, "usecond": 1e3,
                     "msecond": 1e6, "ns": 1, "us": 1e3, "ms": 1e6}.get(r["Metric Unit"], 1)
            try:
                e[r["Metric Name"]] = float(r["Metric Value"].replace(",", "")) * scale
            except ValueError:
                pass
    first, last_k = STEP_BOUNDS[step_kind(args.workload)]
    layers, cur = [], None
    for i in sorted(launches):
        e = launches[i]
        base = e["name"].split("<")[0]
        if base.startswith(first) and cur is None:
            cur = []
        if cur is None:
            continue
        cur.append(e)
        if base == last_k:
            layers.append(cur)
            cur = None
    if not layers:
        raise SystemExit("no complete step (%s ... %s) in %s" % (first, last_k, args.record_traffic))
    per_layer = [sum(e.get("dram__bytes_read.sum", 0) + e.get("dram__bytes_write.sum", 0) for e in L) for L in layers]
    last = {e["name"]: {"read": int(e.get("dram__bytes_read.sum", 0)), "write": int(e.get("dram__bytes_write.sum", 0)),
                        "ns": int(e.get("gpu__time_duration.sum", 0))} for e in layers[-1]}
    out = {"workload": args.workload, "command": args.ncu_command,
           "note": "sum of DRAM read+write bytes over one layer's launches, mean over the %d layers in the "
                   "capture; the writes include write-backs of the benchmark's own L2-flush buffer" % len(layers),
           "kernel_source_hash": layer_source_hash(args.workload), "dram_bytes_per_layer": int(sum(per_layer) / len(per_layer)),
           "per_kernel_last_layer": last}
    path = os.path.join(ROOT, "profiles", "layer_%s_traffic.json" % args.workload)
    with open(path, "w") as f:
        json.dump(out, f, indent=1)
        f.write("\n")
    print(json.dumps(out))


# ----------------------------------------------------------------------------- workloads
def layer_bytes(d, n_touched):
    """Algorithmic bytes of one MoE layer: router, touched routed and shared expert weights, x in, out."""
    return d.E * d.H * 2 + (n_touched + d.S) * 3 * d.H * d.I * 2 + 2 * d.T * d.H * 2


def layer_flops(d):
    return 2.0 * d.T * (d.k + d.S) * 3 * d.H * d.I + 2.0 * d.T * d.E * d.H


def describe(w, layers=1):
    d = w.dims
    s = "MoE layer T=%d, H=%d, E=%d top-%d, S=%d, I=%d" % (d.T, d.H, d.E, d.k, d.S, d.I)
    if layers > 1:
        s = "%d x %s, Zipf(%.1f) routing, residual + RMSNorm" % (layers, s, w.zipf_s)
    if w.V:
        s += "; then greedy acceptance over [%d,%d,%d] bf16 logits (B=%d, K=%d)" % (w.B, w.K + 1, w.V, w.B, w.K)
    return s


class DeviceStep:
    """One workload on the device: `layer()` and `accept()` (each graph-capturable),
    `e2e()` through the public API with host buffers, plus the accounting."""

    def __init__(self, name, w, seed, dev):
        import torch
        from lossless_speculative_verification_gb300 import api, synth
        self.name, self.w, self.dev = name, w, dev
        self.api = api
        d = w.dims
        self.T = d.T
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.sh = api.shape(d.T, d.H, d.E, d.k, d.S, d.I)
        self.ws = api.workspace(self.sh, dev)
        self.layers = []
        if w.layers > 1:
            st = synth.stack_problem(w, seed=seed)
            for L in st["layers"]:
                self.layers.append(api.weights(*[t(L[n]) for n in ("w_router", "w_gate_up", "w_down",
                                                                    "ws_gate_up", "ws_down")]))
            self.x0, self.h0 = t(st["x0"]), t(st["h0"])
        else:
            prob = synth.moe_problem(w, seed=seed)
            self.layers.append(api.weights(*[t(a) for a in (prob.w_router, prob.w_gate_up, prob.w_down,
                                                             prob.ws_gate_up, prob.ws_down)]))
            self.x0 = self.h0 = t(prob.x)
        self.x = torch.empty_like(self.x0)
        self.h = torch.empty_like(self.x0)
        self.h2 = torch.empty_like(self.x0)
        self.out = torch.empty_like(self.x0)
        self.layer_counts = [torch.empty(d.E, dtype=torch.int32, device=dev) for _ in self.layers]
        if w.V:
            logits, planted, drafts = synth.verify_problem(w, seed=seed)
            self.logits = t(logits)
            self.drafts = torch.from_numpy(drafts).to(dev)
            self.aws = api.spec_verify_workspace(w.B, w.K, w.V, dev)
            self.alen = torch.empty(w.B, dtype=torch.int32, device=dev)
            self.comm = torch.empty((w.B, w.K + 1), dtype=torch.int32, device=dev)
        else:
            self.logits = None
        # our kernel launches per step (the counter memset is not one).  Per layer: up to 256 tokens the
        # router (which places the rows), experts, combine; above, the tensor-core router, the fused
        # permutation + gather (<= 8192 pairs; else count, scatter and prep), experts, combine; plus
        # rmsnorm in the stack.  Acceptance: partials + finalize.
        per_layer = 3 if d.T <= 256 else (4 if d.T * d.k <= 8192 else 6)
        acc = 2 if w.V else 0
        self.launches = len(self.layers) * (per_layer + (1 if w.layers > 1 else 0)) + acc

    def _layers(self, x_in):
        api = self.api
        if len(self.layers) == 1:
            api.moe_verify_layer(x_in, self.layers[0], self.sh, self.ws, out=self.out, counts=self.layer_counts[0])
            return
        self.x.copy_(x_in)
        self.h.copy_(self.h0)
        h, h2 = self.h, self.h2
        for L, c in zip(self.layers, self.layer_counts):
            api.moe_verify_layer(h, L, self.sh, self.ws, out=self.out, counts=c)
            api.rmsnorm_residual(self.x, self.out, h=h2)
            h, h2 = h2, h

    def layer(self):
        self._layers(self.x0)

    def accept(self):
        if self.logits is not None:
            self.api.spec_verify_accept(self.logits, self.drafts, self.aws, accept_len=self.alen, committed=self.comm)

    def bytes_and_flops(self):
        d = self.w.dims
        byts = sum(layer_bytes(d, int((c > 0).sum().item())) for c in self.layer_counts)
        flops = layer_flops(d) * len(self.layers)
        acc = self.w.B * (self.w.K + 1) * self.w.V * 2 if self.logits is not None else 0
        return byts, flops, acc

    def setup_e2e(self):
        import torch
        self.hx = self.x0.cpu().pin_memory()
        self.dx = torch.empty_like(self.x0)
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        h2d, d2h = self.hx.numel() * 2, self.h_out.numel() * 2
        if self.logits is not None:
            self.hl = self.logits.cpu().pin_memory()
            self.hd = self.drafts.cpu().pin_memory()
            self.dl, self.dd = torch.empty_like(self.logits), torch.empty_like(self.drafts)
            self.h_len = torch.empty_like(self.alen, device="cpu").pin_memory()
            self.h_comm = torch.empty_like(self.comm, device="cpu").pin_memory()
            h2d += self.hl.numel() * 2 + self.hd.numel() * 4
            d2h += self.h_len.numel() * 4 + self.h_comm.numel() * 4
        return h2d, d2h

    def e2e(self):
        import torch
        cur = torch.cuda.current_stream(self.dev)
        if self.logits is not None:
            # the acceptance's inputs travel on a second stream while the layer runs
            if not hasattr(self, "copy_stream"):
                self.copy_stream = torch.cuda.Stream(self.dev)
            self.copy_stream.wait_stream(cur)
            with torch.cuda.stream(self.copy_stream):
                self.dl.copy_(self.hl, non_blocking=True)
                self.dd.copy_(self.hd, non_blocking=True)
        self.dx.copy_(self.hx, non_blocking=True)
        self._layers(self.dx)
        if self.logits is not None:
            cur.wait_stream(self.copy_stream)
            self.api.spec_verify_accept(self.dl, self.dd, self.aws, accept_len=self.alen, committed=self.comm)
            self.h_len.copy_(self.alen, non_blocking=True)
            self.h_comm.copy_(self.comm, non_blocking=True)
        self.h_out.copy_(self.out, non_blocking=True)


def greedy_row_check(device, min_gap=1e-3):
    """Input generation for the output-layer workload: the greedy tokens of the exact bf16 inputs by
    torch in fp32 (chunked over the vocabulary), and the rows whose top two logits are min_gap apart,
    so that the drafts can be planted with the pages' acceptances.  Plumbing for the synthetic
    inputs only: the timed path is the library's kernel, and parity lives in the tests."""
    import torch

    def row_check(hidden, w_vocab):
        h = torch.from_numpy(np.ascontiguousarray(hidden).view(np.int16)).view(torch.bfloat16).to(device).float()
        best = torch.full((h.shape[0], 2), -float("inf"), device=device)
        arg = torch.zeros(h.shape[0], dtype=torch.int64, device=device)
        for v0 in range(0, w_vocab.shape[0], 16384):
            w = torch.from_numpy(np.ascontiguousarray(w_vocab[v0:v0 + 16384]).view(np.int16)).view(torch.bfloat16)
            lg = h @ w.to(device).float().t()
            top = torch.topk(lg, 2, dim=1)
            cand = torch.cat([best, top.values], dim=1)
            new_best = torch.topk(cand, 2, dim=1).values
            arg = torch.where(top.values[:, 0] > best[:, 0], top.indices[:, 0] + v0, arg)
            best = new_best
        return arg.int().cpu().numpy(), (best[:, 0] - best[:, 1] >= min_gap).cpu().numpy()
    return row_check


class LmHeadStep:
    """Greedy verification with the logits made by the verifier's output layer inside the call
    (spec_verify_lmhead): 32 sequences x (K=3)+1 positions, hidden 1280, vocabulary 129,280.
    Same interface as DeviceStep; its `layer()` is empty."""

    B, K, V, H = 32, 3, 129_280, 1280

    def __init__(self, seed, dev):
        import torch
        from lossless_speculative_verification_gb300 import api, synth
        self.name, self.dev, self.api = "lmhead", dev, api
        self.w = None
        self.layers = []
        self.T = self.B * (self.K + 1)
        p = synth.lmhead_problem(self.B, self.K, V=self.V, H=self.H, seed=seed, row_check=greedy_row_check(dev))
        self.problem = p
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.hidden, self.w_vocab = t(p.hidden), t(p.w_vocab)
        self.drafts = torch.from_numpy(p.drafts).to(dev)
        self.ws = api.spec_verify_lmhead_workspace(self.B, self.K, self.V, self.H, dev)
        self.alen = torch.empty(self.B, dtype=torch.int32, device=dev)
        self.comm = torch.empty((self.B, self.K + 1), dtype=torch.int32, device=dev)
        self.launches = 2  # the fused output layer + greedy search, then the acceptance rule

    @classmethod
    def host_only(cls, seed):
        """The inputs on the host only (for the CPU oracle)."""
        from lossless_speculative_verification_gb300 import synth
        step = cls.__new__(cls)
        step.T = cls.B * (cls.K + 1)
        step.problem = synth.lmhead_problem(cls.B, cls.K, V=cls.V, H=cls.H, seed=seed, row_check=greedy_row_check("cpu"))
        return step

    def describe(self):
        return ("greedy verification of [%d,%d] positions with the logits made by the output layer [%d,%d] "
                "inside the call (B=%d, K=%d)" % (self.B, self.K + 1, self.V, self.H, self.B, self.K))

    def layer(self):
        pass

    def accept(self):
        self.api.spec_verify_lmhead(self.hidden, self.w_vocab, self.drafts, self.ws, self.K, accept_len=self.alen,
                                    committed=self.comm)

    def bytes_and_flops(self):
        byts = self.V * self.H * 2 + self.T * self.H * 2
        return byts, 2.0 * self.T * self.V * self.H, 0

    def setup_e2e(self):
        import torch
        self.h_hidden = self.hidden.cpu().pin_memory()
        self.h_drafts = self.drafts.cpu().pin_memory()
        self.d_hidden, self.d_drafts = torch.empty_like(self.hidden), torch.empty_like(self.drafts)
        self.h_len = torch.empty_like(self.alen, device="cpu").pin_memory()
        self.h_comm = torch.empty_like(self.comm, device="cpu").pin_memory()
        h2d = self.h_hidden.numel() * 2 + self.h_drafts.numel() * 4
        d2h = self.h_len.numel() * 4 + self.h_comm.numel() * 4
        return h2d, d2h

    def e2e(self):
        self.d_hidden.copy_(self.h_hidden, non_blocking=True)
        self.d_drafts.copy_(self.h_drafts, non_blocking=True)
        self.api.spec_verify_lmhead(self.d_hidden, self.w_vocab, self.d_drafts, self.ws, self.K,
                                    accept_len=self.alen, committed=self.comm)
        self.h_len.copy_(self.alen, non_blocking=True)
        self.h_comm.copy_(self.comm, non_blocking=True)


def lmhead_oracle_sampler(step):
    """The oracle's output layer (numpy fp64 matmul over the vocabulary, chunked) on whole
    positions, cycling over the batch, plus the acceptance rule of their sequences."""
    import oracle
    p = step.problem
    state = {"n": 0}

    def sample(seconds):
        n0 = state["n"]
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            r = state["n"] % step.T
            oracle.lmhead_argmax(p.hidden[r:r + 1], p.w_vocab)
            if r % (step.K + 1) == step.K:
                b = r // (step.K + 1)
                oracle.accept_from_greedy(p.greedy[b:b + 1], p.drafts[b:b + 1])
            state["n"] += 1
        dt = time.perf_counter() - t0
        n = state["n"] - n0
        return {"value": n / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                "kind": "oracle (numpy fp64 matmul; its BLAS may use every core)",
                "sample": "%d positions (cycling over the %d) through the oracle's output layer and greedy "
                          "search, plus the acceptance of their sequences, %.1f s" % (n, step.T, dt)}

    return sample


class AttentionStep:
    """Causal attention of the verified positions over their sequences' caches
    (spec_verify_attention): 32 sequences x (K=3)+1 positions, 10 heads x 128, page-shaped
    prefixes (visual tokens + the page's text so far).  Same interface as LmHeadStep."""

    B, Q, NH, D = 32, 4, 10, 128

    def __init__(self, seed, dev):
        import torch
        from lossless_speculative_verification_gb300 import api, synth
        self.name, self.dev, self.api = "attention", dev, api
        self.w = None
        self.layers = []
        self.T = self.B * self.Q
        p = self.problem = synth.attention_problem(self.B, self.Q, nh=self.NH, d=self.D, seed=seed)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.q, self.k_cache, self.v_cache = t(p.q), t(p.k_cache), t(p.v_cache)
        self.ctx_len = torch.from_numpy(p.ctx_len).to(dev)
        self.ws = api.spec_verify_attention_workspace(self.B, self.Q, p.L, self.NH, self.D, dev)
        self.out = torch.empty_like(self.q)
        self.launches = 2  # the persistent stream over the caches, then the merge of the splits

    @classmethod
    def host_only(cls, seed):
        from lossless_speculative_verification_gb300 import synth
        step = cls.__new__(cls)
        step.T = cls.B * cls.Q
        step.problem = synth.attention_problem(cls.B, cls.Q, nh=cls.NH, d=cls.D, seed=seed)
        return step

    def describe(self):
        p = self.problem
        return ("causal attention of [%d,%d] verified positions (%d heads x %d) over bf16 caches of %d..%d "
                "entries (mean %.0f, capacity %d)" % (self.B, self.Q, self.NH, self.D, p.ctx_len.min(),
                                                      p.ctx_len.max(), p.ctx_len.mean(), p.L))

    def layer(self):
        pass

    def accept(self):
        self.api.spec_verify_attention(self.q, self.k_cache, self.v_cache, self.ctx_len, self.ws, out=self.out)

    def bytes_and_flops(self):
        p = self.problem
        kv = int(p.ctx_len.astype(np.int64).sum()) * self.NH * self.D * 2 * 2
        byts = kv + 2 * self.T * self.NH * self.D * 2 + self.B * 4
        flops = 4.0 * self.Q * self.NH * self.D * float(p.ctx_len.astype(np.int64).sum())
        return byts, flops, 0

    def setup_e2e(self):
        import torch
        self.h_q = self.q.cpu().pin_memory()
        self.h_len = self.ctx_len.cpu().pin_memory()
        self.d_q, self.d_len = torch.empty_like(self.q), torch.empty_like(self.ctx_len)
        self.h_out = torch.empty_like(self.out, device="cpu").pin_memory()
        return self.h_q.numel() * 2 + self.h_len.numel() * 4, self.h_out.numel() * 2

    def e2e(self):
        self.d_q.copy_(self.h_q, non_blocking=True)
        self.d_len.copy_(self.h_len, non_blocking=True)
        self.api.spec_verify_attention(self.d_q, self.k_cache, self.v_cache, self.d_len, self.ws, out=self.out)
        self.h_out.copy_(self.out, non_blocking=True)


def attention_oracle_sampler(step):
    """The oracle's attention (numpy fp64 einsum) on whole sequences, cycling over the batch."""
    import oracle
    p = step.problem
    state = {"n": 0}

    def sample(seconds):
        n0 = state["n"]
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            b = state["n"] % p.B
            oracle.verify_attention(p.q[b:b + 1], p.k_cache[b:b + 1], p.v_cache[b:b + 1], p.ctx_len[b:b + 1],
                                    1.0 / np.sqrt(p.d))
            state["n"] += 1
        dt = time.perf_counter() - t0
        n = state["n"] - n0
        return {"value": n * p.Q / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                "kind": "oracle (numpy fp64 einsum; its BLAS may use every core)",
                "sample": "%d sequences x %d verified positions (cycling over the %d) through the oracle's "
                          "attention, %.1f s" % (n, p.Q, p.B, dt)}

    return sample


class DraftStep:
    """K = 3 recursive applications of the FastMTP draft block to 32 sequences (spec_draft_loop):
    hidden 1280 (10 heads x 128), FFN 7,168, vocabulary 129,280, block caches with the page
    lengths.  The unit is a drafted token (B x K per step)."""

    B, K, H, NH, I, V = 32, 3, 1280, 10, 7168, 129_280

    def __init__(self, seed, dev):
        import torch
        from lossless_speculative_verification_gb300 import api, synth
        self.name, self.dev, self.api = "draft", dev, api
        self.w = None
        self.layers = []
        self.T = self.B * self.K
        p = self.problem = synth.draft_problem(self.B, K=self.K, H=self.H, nh=self.NH, I=self.I, V=self.V, seed=seed)
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
        self.weights = {n: t(p.weights[n]) for n in api.DRAFT_WEIGHTS}
        self.h0, self.k_cache, self.v_cache = t(p.h0), t(p.k_cache), t(p.v_cache)
        self.t0 = torch.from_numpy(p.t0).to(dev)
        self.ctx_len = torch.from_numpy(p.ctx_len).to(dev)
        self.ws = api.spec_draft_workspace(self.B, self.H, self.NH, self.I, self.V, p.L, dev)
        self.drafts = None
        # per step: input norms + W_p + norm + q/k/v + append + attention (2) + W_o + residual norm
        # + gate/up (SwiGLU) + down + residual norm + output layer (2) = 14 kernels, plus the copy of
        # the tokens
        self.launches = 11 * self.K

    @classmethod
    def host_only(cls, seed):
        from lossless_speculative_verification_gb300 import synth
        step = cls.__new__(cls)
        step.T = cls.B * cls.K
        step.problem = synth.draft_problem(cls.B, K=cls.K, H=cls.H, nh=cls.NH, I=cls.I, V=cls.V, seed=seed)
        return step

    def describe(self):
        p = self.problem
        return ("%d recursive draft-block steps for %d sequences: hidden %d (%d heads), FFN %d, vocabulary %d, "
                "block caches of %d..%d entries" % (self.K, self.B, self.H, self.NH, self.I, self.V,
                                                    p.ctx_len.min(), p.ctx_len.max()))

    def layer(self):
        pass

    def accept(self):
        self.drafts = self.api.spec_draft_loop(self.weights, self.h0, self.t0, self.k_cache, self.v_cache,
                                               self.ctx_len, self.K, self.ws)

    def bytes_and_flops(self):
        p = self.problem
        H, I, V = self.H, self.I, self.V
        weights = (2 * H * H + 4 * H * H + 3 * H * I + V * H) * 2        # per step
        cache = int((p.ctx_len.astype(np.int64) + 1).sum()) * H * 2 * 2   # keys and values read per step
        byts = self.K * (weights + cache)
        flops = 2.0 * self.B * self.K * (weights / 2)
        return byts, flops, 0

    def setup_e2e(self):
        import torch
        self.h_h0 = self.h0.cpu().pin_memory()
        self.h_t0 = self.t0.cpu().pin_memory()
        self.d_h0, self.d_t0 = torch.empty_like(self.h0), torch.empty_like(self.t0)
        self.h_drafts = torch.empty((self.B, self.K), dtype=torch.int32).pin_memory()
        return self.h_h0.numel() * 2 + self.h_t0.numel() * 4, self.h_drafts.numel() * 4

    def e2e(self):
        self.d_h0.copy_(self.h_h0, non_blocking=True)
        self.d_t0.copy_(self.h_t0, non_blocking=True)
        d = self.api.spec_draft_loop(self.weights, self.d_h0, self.d_t0, self.k_cache, self.v_cache, self.ctx_len,
                                     self.K, self.ws)
        self.h_drafts.copy_(d, non_blocking=True)


def draft_oracle_sampler(step):
    """The oracle's draft loop (numpy fp64) on one sequence at a time, cycling over the batch."""
    import oracle
    from lossless_speculative_verification_gb300 import synth
    p = step.problem
    state = {"n": 0}

    def sample(seconds):
        n0 = state["n"]
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            b = state["n"] % p.B
            kc = synth.bf16_value(p.k_cache[b:b + 1]).astype(np.float64)
            vc = synth.bf16_value(p.v_cache[b:b + 1]).astype(np.float64)
            oracle.draft_loop(p.h0[b:b + 1], p.t0[b:b + 1], p.weights, kc, vc, p.ctx_len[b:b + 1], p.nh, p.K)
            state["n"] += 1
        dt = time.perf_counter() - t0
        n = state["n"] - n0
        return {"value": n * p.K / dt, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                "kind": "oracle (numpy fp64; its BLAS may use every core)",
                "sample": "%d sequences x %d drafted tokens (cycling over the %d) through the oracle's draft loop, "
                          "%.1f s" % (n, p.K, p.B, dt)}

    return sample


# workloads outside the MoE layer: name -> (step class, oracle sampler)
SIDE_STEPS = {"lmhead": (LmHeadStep, lmhead_oracle_sampler), "attention": (AttentionStep, attention_oracle_sampler),
              "draft": (DraftStep, draft_oracle_sampler)}


def flush_l2(flush, i):
    """Evict the step's data from L2: write a buffer larger than L2, then read it back, so that the
    L2 holds only clean lines of the flush buffer and the step pays no write-back of them."""
    import torch
    flush.fill_(i & 0xFF)
    torch.amax(flush.view(torch.int32))


def measure(step, args, local, world, flush, dist):
    """Warm up, time `steps` graph replays (L2 flushed before each), then the e2e path."""
    import torch
    api = step.api
    stream = torch.cuda.current_stream(step.dev)
    for _ in range(max(args.warmup, 0)):
        step.layer()
        step.accept()
    torch.cuda.synchronize()
    assert api.get_device_error() == 0

    eager_ms = []
    for i in range(min(args.steps, 10)):
        flush_l2(flush, i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step.layer()
        step.accept()
        b.record(stream)
        b.synchronize()
        eager_ms.append(a.elapsed_time(b))

    # The step as one CUDA graph with its timing events recorded as graph nodes.  The step time
    # comes from a graph with events at its start and end only; the layer/acceptance split (for
    # the roofline) from replays of a second graph with one more event between the two, which
    # costs the acceptance its programmatic early launch.  Where torch cannot record events
    # inside a graph: two graphs with events between them.
    try:
        evs = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(5)]
        one_graph = True
    except TypeError:
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        one_graph = False
    if one_graph:
        g_step, g_split = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step):
            evs[0].record()
            step.layer()
            step.accept()
            evs[1].record()
        with torch.cuda.graph(g_split):
            evs[2].record()
            step.layer()
            evs[3].record()
            step.accept()
            evs[4].record()
        graphs = [g_step, g_split]
    else:
        graphs = [torch.cuda.CUDAGraph() for _ in range(2)]
        for g, fn in zip(graphs, (step.layer, step.accept)):
            with torch.cuda.graph(g):
                fn()

    def replay(split):
        if one_graph:
            graphs[1 if split else 0].replay()
        else:
            evs[2].record(stream)
            graphs[0].replay()
            evs[3].record(stream)
            graphs[1].replay()
            evs[4].record(stream)

    for _ in range(max(args.warmup, 0)):
        replay(False)
        replay(True)
    torch.cuda.synchronize()
    assert api.get_device_error() == 0

    step_ms, layer_list, accept_list = [], [], []
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the sampler polls every 100 ms: keep the GPU in the same back-to-back load for a
        # moment before and after the timed steps so that its samples describe them
        clk.wait_first_sample()
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            flush_l2(flush, 0)
            replay(False)
        torch.cuda.synchronize()
        for i in range(args.steps):
            flush_l2(flush, i)
            replay(not one_graph)
            if one_graph:
                evs[1].synchronize()
                step_ms.append(evs[0].elapsed_time(evs[1]))
            else:
                evs[4].synchronize()
                step_ms.append(evs[2].elapsed_time(evs[4]))
        for i in range(args.steps):
            flush_l2(flush, i)
            replay(True)
            evs[4].synchronize()
            layer_list.append(evs[2].elapsed_time(evs[3]))
            accept_list.append(evs[3].elapsed_time(evs[4]))
        t_end = time.perf_counter() + 0.3
        while time.perf_counter() < t_end:
            flush_l2(flush, 0)
            replay(False)
        torch.cuda.synchronize()
    assert api.get_device_error() == 0
    total_ms = sum(step_ms)
    layer_ms = statistics.mean(layer_list)
    accept_ms = statistics.mean(accept_list)

    h2d, d2h = step.setup_e2e()
    for _ in range(max(args.warmup, 1)):
        step.e2e()
    torch.cuda.synchronize()
    e2e_total = 0.0
    for i in range(args.steps):
        flush_l2(flush, i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        step.e2e()
        b.record(stream)
        b.synchronize()
        e2e_total += a.elapsed_time(b)
    assert api.get_device_error() == 0
    if world > 1:
        total_ms, e2e_total = max_over_ranks([total_ms, e2e_total], dist, step.dev)
    return dict(total_ms=total_ms, layer_ms=layer_ms, accept_ms=accept_ms, eager_ms=statistics.mean(eager_ms),
                e2e_total=e2e_total, h2d=h2d, d2h=d2h, clocks=clk.summary(), one_graph=one_graph)


def max_over_ranks(values, dist, device):
    """Element-wise maximum of the ranks' values (the job's time is its slowest replica's)."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def committed_tokens_per_s(accept_len, world, steps, total_ms):
    """The secondary figure: tokens the step commits (each sequence's accepted drafts plus its
    correction or bonus token, sum(accept_len + 1)) per second over the whole job; None when
    the step has no acceptance."""
    if accept_len is None:
        return None
    a = np.asarray(accept_len, dtype=np.int64)
    return float((a + 1).sum()) * world * steps / (total_ms / 1e3)


def job_tokens_per_s(tokens_per_step, world, steps, total_ms):
    """Whole-job throughput: every replica's verified positions over the slowest replica's time."""
    return tokens_per_step * world * steps / (total_ms / 1e3)


def result_line(args, step, m, world, cpu):
    hbm, tflops, peak_src = peaks()
    w = step.w
    byts, flops, acc_bytes = step.bytes_and_flops()
    khash = layer_source_hash(step.name)
    if step.name in SIDE_STEPS:
        achieved = byts / (m["total_ms"] / args.steps / 1e3) / 1e9
        kernel = ("lmhead_argmax_kernel (tcgen05 product of the output layer and the hidden rows, reduced "
                  "to each row's (max, first index) per 176-row vocabulary tile) + accept_finalize_kernel"
                  if step.name == "lmhead" else
                  "attn_split_kernel (persistent: TMA key/value tiles, warp MMAs for scores and weighted values, "
                  "online softmax in fp32, one state per 256-position split) + attn_combine_kernel"
                  if step.name == "attention" else
                  "spec_draft_loop: 11 launches per step (skinny_gemm_kernel split-K projections with q/k/v in "
                  "one launch and the SwiGLU FFN in two, the RMSNorms and residual adds folded into them, "
                  "attention, fused output-layer argmax)")
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "algorithmic_bytes": byts, "algorithmic_flops": flops, "kernel": kernel,
                "peak_source": peak_src, "traffic": ncu_traffic(step.name, khash), "kernel_source_hash": khash}
        if step.name == "draft" and roof["traffic"] is not None:
            roof["traffic"] *= step.K   # the capture sums one recursion step; a launch of the loop runs K

    elif step.name == "prefill":
        achieved = flops / (m["layer_ms"] / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": tflops, "unit": "TFLOP/s", "frac": achieved / tflops,
                "algorithmic_flops": flops}
    else:
        achieved = byts / (m["layer_ms"] / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "algorithmic_bytes": byts}
    if step.name not in SIDE_STEPS:
        roof.update({"kernel": "moe_verify_layer x%d: router, permute+gather, grouped SwiGLU experts (tcgen05), "
                               "combine; one PDL-chained launch sequence per layer" % len(step.layers),
                     "peak_source": peak_src, "traffic": ncu_traffic(step.name, khash), "layer_ms": m["layer_ms"],
                     "kernel_source_hash": khash})
    if acc_bytes:
        # "ms": the acceptance launches between two events (the event costs them their early launch);
        # "in_step_ms": what they add to the step, the step time less the layer's
        in_step = m["total_ms"] / args.steps - m["layer_ms"]
        roof["accept"] = {"ms": m["accept_ms"], "algorithmic_bytes": acc_bytes,
                          "achieved_gbs": acc_bytes / (m["accept_ms"] / 1e3) / 1e9,
                          "in_step_ms": in_step,
                          "in_step_gbs": acc_bytes / (in_step / 1e3) / 1e9 if in_step > 0 else None}
    tokens = step.T * world * args.steps
    line = {
        "metric": METRIC, "value": job_tokens_per_s(step.T, world, args.steps, m["total_ms"]), "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["total_ms"] / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": "%s: %s" % (step.name, describe(w, len(step.layers)) if w is not None else
                                           step.describe()),
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "flushed before every timed step (256 MB written, then read back, outside the events)",
                   "timing": ("step replayed as one CUDA graph with CUDA events recorded as graph nodes at its "
                              "start and end; the layer/acceptance split from K more replays of the same step "
                              "with an event between them" if m["one_graph"] else
                              "step replayed as 2 CUDA graphs (layers, acceptance); CUDA events per step"),
                   "clocks_window": "nvidia-smi every 100 ms over back-to-back steps around the timed ones",
                   "eager_ms_per_step": m["eager_ms"]},
        "roofline": roof,
        "e2e": {"value": tokens / (m["e2e_total"] / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": m["h2d"],
                "d2h_bytes_per_step": m["d2h"]},
        "committed_tokens_per_s": committed_tokens_per_s(
            step.alen.cpu().numpy() if getattr(step, "alen", None) is not None else None, world, args.steps,
            m["total_ms"]),
        "gpu_launches": step.launches * args.steps,
        "clocks": m["clocks"],
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def workloads(name):
    from lossless_speculative_verification_gb300 import synth
    if name in SIDE_STEPS:
        return [(name, None, 0)]
    if name == "sweep":
        return [("sweep", synth.sweep_workload(B, K), synth.sweep_seed(B, K))
                for B in synth.SWEEP_B for K in synth.SWEEP_K]
    return [(name, synth.WORKLOADS[name], 0)]


# ----------------------------------------------------------------------------- CPU oracle (baseline and reference arm)
def oracle_sampler(w, seed):
    """The oracle as it stands, single-threaded, on a bounded sample of the workload: whole tokens
    through every layer (and the acceptance of their sequences), cycling over the batch.  Returns
    sample(seconds) -> cpu_baseline dict; the inputs are generated once, outside any timing."""
    import oracle
    from lossless_speculative_verification_gb300 import synth
    oracle.build()
    d = w.dims
    if w.layers > 1:
        st = synth.stack_problem(w, seed=seed)
        layers, xs, hs = st["layers"], st["x0"], st["h0"]
    else:
        prob = synth.moe_problem(w, seed=seed)
        layers = [dict(w_router=prob.w_router, w_gate_up=prob.w_gate_up, w_down=prob.w_down,
                       ws_gate_up=prob.ws_gate_up, ws_down=prob.ws_down)]
        xs = hs = prob.x
    logits = drafts = None
    if w.V:
        logits, planted, drafts = synth.verify_problem(w, seed=seed)
    state = {"n": 0}

    def sample(seconds):
        n0 = state["n"]
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < seconds:
            t = state["n"] % d.T
            x, h = xs[t:t + 1], hs[t:t + 1]
            for L in layers:
                out, _, _ = oracle.moe_layer(h, L["w_router"], L["w_gate_up"], L["w_down"], L["ws_gate_up"],
                                             L["ws_down"], d.k, d.S)
                if len(layers) > 1:
                    xn, hn = oracle.rmsnorm_residual(x, synth.bf16_bits(out.astype(np.float32)))
                    x, h = synth.bf16_bits(xn.astype(np.float32)), synth.bf16_bits(hn.astype(np.float32))
            if logits is not None and t % (w.K + 1) == 0:
                b = t // (w.K + 1)
                oracle.accept(logits[b:b + 1], drafts[b:b + 1])
            state["n"] += 1
        dt = time.perf_counter() - t0
        n = state["n"] - n0
        return {"value": n / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                "sample": "%d token passes (cycling over the %d tokens) through %d oracle layer(s)%s, %.1f s"
                          % (n, d.T, len(layers), " plus the acceptance of their sequences" if w.V else "", dt)}

    return sample


def k_policy_line(step_ms):
    """Per batch size, the number of drafts the library's policy picks from the measured verify
    step times (K = 0 is the plain greedy step) and the pages' conditional acceptances."""
    from lossless_speculative_verification_gb300 import api, synth
    out = {}
    for B in sorted({b for b, _ in step_ms}):
        ks = sorted(k for b, k in step_ms if b == B)
        if ks != list(range(len(ks))) or len(ks) < 2:
            continue
        cost = [step_ms[(B, k)] for k in ks]
        a = list(synth.PAGE_ACCEPT[:len(ks) - 1])
        k_best, tau, sp = api.spec_k_policy(a, cost)
        out[str(B)] = {"step_ms": cost, "tau": [round(x, 4) for x in tau], "speedup": [round(x, 4) for x in sp],
                       "k_best": k_best}
    return {"metric": "k_policy", "note": "cost = one verify step of the MoE layer plus acceptance (no draft "
            "block, no attention); acceptances 0.830/0.663/0.636 from the pages", "per_batch": out}


def run_spec(args, rank, world, local, dev, flush):
    """Speculative step costs t(B, K) (drafting + verify pass) and the K policy on them."""
    import torch
    from lossless_speculative_verification_gb300 import api, synth
    from lossless_speculative_verification_gb300.decoder import Decoder
    n_layers = 11
    dims = synth._verify_dims(1, 0)
    prob = synth.decoder_problem(n_layers, dims, V=synth.VOCAB, seed=args.seed + 1000 * rank)
    Bmax, Qmax = max(synth.SWEEP_B), max(synth.SWEEP_K) + 1
    L = synth.page_cache_capacity(Qmax)
    dec = Decoder(prob, Bmax, L, dev)
    dec.fill_caches(args.seed + 5)
    rs = synth.streams(args.seed + 77, 4)
    ctx0 = synth.page_context_lengths(rs[0], Bmax, 0)                 # the prefix before the verified positions
    g = torch.Generator(device=dev).manual_seed(args.seed + 9)
    dk = torch.randn((Bmax, L, dec.nh, dec.hd), generator=g, device=dev).to(torch.bfloat16)
    dv = torch.randn_like(dk)
    h_all = torch.from_numpy(synth.hidden_rows(rs[1], Bmax, dec.H, "sphere").view(np.int16)).view(torch.bfloat16).to(dev)
    tok_all = torch.from_numpy(rs[2].integers(0, dec.V, size=(Bmax, Qmax)).astype(np.int32)).to(dev)
    stream = torch.cuda.current_stream(dev)
    step_ms, draft_ms = {}, {}
    for B in synth.SWEEP_B:
        dws = api.spec_draft_workspace(B, dec.H, dec.nh, prob.I_draft, dec.V, L, dev)
        dctx = torch.from_numpy(ctx0[:B].astype(np.int32)).to(dev)
        for K in synth.SWEEP_K:
            Q = K + 1
            tokens = tok_all[:B, :Q].contiguous()                   # the verify pass's inputs (their values
            ctx_after = dctx + Q                                      # do not change the work)
            dr = torch.zeros((B, K), dtype=torch.int32, device=dev)
            h0, t0 = h_all[:B].contiguous(), tokens[:, 0].contiguous()

            def draft():
                if K:
                    api.spec_draft_loop(dec.draft_w, h0, t0, dk[:B], dv[:B], dctx, K, dws, out=dr)

            def step():
                draft()
                dec.verify(tokens, ctx_after, dr)

            for _ in range(max(args.warmup, 1)):
                step()
            torch.cuda.synchronize()
            graphs = []
            for fn in (step, draft):
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr):
                    fn()
                graphs.append(gr)
            for gr in graphs:
                gr.replay()
            torch.cuda.synchronize()
            assert api.get_device_error() == 0
            times = {0: [], 1: []}
            with ClockSampler(local) as clk:
                clk.wait_first_sample()
                for which in (0, 1):
                    if which == 1 and K == 0:
                        continue
                    for i in range(args.steps):
                        flush_l2(flush, i)
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                        a.record(stream)
                        graphs[which].replay()
                        b.record(stream)
                        b.synchronize()
                        times[which].append(a.elapsed_time(b))
            assert api.get_device_error() == 0
            t_step = statistics.median(times[0])
            t_draft = statistics.median(times[1]) if K else 0.0
            step_ms[(B, K)], draft_ms[(B, K)] = t_step, t_draft
            tau = float(api.spec_k_policy(list(synth.PAGE_ACCEPT[:K]) or [0.0], [1.0] * (K + 1) if K else [1.0, 1.0])[1][K])
            launches = dec.launches_per_verify(B, Q) + 11 * K
            if rank == 0:
                print(json.dumps({
                    "metric": "speculative step: %d-layer verify pass over B x (K+1) positions after K draft-block "
                              "steps" % n_layers,
                    "value": B * Q / (t_step / 1e3), "unit": "verified tokens/s", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
                    "dtype": "bf16", "data": "synthetic",
                    "config": {"workload": "spec: B=%d, K=%d; %d layers (attention 10x128 over page-shaped caches "
                                           "+ MoE H=1280, E=64 top-6, S=2, I=896), output layer [129280,1280] fused "
                                           "with acceptance; draft block FFN 7168" % (B, K, n_layers),
                               "l2": "flushed before every timed step",
                               "timing": "median of CUDA-graph replays, CUDA events"},
                    "draft_ms": t_draft, "verify_ms": t_step - t_draft,
                    "expected_committed_tokens_per_s": B * tau / (t_step / 1e3),
                    "gpu_launches": launches * args.steps, "clocks": clk.summary()}), flush=True)
            del graphs
        del dws
        torch.cuda.empty_cache()
    if rank == 0:
        out = {}
        for B in synth.SWEEP_B:
            cost = [step_ms[(B, k)] for k in synth.SWEEP_K]
            k_best, tau, sp = api.spec_k_policy(list(synth.PAGE_ACCEPT), cost)
            out[str(B)] = {"step_ms": [round(c, 4) for c in cost], "draft_ms": [round(draft_ms[(B, k)], 4)
                                                                              for k in synth.SWEEP_K],
                           "tau": [round(x, 4) for x in tau], "speedup": [round(x, 4) for x in sp], "k_best": k_best}
        print(json.dumps({"metric": "k_policy", "note": "cost = one speculative step: K draft-block steps + the "
                          "verify pass of an 11-layer decoder (attention + MoE per layer, output layer fused with "
                          "acceptance) over K+1 positions; acceptances 0.830/0.663/0.636 from the pages",
                          "per_batch": out}), flush=True)


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload == "spec":
        print(json.dumps({"impl": "reference", "workload": "spec",
                          "unavailable": "no bounded oracle sample of the 11-layer speculative step (the oracle takes "
                                         "minutes per step); the component workloads carry the oracle baselines"}))
        return
    for name, w, seed in workloads(args.workload):
        per_step = 2.0 if name != "sweep" else 0.5       # seconds of oracle work per timed step
        if name in SIDE_STEPS:
            cls, sampler = SIDE_STEPS[name]
            step = cls.host_only(seed + args.seed)
            sample = sampler(step)
            w_desc = step.describe()
        else:
            sample = oracle_sampler(w, seed + args.seed)
            w_desc = describe(w, w.layers)
        sample(0.2 * max(args.warmup, 1))                # warm-up
        t0 = time.perf_counter()
        res = sample(per_step * args.steps)
        dt = time.perf_counter() - t0
        line = {
            "impl": "reference", "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "%s: %s" % (name, w_desc), "l2": "n/a (CPU)"},
            "cpu_baseline": res,
            "e2e": {"value": res["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        }
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch
    from lossless_speculative_verification_gb300 import _build
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or not os.path.exists(_build.LIB):
        _build.build()
    if world > 1:
        dist.barrier()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    if args.workload == "spec":
        run_spec(args, rank, world, local, dev, flush)
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return
    step_ms = {}
    for name, w, seed in workloads(args.workload):
        if name in SIDE_STEPS:
            step = SIDE_STEPS[name][0](seed + args.seed + 1000 * rank, dev)
        else:
            step = DeviceStep(name, w, seed + args.seed + 1000 * rank, dev)
        m = measure(step, args, local, world, flush, dist)
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            sampler = SIDE_STEPS[name][1](step) if name in SIDE_STEPS else oracle_sampler(w, seed + args.seed)
            cpu = sampler(12.0 if args.workload != "sweep" else 2.0)
        if rank == 0:
            print(json.dumps(result_line(args, step, m, world, cpu)), flush=True)
        if name == "sweep":
            step_ms[(w.B, w.K)] = m["total_ms"] / args.steps
        del step
        torch.cuda.empty_cache()
    if rank == 0 and step_ms:
        print(json.dumps(k_policy_line(step_ms)), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def main():
    args = parse()
    if args.record_traffic:
        record_traffic(args)
        return
    rank, world, local = dist_env()
    if args.warmup < 0 or args.steps <= 0:
        raise SystemExit("steps must be positive")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
