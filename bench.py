#!/usr/bin/env python
"""Benchmark: GDN chunked-prefill forward + backward through the C ABI.

One step = gdr_fwd (o, final_state, A) followed by gdr_bwd (dq, dk, dv, dbeta,
dg, dh0) over one synthetic batch: every step of the hot path.  The default
workload is the largest one, the training case B=2, T=16384, Hq=32, Hv=64,
K=V=128 (bf16 q/k/v, fp32 g/beta, 30% of v-heads with g == 0, h0 ~ N(0, 0.1),
do ~ N(0, 1), dht ~ N(0, 0.1)).  The same line carries, under
``fwd_workloads``, the forward alone on the long-context case (B=1, T=262144,
Hq=8, Hv=16, o fp32) and the 4-sequence varlen case (Hq=16, Hv=32), each with
the context-parallel warm-up starts the planner chose and, beside it, with the
exact split only (cp_warmup = -1).

Timing: W untimed warm-up steps, then K steps bracketed by a barrier and
torch.cuda.synchronize() on both sides; each step is timed with CUDA events on
the launching stream after an L2 flush (a 256 MiB write), and the value is the
tokens of all ranks divided by the slowest rank's summed step time.  K more
steps follow with every kernel bracketed by caller-owned events
(gdr_opts.events; kept out of the timed steps, whose time the extra event
records would inflate): the dominant kernel's algorithmic work over its
measured duration gives the roofline fraction, and their launch count (the
same calls as the K timed steps) is gpu_launches, the count over the K steps.

``--impl reference`` times the fp64 CPU oracle (the pages ship no code to
run, so the oracle is the reference arm) on a bounded sample of the same
workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "GDN chunked-prefill fwd/bwd Mtokens/s at 1 GB300; % of bf16 roofline"
DEFAULT_WORKLOAD = "bwd_bf16_B2_T16384_hq32_hv64_d128"
FWD_EXTRAS = ("fwd_bf16_T262144_hq8_hv16_d128", "fwd_bf16_varlen4_hq16_hv32_d128")
FLUSH_BYTES = 256 << 20


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            pk = json.load(f)
        return {"hbm_gbs": pk["hbm_gbs"], "bf16_tflops": pk["bf16_tflops"],
                "bf16_tflops_sustained": pk.get("bf16_tflops_sustained", pk["bf16_tflops"]),
                "sm_max_mhz": pk.get("sm_max_mhz", 2070.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0,
            "source": "fallback"}


# ---------------------------------------------------------------------------
# algorithmic work per kernel launch (inputs read once, outputs written once)
# ---------------------------------------------------------------------------
C = 64


def kernel_work(name, spec, in_bytes, o_bytes, nchunk_heads, with_A=True):
    """(flops, bytes) of one launch of kernel `name` over the whole problem
    (`with_A`: the forward's chunk kernel writes A for a backward).

    Unit: one (chunk, v-head) pair of C = 64 tokens.  Flops count the dense
    contractions the kernel's step of the method needs (2 per MAC, causal
    products halved), not the extra terms of split operands; bytes count its
    inputs read once and outputs written once (the workspace tiles it passes to
    the next kernel are not algorithmic).  Overhead kernels (the context-parallel
    summaries and combines, the tables, the group sums) count zero."""
    K, V, Hv, Hq = spec.K, spec.V, spec.Hv, spec.Hq
    G = Hv // Hq
    th = spec.tokens * Hv                      # token-heads
    qk = spec.tokens * Hq * K * in_bytes       # one of q or k
    vv = spec.tokens * Hv * V * in_bytes       # one of v, o (input dtype) or do
    gb = spec.tokens * Hv * 4                  # one of g, beta, dg, dbeta
    A = spec.tokens * Hv * C * 4
    st = spec.n_seqs * Hv * K * V * 4          # one state tensor
    n = nchunk_heads
    mac = {
        # [K;Q] K^T (shared by the group), the triangular inverse
        "chunk": n * (2 * C * C * K / G + C ** 3 / 3),
        # K S0, Q S0, K^T Y; A R; P Ut (causal)
        "scan": n * (3 * C * K * V + C * C * V + C * C * V / 2),
        "scan_states": n * (2 * C * K * V + C * C * V),
        # dS1 K^T, X [Q ; K]; dO^T P (causal); dUt A
        "dh": n * (3 * C * K * V + C * C * V / 2 + C * C * V),
        # K S0, dO S0^T, dKS S0^T, Y dS1^T; A R, A^T dUt, dUt R^T, dO Y^T;
        # Q K^T, K K^T, dP'' K, dP''^T Q, MM K, MM^T K; A^T dA A^T
        "bwd_chunk": n * (4 * C * K * V + 3.5 * C * C * V + 6 * C * C * K + 2 * C ** 3),
    }
    byt = {
        "chunk": 2 * qk + 2 * gb + (A if with_A else 0),
        "chunk_from_A": 2 * qk + 2 * gb + A,
        "scan": 2 * qk + vv + th * V * o_bytes + st,
        "scan_states": qk + vv,
        "dh": 2 * qk + vv + 2 * st,
        "bwd_chunk": 2 * qk + 2 * vv + A + 2 * gb + (2 * qk + vv) + 2 * gb,
    }
    raw = name.split("_", 1)[1] if name.startswith(("tc_", "mma_", "simt_")) else name
    from_A = raw in ("chunk_from_A", "wy_from_A")  # the backward's pass reads A
    base = {"chunk_from_A": "chunk", "wy": "chunk", "wy_from_A": "chunk"}.get(raw, raw)
    if base in mac:
        return 2.0 * mac[base], float(byt["chunk_from_A" if from_A else base])
    return 0.0, 0.0


# DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum) from one
# ncu capture of the kernel on the workload; an entry is removed whenever the
# kernel changes (the summaries under profiles/ give the commands).
TRAFFIC = {
    ("tc_bwd_chunk", "bwd_bf16_B2_T16384_hq32_hv64_d128"): 7.54e9 + 2.14e9,
}


# ---------------------------------------------------------------------------
# clocks sampler
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0, t1):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = [l for (ts, l) in self.lines if t0 - 0.15 <= ts <= t1 + 0.15] or [l for (_, l) in self.lines]
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the CPU oracle arm
# ---------------------------------------------------------------------------
def oracle_sample(x, spec, t_sample, heads_sample, nthreads=None):
    """Run the fp64 oracle forward+backward on the first t_sample tokens of the
    first sequence, over the first `heads_sample` qk-heads and their v-heads.
    Returns (full-workload Mtokens/s, seconds, tokens, threads)."""
    import oracle
    G = spec.Hv // spec.Hq
    hq = slice(0, heads_sample)
    hv = slice(0, heads_sample * G)
    T = min(t_sample, spec.T if spec.lengths is None else spec.lengths[0])
    q = x["q"][:1, :T, hq]
    k = x["k"][:1, :T, hq]
    v = x["v"][:1, :T, hv]
    g = x["g"][:1, :T, hv]
    beta = x["beta"][:1, :T, hv]
    h0 = None if x["h0"] is None else x["h0"][:1, hv]
    do = x["do"][:1, :T, hv]
    dht = x["dht"][:1, hv]
    nthreads = nthreads or os.cpu_count() or 1
    t0 = time.perf_counter()
    oracle.fwd(q, k, v, g, beta, x["scale"], h0=h0, nthreads=nthreads, vblock=16)
    oracle.bwd(q, k, v, g, beta, x["scale"], do, dht=dht, h0=h0, nthreads=nthreads)
    dt = time.perf_counter() - t0
    # throughput in full-workload tokens: each token carries Hv heads of work
    eq_tokens = T * (heads_sample * G) / spec.Hv
    return eq_tokens / dt / 1e6, dt, T, nthreads


def run_reference(args, spec, rank, world):
    """The oracle as it stands on the host cores: each step one bounded sample
    (the first --ref-tokens tokens of sequence 0, every v-head) of the workload."""
    from gated_deltanet_chunked_delta_gb300 import inputs
    if rank != 0:
        return
    x = inputs.make(spec, seed=0)
    import oracle
    oracle.build()
    t_sample, heads = args.ref_tokens, spec.Hq
    vals, secs = [], []
    for i in range(args.warmup + args.steps):
        v, dt, T, nth = oracle_sample(x, spec, t_sample, heads)
        if i >= args.warmup:
            vals.append(v)
            secs.append(dt)
    value = statistics.mean(vals)
    line = {"metric": METRIC, "impl": "reference", "value": value, "unit": "Mtokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(secs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(spec, args),
            "ms_per_full_step_extrapolated": spec.tokens / (value * 1e6) * 1e3,
            "cpu_baseline": {"value": value, "unit": "Mtokens/s", "cores": nth, "kind": "oracle",
                             "sample": f"each step: oracle fwd+bwd on tokens [0,{T}) of sequence 0, all {spec.Hv} "
                                       f"v-heads; ms_per_step is that sample's time, value its throughput in "
                                       f"full-workload tokens"},
            "e2e": {"value": value, "unit": "Mtokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def aggregate(total_ms, tokens, steps, device):
    """Whole-job throughput over ranks: the slowest rank's summed step time and
    the tokens of all ranks.  Returns (Mtokens/s, max total ms)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([float(total_ms)], dtype=torch.float64, device=device)
        n = torch.tensor([float(tokens)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        total_ms, tokens = float(t.item()), float(n.item())
    return tokens * steps / (total_ms / 1e3) / 1e6, total_ms


STEP_DESC = {"both": "gdr_fwd(o, final_state, A) + gdr_bwd(dq, dk, dv, dbeta, dg, dh0)",
             "fwd": "gdr_fwd(o, final_state)",
             "bwd": "gdr_bwd(dq, dk, dv, dbeta, dg, dh0)"}


def _config(spec, args, mode=None):
    return {"workload": spec.name, "B": spec.B, "T": spec.T, "Hq": spec.Hq, "Hv": spec.Hv, "K": spec.K,
            "V": spec.V, "lengths": list(spec.lengths) if spec.lengths else None,
            "in_dtype": spec.in_dtype, "o_dtype": spec.out_dtype,
            "step": STEP_DESC[mode or getattr(args, "mode", "both")],
            "l2": f"flushed before every timed step ({FLUSH_BYTES >> 20} MiB write)",
            "parallelism": f"independent replicas x{args.gpus} (no collective)"}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
class Workload:
    """Device inputs, outputs and workspaces of one workload, and its step."""

    def __init__(self, gdr, spec, mode, dev, path, cp, cp_warmup=0):
        self.gdr, self.spec, self.mode, self.path, self.cp, self.cp_warmup = gdr, spec, mode, path, cp, cp_warmup
        x = inputs_make(spec)
        self.x = x
        keys = ("q", "k", "v", "g", "beta", "h0", "do", "dht", "cu_seqlens")
        self.d = d = {k: (x[k].to(dev) if torch.is_tensor(x.get(k)) else None) for k in keys}
        self.cu_host = x["cu_seqlens"]
        o_dtype = torch.float32 if spec.out_dtype == "f32" else torch.bfloat16
        self.prob = prob = gdr.Problem(d["q"], d["v"], d["cu_seqlens"], self.cu_host)
        self.opts = opts = gdr.make_opts(cp, path, cp_warmup=cp_warmup)
        self.plan = gdr.get_plan(prob, gdr.GDR_BF16 if spec.in_dtype == "bf16" else gdr.GDR_F32, opts)
        self.ws_f = gdr.alloc_workspace(gdr.fwd_workspace_size(prob, opts), dev)
        self.ws_b = gdr.alloc_workspace(gdr.bwd_workspace_size(prob, opts), dev) if mode != "fwd" else None
        N, B, T, Hv, K, V = prob.N, spec.B, spec.T, spec.Hv, spec.K, spec.V
        # A is written only where a backward reads it: the forward-only workloads
        # return o and final_state
        self.want_A = mode != "fwd"
        self.out_f = {"o": torch.empty(B, T, Hv, V, device=dev, dtype=o_dtype),
                      "final_state": torch.empty(N, Hv, K, V, device=dev),
                      "A": torch.empty(B, T, Hv, 64, device=dev) if self.want_A else None}
        self.out_b = None
        if mode != "fwd":
            self.out_b = {"dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["k"]),
                          "dv": torch.empty_like(d["v"]), "dbeta": torch.empty_like(d["g"]),
                          "dg": torch.empty_like(d["g"]), "dh0": torch.empty(N, Hv, K, V, device=dev)}
        if mode == "bwd":
            self.run_fwd()  # A for the backward, untimed

    def buffers(self):
        """This workload's device inputs and outputs: (d, out_f, out_b)."""
        return self.d, self.out_f, self.out_b

    def clone_buffers(self):
        """A second set of device inputs and outputs of the same shapes (contents
        copied), for steps whose copies overlap another step's kernels."""
        d = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in self.d.items()}
        out_f = {k: (v.clone() if v is not None else None) for k, v in self.out_f.items()}
        out_b = {k: v.clone() for k, v in self.out_b.items()} if self.out_b else None
        return d, out_f, out_b

    def run_fwd(self, timer=None, bufs=None):
        d, out_f, _ = bufs or self.buffers()
        self.gdr.gdr_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], self.x["scale"], h0=d["h0"],
                         cu_seqlens=d["cu_seqlens"], cu_seqlens_host=self.cu_host, out=out_f,
                         want_A=self.want_A, workspace=self.ws_f, cp_segments=self.cp, path=self.path,
                         timer=timer, cp_warmup=self.cp_warmup)

    def run_bwd(self, timer=None, bufs=None):
        d, out_f, out_b = bufs or self.buffers()
        self.gdr.gdr_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], out_f["A"], d["do"], dht=d["dht"],
                         scale=self.x["scale"], h0=d["h0"], cu_seqlens=d["cu_seqlens"],
                         cu_seqlens_host=self.cu_host, out=out_b, workspace=self.ws_b, cp_segments=self.cp,
                         path=self.path, timer=timer, cp_warmup=self.cp_warmup)

    def step(self, timer_f=None, timer_b=None):
        if self.mode in ("both", "fwd"):
            self.run_fwd(timer_f)
        if self.mode in ("both", "bwd"):
            self.run_bwd(timer_b)


def e2e_pipelined(w, mode, steps, stream, dev):
    """End-to-end steps through the public calls: each step copies its inputs
    in from pinned host memory and its results out to pinned host memory, and
    every copy lies between the timed region's two events.  The steps run as a
    software pipeline over two device buffer sets, the way a training loop
    prefetches its next batch: step i + 1's inputs go in on a copy-in stream
    and step i's results come out on a copy-out stream while the kernels of
    the neighbouring steps run (the link carries both directions at once).
    The results are o and final_state of the forward and every gradient of
    the backward; A, which the backward reads, stays on the device.  Returns
    (total ms of `steps` steps, h2d bytes per step, d2h bytes per step)."""
    x = w.x
    in_f = [k for k in ("q", "k", "v", "g", "beta", "h0") if torch.is_tensor(x.get(k))]
    in_b = [k for k in ("do", "dht") if torch.is_tensor(x.get(k))] if mode != "fwd" else []
    out_f_keys = ["o", "final_state"] if mode != "bwd" else []
    out_b_keys = ["dq", "dk", "dv", "dbeta", "dg", "dh0"] if mode != "fwd" else []
    sets = [w.buffers(), w.clone_buffers()]

    def dst(bufs, k):
        d, out_f, _ = bufs
        return out_f["A"] if k == "A" else d[k]

    def src(bufs, k):
        _, out_f, out_b = bufs
        return out_f[k] if k in out_f else out_b[k]

    hin = {k: x[k].pin_memory() for k in in_f + in_b}
    if mode == "bwd":  # the backward alone reads the forward's A as an input
        in_f.append("A")
        hin["A"] = w.out_f["A"].cpu().pin_memory()
    hout = {k: torch.empty(src(sets[0], k).shape, dtype=src(sets[0], k).dtype, pin_memory=True)
            for k in out_f_keys + out_b_keys}
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = sum(t.numel() * t.element_size() for t in hout.values())
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def run(n):
        e_in_f, e_in_b, e_fwd, e_done, e_out = ([None] * n for _ in range(5))
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        cin.wait_event(t0)
        cout.wait_event(t0)
        for i in range(n):
            b = sets[i % 2]
            with torch.cuda.stream(cin):
                if i >= 2:
                    cin.wait_event(e_done[i - 2])  # step i - 2 has read this set's inputs
                for k in in_f:
                    dst(b, k).copy_(hin[k], non_blocking=True)
                e_in_f[i] = torch.cuda.Event()
                e_in_f[i].record(cin)
                for k in in_b:
                    dst(b, k).copy_(hin[k], non_blocking=True)
                e_in_b[i] = torch.cuda.Event()
                e_in_b[i].record(cin)
            stream.wait_event(e_in_f[i])
            if i >= 2:
                stream.wait_event(e_out[i - 2])  # step i - 2's results are out of this set
            if mode != "bwd":
                w.run_fwd(bufs=b)
            e_fwd[i] = torch.cuda.Event()
            e_fwd[i].record(stream)
            if mode != "fwd":
                stream.wait_event(e_in_b[i])
                w.run_bwd(bufs=b)
            e_done[i] = torch.cuda.Event()
            e_done[i].record(stream)
            with torch.cuda.stream(cout):
                cout.wait_event(e_fwd[i])
                for k in out_f_keys:
                    hout[k].copy_(src(b, k), non_blocking=True)
                cout.wait_event(e_done[i])
                for k in out_b_keys:
                    hout[k].copy_(src(b, k), non_blocking=True)
                e_out[i] = torch.cuda.Event()
                e_out[i].record(cout)
        stream.wait_event(e_out[n - 1])
        t1.record(stream)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1)

    run(2)  # warm-up: first touch of the pinned buffers and the second set
    total = run(steps)
    del sets[1]
    return total, h2d, d2h


def inputs_make(spec):
    from gated_deltanet_chunked_delta_gb300 import inputs
    return inputs.make(spec, seed=0)


def timed_steps(w, steps, warmup, flush, stream, world, clocks=None):
    """W warm-up steps, then `steps` timed ones (barrier + synchronize on both
    sides of the run, an L2 flush before each step, CUDA events on the
    launching stream; the steps are enqueued back to back, so that a host-side
    stall cannot fall between a step's start event and its kernels); then as
    many steps again with every kernel bracketed by caller-owned events.
    Returns (per-step ms, per-kernel ms lists, launches over the `steps` steps,
    wall seconds, clocks)."""
    gdr = w.gdr
    for _ in range(warmup):
        flush.zero_()
        w.step()
    torch.cuda.synchronize()
    gdr.check_status()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    for i in range(steps):
        flush.zero_()
        e0[i].record(stream)
        w.step()
        e1[i].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t1 = time.time()
    clk = clocks.stop(t0, t1) if clocks else None
    step_ms = [a.elapsed_time(b) for a, b in zip(e0, e1)]
    # per-kernel durations from separate steps with caller-owned events around
    # every launch (kept out of the timed steps, whose time they would inflate)
    tf, tb = gdr.KernelTimer(32), gdr.KernelTimer(32)
    per_kernel, launches = {}, 0
    for i in range(steps):
        flush.zero_()
        w.step(tf, tb)
        torch.cuda.synchronize()
        for timer in (tf, tb):
            launches += timer.count.value
            for nm, ms in timer.elapsed():
                per_kernel.setdefault(nm, []).append(ms)
    gdr.check_status()
    return step_ms, per_kernel, launches, t1 - t0, clk


def rooflines(spec, mode, per_kernel, peaks, nch_heads, step_ms_mean):
    """The dominant kernel's roofline object and the whole step's fraction of
    max(flops / bf16 peak, bytes / HBM peak)."""
    K, V, Hv = spec.K, spec.V, spec.Hv
    tokens = spec.tokens
    in_b = 2 if spec.in_dtype == "bf16" else 4
    o_b = 4 if spec.out_dtype == "f32" else 2
    agg = {nm: (sum(v), len(v)) for nm, v in per_kernel.items()}
    # the dominant kernel among those with algorithmic work (the context-parallel
    # summaries and combines, the tables and the group sums count none)
    top = max(agg, key=lambda n: agg[n][0])
    working = [n for n in agg if kernel_work(n, spec, in_b, o_b, nch_heads, mode != "fwd") != (0.0, 0.0)]
    dom = max(working, key=lambda n: agg[n][0]) if working else top
    dom_ms = agg[dom][0] / agg[dom][1]
    fl, by = kernel_work(dom, spec, in_b, o_b, nch_heads, with_A=mode != "fwd")
    tc_peak = peaks["bf16_tflops"]
    alu_peak = 152 * 128 * 2 * peaks["sm_max_mhz"] * 1e6 / 1e12  # fp32 FFMA, TFLOP/s
    if dom.startswith("simt"):
        t_c, t_m = fl / (alu_peak * 1e12), by / (peaks["hbm_gbs"] * 1e9)
        if t_c >= t_m:
            roof = {"bound": "alu", "achieved": fl / (dom_ms / 1e3) / 1e12, "peak": alu_peak, "unit": "TFLOP/s"}
        else:
            roof = {"bound": "hbm", "achieved": by / (dom_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        t_c, t_m = fl / (tc_peak * 1e12), by / (peaks["hbm_gbs"] * 1e9)
        if t_c >= t_m:
            roof = {"bound": "tensor", "achieved": fl / (dom_ms / 1e3) / 1e12, "peak": tc_peak, "unit": "TFLOP/s"}
        else:
            roof = {"bound": "hbm", "achieved": by / (dom_ms / 1e3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = TRAFFIC.get((dom, spec.name))
    roof["algorithmic_bytes"] = by
    roof["algorithmic_flops"] = fl
    roof["kernel"] = dom
    roof["kernel_ms"] = dom_ms
    if top != dom:
        roof["longest_kernel"] = top  # an overhead kernel took longer
    roof["peak_source"] = peaks["source"]

    # whole-step roofline (the metric's "% of bf16 roofline"): algorithmic flops
    # (forward 166.6 kflop and backward 491.5 kflop per token-head at K = V = 128,
    # G = 2) and bytes (inputs read once, outputs written once)
    N = spec.n_seqs
    th = tokens * Hv
    qk_b, v_b, gb_b = tokens * spec.Hq * K * in_b, tokens * Hv * V * in_b, tokens * Hv * 4
    A_b, st_b = tokens * Hv * 64 * 4, N * Hv * K * V * 4
    f_fl, b_fl = th * 166.6e3, th * 491.5e3
    # the forward writes A only when a backward follows in the step
    f_by = (2 * qk_b + v_b + 2 * gb_b + (st_b if spec.h0 else 0) + tokens * Hv * V * o_b + st_b
            + (A_b if mode != "fwd" else 0))
    b_by = (2 * qk_b + 2 * v_b + 2 * gb_b + A_b + (2 * st_b if spec.h0 else st_b)
            + 2 * qk_b + v_b + 2 * gb_b + st_b)
    step_flops = (f_fl if mode != "bwd" else 0) + (b_fl if mode != "fwd" else 0)
    step_bytes = (f_by if mode != "bwd" else 0) + (b_by if mode != "fwd" else 0)
    step_roof_ms = max(step_flops / (tc_peak * 1e12), step_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3
    total = sum(a for a, _ in agg.values())
    kernels = {nm: {"launches": n, "ms_total": round(t, 4), "share": round(t / total, 4)}
               for nm, (t, n) in sorted(agg.items(), key=lambda kv: -kv[1][0])}
    step = {"flops": step_flops, "bytes": step_bytes, "ms": step_roof_ms,
            "bound": "tensor" if step_flops / (tc_peak * 1e12) * 1e3 >= step_roof_ms else "hbm"}
    return roof, step_roof_ms / step_ms_mean, step, kernels


def unflushed_steps(w, steps, stream):
    """Per-step ms of `steps` more steps enqueued back to back with no L2 flush
    between them (reported beside the flushed value, not as it)."""
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        e0[i].record(stream)
        w.step()
        e1[i].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(e0, e1)]


def fwd_extra(gdr, name, args, dev, path, flush, stream, peaks):
    """Forward-only figures of one workload: with the planner's warm-up starts
    and with the exact context-parallel split only."""
    from gated_deltanet_chunked_delta_gb300 import inputs
    spec = inputs.resolve(name)
    res = {"workload": name, "mode": "fwd", "step": STEP_DESC["fwd"]}
    steps, warmup = max(3, args.steps // 2), max(3, min(args.warmup, 5))
    for key, cw in (("planned", 0), ("exact_cp", -1)):
        w = Workload(gdr, spec, "fwd", dev, path, args.cp, cw)
        step_ms, per_kernel, launches, _, _ = timed_steps(w, steps, warmup, flush, stream, 1)
        ms = statistics.mean(step_ms)
        roof, frac, sroof, kernels = rooflines(spec, "fwd", per_kernel, peaks, w.prob.num_chunks() * spec.Hv, ms)
        r = {"value": spec.tokens / (ms / 1e3) / 1e6, "unit": "Mtokens/s", "ms_per_step": ms,
             "step_roofline_frac": frac, "cp_warmup": w.plan["cp_warmup"], "cp_segments": w.plan["n_segments"],
             "seg_len": w.plan["seg_len"], "gpu_launches": launches, "gpu_launches_per_step": launches // steps,
             "kernels": kernels}
        if key == "planned":
            r.update({"roofline": roof, "step_roofline": sroof})
        res[key] = r
        del w
        torch.cuda.empty_cache()
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gdr", choices=["gdr", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--path", default="auto", choices=["auto", "simt", "tc"])
    ap.add_argument("--cp", type=int, default=0, help="cp_segments (0 auto, 1 off, n forced)")
    ap.add_argument("--cp-warmup", type=int, default=0, help="cp_warmup (0 planner's choice, -1 off, n chunks)")
    ap.add_argument("--mode", default="both", choices=["both", "fwd", "bwd"],
                    help="step = forward + backward (default), forward only, or backward only")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true", help="skip the forward-only workloads")
    ap.add_argument("--ref-tokens", type=int, default=1024, help="tokens per oracle step (reference arm)")
    ap.add_argument("--cpu-tokens", type=int, default=4096,
                    help="tokens of the all-cores cpu_baseline sample (0: the whole first sequence)")
    ap.add_argument("--cpu-tokens-1core", type=int, default=1024,
                    help="tokens of the one-core cpu_baseline sample (over 8 v-heads at most)")
    ap.add_argument("--T", type=int, default=0,
                    help="shorter sequences of the same fixed-length workload (profiling captures)")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from gated_deltanet_chunked_delta_gb300 import inputs
    base = inputs.resolve(args.workload)
    from dataclasses import replace
    spec = replace(base, bwd=True)
    if args.T:
        if spec.lengths is not None:
            raise SystemExit("--T applies to fixed-length workloads")
        spec = replace(spec, T=args.T, name=f"{spec.name}@T{args.T}")

    if args.impl == "reference":
        run_reference(args, spec, rank, world)
        return

    import gated_deltanet_chunked_delta_gb300 as gdr
    gdr.load()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    path = {"auto": gdr.GDR_PATH_AUTO, "simt": gdr.GDR_PATH_SIMT, "tc": gdr.GDR_PATH_TC}[args.path]
    peaks = _peaks()
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    w = Workload(gdr, spec, args.mode, dev, path, args.cp, args.cp_warmup)
    x, d, out_f, out_b = w.x, w.d, w.out_f, w.out_b
    clocks = Clocks(local)
    step_ms, per_kernel, launches, _, clk = timed_steps(w, args.steps, args.warmup, flush, stream, world, clocks)
    tokens = spec.tokens
    value, total_ms = aggregate(sum(step_ms), tokens, args.steps, dev)
    unfl_ms = statistics.median(unflushed_steps(w, args.steps, stream))

    # e2e: every step's inputs in from pinned host memory and its results out,
    # inside the timed region, steps pipelined over two buffer sets
    e2e_steps = max(4, args.steps)
    e2e_total, h2d, d2h = e2e_pipelined(w, args.mode, e2e_steps, stream, dev)
    e2e_val, _ = aggregate(e2e_total, tokens, e2e_steps, dev)
    gdr.check_status()

    roof, step_frac, sroof, kernels = rooflines(spec, args.mode, per_kernel, peaks,
                                                w.prob.num_chunks() * spec.Hv, total_ms / args.steps)
    cfg = _config(spec, args)
    cfg["cp_warmup"] = w.plan["cp_warmup"]
    cfg["cp_segments"] = w.plan["n_segments"]
    line = {"metric": METRIC, "value": value, "unit": "Mtokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if spec.in_dtype == "bf16" else "f32",
            "data": "synthetic", "config": cfg,
            "roofline": roof,
            "step_roofline_frac": step_frac,
            "step_roofline": sroof,
            "kernels": kernels,
            "e2e": {"value": e2e_val, "unit": "Mtokens/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "steps": e2e_steps, "ms_per_step": e2e_total / e2e_steps,
                    "copies": ("pinned host buffers; steps pipelined over two device buffer sets: the next "
                               "step's inputs in on a copy-in stream and each step's results out on a copy-out "
                               "stream while kernels run; results are o, final_state and the gradients "
                               "(A stays on the device)")},
            "gpu_launches": launches, "gpu_launches_per_step": launches // args.steps, "clocks": clk,
            "unflushed": {"ms_per_step": unfl_ms, "value": tokens * world / (unfl_ms / 1e3) / 1e6,
                          "note": "median of as many steps again with no L2 flush between them (this rank)"}}
    del out_f, out_b, d
    if rank == 0 and world == 1 and not args.no_extras and args.workload == DEFAULT_WORKLOAD:
        del w
        torch.cuda.empty_cache()
        line["fwd_workloads"] = [fwd_extra(gdr, nm, args, dev, path, flush, stream, peaks) for nm in FWD_EXTRAS]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        v, dt, Ts, nth = oracle_sample(x, spec, args.cpu_tokens or (1 << 30), spec.Hq)
        h1 = max(1, min(spec.Hq, 8 // max(1, spec.Hv // spec.Hq)))
        v1, dt1, T1, _ = oracle_sample(x, spec, args.cpu_tokens_1core, h1, nthreads=1)
        line["cpu_baseline"] = {"value": v, "unit": "Mtokens/s", "cores": nth, "kind": "oracle",
                                "sample": f"oracle fwd+bwd on tokens [0,{Ts}) of sequence 0, all {spec.Hv} "
                                          f"v-heads ({dt:.1f} s); throughput in full-workload tokens",
                                "one_core": {"value": v1, "unit": "Mtokens/s", "cores": 1,
                                             "sample": f"oracle fwd+bwd on tokens [0,{T1}) of sequence 0, "
                                                       f"{h1 * (spec.Hv // spec.Hq)} v-heads ({dt1:.1f} s); "
                                                       f"throughput in full-workload tokens"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
