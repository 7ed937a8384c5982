#!/usr/bin/env python
"""Throughput of the causal linear-attention hot path on GB300.

Headline: Hedgehog chunked prefill on the Llama-2-7B attention shape
(B=1, H=32, n=4096, d=128, bf16 in / fp32 accumulate), the largest prefill
workload, in tokens/s, where a token is one sequence position of one batch
element across all H heads.
Inputs rotate through enough resident copies to exceed twice the L2 size, so
every step streams from HBM.  Steps are replayed from CUDA graphs (each step
is one hh_linattn_fwd_causal call through the C ABI) and timed with CUDA
events on the launching stream.

The other hot-path rows (GPT-2-shaped prefill, Taylor prefill, recurrent
decode, the float32 workload, the loss and its gradient) are measured in the
same run and reported under "rows".

``--impl reference`` times the fp64 CPU oracle on bounded samples of the
same workload (the baseline arm; no GPU work).
"""

from __future__ import annotations

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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "llama2_prefill_1x32x4096_d128"
METRIC = "causal linear-attn prefill tokens/s (+% BF16 TC peak); decode GB/s (+% HBM)"


# ---------------------------------------------------------------------------
# peaks, clocks, bookkeeping
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background (200 ms period)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        inside = [s for t, s in self.samples
                  if self.t_start is not None and self.t_start - 0.2 <= t <= (self.t_end or t) + 0.2]
        use = inside or [s for _, s in self.samples]

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[1]) for s in use if len(s) > 1 and num(s[1]) is not None]
        mx = [num(s[2]) for s in use if len(s) > 2 and num(s[2]) is not None]
        pw = [num(s[3]) for s in use if len(s) > 3 and num(s[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i - 5] for s in use for i in range(5, min(9, len(s)))
                          if s[i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "reasons": reasons, "samples": len(use), "samples_in_region": len(inside)}


def source_digest(files=None):
    """Hash of CUDA sources (the named files of csrc/, else all of them), to
    tell whether stored ncu counters are current."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "softmax_mimicking_feature_gb300", "csrc")
    for name in sorted(files if files else os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from profiles/dram_traffic.json when still current."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            entries = json.load(f)
    except Exception:
        return None
    for e in entries:
        if e.get("kernel") != kernel or e.get("workload") != workload:
            continue
        try:
            current = source_digest(e.get("sources"))
        except OSError:
            continue
        if e.get("source") == current:
            return e.get("bytes_per_launch")
    return None


# ---------------------------------------------------------------------------
# per-workload algorithmic counts (per token-head unless stated)
# ---------------------------------------------------------------------------

def prefill_counts(w):
    """Algorithmic bytes and FLOP of one prefill call on workload w.

    Bytes: q, k, v read and y written once (d elements each).  FLOP per
    token-head (chunk C, feature dim d'): Hedgehog feature maps 4d^2, intra-
    chunk scores and A.V over the causal half C/2 each way plus the diagonal
    (d'(C+1) + d(C+1)), inter-chunk readout and state update 4 d' d.  The
    Taylor feature construction on CUDA cores is not counted."""
    esz = 4 if w.dtype == "f32" else 2
    d = w.d
    dp = 2 * d if w.kind == "hedgehog" else 1 + d + d * d
    C = w.chunk
    th = w.B * w.H * w.n
    fmap = 4 * d * d if w.kind == "hedgehog" else 0
    flops = th * (fmap + dp * (C + 1) + d * (C + 1) + 4 * dp * d)
    return {"bytes": th * 4 * d * esz, "flops": flops}


def decode_counts(w):
    """Bytes per step: S and z read + written in fp32, q, k, v read and y written."""
    dp = 2 * w.d if w.kind == "hedgehog" else 1 + w.d + w.d * w.d
    per = 2 * 4 * (dp * w.d + dp) + 4 * w.d * 2
    flops = 4 * w.d * w.d + 4 * dp * w.d
    return {"bytes": w.B * w.H * per, "flops": w.B * w.H * flops}


def loss_counts(w):
    d = w.d
    dp = 2 * d
    pairs = w.B * w.H * w.n * (w.n + 1) // 2
    return {"pairs": pairs, "flops": pairs * 2 * (d + dp), "bytes": w.B * w.H * w.n * 2 * d * 2}


def grad_counts(w):
    """Gradient of the summed loss w.r.t. W, b (bf16 Hedgehog).

    Algorithmic FLOP per causal pair: the scores s and a (2d + 2d') once and the
    two feature-side contractions dPhi(q) += g phi(k), dPhi(k) += g phi(q)
    (2 x 2d').  Executed: s and a three times (row statistics, query side, key
    side) plus the two contractions."""
    d = w.d
    dp = 2 * d
    pairs = w.B * w.H * w.n * (w.n + 1) // 2
    return {"pairs": pairs, "flops": pairs * (2 * d + 2 * dp + 4 * dp),
            "flops_executed": pairs * (3 * (2 * d + 2 * dp) + 4 * dp)}


# ---------------------------------------------------------------------------
# GPU timing helpers
# ---------------------------------------------------------------------------

def _fm(hh, w, x, kind=None):
    kind = kind or w.kind
    if kind == "hedgehog":
        return hh.FeatureMap("hedgehog", w.d, x["W"], x["b"])
    if kind == "hedgehog_softmax":
        return hh.FeatureMap("hedgehog_softmax", w.d, x["W"])
    return hh.FeatureMap("taylor2", w.d)


def time_graphs(torch, step_fns, K, W, sampler=None, dist=None, cap=240):
    """Run W warm-up steps, then time exactly K steps replayed from CUDA graphs.

    step_fns[i] enqueues step i of a rotation.  The K steps run back to back
    from at most two graphs: one of min(K, cap) consecutive steps replayed
    K // that many times, and one holding the remaining steps, so that no step
    pays a graph-launch gap of its own for any K."""
    R = len(step_fns)
    for i in range(W):
        step_fns[i % R]()
    torch.cuda.synchronize()
    per = min(K, max(R, cap - cap % R))
    n_big, rem = divmod(K, per)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())

    def capture(count):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                for i in range(count):
                    step_fns[i % R]()
        return g

    big = capture(per)
    tail = capture(rem) if rem else None
    torch.cuda.synchronize()
    big.replay()
    if tail is not None:
        tail.replay()
    torch.cuda.synchronize()
    if sampler:
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if sampler:
        sampler.mark("start")
    e0.record(stream)
    for _ in range(n_big):
        big.replay()
    if tail is not None:
        tail.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("end")
    if dist is not None:
        dist.barrier()
    return e0.elapsed_time(e1)  # ms


def job_time_ms(torch, ms, dist, device):
    """The whole job's time for N ranks: the largest per-rank time, which
    every rank receives (one all-reduce; the ranks run independent replicas,
    so nothing else is exchanged)."""
    if dist is None:
        return ms
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(K, B, n, world, ms):
    """Tokens per second of the whole job: every rank's K calls of B x n tokens
    within the job's time."""
    return K * B * n * world / (ms / 1e3)


def n_rotation(bytes_per_set, l2_bytes):
    return max(2, math.ceil(2.2 * l2_bytes / max(bytes_per_set, 1)))


# ---------------------------------------------------------------------------
# rows
# ---------------------------------------------------------------------------

def bench_prefill(torch, hh, wl, w, K, W, dev, sampler=None, dist=None, l2=0, kind=None):
    cnt = prefill_counts(w)
    esz = 4 if w.dtype == "f32" else 2
    per_set = cnt["bytes"]
    R = n_rotation(per_set, l2)
    sets = [wl.make_inputs(w, seed=100 + i, device=dev) for i in range(R)]
    fm = _fm(hh, w, sets[0], kind)
    ys = [torch.empty_like(x["q"]) for x in sets]
    need = hh.fwd_workspace_bytes(fm, w.torch_dtype, w.B, w.H, w.n, w.chunk)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    segs, launches = hh.fwd_plan(fm, w.torch_dtype, w.B, w.H, w.n, w.chunk)
    fns = [(lambda x=x, y=y: hh.linattn_fwd_causal(fm, x["q"], x["k"], x["v"], chunk=w.chunk,
                                                    y=y, workspace=ws)) for x, y in zip(sets, ys)]
    ms = time_graphs(torch, fns, K, W, sampler, dist)
    return {"ms_total": ms, "K": K, "rotation": R, "set_bytes": per_set * R,
            "segments": segs, "launches": launches, "counts": cnt, "sets": sets, "fm": fm, "ws": ws}


def bench_decode(torch, hh, wl, w, K, W, dev):
    # state from an n-token prefill on the device, then K decode steps
    x = wl.make_inputs(w, seed=300, device=dev)
    fm = _fm(hh, w, x)
    _, S, z = hh.linattn_fwd_causal(fm, x["q"], x["k"], x["v"], return_state=True)
    del x
    torch.cuda.synchronize()
    R = 16
    g = torch.Generator(device=dev)
    g.manual_seed(301)
    steps = [tuple((torch.randn(w.B, w.H, w.d, generator=g, device=dev) * w.qk_std).to(w.torch_dtype)
                   for _ in range(3)) for _ in range(R)]
    ys = [torch.empty(w.B, w.H, w.d, dtype=w.torch_dtype, device=dev) for _ in range(R)]
    fns = [(lambda t=t, y=y: hh.linattn_decode_step(fm, t[0], t[1], t[2], S, z, y=y))
           for t, y in zip(steps, ys)]
    ms = time_graphs(torch, fns, K, W)
    return {"ms_total": ms, "K": K, "counts": decode_counts(w)}


def bench_loss(torch, hh, wl, w, K, W, dev):
    x = wl.make_inputs(w, seed=400, device=dev)
    fm = _fm(hh, w, x)
    need = hh.loss_workspace_bytes(fm, w.torch_dtype, w.B, w.H, w.n)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    fns = [lambda: hh.mimicry_loss(fm, x["q"], x["k"], return_rows=False, workspace=ws)]
    ms = time_graphs(torch, fns, K, W)
    return {"ms_total": ms, "K": K, "counts": loss_counts(w)}


def bench_grad(torch, hh, wl, w, K, W, dev, kind=None):
    x = wl.make_inputs(w, seed=500, device=dev)
    fm = _fm(hh, w, x, kind)
    need = hh.loss_grad_workspace_bytes(fm, w.torch_dtype, w.B, w.H, w.n)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    fns = [lambda: hh.mimicry_loss_grad(fm, x["q"], x["k"], workspace=ws)]
    ms = time_graphs(torch, fns, K, W)
    return {"ms_total": ms, "K": K, "counts": grad_counts(w)}


def e2e_prefill(torch, hh, w, sets, fm, ws, E, dev):
    """Same metric through the public API with pinned host buffers, copies timed.

    Every step copies its q, k, v from pinned host memory and reads its y back.
    Steps are double-buffered the way a serving loop runs them: the inputs of
    step i+1 are copied on their own stream while step i computes, and y of
    step i goes back on a third stream, so the two copy directions overlap;
    events keep each buffer's writes after its last reader."""
    host = {t: sets[0][t].cpu().pin_memory() for t in ("q", "k", "v")}
    y_host = [torch.empty_like(host["q"]).pin_memory() for _ in range(2)]
    dev_in = [{t: torch.empty_like(sets[0][t]) for t in ("q", "k", "v")} for _ in range(2)]
    dev_y = [torch.empty_like(sets[0]["q"]) for _ in range(2)]
    comp = torch.cuda.current_stream()
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    in_ready = [ev(), ev()]      # inputs of buffer set b copied
    in_free = [ev(), ev()]       # the prefill has read buffer set b
    y_ready = [ev(), ev()]       # y of buffer set b written
    y_free = [ev(), ev()]        # y of buffer set b copied back
    for b in range(2):
        in_free[b].record(comp)
        y_free[b].record(comp)

    def step(i):
        b = i & 1
        with torch.cuda.stream(h2d):
            h2d.wait_event(in_free[b])
            for t in ("q", "k", "v"):
                dev_in[b][t].copy_(host[t], non_blocking=True)
            in_ready[b].record(h2d)
        comp.wait_event(in_ready[b])
        comp.wait_event(y_free[b])
        hh.linattn_fwd_causal(fm, dev_in[b]["q"], dev_in[b]["k"], dev_in[b]["v"], chunk=w.chunk,
                              y=dev_y[b], workspace=ws)
        in_free[b].record(comp)
        y_ready[b].record(comp)
        with torch.cuda.stream(d2h):
            d2h.wait_event(y_ready[b])
            y_host[b].copy_(dev_y[b], non_blocking=True)
            y_free[b].record(d2h)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    h2d.wait_stream(comp)   # no copy of the timed steps starts before e0
    d2h.wait_stream(comp)
    for i in range(E):
        step(i)
    comp.wait_stream(h2d)
    comp.wait_stream(d2h)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    el = host["q"].numel() * host["q"].element_size()
    return {"value": E * w.B * w.n / (ms / 1e3), "unit": "tokens/s",
            "h2d_bytes_per_step": 3 * el, "d2h_bytes_per_step": el, "steps": E,
            "copies": "double-buffered: h2d, compute and d2h on three streams"}


# ---------------------------------------------------------------------------
# CPU oracle (reported baseline / reference arm)
# ---------------------------------------------------------------------------

def oracle_prefill_sample(w, budget_s, x=None, max_units=None):
    """Time the fp64 oracle on (b, h) units of workload w.

    Units are taken in order, cycling over the workload, until budget_s has
    passed (or max_units units are done)."""
    import oracle as O
    from softmax_mimicking_feature_gb300 import workloads as wl
    if x is None:
        x = wl.make_inputs(w, seed=100, seqs=range(min(w.B, 8)))
    q, k, v = (x[t].double().numpy() for t in ("q", "k", "v"))
    W = None if x["W"] is None else x["W"].double().numpy()
    b = None if x["b"] is None else x["b"].double().numpy()
    units = [(bi, h) for bi in range(q.shape[0]) for h in range(q.shape[1])]
    t0 = time.perf_counter()
    done = 0
    while True:
        bi, h = units[done % len(units)]
        O.fwd_causal(w.kind, q[bi:bi + 1, h:h + 1], k[bi:bi + 1, h:h + 1], v[bi:bi + 1, h:h + 1],
                     None if W is None else W[h:h + 1], None if b is None else b[h:h + 1])
        done += 1
        if (max_units and done >= max_units) or (not max_units and time.perf_counter() - t0 > budget_s):
            break
    dt = time.perf_counter() - t0
    tokens = done * w.n / w.H
    return {"value": tokens / dt, "unit": "tokens/s", "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{done} (batch, head) units x {w.n} tokens of {w.name} "
                      f"(quadratic form, fp64 numpy; BLAS threads = library default)",
            "seconds": dt}


def run_reference(args):
    from softmax_mimicking_feature_gb300 import workloads as wl
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    w = wl.WORKLOADS[args.workload]
    x = wl.make_inputs(w, seed=100, seqs=[0])
    units = 2  # one bounded sample per step
    for _ in range(args.warmup):
        oracle_prefill_sample(w, 1e9, x=x, max_units=units)
    vals, secs = [], 0.0
    for _ in range(args.steps):
        r = oracle_prefill_sample(w, 1e9, x=x, max_units=units)
        secs += r["seconds"]
    tokens = args.steps * units * w.n / w.H
    value = tokens / secs
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
                       "step": f"{units} (batch, head) units of the workload per step"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle",
                             "sample": f"{units} (batch, head) units x {w.n} tokens per step, "
                                       f"fp64 numpy quadratic form"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# main arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    import softmax_mimicking_feature_gb300 as hh
    from softmax_mimicking_feature_gb300 import workloads as wl
    from softmax_mimicking_feature_gb300 import _abi

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    _abi.lib()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 0) or 126 * 2**20)
    peaks = load_peaks()
    w = wl.WORKLOADS[args.workload]

    sampler = ClockSampler(local)
    sampler.start()
    res = bench_prefill(torch, hh, wl, w, args.steps, args.warmup, dev, sampler, dist, l2)
    sampler.stop()

    ms = job_time_ms(torch, res["ms_total"], dist, dev)
    K = args.steps
    value = job_tokens_per_s(K, w.B, w.n, world, ms)
    cnt = res["counts"]
    per_launch_s = (res["ms_total"] / 1e3) / K
    achieved_gbs = cnt["bytes"] / per_launch_s / 1e9
    tflops_alg = cnt["flops"] / per_launch_s / 1e12
    kernel_name = "hh_prefill (whole hh_linattn_fwd_causal call)"
    traffic = stored_traffic("prefill", w.name)
    roofline = {"bound": "hbm", "achieved": achieved_gbs, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved_gbs / peaks["hbm_gbs"], "traffic": traffic,
                "kernel": kernel_name, "launches_per_step": res["launches"],
                "peak_source": peaks["source"],
                "tensor_frac_alg": tflops_alg * 1e12 / (peaks["bf16_tflops"] * 1e12),
                "tensor_tflops_alg": tflops_alg}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "H": w.H, "n": w.n, "d": w.d,
                       "chunk": w.chunk, "feature_map": w.kind, "segments": res["segments"],
                       "l2": f"inputs rotate over {res['rotation']} resident sets "
                             f"({res['set_bytes'] / 1e6:.0f} MB > 2x L2 {l2 / 1e6:.0f} MB)",
                       "timing": "CUDA events around K back-to-back calls replayed from CUDA graphs",
                       "parallelism": f"replicas x{world}"},
            "clocks": sampler.summary(),
            "roofline": roofline,
            "gpu_launches": K * res["launches"]}

    if rank == 0:
        line["e2e"] = e2e_prefill(torch, hh, w, res["sets"], res["fm"], res["ws"],
                                  min(K, 200), dev)
        if world == 1 and not args.no_cpu:
            line["cpu_baseline"] = oracle_prefill_sample(w, args.cpu_seconds)
        if not args.no_rows and world == 1:
            line["rows"] = other_rows(torch, hh, wl, dev, peaks, l2)
    del res
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def other_rows(torch, hh, wl, dev, peaks, l2):
    rows = {}

    def prefill_row(name, K, kind=None):
        w = wl.WORKLOADS[name]
        r = bench_prefill(torch, hh, wl, w, K, 3, dev, l2=l2, kind=kind)
        s = r["ms_total"] / 1e3 / K
        c = r["counts"]
        rows[(kind + ":" if kind else "") + name] = {"tokens_per_s": w.B * w.n / s, "ms_per_call": s * 1e3,
                      "hbm_gbs_alg": c["bytes"] / s / 1e9,
                      "hbm_frac": c["bytes"] / s / 1e9 / peaks["hbm_gbs"],
                      "tensor_frac_alg": c["flops"] / s / 1e12 / peaks["bf16_tflops"],
                      "segments": r["segments"], "launches": r["launches"]}

    for name, K, kind in (("gpt2_prefill_8x12x1024_d64", 200, None),
                          ("taylor2_prefill_4x8x8192_d16", 20, None),
                          ("hedgehog_f32_1x1x256_d64", 50, None),
                          ("gpt2_prefill_8x12x1024_d64", 200, "hedgehog_softmax"),
                          ("llama2_prefill_1x32x4096_d128", 20, "hedgehog_softmax")):
        try:
            prefill_row(name, K, kind)
        except Exception as e:  # report, do not hide
            rows[(kind + ":" if kind else "") + name] = {"error": repr(e)}
        torch.cuda.empty_cache()

    try:
        w = wl.WORKLOADS["llama2_decode_128x32_d128"]
        r = bench_decode(torch, hh, wl, w, 64, 4, dev)
        s = r["ms_total"] / 1e3 / r["K"]
        rows[w.name] = {"gb_per_s": r["counts"]["bytes"] / s / 1e9,
                        "hbm_frac": r["counts"]["bytes"] / s / 1e9 / peaks["hbm_gbs"],
                        "hbm_frac_of_8tbs": r["counts"]["bytes"] / s / 8e12,
                        "us_per_step": s * 1e6, "tokens_per_s": w.B / s,
                        "bytes_per_step": r["counts"]["bytes"]}
    except Exception as e:
        rows["llama2_decode_128x32_d128"] = {"error": repr(e)}
    torch.cuda.empty_cache()

    for name in ("llama2_prefill_1x32x4096_d128", "hedgehog_f32_1x1x256_d64"):
        try:
            w = wl.WORKLOADS[name]
            r = bench_loss(torch, hh, wl, w, 5, 2, dev)
            s = r["ms_total"] / 1e3 / r["K"]
            rows["loss:" + name] = {"ms_per_call": s * 1e3,
                                    "pairs_per_s": r["counts"]["pairs"] / s,
                                    "tensor_frac_alg": r["counts"]["flops"] / s / 1e12 / peaks["bf16_tflops"]}
        except Exception as e:
            rows["loss:" + name] = {"error": repr(e)}
        torch.cuda.empty_cache()

    for key, name, kind in (("grad", "llama2_prefill_1x32x4096_d128", None),
                            ("grad", "gpt2_prefill_8x12x1024_d64", None),
                            ("softmax_grad", "gpt2_prefill_8x12x1024_d64", "hedgehog_softmax")):
        try:
            w = wl.WORKLOADS[name]
            r = bench_grad(torch, hh, wl, w, 5, 2, dev, kind)
            s = r["ms_total"] / 1e3 / r["K"]
            c = r["counts"]
            rows[key + ":" + name] = {"ms_per_call": s * 1e3, "pairs_per_s": c["pairs"] / s,
                                    "tensor_frac_alg": c["flops"] / s / 1e12 / peaks["bf16_tflops"],
                                    "tensor_frac_executed":
                                        c["flops_executed"] / s / 1e12 / peaks["bf16_tflops"]}
        except Exception as e:
            rows[key + ":" + name] = {"error": repr(e)}
        torch.cuda.empty_cache()
    return rows


def run_row(args):
    """One hot-path row alone (for profiling): prefill:, softmax_prefill:, loss:,
    grad:, softmax_grad:<workload>, or decode."""
    import torch
    import softmax_mimicking_feature_gb300 as hh
    from softmax_mimicking_feature_gb300 import workloads as wl
    from softmax_mimicking_feature_gb300 import _abi
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _abi.lib()
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or 126 * 2**20)
    kind, _, name = args.row.partition(":")
    if kind in ("prefill", "softmax_prefill"):
        w = wl.WORKLOADS[name]
        r = bench_prefill(torch, hh, wl, w, args.steps, args.warmup, dev, l2=l2,
                          kind="hedgehog_softmax" if kind == "softmax_prefill" else None)
        s = r["ms_total"] / 1e3 / args.steps
        out = {"row": args.row, "us_per_call": s * 1e6, "tokens_per_s": w.B * w.n / s,
               "hbm_gbs_alg": r["counts"]["bytes"] / s / 1e9, "segments": r["segments"]}
    elif kind == "loss":
        w = wl.WORKLOADS[name]
        r = bench_loss(torch, hh, wl, w, args.steps, args.warmup, dev)
        s = r["ms_total"] / 1e3 / args.steps
        out = {"row": args.row, "us_per_call": s * 1e6, "pairs_per_s": r["counts"]["pairs"] / s}
    elif kind in ("grad", "softmax_grad"):
        w = wl.WORKLOADS[name]
        r = bench_grad(torch, hh, wl, w, args.steps, args.warmup, dev,
                       "hedgehog_softmax" if kind == "softmax_grad" else None)
        s = r["ms_total"] / 1e3 / args.steps
        out = {"row": args.row, "us_per_call": s * 1e6, "pairs_per_s": r["counts"]["pairs"] / s}
    elif kind == "decode":
        w = wl.WORKLOADS["llama2_decode_128x32_d128"]
        if args.decode_seqs:
            w = w.with_(B=args.decode_seqs)
        r = bench_decode(torch, hh, wl, w, args.steps, args.warmup, dev)
        s = r["ms_total"] / 1e3 / args.steps
        out = {"row": args.row, "B": w.B, "us_per_step": s * 1e6,
               "gb_per_s": r["counts"]["bytes"] / s / 1e9}
    else:
        raise SystemExit(f"unknown row {args.row!r}")
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--row", default=None,
                    help="time one row alone: prefill:<workload>, loss:<workload>, "
                         "grad:<workload> or decode")
    ap.add_argument("--decode-seqs", type=int, default=0,
                    help="with --row decode: number of sequences (default: the workload's 128)")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    if args.row:
        return run_row(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
