#!/usr/bin/env python3
"""Benchmark of the GB300 MXFP4 routed-expert MoE layer.

One step = one forward of the whole layer (route -> sort -> Q8(x) -> gate/up +
SwiGLU -> Q8(h) -> down -> combine) over one batch of synthetic tokens, issued
through the library's C ABI and captured once per (layer copy, batch) in a
CUDA graph.  The default workload is single-token decode of the
DeepSeek-V4-Flash routed-expert layer (H 4096, 256 experts, top-6, expert
intermediate 2048, MXFP4 weights with E8M0 per-32 scales, bf16 router and
activations).

L2: a single token touches ~82 MB (< 129 MB of L2), so steps cycle through
NL distinct copies of the layer's weights (3.4 GB each) and distinct token
batches; each copy is re-used only after NL-1 other layers' traffic has gone
through L2, so every step streams its weights from HBM.

Prints ONE JSON line (rank 0).  Multi-GPU (torchrun) runs independent replicas
(the layer does not need a collective for a data-parallel decode batch);
value = tokens of all ranks / max time over ranks.

--impl reference times the CPU oracle (the plain C statement of the layer) on
the host cores instead, on a bounded sample of each step's batch.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, E, K_TOP, I_EXP = 4096, 256, 6, 2048
EXPERT_BYTES = 2 * I_EXP * (H // 2 + H // 32) + H * (I_EXP // 2 + I_EXP // 32)
ROUTER_BYTES = E * H * 2

WORKLOADS = {
    # name: (tokens per step, zipf exponent or None, layer copies cycled)
    "decode-1": (1, None, 8),
    "krow-2": (2, None, 8),
    "krow-3": (3, None, 8),
    "krow-4": (4, None, 8),
    "krow-8": (8, None, 8),
    "krow-16": (16, None, 8),
    "zipf-32": (32, 1.1, 6),
    "zipf-64": (64, 1.1, 6),
    "prefill-512": (512, None, 3),
    "prefill-8192": (8192, None, 2),
}
METRIC = "MoE-layer tokens/s and achieved HBM TB/s (decode 1–16 rows; prefill 512 rows)"

# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# roofline kernel, from one ncu capture of the kernel on a one-layer copy of
# the workload, with the hash of the kernel's sources at that capture: a
# figure whose sources have changed since is reported as null.
NCU_TRAFFIC = {
    # (workload, roofline kernel): (bytes per launch, source hash at capture)
    ("decode-1", "moe_decode_forward"): (84.08e6, "cfb92175ac34c33b"),
}
# sources of each roofline kernel (the files its code comes from)
KERNEL_SOURCES = {
    "moe_decode_forward": ["decode.cu", "mx_device.cuh", "common.cuh"],
    "moe_decode_forward_shared": ["decode.cu", "mx_device.cuh", "common.cuh"],
    "moe_mxfp4_gateup_swiglu": ["tc_expert.cu", "tc_device.cuh", "mxmv.cu", "mx_device.cuh", "common.cuh"],
}
ARITHMETIC = "e2m1*int8 exact int32 block dots, fp32 scale and accumulate"
# batches of 17+ rows: experts of more than 4 rows on the tensor cores
ARITHMETIC_TENSOR = ("e2m1*int8 exact int32 block dots (experts of <= 4 rows); e2m1 weights x six e2m1 planes "
                     "of the Q8 activations, fp32 MMA accumulation (more rows)")


def source_hash(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "mxfp4_mixture_experts_moe_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, kernel: str):
    """Measured DRAM bytes per launch, or None (no capture, or the kernel's
    sources changed since the capture)."""
    rec = NCU_TRAFFIC.get((workload, kernel))
    if rec is None or rec[1] != source_hash(kernel):
        return None
    return rec[0]


def workload_config(workload: str, world: int, shared: bool) -> dict:
    """The workload a line is measured on (the same keys and values on both
    arms)."""
    T, zipf, _ = WORKLOADS[workload]
    return {"workload": workload, "tokens_per_step": T, "hidden": H, "experts": E, "top_k": K_TOP,
            "expert_intermediate": I_EXP, "weights": "MXFP4 E2M1 + E8M0 per 32, random init",
            "activations": "bf16 N(0,1) -> Q8 per 32", "router": "bf16 N(0,0.02)", "zipf_bias": zipf,
            "parallelism": f"replicas{world}", "shared_expert": shared}


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.machine()


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="decode-1")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="layer copies to cycle (default: per workload)")
    ap.add_argument("--graph-steps", type=int, default=16, help="layer forwards captured per CUDA graph")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="target oracle time of each cpu_baseline sample (one core, then every core)")
    ap.add_argument("--no-sub", action="store_true",
                    help="skip the krow-16 and prefill-512 sub-records of the default decode-1 line")
    ap.add_argument("--shared-expert", action="store_true",
                    help="the layer also has a shared expert (every token, weight 1, joined onto the routed output)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks/throttle sampling while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc:
            time.sleep(0.06)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def make_layer(moe, torch, seed, zipf, device, shared=False):
    """Random-init layer in the boundary layout, generated on the device
    (with a shared expert of the same format when ``shared``)."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    wr = (torch.randn(E, H, generator=g, device=device) * 0.02).to(torch.bfloat16)
    bias = None
    if zipf:
        perm = torch.randperm(E, generator=g, device=device)
        rank = torch.empty(E, dtype=torch.float64, device=device)
        rank[perm] = torch.arange(E, dtype=torch.float64, device=device)
        p = (rank + 1.0) ** (-zipf)
        bias = torch.log(p / p.sum()).float()

    def nib(*shape):
        return torch.randint(0, 256, shape, generator=g, device=device, dtype=torch.uint8)

    def sc(*shape):
        return (123 + torch.randint(0, 5, shape, generator=g, device=device)).to(torch.uint8)

    sh = None
    if shared:
        sh = moe.SharedExpertWeights(wg=nib(1, I_EXP, H // 2), sg=sc(1, I_EXP, H // 32),
                                     wu=nib(1, I_EXP, H // 2), su=sc(1, I_EXP, H // 32),
                                     wd=nib(1, H, I_EXP // 2), sd=sc(1, H, I_EXP // 32))
    return moe.LayerWeights(wr=wr, bias=bias, k=K_TOP,
                            wg=nib(E, I_EXP, H // 2), sg=sc(E, I_EXP, H // 32),
                            wu=nib(E, I_EXP, H // 2), su=sc(E, I_EXP, H // 32),
                            wd=nib(E, H, I_EXP // 2), sd=sc(E, H, I_EXP // 32), shared=sh)


# ------------------------------------------------------------------ oracle timing

class OracleSample:
    """The CPU oracle on a pool of tokens of the same workload (inputs from the
    seeded generator), timed per assignment so any step budget can be met."""

    def __init__(self, T, zipf, pool=8, shared=False):
        import oracle
        import synth
        self.oracle, self.synth = oracle, synth
        self.spec = synth.DSV4_ZIPF if zipf else synth.DSV4
        self.k = self.spec.k
        self.x = synth.activations(self.spec, pool, token0=123456)
        self.wr = synth.router_weights(self.spec)
        self.bias = synth.router_bias(self.spec)
        _, self.ids, _ = oracle.route(self.x, self.wr, self.k, self.bias)
        self.experts = {int(e): synth.expert(self.spec, int(e)) for e in np.unique(self.ids)}
        self.shared = synth.shared_expert(self.spec) if shared else None
        self.units = self.k + (1 if shared else 0)  # expert passes per token
        self.pool = pool
        self.T = T

    def run_assignments(self, n_assign, start=0):
        """One token through the oracle: the whole layer (with the shared
        expert, if any) when n_assign == units, else routing, Q8(x) and
        n_assign of its routed slots (gate/up, SwiGLU, Q8(h), down).  Returns
        seconds."""
        o = self.oracle
        t = start % self.pool
        xt = self.x[t:t + 1]
        t0 = time.perf_counter()
        if n_assign >= self.units:
            o.layer(xt, self.wr, self.bias, self.k, self.experts, shared=self.shared)
            return time.perf_counter() - t0
        _, ids, _ = o.route(xt, self.wr, self.k, self.bias)
        xq, xs = o.quant_q8(xt)
        for j in range(min(n_assign, self.k)):
            e = self.experts[int(ids[0, j])]
            G, U = o.expert_gateup(xq[0], xs[0], e.wg, e.sg, e.wu, e.su)
            h = np.array([o.silu(g) * u for g, u in zip(G, U)], dtype=np.float32)
            hq, hs = o.quant_q8(h[None])
            o.expert_down(hq[0], hs[0], e.wd, e.sd)
        return time.perf_counter() - t0


def oracle_rate(T, zipf, seconds, shared=False, threads=1):
    """tokens/s of the oracle over ~`seconds` of work, the whole layer per
    token, with `threads` host threads taking tokens in turn (the C oracle
    releases the interpreter lock while it runs)."""
    s = OracleSample(T, zipf, pool=max(8, threads), shared=shared)
    s.run_assignments(s.units)  # warm (and its one-time tables) before any thread starts
    counts = [0] * threads
    stop = time.perf_counter() + seconds

    def worker(i):
        j = i
        while time.perf_counter() < stop:
            s.run_assignments(s.units, j)
            counts[i] += 1
            j += threads

    t0 = time.perf_counter()
    if threads == 1:
        worker(0)
    else:
        with cf.ThreadPoolExecutor(threads) as ex:
            list(ex.map(worker, range(threads)))
    wall = time.perf_counter() - t0
    return sum(counts) / wall, sum(counts), s.pool


def cpu_baseline(T, zipf, seconds, shared=False):
    """The oracle on this host: one core, then one thread per host CPU."""
    ncpu = os.cpu_count() or 1
    r1, n1, pool = oracle_rate(T, zipf, seconds, shared, 1)
    rn, nn, _ = oracle_rate(T, zipf, seconds, shared, ncpu)
    return {"value": rn, "unit": "tokens/s", "cores": ncpu, "kind": "oracle",
            "sample": f"{nn} tokens of the {T}-token workload in ~{seconds:.0f} s with {ncpu} threads (whole layer "
                      f"per token, tokens in turn over a {max(8, ncpu)}-token pool); one core: {n1} tokens",
            "single_core_value": r1, "host_cpus": ncpu, "cpu_model": cpu_model()}


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    T, zipf, _ = WORKLOADS[args.workload]
    if rank != 0:
        return
    s = OracleSample(T, zipf, shared=args.shared_expert)
    t1 = s.run_assignments(1)
    budget = 150.0 / max(1, args.steps + args.warmup)
    m = int(max(1, min(s.units, budget // max(t1, 1e-6))))
    for i in range(args.warmup):
        s.run_assignments(m, i)
    tot = 0.0
    for i in range(args.steps):
        tot += s.run_assignments(m, i)
    tok = args.steps * m / s.units
    value = tok / tot
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": workload_config(args.workload, world, args.shared_expert),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: routing + {m} of the {s.units} expert passes of one token "
                                       f"(tokens/s scaled by {m}/{s.units}); single-threaded C oracle",
                             "host_cpus": os.cpu_count(), "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ our arm

def max_over_ranks(dist, seconds: float) -> float:
    """The largest of the ranks' times (every rank gets it); the value itself
    without a process group."""
    if not dist:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_workload(moe, torch, dev, stream, layers, workload, K, warmup, graph_steps, nx, shared, seed,
                  dist=None, clocks=None, keep_warm_s=0.3):
    """K timed steps of `workload` on the given layer copies (its first NL).

    Step s of the run uses pair s % NG = (layer copy, token batch).
    Single-step graphs serve the routing pass and any remainder; the timed
    steps replay multi-step graphs of S consecutive steps, so the per-graph
    launch cost is paid once per S layer forwards (as in a model whose whole
    decode step is one graph).  Single-launch path: no events inside the
    timed graphs, its kernel time is the timed region over the K launches.
    Stage path: events bracket the gate/up launches of the first step of
    each graph."""
    T, zipf, NL = WORKLOADS[workload]
    layers = layers[:NL]
    NL = len(layers)  # fewer copies when the run was given --layers
    NX = nx
    NG = NL * NX if T <= 64 else NL
    gx = torch.Generator(device=dev)
    gx.manual_seed(seed)
    xs = torch.randn(NX, T, H, generator=gx, device=dev).to(torch.bfloat16)
    ws = moe.Workspace(T, layers[0], dev)
    torch.cuda.synchronize(dev)
    try:
        mk_ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        mk_ev()
        in_graph_events = True
    except TypeError:
        in_graph_events = False
    ml = moe.MoeLayer(layers[0])
    fused = ml.use_fused(T)
    one_launch = fused and (not shared or ml.shared_in_one_launch(T))
    stage = "decode" if fused else "gateup"   # the dominant kernel
    S = graph_steps if (graph_steps > 1 and NG % graph_steps == 0) else 1

    def pair(s):
        return layers[s % NG % NL], xs[(s % NG // NL) % NX]

    singles, multis, multi_events = [], [], []
    with torch.cuda.stream(stream):
        for gi in range(NG):
            lw, x = pair(gi)
            layer = moe.MoeLayer(lw)
            layer.forward(x, ws, stream)  # warm / first-call set-up outside capture
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                layer.forward(x, ws, stream)
            singles.append(g)
        for gj in range(NG // S):
            ev = {stage: (mk_ev(), mk_ev())} if (in_graph_events and not one_launch) else None
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(S):
                    lw, x = pair(gj * S + i)
                    moe.MoeLayer(lw).forward(x, ws, stream, events=ev if i == 0 else None)
            multis.append(g)
            multi_events.append(ev)
    torch.cuda.synchronize(dev)

    # routing of every step pair (for the algorithmic bytes)
    uniq = []
    for g in singles:
        g.replay()
        torch.cuda.synchronize(dev)
        uniq.append(int(torch.unique(ws.ids).numel()))
    A = T * K_TOP
    step_bytes = [ROUTER_BYTES + u * EXPERT_BYTES + T * H * 2 + T * H * 4 for u in uniq]
    routed_bytes = list(step_bytes)
    if shared:  # its weights, and its h and output rows
        step_bytes = [b + EXPERT_BYTES + T * I_EXP * 4 * 2 + T * H * 4 * 2 for b in step_bytes]
    if one_launch:  # the one kernel moves the whole layer (shared expert included)
        gu_bytes = list(step_bytes)
    elif fused:  # the single launch moves the routed layer; the shared expert's calls follow
        gu_bytes = routed_bytes
    else:
        gu_bytes = [u * 2 * I_EXP * (H // 2 + H // 32) + T * (H + H // 32 * 4) + A * I_EXP * 4 for u in uniq]

    def run(n, start=0):
        s, end = start, start + n
        while s < end:
            if s % S == 0 and end - s >= S:
                multis[(s % NG) // S].replay()
                s += S
            else:
                singles[s % NG].replay()
                s += 1

    with torch.cuda.stream(stream):
        run(max(3, warmup))
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < keep_warm_s:
            run(NG)
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    # timed region: exactly K steps, starting at step 0 of the cycle
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if clocks is not None:
        clocks.__enter__()
    try:
        if dist:
            dist.barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            ev0.record(stream)
            run(K)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
        if dist:
            dist.barrier()
    finally:
        if clocks is not None:
            clocks.__exit__(None, None, None)
    ms = ev0.elapsed_time(ev1)
    if one_launch:
        # one launch per step: the kernel's average duration over the timed
        # region (launch gaps included, so an upper bound)
        gu_steps, gu_ms = list(range(K)), [ms / K] * K
    elif in_graph_events:
        firsts = [s for s in range(0, K - K % S, S)][-len(multis):]
        gu_steps = firsts
        gu_ms = [multi_events[(s % NG) // S][stage][0].elapsed_time(multi_events[(s % NG) // S][stage][1])
                 for s in firsts]
    else:
        gu_steps, gu_ms = [], []
    ms = max_over_ranks(dist, ms)
    bytes_mean = sum(step_bytes[s % NG] for s in range(K)) / K
    if one_launch and shared:
        rk = "moe_decode_forward_shared"
    elif fused:
        rk = "moe_decode_forward"
    else:
        rk = "moe_mxfp4_gateup_swiglu"
    return dict(T=T, NL=NL, NX=NX, S=S, ms=ms, fused=fused, one_launch=one_launch, uniq=uniq,
                bytes_mean=bytes_mean, gu_steps=gu_steps, gu_ms=gu_ms, gu_bytes=gu_bytes, NG=NG, kernel=rk,
                launches=K * ml.kernels_per_forward(T), xs=xs, ws=ws)


def roofline_of(r, workload, hbm_peak, peak_kind):
    if not r["gu_ms"]:
        return None
    NG = r["NG"]
    gb = sum(r["gu_bytes"][s % NG] for s in r["gu_steps"])
    sec = sum(r["gu_ms"]) * 1e-3
    achieved = gb / sec / 1e9
    rk = r["kernel"]
    traffic = ncu_traffic(workload, rk)
    return {"kernel": rk, "bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": traffic, "peak_kind": peak_kind,
            "launches_timed": len(r["gu_ms"]), "avg_launch_us": 1e6 * sec / len(r["gu_ms"]),
            "algorithmic_bytes_per_launch": gb / len(r["gu_ms"])}


def mxf4_peak(moe, torch, stream):
    """Measured dense FP4 tensor-core rate (TFLOP/s) of the instruction the
    tensor-core path issues, at N = 256 (the dense peak) and at N = 64 (the
    expert kernel's shape); best of three launches each."""
    out = {}
    for n in (256, 64):
        best = 0.0
        with torch.cuda.stream(stream):
            moe.moe_mxf4_mma_probe(n, 1 << 12, stream)
            for _ in range(3):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fl = moe.moe_mxf4_mma_probe(n, 1 << 17, stream)
                e1.record(stream)
                e1.synchronize()
                best = max(best, fl / (e0.elapsed_time(e1) * 1e-3) / 1e12)
        out[n] = best
    return out


def sub_record(moe, torch, dev, stream, layers, workload, hbm_peak, peak_kind, fp4_peak):
    """A short measurement of another workload of the metric's range on the
    same layer copies (no clocks sampler, no e2e): its own tokens/s, layer
    GB/s and roofline of its dominant kernel."""
    T = WORKLOADS[workload][0]
    K = 32 if T <= 64 else 8
    r = time_workload(moe, torch, dev, stream, layers, workload, K, 3, 16, 2, False, seed=11, keep_warm_s=0.1)
    ms_step = r["ms"] / K
    layer_gbs = r["bytes_mean"] / (ms_step * 1e-3) / 1e9
    rec = {"workload": workload, "value": T * K / (r["ms"] * 1e-3), "unit": "tokens/s", "steps": K,
           "ms_per_step": ms_step, "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / hbm_peak,
           "roofline": roofline_of(r, workload, hbm_peak, peak_kind),
           "distinct_experts_mean": sum(r["uniq"]) / len(r["uniq"]),
           "path": "fused single-launch decode" if r["fused"] else "stage calls",
           "gpu_launches": r["launches"]}
    if rec["roofline"] and not r["fused"] and fp4_peak:
        # the gate/up projections as tensor work: useful multiply-adds (x2)
        # over the measured dense FP4 rate of the tensor-core instruction
        fl = 2.0 * T * K_TOP * 2 * I_EXP * H
        tf = fl / (rec["roofline"]["avg_launch_us"] * 1e-6) / 1e12
        rec["tensor"] = {"achieved": tf, "peak": fp4_peak, "unit": "TFLOP/s", "frac": tf / fp4_peak,
                         "peak_kind": "measured (moe_mxf4_mma_probe, N=256)",
                         "flops_per_launch": fl}
    return rec


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    import torch
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
        if dist:
            dist.barrier()
            dist.destroy_process_group()
        return

    import __graft_entry__
    __graft_entry__.build()
    import mxfp4_mixture_experts_moe_gb300 as moe
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    T, zipf, NL = WORKLOADS[args.workload]
    if args.layers > 0:
        NL = args.layers
        WORKLOADS[args.workload] = (T, zipf, NL)
    NX = 16 if T <= 64 else 2          # distinct token batches
    layers = [make_layer(moe, torch, 1000 * rank + l, zipf, dev, shared=args.shared_expert) for l in range(NL)]
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)  # weights are written on the default stream

    clocks = ClockSampler(local)
    r = time_workload(moe, torch, dev, stream, layers, args.workload, args.steps, args.warmup, args.graph_steps, NX,
                      args.shared_expert, seed=7 + rank, dist=dist, clocks=clocks)
    K = args.steps
    ms = r["ms"]
    ms_step = ms / K
    value = world * T * K / (ms * 1e-3)
    hbm_peak, peak_kind = peaks()
    roofline = roofline_of(r, args.workload, hbm_peak, peak_kind)
    layer_gbs = r["bytes_mean"] / (ms_step * 1e-3) / 1e9

    # ---- end to end: pinned host x in, host out, synchronised every step
    e2e = None
    if not args.no_e2e:
        xs, ws = r["xs"], r["ws"]
        xh = torch.empty(NX, T, H, dtype=torch.bfloat16).pin_memory()
        xh.copy_(xs.cpu())
        outh = torch.empty(T, H, dtype=torch.float32).pin_memory()
        xin = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        eg = []
        with torch.cuda.stream(stream):
            for l in range(NL):
                layer = moe.MoeLayer(layers[l])
                layer.forward(xin, ws, stream)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    layer.forward(xin, ws, stream)
                eg.append(g)
            torch.cuda.synchronize(dev)
            Ke = min(K, 2000)
            for s in range(5):
                xin.copy_(xh[s % NX], non_blocking=True)
                eg[s % NL].replay()
                outh.copy_(ws.out, non_blocking=True)
                stream.synchronize()
            if dist:
                dist.barrier()
            t0 = time.perf_counter()
            for s in range(Ke):
                xin.copy_(xh[s % NX], non_blocking=True)
                eg[s % NL].replay()
                outh.copy_(ws.out, non_blocking=True)
                stream.synchronize()
            e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(dist, e2e_s)
        n_k = moe.MoeLayer(layers[0]).kernels_per_forward(T)
        path = "the single fused launch" if n_k == 1 else f"the stage calls ({n_k} kernels)"
        e2e = {"value": world * T * Ke / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
               "d2h_bytes_per_step": T * H * 4,
               "how": f"pinned host x -> device, graph replay of {path}, out -> pinned host, stream sync, every step"}

    # ---- the rest of the metric's range on the same layer copies, and the
    # measured FP4 tensor rate the prefill projections are reported against
    subs, fp4 = None, None
    if rank == 0 and world == 1 and args.workload == "decode-1" and not args.shared_expert and not args.no_sub:
        fp4 = mxf4_peak(moe, torch, stream)
        subs = [sub_record(moe, torch, dev, stream, layers, w, hbm_peak, peak_kind, fp4[256])
                for w in ("krow-16", "prefill-512")]

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(T, zipf, args.cpu_seconds, shared=args.shared_expert)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": ARITHMETIC if T < 17 else ARITHMETIC_TENSOR, "data": "synthetic",
            "config": workload_config(args.workload, world, args.shared_expert),
            "run": {"l2": f"{NL} layer copies x {r['NX']} token batches cycled ({NL * 3.42:.1f} GB of weights > L2)",
                    "graph": f"CUDA graphs of {r['S']} consecutive layer forwards (distinct layer copies), "
                             "replayed back to back",
                    "path": ("fused single-launch decode" if r["fused"] else "stage calls")
                            + ("" if not args.shared_expert else " with the shared expert" if r["one_launch"]
                               else " + the shared expert's stage calls"),
                    "distinct_experts_mean": sum(r["uniq"]) / len(r["uniq"])},
            "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / hbm_peak,
            "roofline": roofline,
            "sub_records": subs,
            "tensor_peak_tflops": None if fp4 is None else {"mxf4_n256": fp4[256], "mxf4_n64": fp4[64],
                                                           "how": "moe_mxf4_mma_probe, best of 3 launches"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": r["launches"],
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
