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
import json
import os
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
# roofline kernel, from one ncu capture of the current kernels on a one-layer
# copy of the workload; workloads without a capture report null.
NCU_TRAFFIC = {
    ("decode-1", "moe_decode_forward"): 84.02e6,
    ("decode-1", "moe_decode_forward_shared"): 98.02e6,
    ("prefill-512", "moe_mxfp4_gateup_swiglu"): 2.3209e9,
}


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
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target oracle time of the cpu_baseline sample")
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


def oracle_rate(T, zipf, seconds, shared=False):
    """tokens/s of the oracle over ~`seconds` of CPU work (one core)."""
    s = OracleSample(T, zipf, shared=shared)
    s.run_assignments(1)  # warm
    done_tok, spent, i = 0.0, 0.0, 0
    while spent < seconds:
        spent += s.run_assignments(s.units, i)
        done_tok += 1
        i += 1
    return done_tok / spent, f"{int(done_tok)} tokens of the {T}-token workload (whole layer per token, " \
                             f"{s.pool}-token pool), oracle single-threaded"


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
            "config": {"workload": args.workload, "tokens_per_step": T, "hidden": H, "experts": E, "top_k": K_TOP,
                       "expert_intermediate": I_EXP, "shared_expert": args.shared_expert},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                             "sample": f"each step: routing + {m} of the {s.units} expert passes of one token "
                                       f"(tokens/s scaled by {m}/{s.units}); single-threaded C oracle"},
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
    NX = 16 if T <= 64 else 2          # distinct token batches
    NG = NL * NX if T <= 64 else NL    # graphs: (layer copy, batch) pairs
    layers = [make_layer(moe, torch, 1000 * rank + l, zipf, dev, shared=args.shared_expert) for l in range(NL)]
    gx = torch.Generator(device=dev)
    gx.manual_seed(7 + rank)
    xs = torch.randn(NX, T, H, generator=gx, device=dev).to(torch.bfloat16)
    ws = moe.Workspace(T, layers[0], dev)
    stream = torch.cuda.Stream(device=dev)
    torch.cuda.synchronize(dev)  # weights, inputs and workspace are written on the default stream

    # ---- graphs.  Step s of the run uses pair s % NG = (layer copy, batch).
    # Single-step graphs serve the routing pass and any remainder; the timed
    # steps replay multi-step graphs of S consecutive steps, so the per-graph
    # launch cost is paid once per S layer forwards (as in a model whose whole
    # decode step is one graph).  Fused path: no events inside the timed
    # graphs, its kernel time is the timed region over K launches.  Stage
    # path: events bracket the gate/up kernel of the first step of each graph.
    try:
        mk_ev = lambda: torch.cuda.Event(enable_timing=True, external=True)  # noqa: E731
        mk_ev()
        in_graph_events = True
    except TypeError:
        in_graph_events = False
    fused = moe.MoeLayer(layers[0]).use_fused(T)
    # one launch per step (the shared expert, if any, inside it): its time is
    # the timed region over the steps; else events bracket the dominant kernel
    one_launch = fused and (not args.shared_expert or moe.MoeLayer(layers[0]).shared_in_one_launch(T))
    stage = "decode" if fused else "gateup"   # the dominant kernel
    S = args.graph_steps if (args.graph_steps > 1 and NG % args.graph_steps == 0) else 1

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

    # ---- routing of every step pair (for algorithmic bytes)
    uniq = []
    for g in singles:
        g.replay()
        torch.cuda.synchronize(dev)
        uniq.append(int(torch.unique(ws.ids).numel()))
    A = T * K_TOP
    step_bytes = [ROUTER_BYTES + u * EXPERT_BYTES + T * H * 2 + T * H * 4 for u in uniq]
    routed_bytes = list(step_bytes)
    if args.shared_expert:  # its weights, and its h and output rows
        step_bytes = [b + EXPERT_BYTES + T * I_EXP * 4 * 2 + T * H * 4 * 2 for b in step_bytes]
    if one_launch:  # the one kernel moves the whole layer (shared expert included)
        gu_bytes = list(step_bytes)
    elif fused:  # the single launch moves the routed layer; the shared expert's calls follow
        gu_bytes = routed_bytes
    else:
        gu_bytes = [u * 2 * I_EXP * (H // 2 + H // 32) + T * (H + H // 32 * 4) + A * I_EXP * 4 for u in uniq]

    def run(n, start=0):
        """Steps start .. start+n-1: whole multi-step graphs where they line
        up, single-step graphs for the rest."""
        s, end = start, start + n
        while s < end:
            if s % S == 0 and end - s >= S:
                multis[(s % NG) // S].replay()
                s += S
            else:
                singles[s % NG].replay()
                s += 1

    # ---- warm-up: W steps, plus enough to bring clocks up (~0.3 s)
    with torch.cuda.stream(stream):
        run(max(3, args.warmup))
        t0 = time.perf_counter()
        while time.perf_counter() - t0 < 0.3:
            run(NG)
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)

    # ---- timed region: exactly K steps, starting at step 0 of the cycle
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    with clocks:
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
    ms = ev0.elapsed_time(ev1)
    if one_launch:
        # one launch per step: the kernel's average duration over the timed
        # region (launch gaps included, so an upper bound)
        gu_steps = list(range(K))
        gu_ms = [ms / K] * K
    elif in_graph_events:
        # the dominant launches (gate/up; or the routed single launch when the
        # shared expert's calls follow it) of the first step of the last
        # multi-step graphs replayed
        firsts = [s for s in range(0, K - K % S, S)][-len(multis):]
        gu_steps = firsts
        gu_ms = [multi_events[(s % NG) // S][stage][0].elapsed_time(multi_events[(s % NG) // S][stage][1])
                 for s in firsts]
    else:
        gu_steps, gu_ms = [], []
    ms = max_over_ranks(dist, ms)
    ms_step = ms / K
    bytes_mean = sum(step_bytes[s % NG] for s in range(K)) / K
    value = world * T * K / (ms * 1e-3)

    # ---- end to end: pinned host x in, host out, synchronised every step
    e2e = None
    if not args.no_e2e:
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
        e2e_value = world * T * Ke / e2e_s

        e2e = {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
               "d2h_bytes_per_step": T * H * 4,
               "how": "pinned host x -> device, graph replay of the six ABI calls, out -> pinned host, "
                      "stream sync, every step"}

    hbm_peak, peak_kind = peaks()
    roofline = None
    if gu_ms:
        gb = sum(gu_bytes[s % NG] for s in gu_steps)
        achieved = gb / (sum(gu_ms) * 1e-3) / 1e9
        rk = ("moe_decode_forward_shared" if one_launch and args.shared_expert else "moe_decode_forward") if fused \
            else "moe_mxfp4_gateup_swiglu"
        roofline = {"kernel": rk, "bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                    "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": NCU_TRAFFIC.get((args.workload, rk)),
                    "peak_kind": peak_kind, "launches_timed": len(gu_ms),
                    "avg_launch_us": 1e3 * sum(gu_ms) / len(gu_ms),
                    "algorithmic_bytes_per_launch": gb / len(gu_ms)}
    layer_gbs = bytes_mean / (ms_step * 1e-3) / 1e9

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, sample = oracle_rate(T, zipf, args.cpu_seconds, shared=args.shared_expert)
        cpu = {"value": rate, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {"workload": args.workload, "tokens_per_step": T, "hidden": H, "experts": E, "top_k": K_TOP,
                       "expert_intermediate": I_EXP, "weights": "MXFP4 E2M1 + E8M0/32, random init",
                       "activations": "bf16 N(0,1) -> Q8 per 32", "router": "bf16",
                       "zipf_bias": zipf, "parallelism": f"replicas{world}",
                       "l2": f"{NL} layer copies x {NX} token batches cycled ({NL * 3.42:.1f} GB of weights > L2)",
                       "graph": f"CUDA graphs of {S} consecutive layer forwards (distinct layer copies), replayed back to back",
                       "path": ("fused single-launch decode" if fused else "six stage calls (8 kernels)")
                               + ("" if not args.shared_expert else " with the shared expert" if one_launch
                                  else " + the shared expert's stage calls"),
                       "shared_expert": args.shared_expert,
                       "distinct_experts_mean": sum(uniq) / len(uniq)},
            "layer_hbm_gbs": layer_gbs, "layer_hbm_frac": layer_gbs / hbm_peak,
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": K * moe.MoeLayer(layers[0]).kernels_per_forward(T),
            "clocks": clocks.summary(),
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
