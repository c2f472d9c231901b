"""Throughput benchmark of the MiTA forward operator on B300.

One step = one ``mita_forward`` over the whole batch of the workload (all
six steps of the operator).  Default workload: the DeiT-S-shaped layer
(B=256, H=6, N=196 on a 14x14 grid, d=64, m=25 from 5x5 pooling, k=25,
bf16, clustered tokens).  Metric: query-heads per second (B*H*N per step
divided by the step time).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mita|reference]
Under torchrun each rank runs its own copy of the workload (heads are
independent, so the batch shards over ranks with no collective on the data
path: weak scaling); the timing is the max over ranks.

``--impl reference`` times the CPU oracle (the plain fp64 restatement the
tests use) on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math

import numpy as np
import os
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mixture_top_attention_mita_b300 import synth  # noqa: E402

METRIC = "MiTA fwd query-heads/s at DeiT-S shape (m=k=25); % of HBM/tensor roofline"
L2_BYTES = 126 * 1024 * 1024


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="mita", choices=["mita", "reference"])
    ap.add_argument("--workload", default="deit_s", choices=sorted(synth.WORKLOADS))
    ap.add_argument("--path", default="auto", choices=["auto", "staged", "fused", "tiled"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time K stream launches instead of one CUDA graph of the K steps")
    ap.add_argument("--routing-only", action="store_true",
                    help="the routing-only variant: the shared expert dropped from every query's softmax")
    ap.add_argument("--routes", type=int, default=1,
                    help="experts per query (s > 1 runs on the staged path)")
    ap.add_argument("--long-sweep", action="store_true",
                    help="long-sequence throughput against full attention (one JSON line per length)")
    ap.add_argument("--backward", action="store_true",
                    help="time mita_backward (input gradients for an output gradient) instead of the forward")
    ap.add_argument("--no-soak", action="store_true", help="skip the untimed repeats that extend clock sampling")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the graph-timed forwards of the other workloads reported beside the main line")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch B (smaller cases for profiler captures)")
    ap.add_argument("--heads", type=int, default=None, help="override the workload's head count H")
    return ap.parse_args()


def algorithmic(w, backward=False):
    """Compulsory HBM bytes and algorithmic FLOPs per step: read Q, K, V once,
    write out, expert indices and routes; FLOPs of the six contractions
    (landmark scores, landmark values, query-landmark scores reused for the
    route, shared and routed QK and PV).  Backward: read Q, K, V and dOut,
    write fp32 dQ, dK, dV; the forward's contractions once (recomputed) and
    twice more for the gradients."""
    e = 2 if w.dtype == "bf16" else 4
    per_head_flops = 4 * w.N * w.d * (2 * w.m + w.k)
    if backward:
        return (4 * w.N * w.d * e + 3 * w.N * w.d * 4) * w.heads, 3 * per_head_flops * w.heads
    per_head_bytes = 4 * w.N * w.d * e + 4 * w.m * w.k + 4 * w.N
    return per_head_bytes * w.heads, per_head_flops * w.heads


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained"), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def workload_desc(w, routes=1):
    grid = f"{w.gh}x{w.gw}" if w.gh > 1 else f"1-D {w.N}"
    return (f"{w.name}: B={w.B} H={w.H} N={w.N} ({grid}) d={w.d} m={w.m} ({w.ph}x{w.pw}) k={w.k} "
            f"s={routes} {w.dtype} {w.gen}")


# Sources each recorded kernel is compiled from (its DRAM traffic changes only
# with these); any other tag hashes every CUDA source.
KERNEL_SOURCES = {"mita_fused": ["csrc/fused.cu", "csrc/fused.cuh", "csrc/common.cuh", "../include/mita.h"]}


def source_hash(kernel_tag=None):
    import hashlib
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "mixture_top_attention_mita_b300")
    csrc = os.path.join(pkg, "csrc")
    if kernel_tag in KERNEL_SOURCES:
        files = [os.path.normpath(os.path.join(pkg, f)) for f in KERNEL_SOURCES[kernel_tag]]
    else:
        files = [os.path.join(csrc, fn) for fn in sorted(os.listdir(csrc)) if fn.endswith((".cu", ".cuh"))]
    for fn in files:
        h.update(open(fn, "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profiles(kernel_tag, workload):
    """DRAM bytes per launch recorded from an ncu capture of this kernel on
    this workload, or None when none is recorded or the kernel sources have
    changed since."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    want = source_hash(kernel_tag)
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        f = dict(kv.split("=", 1) for kv in line.split())
        if f.get("kernel") == kernel_tag and f.get("workload") == workload and f.get("src") == want:
            return float(f["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = max(mx, float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


def variant_name(args):
    """The operator variant a run measures: mita, routing_only, routes_s<S>, backward."""
    parts = (["routing_only"] if args.routing_only else []) + ([f"routes_s{args.routes}"] if args.routes > 1 else [])
    parts += ["backward"] if getattr(args, "backward", False) else []
    return "+".join(parts) if parts else "mita"


def _oracle_sample(w, seconds, threads, shared=True, routes=1, backward=False):
    """Time the CPU oracle (fp64) on ``threads`` host threads, whole heads of
    the workload spread over the threads, until about ``seconds`` of work.
    Returns (query-heads/s, description of the sample).  A long sequence
    (N > 16384) takes all landmark work of one head over the threads and the
    route and attend steps of a slice of its queries; the per-query time is
    scaled to all N queries run on the same threads, which the description
    says."""
    import oracle
    if w.N > 16384 and not backward:
        Q, K, V = synth.make_inputs(w.scaled(B=1, H=1))
        nq = 256
        qs = list(range(0, w.N, w.N // nq))[:nq]
        t0 = time.perf_counter()
        oracle.head_threaded(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io=w.dtype, queries=qs[:1],
                             shared=shared, threads=threads)
        t_land = time.perf_counter() - t0
        t1 = time.perf_counter()
        oracle.head_threaded(Q[0, 0], K[0, 0], V[0, 0], w.grid, w.m, w.k, io=w.dtype, queries=qs, shared=shared,
                             threads=threads)
        per_q = max(0.0, (time.perf_counter() - t1 - t_land) / (nq - 1))
        per_head = t_land + per_q * w.N / threads
        return w.N / per_head, (f"1 head of {w.name}: every landmark row on {threads} thread(s), route+attend of "
                                f"{nq} queries; per-query time scaled to {w.N} queries over {threads} thread(s)")
    n_heads = 16 * threads   # enough heads per batch that every thread stays busy
    H = min(w.H, n_heads)
    B = -(-n_heads // H)
    sample = w.scaled(B=B, H=H)
    Q, K, V = synth.make_inputs(sample)
    heads = [(b, h) for b in range(B) for h in range(H)]
    G = None
    if backward:
        G = np.random.default_rng(0).standard_normal((w.N, w.d))
    done, t0 = 0, time.perf_counter()
    while True:
        if backward:
            from concurrent.futures import ThreadPoolExecutor
            Qf, Kf, Vf = Q.double().numpy(), K.double().numpy(), V.double().numpy()
            with ThreadPoolExecutor(max_workers=threads) as ex:
                list(ex.map(lambda bh: oracle.backward(Qf[bh], Kf[bh], Vf[bh], G, w.grid, w.m, w.k, io=w.dtype,
                                                       shared=shared), heads))
            done += len(heads)
        else:
            done += oracle.forward_heads_threaded(Q, K, V, w.grid, w.m, w.k, heads, io=w.dtype, shared=shared,
                                                  s=routes, threads=threads)
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return done * w.N / el, f"{done} whole heads of {w.name} ({done * w.N} query-heads) on {threads} thread(s), {el:.1f} s"


def cpu_baseline(w, seconds, shared=True, routes=1, backward=False):
    """The CPU oracle timed on the host cores: on every core the process may
    run on (``cores``, one thread each, heads spread over them) and on one
    core (``value_1core``), about ``seconds`` of work in all; query-heads/s
    (``shared=False``: the routing-only variant)."""
    import oracle
    cores = oracle.threads_available()
    vn, sn = _oracle_sample(w, seconds / 2, cores, shared, routes, backward)
    v1, s1 = _oracle_sample(w, seconds / 2, 1, shared, routes, backward)
    return {"value": vn, "unit": "query-heads/s", "cores": cores, "kind": "oracle", "value_1core": v1,
            "sample": f"{sn}; one core: {s1}"}


def bench_config(w, ws, routes, variant):
    """The ``config`` object both arms print: the workload, its batch and
    sequence length, the sharding and the L2 rule of the timed loop."""
    e = 2 if w.dtype == "bf16" else 4
    set_bytes = 4 * w.heads * w.N * w.d * e
    nsets = min(8, max(2, math.ceil(3 * L2_BYTES / set_bytes) + 1))
    return {"workload": workload_desc(w, routes), "global_batch": w.B * ws, "seq_len": w.N,
            "parallelism": f"heads sharded over {ws} GPU(s), no collective", "variant": variant,
            "l2": f"inputs rotate over {nsets} buffer sets ({nsets * set_bytes / 1e6:.0f} MB > 126 MB L2)"}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, ws, device):
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, ms_per_rank, ws, device):
    """Whole-job throughput: every rank processes units_per_rank units; the
    job takes as long as its slowest rank (max over ranks)."""
    ms = max_over_ranks(ms_per_rank, ws, device)
    return ws * units_per_rank / (ms / 1000.0), ms


def run_reference(args, w, ws, rank):
    """The reference arm: the CPU oracle on every host core.  Each step runs
    a bounded sample of the workload's heads (sized so that all steps take
    about --cpu-seconds) and is timed as it runs; ms_per_step is that time,
    value the sample's query-heads over it (median step).  The time the
    whole workload would take at that rate is reported apart, labelled as an
    extrapolation."""
    if rank != 0:
        return 0
    import oracle
    cores = oracle.threads_available()
    per_step = max(0.05, args.cpu_seconds / max(1, args.steps + args.warmup))
    rates, times, sample = [], [], ""
    for st in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, sample = _oracle_sample(w, per_step, cores, shared=not args.routing_only, routes=args.routes,
                                   backward=args.backward)
        el = time.perf_counter() - t0
        if st >= args.warmup:
            rates.append(v)
            times.append(el)
    order = sorted(range(len(rates)), key=lambda i: rates[i])
    mid = order[len(order) // 2]
    v, ms = rates[mid], 1000.0 * times[mid]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "query-heads/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded generator, no dataset)",
            "config": bench_config(w, ws, args.routes, variant_name(args)),
            "extrapolated_ms_per_full_workload": round(1000.0 * w.heads * w.N / v, 1),
            "cpu_baseline": {"value": v, "unit": "query-heads/s", "cores": cores, "kind": "oracle",
                             "sample": sample + " per step; median step"},
            "e2e": {"value": v, "unit": "query-heads/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def long_sweep(args):
    """MiTA forward against full attention (torch scaled_dot_product_attention,
    the fused flash kernel) on single-head 1-D sequences with m * k = N / 4,
    d = 128, bf16 (the shape of the method's long-sequence throughput figure).
    One JSON line per length: both times from CUDA events, median of a few
    runs after a warm-up."""
    import mixture_top_attention_mita_b300 as mita
    dev = torch.device("cuda")
    for N, m, k in ((16384, 64, 64), (65536, 128, 128), (262144, 256, 256), (1048576, 256, 1024)):
        w = synth.WORKLOADS["long1d"].scaled(name=f"long_{N}", B=1, H=1, N=N, gw=N, pw=m, m=m, k=k,
                                             span=1024, seed=2000 + N % 997)
        Qc, Kc, Vc = synth.make_inputs(w)
        Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
        out = torch.empty_like(Q)
        plan = mita.Plan.for_workload(w)

        def timed(fn, reps):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            ts = []
            for _ in range(reps):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                fn()
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b))
            return sorted(ts)[len(ts) // 2]

        t_mita = timed(lambda: plan.forward(Q, K, V, out), 5)
        st = plan.status()
        t_sdpa = timed(lambda: torch.nn.functional.scaled_dot_product_attention(Q, K, V), 3 if N > 300000 else 5)
        print(json.dumps({"sweep": "long_sequence", "N": N, "m": m, "k": k, "d": w.d, "dtype": w.dtype,
                          "path": plan.path, "status": st, "mita_ms": round(t_mita, 4),
                          "full_attention_ms": round(t_sdpa, 4), "speedup": round(t_sdpa / t_mita, 2)}))
        plan.close()
        del Q, K, V, out
        torch.cuda.empty_cache()
    return 0


def measure_forward(mita, w, steps, dev, stream):
    """The graph-timed forward of another workload with the main line's
    method: rotating input sets above L2, the K steps captured once into one
    CUDA graph and replayed between CUDA events.  Returns ms per step and the
    roofline fraction of measured peak (the slower of HBM and tensor time)."""
    Qc, Kc, Vc = synth.make_inputs(w)
    set_bytes = 4 * Qc.numel() * Qc.element_size()
    nsets = min(8, max(2, math.ceil(3 * L2_BYTES / set_bytes) + 1))
    sets = []
    for _ in range(nsets):
        Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
        sets.append((Q, K, V, torch.empty_like(Q), torch.empty(w.B, w.H, w.m, w.k, dtype=torch.int32, device=dev),
                     torch.empty(w.B, w.H, w.N, dtype=torch.int32, device=dev)))
    plan = mita.Plan.for_workload(w)
    for i in range(3):
        plan.forward(*sets[i % nsets], stream)
    if plan.status() != mita.MITA_OK:
        raise RuntimeError(f"{w.name}: device status {plan.status()}")
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
        cs = torch.cuda.current_stream()
        for i in range(steps):
            plan.forward(*sets[i % nsets], cs)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    if plan.status() != mita.MITA_OK:
        raise RuntimeError(f"{w.name}: device status after the timed steps")
    ms = e0.elapsed_time(e1) / steps
    nbytes, flops = algorithmic(w)
    pk = peaks()
    t_hbm, t_tc = nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12)
    out = {"workload": workload_desc(w), "path": plan.path, "ms_per_step": round(ms, 5),
           "value": w.heads * w.N / (ms / 1000.0), "unit": "query-heads/s",
           "roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor", "frac": round(max(t_hbm, t_tc) / (ms / 1000.0), 4)},
           "steps": steps, "l2": f"inputs rotate over {nsets} buffer sets"}
    plan.close()
    del sets, g
    torch.cuda.empty_cache()
    return out


def main():
    args = parse()
    ws, rank, local = dist_setup()
    w = synth.WORKLOADS[args.workload]
    if args.batch is not None or args.heads is not None:
        B, H = args.batch or w.B, args.heads or w.H
        w = w.scaled(name=f"{w.name}_B{B}_H{H}", B=B, H=H)
    if args.impl == "reference":
        return run_reference(args, w, ws, rank)
    if args.long_sweep:
        return long_sweep(args) if rank == 0 else 0

    import mixture_top_attention_mita_b300 as mita
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    plan = mita.Plan.for_workload(w)
    plan.set_path(args.path)
    if args.routing_only:
        plan.set_option(mita.OPT_ROUTING_ONLY, 1)
    if args.routes > 1:
        plan.set_option(mita.OPT_ROUTES, args.routes)
    path = "staged" if args.backward else plan.path   # the backward runs the stage-by-stage kernels
    stream = torch.cuda.current_stream()

    # inputs: enough rotating sets that consecutive steps never hit in L2
    Qc, Kc, Vc = synth.make_inputs(w, seed=w.seed + 7919 * rank)
    set_bytes = 4 * Qc.numel() * Qc.element_size()
    nsets = min(8, max(2, math.ceil(3 * L2_BYTES / set_bytes) + 1))   # as bench_config states
    sets = []
    for s in range(nsets):
        Q, K, V = Qc.to(dev), Kc.to(dev), Vc.to(dev)
        out = torch.empty_like(Q)
        idx = torch.empty(w.B, w.H, w.m, w.k, dtype=torch.int32, device=dev)
        route = torch.empty(w.B, w.H, w.N, dtype=torch.int32, device=dev)
        sets.append((Q, K, V, out, idx, route))

    grads = None
    if args.backward:
        gen = torch.Generator("cpu").manual_seed(w.seed + 17)
        dOuts = [torch.randn(Qc.shape, generator=gen).to(Qc.dtype).to(dev) for _ in range(nsets)]
        grads = [torch.empty(Qc.shape, dtype=torch.float32, device=dev) for _ in range(3)]

    def step(i, st=None):
        Q, K, V, out, idx, route = sets[i % nsets]
        if args.backward:
            plan.backward(Q, K, V, dOuts[i % nsets], *grads, st or stream)
        else:
            plan.forward(Q, K, V, out, idx, route, st or stream)

    for i in range(args.warmup):
        step(i)
    st = plan.status()
    if st != mita.MITA_OK:
        raise SystemExit(f"device status {mita.STATUS.get(st, st)}")

    # The K timed steps are captured once into one CUDA graph (step i on
    # buffer set i mod nsets, exactly as the stream loop would launch them)
    # and replayed once: the device runs the K forwards back to back, with
    # no host launch latency between them.  --no-graph times K launches from
    # the host instead; the stream-launched time is reported beside either.
    g, graph_error, launches = None, None, 0
    if not args.no_graph:
        try:
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            l0 = plan.launch_count()
            with torch.cuda.graph(g, stream=side, capture_error_mode="thread_local"):
                cs = torch.cuda.current_stream()
                for i in range(args.steps):
                    step(i, cs)
            launches = plan.launch_count() - l0
            g.replay()                 # untimed: the graph's first upload
            torch.cuda.synchronize()
            st = plan.status()
            if st != mita.MITA_OK:
                raise RuntimeError(f"device status {mita.STATUS.get(st, st)}")
        except Exception as exc:       # reported; the stream loop is timed instead
            g, graph_error = None, str(exc).splitlines()[0][:200]

    def timed_steps(use_graph):
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        if use_graph:
            g.replay()
        else:
            for i in range(args.steps):
                step(i)
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        return e0.elapsed_time(e1) / args.steps

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.2)
    if g is not None:
        ms = timed_steps(True)
    else:
        l0 = plan.launch_count()
        ms = timed_steps(False)
        launches = plan.launch_count() - l0
    # keep the same load running until the clock sampler has seen >= 1 s
    t_end = time.time() + (0.0 if args.no_soak else max(0.0, 1.0 - ms * args.steps / 1000.0))
    while time.time() < t_end:
        if g is not None:
            g.replay()
        else:
            for i in range(args.steps):
                step(i)
        torch.cuda.synchronize()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    st = plan.status()
    if st != mita.MITA_OK:
        raise SystemExit(f"device status {mita.STATUS.get(st, st)}")
    stream_ms = max_over_ranks(timed_steps(False), ws, dev) if g is not None else None
    st = plan.status()
    if st != mita.MITA_OK:
        raise SystemExit(f"device status {mita.STATUS.get(st, st)}")
    qh = w.heads * w.N
    value, ms = whole_job_rate(qh, ms, ws, dev)
    nbytes, flops = algorithmic(w, args.backward)
    pk = peaks()
    # dominant kernel: on the fused path the step is one launch; on the
    # staged path the whole step is reported (kernel-level shares live in
    # the ncu launch list under profiles/).
    kernel_tag = "mita_fused" if path == "fused" and not args.backward else \
        f"mita_{'backward' if args.backward else path}_step"
    t_s = ms / 1000.0
    bw = nbytes / t_s / 1e9
    tf = flops / t_s / 1e12
    hbm_frac = bw / pk["hbm_gbs"]
    roof_t = max(nbytes / (pk["hbm_gbs"] * 1e9), flops / (pk["bf16_tflops"] * 1e12))
    bound = "hbm" if nbytes / (pk["hbm_gbs"] * 1e9) >= flops / (pk["bf16_tflops"] * 1e12) else "tensor"
    traffic = traffic_from_profiles(kernel_tag, w.name if variant_name(args) == "mita" else
                                    w.name + "+" + variant_name(args))
    roofline = {"bound": bound, "achieved": round(bw if bound == "hbm" else tf, 2),
                "peak": pk["hbm_gbs"] if bound == "hbm" else pk["bf16_tflops"],
                "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
                "frac": round((bw / pk["hbm_gbs"]) if bound == "hbm" else tf / pk["bf16_tflops"], 4),
                "traffic": traffic, "kernel": kernel_tag,
                "algorithmic_bytes_per_launch": nbytes, "algorithmic_flops_per_launch": flops,
                "roofline_frac_of_step": round(roof_t / t_s, 4), "peak_source": pk["source"] + " (MEASURED_PEAKS.json)"}

    # end to end through the C ABI's host-memory forward: pinned host
    # inputs -> device -> forward -> host results, every step (the call
    # streams the heads through the device in chunks, copies in and out
    # overlapping the kernels)
    e2e = None
    if not args.no_e2e and not args.backward:
        hQ, hK, hV = Qc.pin_memory(), Kc.pin_memory(), Vc.pin_memory()
        _, _, _, out, idx, route = sets[0]
        hout = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        hidx = torch.empty(idx.shape, dtype=idx.dtype).pin_memory()
        hroute = torch.empty(route.shape, dtype=route.dtype).pin_memory()
        e_steps = max(3, min(args.steps, 20))

        def e2e_step():
            plan.forward_host(hQ, hK, hV, hout, hidx, hroute, stream)

        for _ in range(3):
            e2e_step()
        barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        ems = max_over_ranks(e0.elapsed_time(e1) / e_steps, ws, dev)
        h2d = 3 * Qc.numel() * Qc.element_size()
        d2h = out.numel() * out.element_size() + idx.numel() * 4 + route.numel() * 4
        e2e = {"value": ws * qh / (ems / 1000.0), "unit": "query-heads/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(ems, 4)}

    timing = {"timed": "one CUDA graph of the K steps, replayed once" if g is not None else
              "K stream launches from the host",
              "stream_launched_ms_per_step": round(stream_ms, 5) if stream_ms is not None else round(ms, 5)}
    if graph_error:
        timing["graph_error"] = graph_error

    # the other workloads' forwards, timed the same way,
    # beside the main line (default run only)
    others = None
    if (not args.no_others and not args.backward and not args.routing_only and args.routes == 1
            and args.path == "auto" and rank == 0):
        others = {}
        for name in ("deit_s", "deit_t", "hires56", "long1d"):
            if name == args.workload:
                continue
            try:
                others[name] = measure_forward(mita, synth.WORKLOADS[name], args.steps, dev, stream)
            except Exception as exc:
                others[name] = {"error": str(exc).splitlines()[0][:200]}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds, shared=not args.routing_only, routes=args.routes,
                           backward=args.backward)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": "query-heads/s", "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded generator, no dataset)",
                "config": bench_config(w, ws, args.routes, variant_name(args)), "path": path,
                "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "timing": timing, "gpu_launches": launches,
                "other_workloads": others,
                "clocks": clocks, "achieved_tflops": round(tf, 2), "achieved_hbm_gbs": round(bw, 1),
                "hbm_frac": round(hbm_frac, 4)}
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
