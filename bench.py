"""Benchmark of the routing-and-combine step of a decode-step latent-MoE layer.

One step = router logits -> sigmoid+bias top-16 -> routing lists -> MXFP8 of the
latent -> Finalize, on the wide decode batch (T = 1020 tokens = 204 requests x 5
speculative tokens, hidden 7168, latent 3584, 896 experts, top-16), seeded synthetic
inputs resident in HBM. Metric: tokens per second.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0). Under torchrun every rank runs its own replica of the
step on its own GPU (the path shards by token: no data-path collective); value is the
tokens of all ranks over the slowest rank's time. ``--impl reference`` times the CPU
oracle (the plain C reference) on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

T_WIDE = 1020
WORKLOAD = "wide decode step: T=1020 tokens (204 requests x 5 speculative), hidden 7168, latent 3584, 896 experts, top-16"
METRIC = "route+finalize tokens/s at T=1020 (1 GB300)"
FLUSH_BYTES = 256 << 20  # > 129 MB L2


def algorithmic_bytes(T, H=synth.H, L=synth.L, E=synth.E, K=synth.K):
    """Bytes each step must move (inputs read once, outputs written once)."""
    b = {
        "router": T * H * 2 + E * H * 2 + T * E * 4,
        "topk": T * E * 4 + E * 4 + T * K * (4 + 4 + 2),
        "lists": T * K * 4 + (E + 1) * 4 + T * K * 4,
        "mxfp8": T * L * 2 + T * L + T * L // 32,
        "finalize": T * K * L * 2 + T * K * 2 + T * L * 2,
    }
    b["topk+mxfp8"] = b["topk"] + b["mxfp8"]
    return b


def chain_bytes(ab):
    return sum(v for k, v in ab.items() if k != "topk+mxfp8")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained", d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, 1700.0, "fallback"


def kernel_traffic(name):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel's
    source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f).get(name)
    if not d:
        return None
    src = os.path.join(ROOT, "latent_moe_decode_gb300", "csrc", d["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest()[:16] != d["source_sha256_16"]:
        return None
    return d["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def __enter__(self):
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits", "-lms", "200", "-i", str(self.index)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if not self.proc or not self.path:
            return None
        rows = []
        for line in open(self.path):
            f = [v.strip() for v in line.split(",")]
            if len(f) < 7:
                continue
            try:
                rows.append((float(f[0]), float(f[1]), f[3:7]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return None
        mx = max(r[1] for r in rows)
        load = [r[0] for r in rows] or [0.0]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": float(np.median(load)), "sm_max_mhz": mx, "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
class Step:
    """Device-resident inputs and preallocated buffers of one routing-and-combine step,
    plus the step captured as a CUDA graph. With nsets > 1 the inputs are held in
    nsets separate copies (same values, distinct memory), each with its own buffers and
    graph, so that steps run back to back in turn find their inputs cold in L2; with
    chain > 1, one more graph holds `chain` consecutive steps (one per copy in turn), as
    a decode loop captures consecutive layers in one graph."""

    def __init__(self, T, device, seed=0, skew=False, router_algo=0, graph=True, nsets=1, chain=1, rest=0):
        import torch

        import latent_moe_decode_gb300 as m

        self.m, self.T, self.device, self.nsets = m, T, device, nsets
        self.host = synth.chain_inputs(T, seed=seed, skew=skew)
        d = self.host
        tob = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)
        self.sets = []
        for _ in range(nsets):
            self.sets.append({"x": tob(d["x"]), "w": tob(d["w"]), "latent": tob(d["latent"]), "rows": tob(d["rows"]),
                              "bias": torch.from_numpy(d["bias"]).to(device),
                              "rf": m.RouteFinalize(T, synth.H, synth.L, synth.E, synth.K, device=device,
                                                    router_algo=router_algo)})
        s0 = self.sets[0]
        self.x, self.w, self.latent, self.rows, self.bias, self.rf = (s0["x"], s0["w"], s0["latent"], s0["rows"],
                                                                      s0["bias"], s0["rf"])
        self.graphs = []
        if graph:
            for i in range(nsets):
                s = torch.cuda.Stream(device)
                s.wait_stream(torch.cuda.current_stream(device))
                with torch.cuda.stream(s):
                    self.run_direct(i)
                torch.cuda.current_stream(device).wait_stream(s)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    self.run_direct(i)
                self.graphs.append(g)
            self.chain_graph, self.warm_graph, self.chain = None, None, chain
            if chain > 1:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(chain):
                        self.run_direct(i)
                self.chain_graph = g
                # the same number of consecutive steps, all on the first input set (no rotation)
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for _ in range(chain):
                        self.run_direct(0)
                self.warm_graph = g
            # a graph of `rest` consecutive steps (a timed count that is not a multiple of
            # `chain`), continuing the rotation
            self.rest_graph = None
            if rest > 0:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    for i in range(rest):
                        self.run_direct(i)
                self.rest_graph = g

    def run_direct(self, i=0):
        st = self.sets[i % self.nsets]
        st["rf"].run(st["x"], st["w"], st["bias"], st["latent"], st["rows"])

    def run(self, i=0):
        if self.graphs:
            self.graphs[i % self.nsets].replay()
        else:
            self.run_direct(i)

    def calls(self, i=0):
        m, T = self.m, self.T
        st = self.sets[i % self.nsets]
        rf, x, w, bias, latent, rows = st["rf"], st["x"], st["w"], st["bias"], st["latent"], st["rows"]
        return {
            "router": lambda: m.router_logits(x, w, out=rf.logits, workspace=rf.router_ws, algo=rf.router_algo),
            "topk": lambda: m.topk_route(rf.logits, bias, synth.K, ids=rf.ids, weights=rf.weights, weights_bf16=rf.weights_bf16),
            "lists": lambda: m.build_routing_lists(rf.ids, synth.E, offsets=rf.offsets, pairs=rf.pairs, workspace=rf.lists_ws),
            "mxfp8": lambda: m.mxfp8_quantize_rows(latent, q=rf.q, scales=rf.scales),
            "topk+mxfp8": lambda: m.topk_route_quantize(rf.logits, bias, synth.K, latent, ids=rf.ids, weights=rf.weights,
                                                        weights_bf16=rf.weights_bf16, q=rf.q, scales=rf.scales),
            "finalize": lambda: m.finalize(rows, rf.weights_bf16, T, synth.K, out=rf.out),
        }


SLEEP_CYCLES = 200_000  # ~100 us of GPU spin so the host is ahead when the timed work starts


def flush_l2(flush, i):
    """Writes the 256 MB buffer (evicting everything), then reads it back, so the dirty
    lines of the write are written back here and the timed kernels start on a cold,
    clean L2 (as a profiler's cache flush leaves it)."""
    import torch

    flush.fill_(i & 0xFF)
    torch.sum(flush.view(torch.int64))


def time_region(fn, n, flush, stream):
    """CUDA-event times of fn() over n repetitions; before each one L2 is flushed and
    the GPU spins briefly (both outside the events) so the launch is already queued."""
    import torch

    evs = []
    for i in range(n):
        flush_l2(flush, i)
        torch.cuda._sleep(SLEEP_CYCLES)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        evs.append((a, b))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in evs]


def max_over_ranks(values, world, device):
    """Each value's maximum over the ranks (the slowest rank's time); the identity on
    one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch

    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_rate(T, world, ms):
    """Tokens per second of all ranks together: each rank runs its own T-token step
    (the path shards by token, no exchange), timed by the slowest rank."""
    return world * T / (ms * 1e-3)


COLD_FACTOR = 3  # a rotation of input copies moves at least this many L2 capacities
STEPS_PER_GRAPH = 12  # consecutive steps (layers) one CUDA graph holds in the timed run
L2_BYTES = 129 << 20


def time_back_to_back(fns, stream):
    """CUDA-event time of the launches fns[0](), fns[1](), ... issued back to back, in
    ms per launch. The GPU first spins (outside the events) for longer than the host
    takes to issue them all, so the timed region holds only their execution."""
    import torch

    t0 = time.perf_counter()
    for f in fns[:4]:
        f()
    per_call = (time.perf_counter() - t0) / 4
    torch.cuda.synchronize()
    host_s = per_call * len(fns)
    torch.cuda._sleep(int(max(SLEEP_CYCLES, 3.0 * host_s * 2.1e9)))
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for f in fns:
        f()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / len(fns)


def n_copies(bytes_per_launch):
    return max(2, -(-COLD_FACTOR * L2_BYTES // max(1, bytes_per_launch)))


def rotations(step, K):
    """For each call: K launches rotating over enough copies of its inputs that every
    launch reads them cold from HBM (a rotation moves >= 3 L2 capacities)."""
    import torch

    m, T, rf = step.m, step.T, step.rf
    cl = lambda t, n: [t] + [t.clone() for _ in range(n - 1)]
    ab = algorithmic_bytes(T)
    nr, nq, nf = n_copies(ab["router"]), n_copies(ab["topk+mxfp8"]), n_copies(ab["finalize"])
    xs, ws = cl(step.x, nr), cl(step.w, nr)
    lg, lat = cl(rf.logits, nq), cl(step.latent, nq)
    rows = cl(step.rows, nf)
    ids = cl(rf.ids, 4)
    rot = {
        "router": [lambda i=i: m.router_logits(xs[i], ws[i], out=rf.logits, workspace=rf.router_ws, algo=rf.router_algo)
                   for i in range(nr)],
        "topk": [lambda i=i: m.topk_route(lg[i], step.bias, synth.K, ids=rf.ids, weights=rf.weights,
                                          weights_bf16=rf.weights_bf16) for i in range(nq)],
        "lists": [lambda i=i: m.build_routing_lists(ids[i], synth.E, offsets=rf.offsets, pairs=rf.pairs,
                                                    workspace=rf.lists_ws) for i in range(4)],
        "mxfp8": [lambda i=i: m.mxfp8_quantize_rows(lat[i], q=rf.q, scales=rf.scales) for i in range(nq)],
        "topk+mxfp8": [lambda i=i: m.topk_route_quantize(lg[i], step.bias, synth.K, lat[i], ids=rf.ids, weights=rf.weights,
                                                         weights_bf16=rf.weights_bf16, q=rf.q, scales=rf.scales)
                       for i in range(nq)],
        "finalize": [lambda i=i: m.finalize(rows[i], rf.weights_bf16, T, synth.K, out=rf.out) for i in range(nf)],
    }
    return {k: [v[i % len(v)] for i in range(K)] for k, v in rot.items()}, {"router": nr, "topk+mxfp8": nq, "finalize": nf}


def shared_bytes(d):
    """Algorithmic bytes of Finalize with the shared expert: the rows not skipped (index
    -1) read once, indices, weights and shared rows read once, the output written once."""
    T, K, H = d["T"], d["K"], d["H"]
    live = int(np.count_nonzero(d["row_index"] != -1))
    return live * H * 2 + T * K * 4 + T * K * 2 + T * H * 2 + T * H * 2


def time_finalize_shared(dev, steps, warmup):
    """Finalize with the shared expert at its own workload (T=512, K=8, H=7168, 5 % -1
    indices, routed scale 2.5, shared row), launches back to back over enough input
    copies that every launch reads cold inputs."""
    import torch

    import latent_moe_decode_gb300 as m

    d = synth.finalize_shared_inputs()
    T, K = d["T"], d["K"]
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    by = shared_bytes(d)
    n = n_copies(by)
    rows = [bf(d["rows"]) for _ in range(n)]
    shared = [bf(d["shared"]) for _ in range(n)]
    idx = torch.from_numpy(d["row_index"]).to(dev)
    w = bf(d["weights"])
    out = torch.empty(T, d["H"], dtype=torch.bfloat16, device=dev)
    calls = [lambda i=i: m.finalize(rows[i % n], w, T, K, row_index=idx, shared=shared[i % n], scale=d["scale"], out=out)
             for i in range(steps)]
    for c in calls[: max(warmup, n)]:
        c()
    ms = time_back_to_back(calls, torch.cuda.current_stream())
    hbm = load_peaks()[0]
    gbs = by / (ms * 1e-3) / 1e9
    del rows, shared
    torch.cuda.empty_cache()
    return {"workload": "Finalize with shared expert: T=512, K=8, H=7168, routed rows [4096,7168] gathered by "
                        "permuted indices with 5 % -1, BF16 weights, routed_scaling_factor 2.5, shared rows [512,7168]",
            "us": round(ms * 1e3, 2), "alg_bytes": by, "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3),
            "timing": f"{steps} launches back to back over {n} input copies (cold inputs every launch)",
            "traffic": kernel_traffic("finalize_shared")}


def percentiles(v):
    v = np.asarray(v, dtype=np.float64)
    return {"p10": round(float(np.percentile(v, 10)), 5), "p50": round(float(np.percentile(v, 50)), 5),
            "p90": round(float(np.percentile(v, 90)), 5), "n": int(v.size)}


def time_replays(g, n, stream, per):
    """CUDA-event time of each of n consecutive replays of graph g, in ms per step
    (a replay holds `per` steps)."""
    import torch

    torch.cuda._sleep(SLEEP_CYCLES)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    evs[0].record(stream)
    for i in range(n):
        g.replay()
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    return [evs[i].elapsed_time(evs[i + 1]) / per for i in range(n)]


def run_ours(args, rank, world, local_rank):
    import torch

    import latent_moe_decode_gb300 as m

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    m.load()
    T = T_WIDE
    nsets = n_copies(chain_bytes(algorithmic_bytes(T)))
    step = Step(T, dev, seed=rank, nsets=nsets, chain=STEPS_PER_GRAPH, rest=args.steps % STEPS_PER_GRAPH)
    rf = step.rf
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    for i in range(args.warmup * nsets):
        step.run(i)
    for _ in range(args.warmup):
        step.chain_graph.replay()
    barrier()
    rot, copies = rotations(step, args.steps)
    for fns in rot.values():
        for f in fns[:args.warmup]:
            f()
    barrier()

    with ClockSampler(local_rank) as clk:
        # (a) K whole steps back to back, rotating over input sets that together exceed
        #     L2 (every step reads its inputs cold): CUDA graphs of STEPS_PER_GRAPH
        #     consecutive steps, then one graph of the remaining K mod STEPS_PER_GRAPH steps
        barrier()
        full, rest = divmod(args.steps, STEPS_PER_GRAPH)
        fns = [step.chain_graph.replay] * full + ([step.rest_graph.replay] if rest else [])
        ms = time_back_to_back(fns, stream) * len(fns) / args.steps
        barrier()
        # (b) each call alone, K launches back to back over rotated input copies
        per_ms = {k: time_back_to_back(fns, stream) for k, fns in rot.items()}
        # (c) for reference: one step at a time, L2 flushed before each (outside events)
        flushed_ms = float(np.mean(time_region(step.run, args.steps, flush, stream)))
        # (d) spread: each replay of a 12-step graph timed on its own (cold inputs), and the
        #     same with every step on one input set (no rotation: what stays in L2 helps)
        spread = time_replays(step.chain_graph, 15, stream, STEPS_PER_GRAPH)
        for _ in range(2):
            step.warm_graph.replay()
        warm = time_replays(step.warm_graph, 15, stream, STEPS_PER_GRAPH)
    clocks = clk.summary()
    assert m.device_error(clear=True) == 0
    shared_line = time_finalize_shared(dev, args.steps, args.warmup)
    assert m.device_error(clear=True) == 0

    # (c) end to end through the public API: every step copies its inputs in from pinned
    #     host memory, runs (one moe_route_finalize call) and copies its results out.
    #     Consecutive steps overlap on three streams (host->device copies, the step,
    #     device->host copies) with two sets of device inputs and host outputs, as a
    #     serving loop would; the timed region spans K whole steps.
    d = step.host
    hx = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hl = torch.from_numpy(d["latent"].view(np.int16)).view(torch.bfloat16).pin_memory()
    hr = torch.from_numpy(d["rows"].view(np.int16)).view(torch.bfloat16).pin_memory()
    sets = step.sets[:2]
    outs = [[st["rf"].out, st["rf"].ids, st["rf"].weights_bf16, st["rf"].offsets, st["rf"].pairs, st["rf"].q,
             st["rf"].scales] for st in sets]
    houts = [[torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in os_] for os_ in outs]
    h2d = sum(t.numel() * t.element_size() for t in (hx, hl, hr))
    d2h = sum(t.numel() * t.element_size() for t in houts[0])
    copy_in, copy_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_steps(n):
        ev = lambda: torch.cuda.Event()
        ev_in, ev_run, ev_out = [ev() for _ in range(n)], [ev() for _ in range(n)], [ev() for _ in range(n)]
        copy_in.wait_stream(stream)
        copy_out.wait_stream(stream)
        for i in range(n):
            b, st = i % 2, sets[i % 2]
            with torch.cuda.stream(copy_in):
                if i >= 2:
                    copy_in.wait_event(ev_run[i - 2])  # step i-2 no longer reads these inputs
                st["x"].copy_(hx, non_blocking=True)
                st["latent"].copy_(hl, non_blocking=True)
                st["rows"].copy_(hr, non_blocking=True)
                ev_in[i].record(copy_in)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # step i-2's results have been copied out
            st["rf"].run(st["x"], st["w"], st["bias"], st["latent"], st["rows"], stream=stream)
            ev_run[i].record(stream)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(ev_run[i])
                for h, o in zip(houts[b], outs[b]):
                    h.copy_(o, non_blocking=True)
                ev_out[i].record(copy_out)
        stream.wait_stream(copy_in)
        stream.wait_stream(copy_out)

    e2e_steps(4)
    barrier()
    e_a, e_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_a.record(stream)
    e2e_steps(args.steps)
    e_b.record(stream)
    barrier()
    e2e_ms = e_a.elapsed_time(e_b) / args.steps

    ms, e2e_ms = max_over_ranks([ms, e2e_ms], world, dev)
    if rank != 0:
        return None

    hbm, bf16, bf16_sus, peak_src = load_peaks()
    ab = algorithmic_bytes(T)
    fin_gbs = ab["finalize"] / (per_ms["finalize"] * 1e-3) / 1e9
    traffic = kernel_traffic("finalize")
    steps = {}
    for k in per_ms:
        gbs = ab[k] / (per_ms[k] * 1e-3) / 1e9
        steps[k] = {"us": round(per_ms[k] * 1e3, 2), "alg_bytes": ab[k], "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 3)}
    flops = 2.0 * T * synth.E * synth.H
    steps["router"]["TFLOP/s"] = round(flops / (per_ms["router"] * 1e-3) / 1e12, 1)
    steps["router"]["frac_bf16"] = round(flops / (per_ms["router"] * 1e-3) / 1e12 / bf16, 3)
    line = {
        "metric": METRIC,
        "value": round(whole_job_rate(T, world, ms), 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded; shapes and distributions of the pages' wide decode batch)",
        "config": {"workload": WORKLOAD, "T": T, "hidden": synth.H, "latent": synth.L, "experts": synth.E, "top_k": synth.K,
                   "l2": f"inputs larger than L2: steps run back to back over {nsets} copies of the inputs "
                         f"({nsets * chain_bytes(ab) / 1e6:.0f} MB in rotation > 129 MB L2), so each step reads them cold; "
                         f"each call alone likewise over {copies} copies",
                   "launch": f"CUDA graphs of {STEPS_PER_GRAPH} consecutive steps (as a decode loop captures "
                             "consecutive layers; the steps past a multiple of 12 in one more graph), replayed back "
                             "to back; programmatic dependent launch between the kernels of a step",
                   "parallelism": f"replicas x{world} (token-sharded, no collective)"},
        "chain_GB/s": round(chain_bytes(ab) / (ms * 1e-3) / 1e9, 1),
        "ms_per_step_flushed": round(flushed_ms, 5),
        "ms_per_step_spread": dict(percentiles(spread), method="15 replays of a 12-step graph, each timed on its own "
                                   "with CUDA events; cold inputs (rotation over the input copies)"),
        "ms_per_step_warm": dict(percentiles(warm), method="the same with all 12 steps on one input set: the second "
                                 "step onwards finds what L2 kept of the first (170 MB per step > 129 MB L2)"),
        "roofline": {"kernel": "finalize", "bound": "hbm", "achieved": round(fin_gbs, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(fin_gbs / hbm, 3), "traffic": traffic, "alg_bytes_per_launch": ab["finalize"],
                     "peak_source": f"{peak_src}: copy bandwidth (MEASURED_PEAKS.json hbm_gbs)" if peak_src == "measured" else "fallback"},
        "steps_alone": steps,
        "finalize_shared": shared_line,
        "e2e": {"value": round(whole_job_rate(T, world, e2e_ms), 1), "unit": "tokens/s", "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "method": "moe_route_finalize per step; inputs in from pinned host memory and all results out, every "
                          "step, consecutive steps overlapped on copy-in / compute / copy-out streams"},
        "gpu_launches": args.steps * rf.launches,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return line


def sweep_lines(Ts, args, skew=True, label="skew sweep"):
    """The whole step per T (Zipf(1.1) expert popularity with skew, else the uniform
    correction bias), plus each call alone and the stock router; one JSON line per T."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    stream = torch.cuda.current_stream()
    hbm = load_peaks()[0]
    for T in Ts:
        for algo in ([0] if not args.router_algos else [int(a) for a in args.router_algos.split(",")]):
            ab = algorithmic_bytes(T)
            nsets = n_copies(chain_bytes(ab))
            step = Step(T, dev, skew=skew, router_algo=algo, nsets=nsets)
            for i in range(args.warmup * nsets):
                step.run(i)
            # K steps back to back over input copies larger than L2, as the main line
            ms = time_back_to_back([lambda i=i: step.run(i) for i in range(args.steps)], stream)
            rot, _ = rotations(step, args.steps)
            per = {k: round(time_back_to_back(fns, stream) * 1e3, 2) for k, fns in rot.items()}
            frac = {k: round(ab[k] / (v * 1e-6) / 1e9 / hbm, 3) for k, v in per.items()}
            stock = None
            try:  # the stock router call (cuBLAS through torch), timed the same way, for context
                nr = n_copies(ab["router"])
                xs = [step.x] + [step.x.clone() for _ in range(nr - 1)]
                ws = [step.w] + [step.w.clone() for _ in range(nr - 1)]
                out = torch.empty(T, synth.E, dtype=torch.float32, device=dev)
                mms = [lambda i=i: torch.mm(xs[i % nr], ws[i % nr].t(), out_dtype=torch.float32, out=out)
                       for i in range(args.steps)]
                mms[0]()
                stock = round(time_back_to_back(mms, stream) * 1e3, 2)
                del xs, ws
            except Exception:
                pass
            loads = np.bincount(step.rf.ids.cpu().numpy().ravel(), minlength=synth.E)
            print(json.dumps({"config": label, "T": T, "router_algo": algo, "us_per_step": round(ms * 1e3, 2),
                              "tokens/s": round(T / (ms * 1e-3), 1), "chain_GB/s": round(chain_bytes(ab) / (ms * 1e-3) / 1e9, 1),
                              "frac_hbm_chain": round(chain_bytes(ab) / (ms * 1e-3) / 1e9 / hbm, 3), "us_alone": per,
                              "frac_hbm_alone": frac, "us_stock_router_torch_mm": stock,
                              "expert_load_max_over_mean": round(float(loads.max() / max(loads.mean(), 1e-9)), 2),
                              "timing": "back to back over input copies larger than L2 (cold inputs every launch)"}),
                  flush=True)
            assert m.device_error(clear=True) == 0
            del step, rot
            torch.cuda.empty_cache()


def run_sweep(args):
    sweep_lines([int(t) for t in args.sweep.split(",")], args)


def run_configs(args):
    """Every workload of the path, one JSON line each: tiny (T = 8), narrow (64) and wide
    (1020) decode steps, Finalize with the shared expert (T = 512, K = 8, H = 7168), and
    the Zipf(1.1) skew sweep (T = 1, 16, 64, 256, 1020, 4096)."""
    import torch

    for T, name in ((8, "tiny"), (64, "narrow"), (1020, "wide")):
        sweep_lines([T], args, skew=False, label=name)
    print(json.dumps(dict(config="finalize with shared expert", **time_finalize_shared(torch.device("cuda", 0),
                                                                                        args.steps, args.warmup))),
          flush=True)
    sweep_lines([1, 16, 64, 256, 1020, 4096], args, skew=True)


def front_flops_bytes(T, H=synth.H, E=synth.E, L=synth.L):
    """Algorithmic FLOPs and bytes of the front projection: x and both weights read
    once, FP32 logits and BF16 latent written once."""
    return 2.0 * T * (E + L) * H, 2.0 * T * H + 2.0 * (E + L) * H + 4.0 * T * E + 2.0 * T * L


def run_front(args):
    """The front projection (router logits + latent down projection in one launch), one
    JSON line per T: back to back over input copies larger than L2, against the
    measured bf16 tensor peak, with the two stock torch.mm calls for context."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    stream = torch.cuda.current_stream()
    hbm, tflops = load_peaks()[:2]
    wr = torch.from_numpy(synth.router_weight().view(np.int16)).view(torch.bfloat16).to(dev)
    wd = torch.from_numpy(synth.latent_down_weight().view(np.int16)).view(torch.bfloat16).to(dev)
    for T in [int(t) for t in args.front.split(",")]:
        x = torch.from_numpy(synth.hidden_rows(T).view(np.int16)).view(torch.bfloat16).to(dev)
        fl, by = front_flops_bytes(T)
        n = n_copies(int(by))
        xs, wrs, wds = [x] + [x.clone() for _ in range(n - 1)], [wr] + [wr.clone() for _ in range(n - 1)], \
            [wd] + [wd.clone() for _ in range(n - 1)]
        logits = torch.empty(T, synth.E, dtype=torch.float32, device=dev)
        latent = torch.empty(T, synth.L, dtype=torch.bfloat16, device=dev)
        ws = torch.empty(max(1, m.front_projection_workspace(T, synth.H, synth.E, synth.L)), dtype=torch.uint8, device=dev)
        calls = [lambda i=i: m.front_projection(xs[i % n], wrs[i % n], wds[i % n], logits=logits, latent=latent,
                                                workspace=ws) for i in range(args.steps)]
        for c in calls[: max(args.warmup, n)]:
            c()
        ms = time_back_to_back(calls, stream)
        stock = [lambda i=i: (torch.mm(xs[i % n], wrs[i % n].t(), out_dtype=torch.float32, out=logits),
                              torch.mm(xs[i % n], wds[i % n].t(), out=latent)) for i in range(args.steps)]
        for c in stock[: max(args.warmup, n)]:
            c()
        ms_stock = time_back_to_back(stock, stream)
        ach = fl / (ms * 1e-3) / 1e12
        print(json.dumps({"T": T, "us": round(ms * 1e3, 2), "TFLOP/s": round(ach, 1), "peak_TFLOP/s": tflops,
                          "frac_tensor": round(ach / tflops, 3), "GB/s": round(by / (ms * 1e-3) / 1e9, 1),
                          "frac_hbm": round(by / (ms * 1e-3) / 1e9 / hbm, 3),
                          "us_stock_two_torch_mm": round(ms_stock * 1e3, 2), "GFLOP": round(fl / 1e9, 2),
                          "MB": round(by / 1e6, 2),
                          "timing": "back to back over input copies larger than L2 (cold inputs every launch)"}),
              flush=True)
        assert m.device_error(clear=True) == 0
        del xs, wrs, wds
        torch.cuda.empty_cache()


def run_norm(args):
    """Finalize with the RMSNorm epilogue (routed latent and its normalised copy), one
    JSON line per T: back to back over input copies larger than L2, against the
    measured HBM copy bandwidth, with plain Finalize timed the same way."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    stream = torch.cuda.current_stream()
    hbm = load_peaks()[0]
    K, L = synth.K, synth.L
    g = torch.from_numpy(synth.norm_weight().view(np.int16)).view(torch.bfloat16).to(dev)
    for T in [int(t) for t in args.norm.split(",")]:
        rows = torch.from_numpy(synth.expert_rows(T).view(np.int16)).view(torch.bfloat16).to(dev)
        u = synth.rng(0, synth.WEIGHTS).random((T, K)).astype(np.float32)
        w = torch.from_numpy(synth.f32_to_bf16_bits(u / u.sum(1, keepdims=True)).view(np.int16)).view(torch.bfloat16).to(dev)
        by = 2.0 * T * K * L + 2.0 * T * K + 2.0 * L + 2 * 2.0 * T * L
        n = n_copies(int(by))
        rs = [rows] + [rows.clone() for _ in range(n - 1)]
        routed = torch.empty(T, L, dtype=torch.bfloat16, device=dev)
        out = torch.empty(T, L, dtype=torch.bfloat16, device=dev)
        calls = [lambda i=i: m.finalize_rmsnorm(rs[i % n], w, T, K, g, routed=routed, out=out) for i in range(args.steps)]
        plain = [lambda i=i: m.finalize(rs[i % n], w, T, K, out=routed) for i in range(args.steps)]
        for c in calls[: max(args.warmup, n)] + plain[: max(args.warmup, n)]:
            c()
        ms = time_back_to_back(calls, stream)
        ms_plain = time_back_to_back(plain, stream)
        gbs = by / (ms * 1e-3) / 1e9
        print(json.dumps({"T": T, "us": round(ms * 1e3, 2), "GB/s": round(gbs, 1), "peak_GB/s": hbm,
                          "frac_hbm": round(gbs / hbm, 3), "MB": round(by / 1e6, 2),
                          "us_finalize_alone": round(ms_plain * 1e3, 2),
                          "timing": "back to back over input copies larger than L2 (cold inputs every launch)"}),
              flush=True)
        assert m.device_error(clear=True) == 0
        del rs
        torch.cuda.empty_cache()


def run_ncu_norm(args):
    """Finalize with the RMSNorm epilogue at T (default 1020), untimed."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    T = args.T or T_WIDE
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    rows, g = bf(synth.expert_rows(T)), bf(synth.norm_weight())
    u = synth.rng(0, synth.WEIGHTS).random((T, synth.K)).astype(np.float32)
    w = bf(synth.f32_to_bf16_bits(u / u.sum(1, keepdims=True)))
    for _ in range(args.warmup + args.steps):
        m.finalize_rmsnorm(rows, w, T, synth.K, g)
    torch.cuda.synchronize()


def units_inputs(T, dev):
    """Routing lists of the wide batch's top-16 (oracle-free: the library's own chain
    at seed 0) for the unit-window timings."""
    import latent_moe_decode_gb300 as m

    step = Step(T, dev, graph=False)
    step.run()
    return step.rf.offsets.clone(), m.unit_windows_capacity(T, synth.K, synth.E, 8)


def run_units(args):
    """Unit windows (8 pairs per unit) from the routing lists, one JSON line per T, each
    call timed back to back."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    stream = torch.cuda.current_stream()
    for T in [int(t) for t in args.units.split(",")]:
        off, cap = units_inputs(T, dev)
        bufs = [torch.empty(cap, dtype=torch.int32, device=dev) for _ in range(3)]
        uo = torch.empty(synth.E + 1, dtype=torch.int32, device=dev)
        call = lambda: m.unit_windows(off, 8, max_units=cap, unit_offsets=uo, unit_expert=bufs[0], unit_start=bufs[1],
                                      unit_len=bufs[2])
        for _ in range(args.warmup):
            call()
        ms = time_back_to_back([call] * args.steps, stream)
        n = int(uo[-1].item())
        print(json.dumps({"T": T, "us": round(ms * 1e3, 2), "units": n, "pairs": T * synth.K,
                          "bytes": 4 * (synth.E + 1) * 2 + 12 * n, "timing": "back to back, one call per launch"}),
              flush=True)
        assert m.device_error(clear=True) == 0


def run_ncu_units(args):
    """Unit windows at T (default 1020), untimed (for profiler captures)."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    off, cap = units_inputs(args.T or T_WIDE, dev)
    for _ in range(args.warmup + args.steps):
        m.unit_windows(off, 8, max_units=cap)
    torch.cuda.synchronize()


def run_ncu_step(args):
    """The wide step, untimed, warmup + steps times (for profiler captures)."""
    import torch

    dev = torch.device("cuda", 0)
    step = Step(args.T or T_WIDE, dev, graph=False, router_algo=args.router_algo)
    for _ in range(args.warmup + args.steps):
        step.run()
    torch.cuda.synchronize()


def run_ncu_front(args):
    """The front projection at T (default 1020), untimed, warmup + steps times."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    T = args.T or T_WIDE
    bf = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
    x, wr, wd = bf(synth.hidden_rows(T)), bf(synth.router_weight()), bf(synth.latent_down_weight())
    for _ in range(args.warmup + args.steps):
        m.front_projection(x, wr, wd)
    torch.cuda.synchronize()


def run_ncu_call(args):
    """One public call at T (default 1020), untimed, warmup + steps times (for profiler
    captures of a single kernel): router, topk, lists, mxfp8, mxfp8_tcgen05, finalize,
    finalize_shared (the Finalize-with-shared-expert workload)."""
    import torch

    import latent_moe_decode_gb300 as m

    dev = torch.device("cuda", 0)
    m.load()
    T = args.T or T_WIDE
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    name = args.ncu_call
    if name == "finalize_shared":
        d = synth.finalize_shared_inputs()
        rows, w, sh = bf(d["rows"]), bf(d["weights"]), bf(d["shared"])
        idx = torch.from_numpy(d["row_index"]).to(dev)
        call = lambda: m.finalize(rows, w, d["T"], d["K"], row_index=idx, shared=sh, scale=d["scale"])
    else:
        step = Step(T, dev, graph=False)
        step.run()
        torch.cuda.synchronize()
        calls = step.calls()
        if name == "mxfp8_tcgen05":
            call = lambda: m.mxfp8_quantize_rows_tcgen05(step.latent)
        else:
            call = calls[name]
    for _ in range(args.warmup + args.steps):
        call()
    torch.cuda.synchronize()
    assert m.device_error(clear=True) == 0


# ---------------------------------------------------------------------------
ORACLE_STEPS = ("router", "topk", "lists", "mxfp8", "finalize")
REF_TOKENS = 16  # tokens per reference-arm step (a fixed slice of the wide batch)


def oracle_step(d, tokens):
    """The oracle's whole step over the given token rows of the wide batch, single
    threaded; returns each step's seconds."""
    import oracle

    clk, t = time.perf_counter, {}
    x, lat = d["x"][tokens], d["latent"][tokens]
    rows = d["rows"].reshape(T_WIDE, synth.K, synth.L)[tokens].reshape(-1, synth.L)
    t0 = clk()
    logits, _ = oracle.router_logits(x, d["w"], threads=1)
    t["router"] = clk() - t0
    logits = logits.astype(np.float32)
    t0 = clk()
    ids, wf, wb = oracle.topk_route(logits, d["bias"], synth.K)
    t["topk"] = clk() - t0
    t0 = clk()
    oracle.routing_lists(ids, synth.E)
    t["lists"] = clk() - t0
    t0 = clk()
    oracle.mxfp8_quantize(lat)
    t["mxfp8"] = clk() - t0
    t0 = clk()
    oracle.finalize(rows, wb, len(tokens), synth.K)
    t["finalize"] = clk() - t0
    return t


class OneCore:
    """Pins this process to one host core for the oracle's timings (restored on exit)."""

    def __enter__(self):
        self.saved = None
        try:
            self.saved = os.sched_getaffinity(0)
            os.sched_setaffinity(0, {min(self.saved)})
        except (AttributeError, OSError):
            pass
        return self

    def __exit__(self, *a):
        if self.saved:
            os.sched_setaffinity(0, self.saved)


def cpu_baseline(seconds):
    """The oracle as it stands, single-threaded and pinned to one host core, on a
    consecutive slice of the wide batch sized to about `seconds` of CPU work over three
    passes; each step's time is the median of the three."""
    import oracle

    oracle.build()
    d = synth.chain_inputs(T_WIDE)
    with OneCore():
        probe = sum(oracle_step(d, np.arange(4)).values()) / 4
        n = int(min(T_WIDE, max(4, seconds / 3 / max(probe, 1e-6))))
        tok = np.arange(n)
        runs = [oracle_step(d, tok) for _ in range(3)]
    per = {k: float(np.median([r[k] for r in runs])) for k in ORACLE_STEPS}
    total = float(np.median([sum(r.values()) for r in runs]))
    return {"value": round(n / total, 2), "unit": "tokens/s", "cores": 1, "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"tokens 0..{n - 1} of the {T_WIDE}-token wide batch, whole step, three passes "
                      f"({3 * total:.1f} s), pinned to one core",
            "per_step_ms": {k: round(v * 1e3, 2) for k, v in per.items()},
            "per_step_us_per_token": {k: round(v * 1e6 / n, 1) for k, v in per.items()}}


def run_reference(args, rank):
    """The reference arm: the oracle (the plain C reference of the path), pinned to one
    host core; every step is the whole routing-and-combine step over a fixed slice of
    REF_TOKENS tokens of the wide batch. W untimed steps, then K timed steps."""
    if rank != 0:
        return None
    import oracle

    oracle.build()
    d = synth.chain_inputs(T_WIDE)
    tok = np.arange(REF_TOKENS)
    with OneCore():
        for _ in range(args.warmup):
            oracle_step(d, tok)
        runs = []
        t0 = time.perf_counter()
        for _ in range(args.steps):
            runs.append(oracle_step(d, tok))
        wall = time.perf_counter() - t0
    ms = wall / args.steps * 1e3
    v = round(REF_TOKENS / (wall / args.steps), 2)
    base = {"value": v, "unit": "tokens/s", "cores": 1, "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"each step: tokens 0..{REF_TOKENS - 1} of the {T_WIDE}-token wide batch, whole step "
                      f"(router, top-16, lists, MXFP8, Finalize), pinned to one core",
            "per_step_ms": {k: round(float(np.median([r[k] for r in runs])) * 1e3, 3) for k in ORACLE_STEPS}}
    return {
        "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 router / f32 rest", "data": "synthetic (seeded)", "impl": "reference",
        "config": {"workload": WORKLOAD, "T": T_WIDE, "hidden": synth.H, "latent": synth.L, "experts": synth.E,
                   "top_k": synth.K, "parallelism": "one host core (rank 0 only)",
                   "sample": f"{REF_TOKENS} tokens per step"},
        "cpu_baseline": base,
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", default=None, help="comma-separated T list: the skew sweep, one JSON line per T")
    ap.add_argument("--configs", action="store_true", help="every workload (tiny, narrow, wide, Finalize with shared "
                    "expert, skew sweep), one JSON line each")
    ap.add_argument("--router-algos", default=None, help="with --sweep: router kernel families to time (0 auto, 1 simt, 2 tcgen05)")
    ap.add_argument("--ncu-step", action="store_true", help="run the step untimed (for profiler captures)")
    ap.add_argument("--front", default=None, help="comma-separated T list: time the front projection, one JSON line per T")
    ap.add_argument("--ncu-front", action="store_true", help="run the front projection untimed (for profiler captures)")
    ap.add_argument("--norm", default=None, help="comma-separated T list: time Finalize with the RMSNorm epilogue")
    ap.add_argument("--ncu-norm", action="store_true", help="run Finalize with the RMSNorm epilogue untimed (profiling)")
    ap.add_argument("--units", default=None, help="comma-separated T list: time the unit windows of the routing lists")
    ap.add_argument("--ncu-units", action="store_true", help="run the unit windows untimed (for profiler captures)")
    ap.add_argument("--ncu-call", default=None, choices=["router", "topk", "lists", "mxfp8", "mxfp8_tcgen05", "finalize",
                                                         "finalize_shared"],
                    help="run one public call untimed (for profiler captures of one kernel)")
    ap.add_argument("--T", type=int, default=0, help="with --ncu-step / --ncu-call: token count (default 1020)")
    ap.add_argument("--router-algo", type=int, default=0, help="with --ncu-step: router kernel family")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.ncu_step:
        run_ncu_step(args)
        return
    if args.ncu_call:
        run_ncu_call(args)
        return
    if args.ncu_front:
        run_ncu_front(args)
        return
    if args.front:
        run_front(args)
        return
    if args.ncu_norm:
        run_ncu_norm(args)
        return
    if args.ncu_units:
        run_ncu_units(args)
        return
    if args.units:
        run_units(args)
        return
    if args.norm:
        run_norm(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.configs:
        run_configs(args)
        return
    if args.impl == "reference":
        line = run_reference(args, rank)
    else:
        if world > 1:
            import torch

            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
