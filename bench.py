#!/usr/bin/env python3
"""Throughput of the W4A16 routed-expert MoE layer on GB300.

One step = the whole layer on one batch of synthetic tokens, one
moe_layer_forward call: the router (GEMM, softmax, top-k, renormalised
weights) and the routed experts (permute, INT4 expert GEMMs with SiLU*up,
weighted combine); for decode batches one kernel runs both. The stack
workloads run 48 such layers, each followed by the residual + RMS rescale.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

Prints one JSON line. Workloads (shapes from "Running 125B MoE on Three
3090s - vLLM Edition", section 1): decode1 (T=1, the default), decode4,
decode64, prefill512 (Zipf-skewed routing), stack_prefill4096 and
stack_decode4 (48 layers).

Timing: inputs resident in HBM; steps rotate over independent weight sets so
that no step finds its experts in L2 (their total exceeds the 129 MB L2); a
CUDA graph holds one pass over the sets (consecutive steps, as consecutive
layers of a model run), and K steps are whole replays plus one graph of the
remainder; CUDA events on the launching stream; >= 3 warm-up steps. The
expert kernel's own time is taken from events that the library records
around it in separate one-step graphs, replayed after the timed region; where
the layer is that one kernel (the router inside), from the timed region.
`e2e` repeats the timing through the same public calls with every step's
tokens copied in from pinned host memory and its output copied back, inside
the timed region; the copies run on a second stream, so that a step's kernels
overlap the copy-out of the step before it, as a serving loop would run them.
The CPU baseline is the fp64 oracle on a bounded sample of the workload.
Multi-GPU: independent replicas (the layer has no exchange step).
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
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

EXPERT_BYTES = 2_534_400          # packed INT4 + bf16 scales of one full-shape expert
L2_BYTES = 129 * 2**20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# Batches the library runs through its fused decode kernel (larger ones take the
# tensor-core grouped GEMM pipeline).
FUSED_MAX_T = 7


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="decode1", choices=sorted(synth.WORKLOADS) + sorted(EXTRA))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--sets", type=int, default=0, help="weight sets to rotate over (0: enough to exceed L2)")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers of a stack workload (0: its own, 48); fewer only to profile a small case")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target length of the CPU-baseline sample")
    ap.add_argument("--clock-ms", type=float, default=1000.0,
                    help="length of the load window, ending with the timed region, over which clocks are sampled")
    ap.add_argument("--no-per-config", dest="per_config", action="store_false",
                    help="measure the headline workload only (by default a decode1 run also measures %s)"
                    % ", ".join(("decode64", "stack_prefill4096")))
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ clocks --

class Clocks:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ distributed --

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    """Largest v over the ranks (NCCL on the GPUs, or gloo on the host)."""
    if world == 1:
        return v
    import torch.distributed as dist
    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU baseline --

def cpu_baseline(wl, seed: int, target_s: float):
    """The fp64 oracle, as it stands, on a bounded sample of the workload's tokens (tok/s).

    The layer is independent per token, so a sample of n tokens through one layer
    measures the same per-token work as the workload; n is sized from a short
    probe so that the timed run takes about target_s seconds.
    """
    import oracle
    T, H, E, k, I = wl.dims
    oracle.build()
    cores = oracle.max_threads()
    wr = synth.router(E + 1 if wl.shared else E, H, seed=seed, layer=0)
    bias = synth.zipf_bias(E, wl.zipf, seed=seed) if wl.zipf else None
    sh = synth.expert_weights(E + 1, H, I, seed=seed, layer=0, experts=[E]) if wl.shared else None

    def run(n):
        xs = synth.hidden(n, H, seed=seed, layer=101)
        ids, w, _ = oracle.route(xs, wr[:E], k, bias)
        held = np.unique(ids)
        row = np.full(E, -1, np.int32)
        row[held] = np.arange(len(held))
        wts = synth.expert_weights(E, H, I, seed=seed, layer=0, experts=held)
        t0 = time.perf_counter()
        oracle.route(xs, wr[:E], k, bias)
        out = oracle.expert_forward(xs, ids, w.astype(np.float32), wts["w1_packed"], wts["w1_scales"],
                                    wts["w2_packed"], wts["w2_scales"], E, I, expert_row=row)
        if sh is not None:
            gate, y = oracle.shared_expert(xs, wr[E], sh["w1_packed"][0], sh["w1_scales"][0], sh["w2_packed"][0],
                                           sh["w2_scales"][0], I)
            oracle.shared_combine(out, gate, y)
        return time.perf_counter() - t0

    n = cores
    t = run(n)
    n = max(cores, min(8192, int(n * target_s / max(t, 1e-3)) // cores * cores))
    t = run(n)
    return {"value": n / t / wl.layers, "unit": "tok/s", "cores": min(cores, n), "kind": "oracle",
            "sample": "%d seeded tokens through one layer of workload %s (route + experts%s), fp64, %.1f s%s"
                      % (n, wl.name, " + shared expert" if wl.shared else "", t,
                         "; per-token rate divided by %d layers" % wl.layers
                         if wl.layers > 1 else "")}


# ------------------------------------------------------------- our arm -----

def source_hash(names=None) -> str:
    """Hash of the named csrc files (all of them by default)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "w4a16_mixture_experts_gb300", "csrc")
    for name in sorted(names if names is not None else os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: str):
    """DRAM bytes per launch of the workload's dominant kernel from a committed ncu capture
    (profiles/traffic.json), if it was taken on the current sources of that kernel (its
    file and the headers it includes, listed with the entry); else None."""
    return recorded_counter(config, "dram_bytes_per_launch")


def binding_roofline(bytes_per_launch, flops_per_launch, hbm_gbs, tc_tflops):
    """'tensor' if the flops at the tensor rate take longer than the bytes at
    the copy rate, else 'hbm': the roofline that bounds the launch."""
    return "tensor" if flops_per_launch / (tc_tflops * 1e12) > bytes_per_launch / (hbm_gbs * 1e9) else "hbm"


def launches_per_layer(T: int, E: int, routes_itself: bool = False) -> int:
    """Kernels one layer launches: one when the decode kernel runs the router
    itself; else the router is one kernel for T <= 8 (logits, then top-k in the
    last CTA), or logits + top-k, and the forward one fused kernel (the
    library's decode path, T <= 8), or permute 3 + x gather + chunk table +
    gate_up + down + conversion."""
    if routes_itself:
        return 1
    return (1 if T <= 8 else 2) + (1 if T <= FUSED_MAX_T else 8)


def measure(args, wl, steps, rank, world, local):
    """Times `steps` steps of workload wl on this rank; returns the JSON fields."""
    import dataclasses
    import w4a16_mixture_experts_gb300 as moe
    if wl.layers > 1 and args.layers:
        wl = dataclasses.replace(wl, layers=args.layers)
    moe.build()
    moe.lib()
    T, H, E, k, I = wl.dims
    stack = wl.layers > 1
    dev = torch.device("cuda", torch.cuda.current_device())

    # weight sets: the stack's 48 layers, or enough single layers to exceed L2
    if stack:
        nsets = wl.layers
    elif args.sets:
        nsets = args.sets
    else:
        touched = (min(E, T * k) + (1 if wl.shared else 0)) * EXPERT_BYTES
        nsets = max(2, min(16, math.ceil(2.5 * L2_BYTES / touched)))
    seed = args.seed + 1000 * rank
    # with a shared expert the forward runs over E + 1 experts and k + 1 slots
    Ef, kf = (E + 1, k + 1) if wl.shared else (E, k)
    sets = []
    for i in range(nsets):
        d = synth.shared_layer_inputs(wl, seed=seed, layer=i) if wl.shared else synth.layer_inputs(wl, seed=seed, layer=i)
        if not stack:
            d["hidden"] = synth.hidden(T, H, seed=seed, layer=i)
        sets.append({key: (v.to(dev) if v is not None else None) for key, v in d.items()})
        if stack and i > 0:
            sets[i]["hidden"] = None
        del d
    x0 = sets[0]["hidden"]
    ws = moe.shared_workspace(T, H, E, k, I, dev) if wl.shared else moe.workspace(T, H, E, k, I, dev)
    ids = torch.empty(T, kf, dtype=torch.int32, device=dev)
    w = torch.empty(T, kf, dtype=torch.float32, device=dev)
    outs = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(1 if stack else nsets)]
    act = [torch.empty(T, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    stream = torch.cuda.Stream(device=dev)
    ev_b = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nsets)]
    ev_a = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(nsets)]
    unique = [0] * nsets
    for e in ev_b + ev_a:       # torch only lets recorded events be timed; the library re-records them
        e.record(stream)

    # one call per layer: where the decode kernel runs the router itself, that
    # one kernel is the layer, and its time includes the router's bytes
    plan = moe.moe_forward_plan(T, H, Ef, kf, I)
    routes_itself = bool(plan and plan[3])
    router_bytes = Ef * H * 2 + (E * 4 if wl.zipf else 0)

    def layer_call(x, s, nxt=None, out=None):
        moe.moe_layer_forward(x, s["router_w"], k, s["w1_packed"], s["w1_scales"], s["w2_packed"], s["w2_scales"],
                              bias=s["bias"], shared=wl.shared, rms=nxt is not None, eps=1e-6,
                              out=nxt if nxt is not None else out, topk_ids=ids, topk_w=w, ws=ws)

    def step(i, profile=False, x_in=None):
        """Enqueue one step (set i for single layers; all layers for the stack)."""
        if stack:
            x = x0 if x_in is None else x_in
            for l in range(wl.layers):
                if profile:
                    moe.moe_profile_events(ev_b[l], ev_a[l])
                nxt = act[l % 2]
                layer_call(x, sets[l], nxt=nxt)
                x = nxt
            return x
        if profile:
            moe.moe_profile_events(ev_b[i], ev_a[i])
        layer_call(sets[i]["hidden"] if x_in is None else x_in, sets[i], out=outs[i])
        return outs[i]

    with torch.cuda.stream(stream):
        # warm-up, and the unique experts each set touches
        for i in range(max(args.warmup, nsets if not stack else 1)):
            step(i % nsets)
            if not stack and i < nsets:
                torch.cuda.current_stream().synchronize()
                unique[i] = len(torch.unique(ids).tolist())
        stream.synchronize()
        if stack:
            # unique experts per layer along the stack's own routing
            x = x0
            for l in range(wl.layers):
                layer_call(x, sets[l], nxt=act[l % 2])
                stream.synchronize()
                unique[l] = len(torch.unique(ids).tolist())
                x = act[l % 2]
        assert moe.moe_check_device_error(ws, stream) == 0

        # Timed graphs hold consecutive steps over the weight sets (like consecutive
        # layers of a model) with no profiling nodes; K steps = full replays plus one
        # graph of the remainder. Separate one-step graphs with the library's events
        # around the expert kernel give its duration. The e2e graphs add, to every
        # step, the copy of its tokens from pinned host memory and of its output back.
        n_in = 1 if stack else nsets
        h_in = [(x0 if stack else sets[i]["hidden"]).cpu().pin_memory() for i in range(n_in)]
        h_out = [torch.empty(T, H, dtype=torch.bfloat16).pin_memory() for _ in range(n_in)]
        dst_in = [x0 if stack else sets[i]["hidden"] for i in range(n_in)]
        finals = [act[(wl.layers - 1) % 2]] if stack else outs
        copy_stream = torch.cuda.Stream(device=dev)
        ev_fork, ev_join = torch.cuda.Event(), torch.cuda.Event()
        ev_in = [torch.cuda.Event() for _ in range(n_in)]
        ev_done = [torch.cuda.Event() for _ in range(n_in)]

        def enqueue(seq, profile=False, e2e=False):
            if not e2e:
                for i in seq:
                    step(i, profile=profile)
                if profile:
                    moe.moe_profile_events(None, None)
                return
            # every step copies its tokens in from pinned host memory and its output
            # back, on a copy stream: the copy-in of later steps and the copy-out of
            # earlier ones overlap a step's kernels, as a serving loop would
            cur = torch.cuda.current_stream()
            ev_fork.record(cur)
            copy_stream.wait_event(ev_fork)
            with torch.cuda.stream(copy_stream):
                for i in seq:
                    dst_in[i].copy_(h_in[i], non_blocking=True)
                    ev_in[i].record(copy_stream)
            for i in seq:
                cur.wait_event(ev_in[i])
                step(i)
                ev_done[i].record(cur)
                copy_stream.wait_event(ev_done[i])
                with torch.cuda.stream(copy_stream):
                    h_out[i].copy_(finals[i], non_blocking=True)
            ev_join.record(copy_stream)
            cur.wait_event(ev_join)

        use_graph = not args.no_graph
        per = n_in                      # steps per full graph
        rem = steps % per
        G = {}
        if use_graph:
            try:
                for key, seq, prof, e2e in [("all", range(per), False, False), ("rem", range(rem), False, False),
                                            ("e2e_all", range(per), False, True), ("e2e_rem", range(rem), False, True)] + \
                                           [("prof%d" % i, [i], True, False) for i in range(per)]:
                    if len(seq) == 0:
                        continue
                    g = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(g, stream=stream):
                        enqueue(seq, profile=prof, e2e=e2e)
                    G[key] = g
            except Exception as exc:  # capture not possible: time eager launches
                moe.moe_profile_events(None, None)
                print("graph capture failed (%s); timing eager launches" % exc, file=sys.stderr)
                G, use_graph = {}, False

        def run_steps(nsteps, e2e=False):
            """Exactly nsteps steps, set i % per for step i."""
            if use_graph:
                pre = "e2e_" if e2e else ""
                for _ in range(nsteps // per):
                    G[pre + "all"].replay()
                if nsteps % per:
                    assert nsteps % per == rem
                    G[pre + "rem"].replay()
            else:
                for i in range(nsteps):
                    enqueue([i % per], e2e=e2e)

        # warm-up: at least W untimed steps, in whole graphs
        for _ in range(-(-max(args.warmup, 1) // per)):
            if use_graph:
                G["all"].replay()
            else:
                enqueue(range(per))
        stream.synchronize()
        barrier(world)

        # The clock sampler runs over a window of back-to-back passes of the same
        # graphs that ends with the timed region, at least args.clock_ms long, so
        # that it sees the GPU under this load even when the timed region is short.
        clocks = Clocks(local)
        clocks.start()
        w0 = time.perf_counter()
        while (time.perf_counter() - w0) * 1e3 < args.clock_ms:
            if use_graph:
                G["all"].replay()
            else:
                enqueue(range(per))
            stream.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        run_steps(steps)
        t1.record(stream)
        stream.synchronize()
        window_ms = (time.perf_counter() - w0) * 1e3
        ms = t0.elapsed_time(t1)
        clk = clocks.stop()
        if clk is not None:
            clk["window_ms"] = round(window_ms, 1)
            clk["window"] = "back-to-back passes of the timed graphs, ending with the timed region"
        assert moe.moe_check_device_error(ws, stream) == 0

        # expert kernel durations: each set's profiled step once, in rotation
        # (so no set finds its experts in L2), after the timed region
        for i in range(per):
            if use_graph:
                G["prof%d" % i].replay()
            else:
                enqueue([i], profile=True)
        stream.synchronize()
        extra = router_bytes if routes_itself else 0
        if stack:
            durs = [ev_b[l].elapsed_time(ev_a[l]) for l in range(wl.layers)]
            bytes_l = [u * EXPERT_BYTES + extra for u in unique]
        else:
            durs = [ev_b[i].elapsed_time(ev_a[i]) for i in range(per)]
            bytes_l = [unique[i] * EXPERT_BYTES + extra for i in range(per)]

        # end to end through the same calls, with the host copies inside the timed region
        run_steps(per, e2e=True)
        stream.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        run_steps(steps, e2e=True)
        e1.record(stream)
        stream.synchronize()
        ms_e2e = e0.elapsed_time(e1)

        # end to end, eager: every step is a copy of its tokens from pinned host
        # memory, the layer's C-ABI calls launched from the host (no graph), and
        # the copy of its output back, in order on one stream
        def eager_step(i):
            j = i % n_in
            dst_in[j].copy_(h_in[j], non_blocking=True)
            res = step(j, x_in=dst_in[j])
            h_out[j].copy_(res, non_blocking=True)

        for i in range(max(args.warmup, 1)):
            eager_step(i)
        stream.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for i in range(steps):
            eager_step(i)
        g1.record(stream)
        stream.synchronize()
        ms_eager = g0.elapsed_time(g1)
        assert moe.moe_check_device_error(ws, stream) == 0

    ms = max_over_ranks(ms, world)
    ms_e2e = max_over_ranks(ms_e2e, world)
    ms_eager = max_over_ranks(ms_eager, world)
    fused = T <= FUSED_MAX_T
    kernel_timing = "CUDA events around the kernel, in one-step graphs replayed after the timed region"
    if routes_itself:
        # the step is this one launch (per layer): its duration is the timed region's
        # events over the launches it holds (the one-step graphs would add a graph
        # launch's start-up to each)
        durs = [ms / (steps * wl.layers)] * len(bytes_l)
        kernel_timing = "CUDA events over the timed region, which holds one launch per layer"
    pk, pk_src = peaks()
    hbm_gbs = sum(bytes_l) / (sum(durs) * 1e-3) / 1e9
    flops_launch = 2.0 * 3 * H * I * T * kf          # algorithmic: gate, up and down over all slots
    expert_kernel = ("decode_fused_kernel (the router inside)" if routes_itself else "decode_fused_kernel") if fused \
        else "prefill_kernel (gate_up + down launches)"
    if wl.shared:
        expert_kernel += ", shared expert as expert E"
    # the binding roofline: whichever of the unique weight bytes at the copy rate
    # and the flops at the tensor rate takes longer. The tensor peak is the dense
    # bf16 burst rate; a stack's fraction of the sustained rate is given beside it.
    tflops = flops_launch * len(durs) / (sum(durs) * 1e-3) / 1e12
    if binding_roofline(statistics.mean(bytes_l), flops_launch, pk["hbm_gbs"], pk["bf16_tflops"]) == "tensor":
        roof = {"kernel": expert_kernel, "bound": "tensor", "achieved": tflops,
                "peak": pk["bf16_tflops"], "peak_source": "%s bf16_tflops (cuBLAS bf16 dense, burst)" % pk_src,
                "unit": "TFLOP/s", "frac": tflops / pk["bf16_tflops"], "traffic": recorded_traffic(wl.name),
                "algorithmic_flops_per_launch": flops_launch,
                "hbm_achieved_gbs": hbm_gbs, "hbm_frac": hbm_gbs / pk["hbm_gbs"]}
        if stack:
            roof["frac_of_sustained"] = tflops / pk["bf16_tflops_sustained"]
    else:
        roof = {"kernel": expert_kernel, "bound": "hbm", "achieved": hbm_gbs, "peak": pk["hbm_gbs"],
                "peak_source": pk_src + " hbm_gbs (copy)", "unit": "GB/s", "frac": hbm_gbs / pk["hbm_gbs"],
                "traffic": recorded_traffic(wl.name),
                "tensor_achieved_tflops": tflops, "tensor_frac": tflops / pk["bf16_tflops"]}
    roof.update({"algorithmic_bytes_per_launch": statistics.mean(bytes_l),
                 "kernel_ms_per_launch": statistics.mean(durs), "launches_measured": len(durs),
                 "unique_experts_per_launch": statistics.mean(unique[:len(durs)]),
                 "router_bytes_per_launch": router_bytes if routes_itself else 0,
                 "kernel_timing": kernel_timing})
    nlaunch = steps * wl.layers * launches_per_layer(T, E, routes_itself)
    return {
        "metric": "MoE layer tok/s (%s)" % wl.name,
        "value": world * T * steps / (ms * 1e-3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": args.warmup,
        "ms_per_step": ms / steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 activations x int4 weights, fp32 accumulate",
        "data": "synthetic (seeded; shapes and distributions of the pages' workload; random weights)",
        "config": {"workload": wl.name, "T": T, "H": H, "E": E, "k": k, "I": I, "layers": wl.layers,
                   "shared_expert": wl.shared,
                   "zipf": wl.zipf, "weight_sets": nsets,
                   "l2": "rotating %d independent weight sets (> L2) between steps" % nsets
                   if not stack else "48 layers x 1.3 GB of weights per step (> L2)",
                   "graph": use_graph, "steps_per_graph": per if use_graph else 1,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "roofline": roof,
        "e2e": {"value": world * T * steps / (ms_e2e * 1e-3), "unit": "tok/s",
                "h2d_bytes_per_step": T * H * 2, "d2h_bytes_per_step": T * H * 2,
                "copies": "pinned host buffers, one copy in and one out per step, on a copy stream; "
                          "the steps replayed from CUDA graphs",
                "eager": {"value": world * T * steps / (ms_eager * 1e-3), "unit": "tok/s",
                          "ms_per_step": ms_eager / steps,
                          "how": "per step: copy in from pinned host memory, moe_layer_forward%s "
                                 "called through the C ABI from the host (no graph), copy out; one stream"
                                 % (" (with the RMS step) x %d layers" % wl.layers if stack else "")}},
        "gpu_launches": nlaunch,
        "clocks": clk,
    }


# ------------------------------------------------ W8A16 and quantiser workloads --
# Outside the MoE layer proper, the pages' INT8 layers and the INT4 quantiser:
#   w8a16_lm_head_decode1: lm_head [248320, 2560] INT8 gs128 at T = 1 (a GEMV, HBM-bound);
#   w8a16_hc_prefill512:   a hyper-connection down + up pair ([320, 10240] and [10240, 320],
#                          INT8 gs64) at T = 512, one weight pair per layer rotated over 48 layers;
#   quantize_experts:      RTN INT4 g128 with a 50-candidate clip search over 32 experts' w1
#                          rows ([40960, 2560] bf16), two sets rotated.
EXTRA = {
    "w8a16_lm_head_decode1": dict(kind="w8a16", T=1, layers=[(248320, 2560, 128)], sets=1),
    "w8a16_hc_prefill512": dict(kind="w8a16", T=512, layers=[(320, 10240, 64), (10240, 320, 64)], sets=48),
    "quantize_experts": dict(kind="quant", N=32 * 1280, K=2560, nclip=50, sets=2),
}
ISSUE_PER_SMSP = 1.0   # warp instructions issued per cycle per SM sub-partition (4 per SM)


def recorded_counter(config: str, key: str):
    """A per-launch counter of a committed ncu capture, if taken on the current sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(config)
    if not e or e.get("source_hash") != source_hash(e.get("sources", [])):
        return None
    return e.get(key)


def graph_timing(args, stream, one_step, steps, local, world, copy_in=None, copy_out=None):
    """Times `steps` replays of a one-step CUDA graph (and of a graph that adds the host
    copies), with the clock window of measure(). Returns (ms, ms_e2e, clocks)."""
    with torch.cuda.stream(stream):
        for _ in range(max(args.warmup, 1)):
            one_step()
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            one_step()
        ge = None
        if copy_in is not None:
            ge = torch.cuda.CUDAGraph()
            with torch.cuda.graph(ge, stream=stream):
                copy_in()
                one_step()
                copy_out()
        for _ in range(max(args.warmup, 3)):
            g.replay()
        stream.synchronize()
        barrier(world)
        clocks = Clocks(local)
        clocks.start()
        w0 = time.perf_counter()
        while (time.perf_counter() - w0) * 1e3 < args.clock_ms:
            for _ in range(8):
                g.replay()
            stream.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            g.replay()
        t1.record(stream)
        stream.synchronize()
        window = (time.perf_counter() - w0) * 1e3
        ms = t0.elapsed_time(t1)
        clk = clocks.stop()
        if clk is not None:
            clk["window_ms"] = round(window, 1)
            clk["window"] = "back-to-back replays of the timed graph, ending with the timed region"
        ms_e2e = None
        if ge is not None:
            for _ in range(2):
                ge.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(steps):
                ge.replay()
            e1.record(stream)
            stream.synchronize()
            ms_e2e = e0.elapsed_time(e1)
    return max_over_ranks(ms, world), (max_over_ranks(ms_e2e, world) if ms_e2e is not None else None), clk


def measure_w8a16(args, name, steps, rank, world, local):
    import w4a16_mixture_experts_gb300 as moe
    moe.build()
    moe.lib()
    cfg = EXTRA[name]
    T, layers, nsets = cfg["T"], cfg["layers"], args.sets or cfg["sets"]
    dev = torch.device("cuda", torch.cuda.current_device())
    seed = args.seed + 1000 * rank
    K0 = layers[0][1]
    W = []
    for s in range(nsets):
        W.append([{k: v.to(dev) for k, v in synth.int8_weights(N, K, gs, seed=seed, layer=100 * s + j).items()}
                  for j, (N, K, gs) in enumerate(layers)])
    x = synth.hidden(T, K0, seed=seed).to(dev)
    bufs = [torch.empty(T, N, dtype=torch.bfloat16, device=dev) for (N, K, gs) in layers]
    ws = torch.zeros(max(moe.moe_w8a16_workspace_size(T, N, K, gs) for (N, K, gs) in layers), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(device=dev)
    h_in = x.cpu().pin_memory()
    h_out = torch.empty_like(bufs[-1], device="cpu").pin_memory()

    def one_step():
        # one pass over the weight sets (the sets are consecutive layers of a model)
        for s in range(nsets):
            inp = x
            for j, (N, K, gs) in enumerate(layers):
                moe.moe_w8a16_linear(inp, W[s][j]["w_packed"], W[s][j]["scales"], gs, y=bufs[j], ws=ws)
                inp = bufs[j]

    ms, ms_e2e, clk = graph_timing(args, stream, one_step, steps, local, world,
                                   copy_in=lambda: x.copy_(h_in, non_blocking=True),
                                   copy_out=lambda: h_out.copy_(bufs[-1], non_blocking=True))
    assert moe.moe_check_device_error(ws, stream) == 0
    per_layer_ms = ms / steps / nsets
    pk, pk_src = peaks()
    nbytes = sum(N * K + N * (K // gs) * 2 for (N, K, gs) in layers)
    flops = sum(2.0 * T * N * K for (N, K, gs) in layers)
    gbs, tfl = nbytes / (per_layer_ms * 1e-3) / 1e9, flops / (per_layer_ms * 1e-3) / 1e12
    kern = "w8a16_gemv_kernel" if T <= 8 else "prefill_kernel<true, false> (dense INT8 GEMM, split over K where it has few tiles)"
    if binding_roofline(nbytes, flops, pk["hbm_gbs"], pk["bf16_tflops"]) == "tensor":
        roof = {"kernel": kern, "bound": "tensor", "achieved": tfl, "peak": pk["bf16_tflops"],
                "peak_source": "%s bf16_tflops (cuBLAS bf16 dense, burst)" % pk_src, "unit": "TFLOP/s",
                "frac": tfl / pk["bf16_tflops"], "hbm_achieved_gbs": gbs, "hbm_frac": gbs / pk["hbm_gbs"]}
    else:
        roof = {"kernel": kern, "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                "peak_source": pk_src + " hbm_gbs (copy)", "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                "tensor_achieved_tflops": tfl, "tensor_frac": tfl / pk["bf16_tflops"]}
    roof.update({"traffic": recorded_counter(name, "dram_bytes_per_launch"), "algorithmic_bytes_per_launch": nbytes,
                 "algorithmic_flops_per_launch": flops, "kernel_ms_per_launch": per_layer_ms,
                 "launches_measured": steps * nsets,
                 "timing": "the step's graph (the layer's launches only) over CUDA events"})
    return {
        "metric": "W8A16 layer tok/s (%s)" % name, "value": world * T * steps / (ms * 1e-3), "unit": "tok/s",
        "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 activations x int8 weights, fp32 accumulate",
        "data": "synthetic (seeded INT8 pack-quantized weights, N(0,1) activations)",
        "config": {"workload": name, "T": T, "layers": [dict(N=N, K=K, gs=gs) for (N, K, gs) in layers],
                   "weight_sets": nsets, "l2": "weights of a step exceed L2" if nbytes * nsets > L2_BYTES else
                   "weights fit L2 (tensor-bound)", "graph": True},
        "roofline": roof,
        "e2e": {"value": world * T * steps / (ms_e2e * 1e-3), "unit": "tok/s", "h2d_bytes_per_step": T * K0 * 2,
                "d2h_bytes_per_step": bufs[-1].numel() * 2,
                "copies": "pinned host buffers, copy in and out inside the replayed graph"},
        "gpu_launches": steps * nsets * sum(1 if T <= 8 or moe.moe_w8a16_workspace_size(T, N, K, gs) == 256 else 2
                                            for (N, K, gs) in layers),
        "clocks": clk,
    }


def measure_quant(args, name, steps, rank, world, local):
    import w4a16_mixture_experts_gb300 as moe
    moe.build()
    moe.lib()
    cfg = EXTRA[name]
    N, K, nclip, nsets = cfg["N"], cfg["K"], cfg["nclip"], args.sets or cfg["sets"]
    dev = torch.device("cuda", torch.cuda.current_device())
    seed = args.seed + 1000 * rank
    Ws = [synth.bf16_weights(N, K, seed=seed, layer=s).to(dev) for s in range(nsets)]
    packed = torch.empty(N, K // 8, dtype=torch.int32, device=dev)
    scales = torch.empty(N, K // 128, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    h_in = Ws[0].cpu().pin_memory()
    h_out = torch.empty_like(packed, device="cpu").pin_memory()

    def one_step():
        for s in range(nsets):
            lib = moe.lib()
            rc = lib.moe_quantize_int4(moe._p(Ws[s]), N, K, nclip, moe._p(packed), moe._p(scales), None,
                                       moe._stream(None))
            assert rc == 0

    ms, ms_e2e, clk = graph_timing(args, stream, one_step, steps, local, world,
                                   copy_in=lambda: Ws[0].copy_(h_in, non_blocking=True),
                                   copy_out=lambda: h_out.copy_(packed, non_blocking=True))
    per_launch_ms = ms / steps / nsets
    pk, pk_src = peaks()
    weights = N * K
    inst = recorded_counter(name, "warp_instructions_per_launch")
    clock_mhz = (clk or {}).get("sm_mhz") or pk.get("sm_max_mhz", 2070.0)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    peak_issue = sms * 4 * ISSUE_PER_SMSP * clock_mhz * 1e6   # warp instructions per second
    roof = {"kernel": "quantize_int4_kernel", "bound": "alu",
            "achieved": inst / (per_launch_ms * 1e-3) if inst else None,
            "peak": peak_issue, "unit": "warp instructions/s",
            "peak_source": "%d SMs x 4 sub-partitions x 1 warp instruction/cycle x %.0f MHz (sampled)" % (sms, clock_mhz),
            "frac": inst / (per_launch_ms * 1e-3) / peak_issue if inst else None,
            "warp_instructions_per_launch": inst,
            "candidate_evaluations_per_s": weights * nclip / (per_launch_ms * 1e-3),
            "hbm_bytes_per_launch": weights * 2 + weights // 2 + (weights // 128) * 2,
            "hbm_frac": (weights * 2 + weights // 2 + (weights // 128) * 2) / (per_launch_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
            "traffic": recorded_counter(name, "dram_bytes_per_launch"), "kernel_ms_per_launch": per_launch_ms,
            "launches_measured": steps * nsets}
    return {
        "metric": "INT4 quantiser weights/s (%s)" % name, "value": world * weights * nsets * steps / (ms * 1e-3),
        "unit": "weights/s", "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": ms / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 in, fp32 search, int4 out",
        "data": "synthetic (seeded N(0, 0.02^2) bf16 weights with outliers)",
        "config": {"workload": name, "N": N, "K": K, "nclip": nclip, "sets": nsets,
                   "l2": "%d sets of %d MB rotated (> L2)" % (nsets, N * K * 2 >> 20), "graph": True},
        "roofline": roof,
        "e2e": {"value": world * weights * steps / (ms_e2e * 1e-3), "unit": "weights/s",
                "h2d_bytes_per_step": N * K * 2, "d2h_bytes_per_step": N * K // 2,
                "copies": "one weight set in and its packed words out, pinned host buffers, inside the graph",
                "note": "the e2e step quantises the %d sets once each after the copy" % nsets},
        "gpu_launches": steps * nsets,
        "clocks": clk,
    }


def cpu_baseline_extra(name, seed, target_s):
    """The oracle on a bounded sample of an EXTRA workload, scaled to its unit."""
    import oracle
    oracle.build()
    cores = oracle.max_threads()
    cfg = EXTRA[name]
    if cfg["kind"] == "w8a16":
        T = cfg["T"]
        # time each layer on a sample of its rows (T = 1) or of the tokens (T > 1), then scale up
        total, parts = 0.0, []
        for (N, K, gs) in cfg["layers"]:
            n = min(N, 4096) if T == 1 else N
            t_tok = T if T == 1 else min(T, 16)
            d = synth.int8_weights(n, K, gs, seed=seed)
            x = synth.hidden(t_tok, K, seed=seed)
            t0 = time.perf_counter()
            oracle.w8a16_linear(x, d["w_packed"], d["scales"], gs)
            dt = time.perf_counter() - t0
            total += dt * (N / n) * (T / t_tok)
            parts.append("%d of %d rows x %d of %d tokens" % (n, N, t_tok, T))
        nsets = cfg["sets"]
        return {"value": T / (total * nsets), "unit": "tok/s", "cores": cores, "kind": "oracle",
                "sample": "fp64 oracle on " + "; ".join(parts) + ", scaled to the whole layer%s" %
                          (" and to the %d layers of a step" % nsets if nsets > 1 else "")}
    N, K, nclip = cfg["N"], cfg["K"], cfg["nclip"]
    n = 64
    w = synth.bf16_weights(n, K, seed=seed)
    t0 = time.perf_counter()
    oracle.quantize_int4(w, nclip)
    dt = time.perf_counter() - t0
    n = max(n, min(N, int(n * target_s / max(dt, 1e-3))))
    w = synth.bf16_weights(n, K, seed=seed)
    t0 = time.perf_counter()
    oracle.quantize_int4(w, nclip)
    dt = time.perf_counter() - t0
    return {"value": n * K / dt, "unit": "weights/s", "cores": cores, "kind": "oracle",
            "sample": "%d rows x %d of the quantiser input, %d clip candidates, %.1f s" % (n, K, nclip, dt)}


# Workloads measured beside the headline one in a default run: the metric's other
# two batch sizes (64 concurrent decode tokens; the 4096-token prefill on the
# 48-layer stack).
PER_CONFIG = ("decode64", "stack_prefill4096", "shared_decode1", "w8a16_lm_head_decode1", "w8a16_hc_prefill512",
              "quantize_experts")


def measure_any(args, name, steps, rank, world, local):
    if name in EXTRA:
        fn = measure_w8a16 if EXTRA[name]["kind"] == "w8a16" else measure_quant
        return fn(args, name, steps, rank, world, local)
    return measure(args, synth.WORKLOADS[name], steps, rank, world, local)


def run_ours(args, rank, world, local):
    res = measure_any(args, args.config, args.steps, rank, world, local)
    if args.per_config and args.config == "decode1":
        res["per_config"] = {}
        for name in PER_CONFIG:
            torch.cuda.empty_cache()
            res["per_config"][name] = measure_any(args, name, args.steps, rank, world, local)
            torch.cuda.empty_cache()
    return res


def baseline_any(name, seed, target_s):
    if name in EXTRA:
        return cpu_baseline_extra(name, seed, target_s)
    return cpu_baseline(synth.WORKLOADS[name], seed, target_s)


def main():
    args = parse()
    if args.impl == "reference":
        # the oracle on the host cores: rank 0 alone runs it, the other ranks leave at once
        rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
        if rank == 0:
            cb = baseline_any(args.config, args.seed, args.cpu_seconds)
            metric = ("MoE layer tok/s (%s)" % args.config if args.config in synth.WORKLOADS else
                      ("W8A16 layer tok/s (%s)" if EXTRA[args.config]["kind"] == "w8a16" else
                       "INT4 quantiser weights/s (%s)") % args.config)
            line = {"impl": "reference", "metric": metric, "value": cb["value"],
                    "unit": cb["unit"], "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                    "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                    "data": "synthetic", "config": {"workload": args.config},
                    "cpu_baseline": cb,
                    "e2e": {"value": cb["value"], "unit": cb["unit"], "h2d_bytes_per_step": 0,
                            "d2h_bytes_per_step": 0}}
            print(json.dumps(line), flush=True)
        return
    rank, world, local = dist_setup(args)
    res = run_ours(args, rank, world, local)
    if rank == 0:
        res["cpu_baseline"] = baseline_any(args.config, args.seed, args.cpu_seconds)
        for name, r in res.get("per_config", {}).items():
            r["cpu_baseline"] = baseline_any(name, args.seed, args.cpu_seconds / 2)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
