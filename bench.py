#!/usr/bin/env python3
"""Benchmark of the MoE decode layer on GB300.

One step = one pass of the whole layer over one batch: router GEMM -> fp32
softmax/top-8 with the SERE reroute fused in (K'=2, rho=0.5) -> expert-sorted
dispatch -> tcgen05 grouped SwiGLU FFN with the combine fused in.  Workload:
the Qwen3-30B-A3B-shaped decode layer (batch 32, hidden 2048, 128 experts,
top-8, intermediate 768, bf16 experts, fp32 router), synthetic seeded inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun every rank runs its own replica
of the layer on its own batches (the path does not shard); the value is the
tokens of all ranks over the slowest rank's time.  `--impl reference` times
the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import signal
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T, H, N, K_TOP, I = 32, 2048, 128, 8, 768
K_PRIMARY, RHO = 2, 0.5
N_BATCHES = 8
N_COPIES = 4  # expert-weight copies rotated per step (--copies)
E2E_GROUP = 16  # end-to-end steps per captured group
STEP_GROUP = 16  # layer steps per captured graph (decode and sweep)
METRIC = "MoE-layer decode tokens/s (SERE K'=2, rho=0.5; top-8 alongside)"
UNIT = "tokens/s"
EXPERT_BYTES = 3 * H * I * 2
# The committed ncu summary of the decode FFN kernel.  Its DRAM traffic is
# reported only while the kernel's sources hash to the value recorded in it.
FFN_PROFILE = os.path.join(ROOT, "profiles", "ffn_decode_kernel_decode_b32_full.md")
FFN_SOURCES = [os.path.join(ROOT, "expert_routing_moe_gb300", "csrc", f)
               for f in ("ffn_decode.cu", "common.cuh", "tmap.h")]


def ffn_sources_sha256():
    import hashlib
    h = hashlib.sha256()
    for f in FFN_SOURCES:
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ffn_traffic_capture():
    """(dram bytes, algorithmic bytes, active experts) of one FFN launch from
    the committed ncu summary, or None when the summary is missing or was
    taken on other kernel sources than the ones built now."""
    if not os.path.exists(FFN_PROFILE):
        return None
    kv = {}
    for line in open(FFN_PROFILE):
        if line.startswith("- ") and ": " in line:
            key, val = line[2:].split(": ", 1)
            kv[key.strip()] = val.strip().strip("`")
    try:
        if kv["sources_sha256"] != ffn_sources_sha256():
            return None
        return (float(kv["traffic_bytes_per_launch"]), float(kv["algorithmic_bytes_per_launch"]),
                int(kv["active_experts"]))
    except (KeyError, ValueError):
        return None


def workload_config(extra=None):
    c = {"workload": "single MoE decode layer, Qwen3-30B-A3B shape: batch 32, hidden 2048, 128 experts, top-8, "
                     "SwiGLU intermediate 768, bf16 experts, fp32 router; SERE K'=2, rho=0.5, 16x8 clustered "
                     "similarity",
         "batch": T, "hidden": H, "experts": N, "top_k": K_TOP, "intermediate": I, "k_primary": K_PRIMARY,
         "rho": RHO,
         "l2": "inputs larger than L2: %d expert-weight copies (%.2f GB) and %d token batches rotated per step"
               % (N_COPIES, N_COPIES * N * EXPERT_BYTES / 1e9, N_BATCHES)}
    if extra:
        c.update(extra)
    return c


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_inputs(rank, config_seed, n_batches):
    """A replica's own inputs: the seed of its device-drawn weight copies and
    the token-stream offsets of its batches.  Ranks never share a batch, so
    N replicas process N times the tokens (weak scaling)."""
    return config_seed + 10 * (rank + 1), [b + 97 * rank for b in range(n_batches)]


def job_throughput(ws, tokens_per_rank_step, steps, max_ms):
    """Whole-job tokens/s: the tokens of every rank over the slowest rank's time."""
    return ws * tokens_per_rank_step * steps / (max_ms / 1e3)


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.send_signal(signal.SIGTERM)
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            p = [v.strip() for v in line.split(",")]
            if len(p) >= 9:
                rows.append(p)
        os.unlink(self.path)
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    return 6800.0, "fallback 6.8 TB/s"


# ---------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline leg)
# ---------------------------------------------------------------------------
def oracle_sample(budget_s: float, max_batches: int = 64, threads: int = 1):
    """Times the oracle layer (router -> rank -> SERE -> permute -> FFN) on
    whole decode batches of the workload until `budget_s` is used, with
    `threads` host threads (0: every core).  Returns (tokens/s, seconds,
    batches, threads used)."""
    import oracle
    from expert_routing_moe_gb300 import synthetic as syn
    nt = oracle.set_threads(threads)
    L = syn.decode(T)
    L.k_primary, L.rho = K_PRIMARY, RHO
    oracle.layer(L, sere_on=True, tokens=np.arange(1))  # load + warm the library
    # the batches are drawn before the clock starts
    batches = []
    for b in range(N_BATCHES):
        Lb = syn.decode(T, with_weights=False, token_stream_offset=b)
        Lb.w_gate, Lb.w_up, Lb.w_down = L.w_gate, L.w_up, L.w_down
        batches.append(Lb)
    toks, t0, nb = 0, time.perf_counter(), 0
    while nb < max_batches:
        oracle.layer(batches[nb % N_BATCHES], sere_on=True)
        toks += T
        nb += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return toks / el, el, nb, nt


def oracle_timed(Ls, budget_s: float, threads: int, sere: bool, capacity: bool = False, tokens=None):
    """Runs oracle.layer over the layers of Ls in turn until `budget_s` is
    used (at least one).  Returns (seconds, layers run, threads used)."""
    import oracle
    nt = oracle.set_threads(threads)
    t0, n = time.perf_counter(), 0
    while True:
        oracle.layer(Ls[n % len(Ls)], sere_on=sere, capacity_on=capacity, tokens=tokens)
        n += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    return time.perf_counter() - t0, n, nt


def cpu_baseline_legs(budget_s: float):
    """The oracle on every host core and on one, each on whole batches of
    the decode workload for about `budget_s` seconds."""
    v, el, nb, nt = oracle_sample(budget_s, threads=0)
    v1, el1, nb1, _ = oracle_sample(budget_s, threads=1)
    what = "whole decode batches of %d tokens through the oracle layer (router, rank, SERE, permute, FFN + combine)"
    return {"value": v, "unit": UNIT, "cores": nt, "kind": "oracle",
            "sample": "%d %s in %.1f s on %d threads (OpenMP over tokens)" % (nb, what % T, el, nt),
            "single_thread": {"value": v1, "unit": UNIT, "cores": 1,
                              "sample": "%d %s in %.1f s on one thread" % (nb1, what % T, el1)}}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from expert_routing_moe_gb300 import synthetic as syn
    oracle.build()
    nt = oracle.set_threads(0)  # every host core (OpenMP over tokens)
    L = syn.decode(T)
    L.k_primary, L.rho = K_PRIMARY, RHO
    # per-step sample: whole batches when the run fits in ~3 minutes, else a token subset
    t0 = time.perf_counter()
    oracle.layer(L, sere_on=True)
    per_batch = time.perf_counter() - t0
    n_steps = args.steps + args.warmup
    budget = 170.0
    ntok = T if per_batch * n_steps <= budget else max(1, int(T * budget / (per_batch * n_steps)))
    batches = [syn.decode(T, with_weights=False, token_stream_offset=b) for b in range(N_BATCHES)]
    for b in batches:
        b.w_gate, b.w_up, b.w_down = L.w_gate, L.w_up, L.w_down
        b.k_primary, b.rho = K_PRIMARY, RHO
    tokens = np.arange(ntok)
    for i in range(args.warmup):
        oracle.layer(batches[i % N_BATCHES], sere_on=True, tokens=tokens)
    t0 = time.perf_counter()
    for i in range(args.steps):
        oracle.layer(batches[i % N_BATCHES], sere_on=True, tokens=tokens)
    el = time.perf_counter() - t0
    value = ntok * args.steps / el
    sample = ("oracle layer per step: router, rank and SERE over the whole batch of %d tokens, FFN + combine for "
              "%d token(s) of it; %d host threads" % (T, ntok, nt))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": nt, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def _gpu_setup():
    import torch
    import expert_routing_moe_gb300 as moe
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    from expert_routing_moe_gb300 import build as b
    b.build()
    moe.load()
    return torch, moe, dev, ws, rank, local


def _device_copies(torch, dev, L, n_copies, seed):
    """Expert weights: the host layer's own copy plus n_copies-1 device-drawn
    N(0, 0.02) bf16 copies of the same shapes (to rotate past the L2)."""
    Nn, Ii, Hh = L.N, L.I, L.H
    copies = [tuple(torch.from_numpy(a).view(torch.bfloat16).to(dev) for a in (L.w_gate, L.w_up, L.w_down))]
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    for _ in range(1, n_copies):
        copies.append(tuple((torch.randn(shape, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
                            for shape in ((Nn, Ii, Hh), (Nn, Ii, Hh), (Nn, Hh, Ii))))
    return copies


def _capture(torch, stream, layers, xs, sere, token_w=None):
    """Per (batch, weight copy): a routing+dispatch graph and an FFN graph."""
    graphs = []
    with torch.cuda.stream(stream):
        for bidx, x in enumerate(xs):
            lay = layers[bidx % len(layers)]
            T = x.shape[0]
            for _ in range(2):  # eager warm-up on the capture stream
                lay.forward(x, sere=sere, token_w=token_w)
            stream.synchronize()
            g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(g1, stream=stream):
                lay.route_and_dispatch(x, sere, token_w)
            with torch.cuda.graph(g2, stream=stream):
                lay.ffn(x)
            graphs.append((g1, g2))
    torch.cuda.synchronize()
    return graphs


def _capture_steps(torch, stream, layers, xs, sere, token_w=None, group=1, starts=None):
    """Graphs of `group` consecutive layer steps each (routing, dispatch and
    FFN per step, chained by programmatic dependent launch), step i on batch
    i mod len(xs) and weight copy (i mod len(xs)) mod len(layers); one graph
    per starting batch in `starts` (default: every batch)."""
    graphs = []
    nb = len(xs)
    with torch.cuda.stream(stream):
        for j, b0 in enumerate(range(nb) if starts is None else starts):
            for i in range(group):
                b = (b0 + i) % nb
                for _ in range(2 if j == 0 else 1):
                    layers[b % len(layers)].forward(xs[b], sere=sere, token_w=token_w)
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for i in range(group):
                    b = (b0 + i) % nb
                    layers[b % len(layers)].forward(xs[b], sere=sere, token_w=token_w)
            graphs.append(g)
    torch.cuda.synchronize()
    return graphs


class StepGraphs:
    """Exactly `steps` layer steps as graph replays: steps // group replays of
    graphs of `group` steps (rotating over the starting batches), then one
    graph of the remaining steps % group steps."""

    def __init__(self, torch, stream, layers, xs, sere, steps, token_w=None, group=STEP_GROUP):
        self.group = group
        self.full = _capture_steps(torch, stream, layers, xs, sere, token_w, group=group)
        self.r = steps % group
        self.rem = (_capture_steps(torch, stream, layers, xs, sere, token_w, group=self.r, starts=[0])[0]
                    if self.r else None)

    def run(self, steps, stream, torch):
        if steps % self.group != self.r:
            raise ValueError("the graphs were captured for a remainder of %d steps, not %d"
                             % (self.r, steps % self.group))
        nb = len(self.full)
        with torch.cuda.stream(stream):
            for i in range(steps // self.group):
                self.full[i % nb].replay()
            if self.rem is not None:
                self.rem.replay()


def _timed_passes(torch, dev, stream, sg, steps, warmup, ws, passes):
    """`passes` timed passes of exactly `steps` steps each (after at least
    `warmup` untimed steps), every pass bracketed by a barrier and a device
    synchronize on both sides and timed with CUDA events on the replay
    stream; each pass's time is the maximum over ranks.  Returns the per-pass
    times (ms)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    nb = len(sg.full)
    with torch.cuda.stream(stream):
        for i in range(-(-warmup // sg.group)):
            sg.full[i % nb].replay()
    out = []
    for _ in range(passes):
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = ev(), ev()
        e0.record(stream)
        sg.run(steps, stream, torch)
        e1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        out.append(_max_over_ranks(torch, dev, ws, e0.elapsed_time(e1)))
    return out


def _pass_summary(ms, steps):
    a = np.asarray(ms) / steps
    return {"passes": len(ms), "steps_per_pass": steps, "ms_per_step_median": float(np.median(a)),
            "ms_per_step_min": float(a.min()), "ms_per_step_max": float(a.max()),
            "spread_pct": float((a.max() - a.min()) / np.median(a) * 100.0)}


def _timed_steps(torch, stream, graphs, steps, warmup, ws, group=1):
    """`steps` layer steps as replays of graphs of `group` steps each (steps
    rounded down to a multiple of group), CUDA events around the run.
    Returns (ms, steps timed)."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    nb = len(graphs)
    reps = max(1, steps // group)
    with torch.cuda.stream(stream):
        for i in range(max(1, warmup // group)):
            graphs[i % nb].replay()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(reps):
            graphs[(i * group) % nb].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    return e0.elapsed_time(e1), reps * group


def _ffn_inline(torch, stream, layers, xs, sere, rounds=3, group=STEP_GROUP):
    """Each FFN call's own duration inside graphs of `group` layer steps:
    timing events captured right before and after every FFN call (external
    event-record nodes), each graph replayed and its events read back, over
    `rounds` passes of every graph.  Returns the durations (ms) and the batch
    index of each, or None where this PyTorch cannot record events in a
    graph."""
    nb = len(xs)
    try:
        graphs, evs = [], []
        with torch.cuda.stream(stream):
            for b0 in range(nb):
                pairs = [(torch.cuda.Event(enable_timing=True, external=True),
                          torch.cuda.Event(enable_timing=True, external=True)) for _ in range(group)]
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for i in range(group):
                        b = (b0 + i) % nb
                        lay = layers[b % len(layers)]
                        lay.route_and_dispatch(xs[b], sere)
                        pairs[i][0].record(stream)
                        lay.ffn(xs[b])
                        pairs[i][1].record(stream)
                graphs.append(g)
                evs.append(pairs)
        torch.cuda.synchronize()
        ms, bidx = [], []
        with torch.cuda.stream(stream):
            for g in graphs:   # warm-up pass
                g.replay()
            torch.cuda.synchronize()
            for _ in range(rounds):
                for b0, g in enumerate(graphs):
                    g.replay()
                    stream.synchronize()
                    for i, (a, e) in enumerate(evs[b0]):
                        ms.append(a.elapsed_time(e))
                        bidx.append((b0 + i) % nb)
        del graphs
        return ms, bidx
    except (TypeError, RuntimeError):
        return None


def _active_counts(torch, moe, stream, layers, xs, sere, token_w=None):
    us, rows = [], []
    for bidx, x in enumerate(xs):
        lay = layers[bidx % len(layers)]
        with torch.cuda.stream(stream):
            lay.forward(x, sere=sere, token_w=token_w)
        stream.synchronize()
        code, detail = lay.device_status()
        if code != 0:
            raise RuntimeError("device status %d (%s) detail %d" % (code, moe.status_string(code, True), detail))
        us.append(int(lay.active[0].item()))
        rows.append(int(lay.offsets[lay.N].item()))
    return us, rows


def _timed(torch, stream, graphs, steps, warmup, ws):
    """Replays `steps` steps (both graphs of one batch each); CUDA events on
    the replay stream around the whole run and around every FFN graph."""
    ev = lambda: torch.cuda.Event(enable_timing=True)
    nb = len(graphs)
    with torch.cuda.stream(stream):
        for i in range(warmup):
            g1, g2 = graphs[i % nb]
            g1.replay()
            g2.replay()
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    f0 = [ev() for _ in range(steps)]
    f1 = [ev() for _ in range(steps)]
    e0, e1 = ev(), ev()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(steps):
            g1, g2 = graphs[i % nb]
            g1.replay()
            f0[i].record(stream)
            g2.replay()
            f1[i].record(stream)
        e1.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    return e0.elapsed_time(e1), [a.elapsed_time(b) for a, b in zip(f0, f1)]


def _max_over_ranks(torch, dev, ws, v):
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def _soak(torch, stream, graphs, seconds):
    """Untimed replays so that the clock record covers a loaded GPU."""
    t_end = time.perf_counter() + seconds
    with torch.cuda.stream(stream):
        i = 0
        while time.perf_counter() < t_end:
            for _ in range(50):
                g1, g2 = graphs[i % len(graphs)]
                g1.replay()
                g2.replay()
                i += 1
            stream.synchronize()


def run_ours(args):
    torch, moe, dev, ws, rank, local = _gpu_setup()
    from expert_routing_moe_gb300 import synthetic as syn

    L = syn.decode(T)
    w_r = torch.from_numpy(L.w_r).to(dev)
    sim = torch.from_numpy(L.sim).to(dev)
    copy_seed, offsets = replica_inputs(rank, 1000 * syn.CONFIG_DECODE, N_BATCHES)
    copies = _device_copies(torch, dev, L, N_COPIES, copy_seed)
    xs = []
    for bidx in range(N_BATCHES):
        Lb = syn.decode(T, with_weights=False, token_stream_offset=offsets[bidx])
        xs.append(torch.from_numpy(Lb.x_bf16).view(torch.bfloat16).to(dev))
    layers = [moe.MoELayer(w_r, *copies[c], k=K_TOP, max_tokens=T, sim=sim, k_primary=K_PRIMARY, rho=RHO)
              for c in range(N_COPIES)]
    stream = torch.cuda.Stream(device=dev)

    us_sere, _ = _active_counts(torch, moe, stream, layers, xs, True)
    us_top8, _ = _active_counts(torch, moe, stream, layers, xs, False)
    s_sere = StepGraphs(torch, stream, layers, xs, True, args.steps)
    s_top8 = StepGraphs(torch, stream, layers, xs, False, args.steps)
    g_sere = _capture(torch, stream, layers, xs, True)
    g_top8 = _capture(torch, stream, layers, xs, False)
    # routing + SERE + permutation in one launch, then the FFN tensor-core kernel (which
    # zeroes y and resets its own counters)
    assert layers[0].decode_layer_ok(xs[0])
    launches_per_step = 2

    clk = ClockSampler(local if ws > 1 else 0)
    clk.start()
    if args.clock_soak > 0:
        _soak(torch, stream, g_sere, args.clock_soak)
    # the headline: exactly args.steps whole layer steps per pass, median of the passes
    p_sere = _timed_passes(torch, dev, stream, s_sere, args.steps, args.warmup, ws, args.passes)
    total_ms, steps_t = float(np.median(p_sere)), args.steps
    # the FFN's own duration: events around every FFN call inside the step graphs (else,
    # where events cannot be captured, a routing graph and an FFN graph with events between)
    inline = _ffn_inline(torch, stream, layers, xs, True)
    if inline is not None:
        ffn_ms, ffn_b = inline
        ffn_how = "events captured around every FFN call inside graphs of %d steps" % STEP_GROUP
    else:
        _, ffn_ms = _timed(torch, stream, g_sere, args.steps, args.warmup, ws)
        ffn_b = [i % N_BATCHES for i in range(args.steps)]
        ffn_how = "events between a routing graph and an FFN graph per step"
    ffn_bytes = [us_sere[b] * EXPERT_BYTES + T * H * 2 + T * H * 4 for b in ffn_b]
    p_top8 = _timed_passes(torch, dev, stream, s_top8, args.steps, args.warmup, ws, args.passes)
    t8_ms = float(np.median(p_top8))
    clocks = clk.stop()
    inline8 = _ffn_inline(torch, stream, layers, xs, False)
    if inline8 is not None:
        t8_ffn_ms, t8_b = inline8
    else:
        _, t8_ffn_ms = _timed(torch, stream, g_top8, args.steps, args.warmup, ws)
        t8_b = [i % N_BATCHES for i in range(args.steps)]
    t8_bytes = [us_top8[b] * EXPERT_BYTES + T * H * 2 + T * H * 4 for b in t8_b]

    # ---- end to end through the public API: pinned host x in, host y out, every step ----
    # The copies run on their own stream, overlapped with the layer: step i+1's
    # input is uploaded while step i computes, and step i's output is read back
    # while step i+1 computes (two output buffers; events order every reuse).
    xs_host = [x.cpu().pin_memory() for x in xs]
    y_host = [torch.empty(T, H, dtype=torch.float32).pin_memory() for _ in range(2)]
    y_dev = [torch.empty(T, H, dtype=torch.float32, device=dev) for _ in range(2)]
    x_dev = [torch.empty_like(x) for x in xs]
    cstream = torch.cuda.Stream(device=dev)
    h2d = [torch.cuda.Event() for _ in range(N_BATCHES)]
    fwd = [torch.cuda.Event() for _ in range(2)]
    d2h = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n, e_start=None):
        if e_start is not None:
            cstream.wait_event(e_start)
        with torch.cuda.stream(cstream):
            x_dev[0].copy_(xs_host[0], non_blocking=True)
            h2d[0].record(cstream)
        for i in range(n):
            b_i, j = i % N_BATCHES, i % 2
            lay = layers[b_i % N_COPIES]
            with torch.cuda.stream(stream):
                stream.wait_event(h2d[b_i])            # this step's input is on the device
                if i >= 2:
                    stream.wait_event(d2h[j])          # y_dev[j] was read back (step i-2)
                lay.forward(x_dev[b_i], sere=True, out=y_dev[j])
                fwd[j].record(stream)
            with torch.cuda.stream(cstream):
                if i + 1 < n:
                    nb = (i + 1) % N_BATCHES           # last read by step i-7, ordered before on this stream
                    x_dev[nb].copy_(xs_host[nb], non_blocking=True)
                    h2d[nb].record(cstream)
                cstream.wait_event(fwd[j])
                y_host[j].copy_(y_dev[j], non_blocking=True)
                d2h[j].record(cstream)
        stream.wait_event(d2h[(n - 1) % 2])
        if n >= 2:
            stream.wait_event(d2h[(n - 2) % 2])

    # the pipelined loop of E2E_GROUP steps is captured once (two streams joined
    # by events) and replayed, as a serving loop would, so that the host enqueues
    # one graph per E2E_GROUP steps instead of every copy and call; a graph of the
    # remaining steps makes every pass exactly args.steps steps
    e2e_steps(2)
    torch.cuda.synchronize()

    def e2e_graph(n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            e_fork = torch.cuda.Event()
            e_fork.record(stream)
            e2e_steps(n, e_fork)
        return g

    g_e2e = e2e_graph(E2E_GROUP)
    g_e2e_rem = e2e_graph(args.steps % E2E_GROUP) if args.steps % E2E_GROUP else None
    with torch.cuda.stream(stream):
        for _ in range(-(-args.warmup // E2E_GROUP)):
            g_e2e.replay()
    p_e2e = []
    for _ in range(args.passes):
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps // E2E_GROUP):
                g_e2e.replay()
            if g_e2e_rem is not None:
                g_e2e_rem.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        p_e2e.append(_max_over_ranks(torch, dev, ws, e0.elapsed_time(e1)))
    e2e_ms = float(np.median(p_e2e))
    for lay in layers:
        code, detail = lay.device_status()
        if code != 0:
            raise RuntimeError("device status %d detail %d after the timed runs" % (code, detail))

    peak, peak_src = load_peaks()
    achieved = sum(ffn_bytes) / (sum(ffn_ms) / 1e3) / 1e9
    cap = ffn_traffic_capture()
    line = {
        "metric": METRIC, "value": job_throughput(ws, T, steps_t, total_ms), "unit": UNIT, "n_gpus": ws,
        "steps": steps_t, "warmup": args.warmup, "ms_per_step": total_ms / steps_t,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Dirichlet-skewed router logits, N(0,0.02) bf16 experts)",
        "config": workload_config({"parallelism": "replicas" if ws > 1 else "single GPU",
                                   "cuda_graphs": "value: graphs of 16 layer steps (and one of the remaining "
                                                  "steps), each step the single-launch router + rank + SERE + "
                                                  "permutation and then the FFN, on its own batch and weight "
                                                  "copy; median of %d timed passes of exactly %d steps; "
                                                  "roofline: %s; e2e: groups of 16 steps, each step uploading "
                                                  "its x from pinned host memory and reading its y back on a "
                                                  "copy stream overlapped with the layer, captured as one graph "
                                                  "and replayed" % (args.passes, args.steps, ffn_how)}),
        "timing": _pass_summary(p_sere, steps_t),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": cap[0] if cap else None,
                     "traffic_launch_algorithmic_bytes": cap[1] if cap else None,
                     "traffic_source": ("ncu capture of the current kernel sources (%d active experts), %s"
                                        % (cap[2], os.path.relpath(FFN_PROFILE, ROOT))) if cap else
                                       "no ncu capture of the current kernel sources",
                     "kernel": "ffn_decode_kernel (moe_ffn_grouped: the tcgen05 FFN with the combine fused in, "
                               "y zeroed inside)",
                     "peak_source": peak_src,
                     "bytes_per_launch_mean": float(np.mean(ffn_bytes)),
                     "ms_per_launch_mean": float(np.mean(ffn_ms))},
        "active_experts": {"sere_mean": float(np.mean(us_sere)), "top8_mean": float(np.mean(us_top8))},
        "top8": {"value": job_throughput(ws, T, args.steps, t8_ms), "ms_per_step": t8_ms / args.steps,
                 "timing": _pass_summary(p_top8, args.steps),
                 "ffn_ms_mean": float(np.mean(t8_ffn_ms)),
                 "ffn_gbs": sum(t8_bytes) / (sum(t8_ffn_ms) / 1e3) / 1e9},
        "e2e": {"value": job_throughput(ws, T, args.steps, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 4, "timing": _pass_summary(p_e2e, args.steps)},
        "gpu_launches": launches_per_step * steps_t,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_legs(args.cpu_budget)
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# Further workloads (not the headline line): batch sweep, prefill, 48-layer stack
# ---------------------------------------------------------------------------
def run_sweep(args):
    """Decode batch sweep with 16 protected experts: top-8 and SERE K'=1, 2 at
    rho = 0.5, batch in --batches (default 1, 8, 32, 64, 128); per-layer time,
    union, FFN GB/s."""
    torch, moe, dev, ws, rank, local = _gpu_setup()
    from expert_routing_moe_gb300 import synthetic as syn
    peak, peak_src = load_peaks()
    stream = torch.cuda.Stream(device=dev)
    rows = []
    L0 = syn.sweep(32)
    copies = _device_copies(torch, dev, L0, N_COPIES, 1000 * syn.CONFIG_SWEEP + 10 * (rank + 1))
    clk = ClockSampler(local if ws > 1 else 0)
    clk.start()
    for B in args.batches:
        Lb0 = syn.sweep(B, with_weights=False)
        w_r = torch.from_numpy(Lb0.w_r).to(dev)
        sim = torch.from_numpy(Lb0.sim).to(dev)
        prot = torch.from_numpy(Lb0.protect).to(dev)
        xs = [torch.from_numpy(syn.sweep(B, with_weights=False, token_stream_offset=b).x_bf16)
              .view(torch.bfloat16).to(dev) for b in range(N_BATCHES)]
        for mode, kp in (("top8", 0), ("sere_k1", 1), ("sere_k2", 2)):
            layers = [moe.MoELayer(w_r, *copies[c], k=K_TOP, max_tokens=B, sim=sim, protect=prot,
                                   k_primary=max(kp, 1), rho=RHO) for c in range(N_COPIES)]
            sere = kp > 0
            us, _ = _active_counts(torch, moe, stream, layers, xs, sere)
            steps_g = _capture_steps(torch, stream, layers, xs, sere, group=STEP_GROUP)
            tot, n_t = _timed_steps(torch, stream, steps_g, args.steps, args.warmup, ws, group=STEP_GROUP)
            graphs = _capture(torch, stream, layers, xs, sere)
            _, ffn = _timed(torch, stream, graphs, args.steps, args.warmup, ws)
            byt = [us[i % N_BATCHES] * EXPERT_BYTES + B * H * 6 for i in range(args.steps)]
            gbs = sum(byt) / (sum(ffn) / 1e3) / 1e9
            rows.append({"batch": B, "mode": mode, "active_experts_mean": float(np.mean(us)),
                         "ms_per_layer": tot / n_t, "tokens_per_s": B * n_t / (tot / 1e3),
                         "ffn_us_mean": float(np.mean(ffn)) * 1e3, "ffn_gbs": gbs, "ffn_frac": gbs / peak})
            del graphs, steps_g, layers
    clocks = clk.stop()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle layer (SERE K'=2) on whole batches of each size, all host cores and one
        Lw = syn.sweep(32)
        cpu = {"kind": "oracle", "unit": "tokens/s", "rows": []}
        for B in args.batches:
            Lb = syn.sweep(B, with_weights=False)
            Lb.w_gate, Lb.w_up, Lb.w_down = Lw.w_gate, Lw.w_up, Lw.w_down
            row = {"batch": B}
            for key, nth in (("all_cores", 0), ("one_core", 1)):
                el, n, nt = oracle_timed([Lb], args.cpu_budget / 5, nth, True)
                row[key] = {"value": B * n / el, "cores": nt, "sample": "%d whole batch(es) in %.1f s" % (n, el)}
            cpu["rows"].append(row)
    if rank == 0:
        print(json.dumps({"workload": "decode batch sweep, 16 protected experts per layer, rho=0.5",
                          "metric": "MoE-layer decode tokens/s and FFN HBM GB/s", "peak_gbs": peak,
                          "peak_source": peak_src, "steps": args.steps, "warmup": args.warmup,
                          "l2": "%d weight copies and %d token batches rotated" % (N_COPIES, N_BATCHES),
                          "rows": rows, "clocks": clocks, "cpu_baseline": cpu}), flush=True)
    return 0


def run_prefill(args):
    """Capacity-mode prefill layer: T=8192 (70% visual tokens with w~Beta(2,5)),
    R=10, gamma=1.25.  Tensor-bound: FFN TFLOP/s = 2*3*H*I*rows / FFN time."""
    torch, moe, dev, ws, rank, local = _gpu_setup()
    from expert_routing_moe_gb300 import synthetic as syn
    L = syn.prefill()
    t = lambda a, dt=None: (torch.from_numpy(a).view(dt) if dt else torch.from_numpy(a)).to(dev)
    lay = moe.MoELayer(t(L.w_r), t(L.w_gate, torch.bfloat16), t(L.w_up, torch.bfloat16),
                       t(L.w_down, torch.bfloat16), k=L.k, max_tokens=L.T, R=L.R, capacity_factor=L.gamma)
    x = t(L.x_bf16, torch.bfloat16)
    tw = t(L.token_w)
    stream = torch.cuda.Stream(device=dev)
    us, rows = _active_counts(torch, moe, stream, [lay], [x], False, token_w=tw)
    steps_g = _capture_steps(torch, stream, [lay], [x], False, token_w=tw)
    graphs = _capture(torch, stream, [lay], [x], False, token_w=tw)
    clk = ClockSampler(local if ws > 1 else 0)
    clk.start()
    steps = max(3, args.steps // 20)
    tot, _ = _timed_steps(torch, stream, steps_g, steps, args.warmup, ws)
    _, ffn = _timed(torch, stream, graphs, steps, args.warmup, ws)
    clocks = clk.stop()
    tf = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))["bf16_tflops"] \
        if os.path.exists(os.path.join(ROOT, "MEASURED_PEAKS.json")) else 1900.0
    # MACS: entropy weights computed in the step, per-expert capacity from a modality grouping
    vis = t(L.is_visual.astype(np.uint8))
    ent = torch.empty(L.T, dtype=torch.float32, device=dev)
    w_ent = torch.empty(L.T, dtype=torch.float32, device=dev)
    rv = torch.empty(1, dtype=torch.float32, device=dev)
    from expert_routing_moe_gb300 import _abi as abi
    ws_tw = torch.empty(max(abi.workspace_size(abi.MOE_OP_TOKEN_WEIGHTS, L.T, 1, 1, 1, 1, 1, False, 0), 256),
                        dtype=torch.uint8, device=dev)
    lay_m = moe.MoELayer(lay.w_router, lay.w_gate, lay.w_up, lay.w_down, k=L.k, max_tokens=L.T, R=L.R,
                         capacity_factor=L.gamma, modality_bias=t(syn.modality_bias(N)), r_v=rv)

    def macs_step():
        moe.moe_token_weights(x, vis, ent, w_ent, rv, 1.0, 1e-6, lay_m.status, workspace=ws_tw)
        lay_m.forward(x, token_w=w_ent)

    with torch.cuda.stream(stream):
        macs_step()
        stream.synchronize()
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm, stream=stream):
            macs_step()
        gw = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gw, stream=stream):
            for _ in range(20):
                moe.moe_token_weights(x, vis, ent, w_ent, rv, 1.0, 1e-6, lay_m.status, workspace=ws_tw)
    code, detail = lay_m.device_status()
    if code != 0:
        raise RuntimeError("device status %d detail %d (MACS step)" % (code, detail))
    rows_m = int(lay_m.offsets[lay_m.N].item())
    t_m, _ = _timed_steps(torch, stream, [gm], steps, args.warmup, ws)
    t_w = _timed_steps(torch, stream, [gw], steps, args.warmup, ws)[0] / 20
    macs = {"ms_per_layer": t_m / steps, "tokens_per_s": L.T * steps / (t_m / 1e3), "rows_admitted": rows_m,
            "r_v": float(rv.item()), "token_weights_us": t_w / steps * 1e3,
            "token_weights_gbs": L.T * H * 2 / (t_w / steps / 1e3) / 1e9,
            "modality_groups": "seeded: 32 visual, 32 text, 64 shared experts"}
    flops = 2.0 * 3 * H * I * rows[0]
    ffn_s = float(np.mean(ffn)) / 1e3
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle layer: router, ranking, capacity and permutation over all 8192 tokens,
        # FFN + combine on a 256-token sample, scaled to the whole batch
        cpu = {"kind": "oracle", "unit": "tokens/s"}
        smp = np.sort(np.random.default_rng(5).choice(L.T, 256, replace=False)).astype(np.int32)
        for key, nth in (("all_cores", 0), ("one_core", 1)):
            el_r, _, nt = oracle_timed([L], 0.0, nth, False, capacity=True, tokens=np.arange(0, dtype=np.int32))
            el_f, _, _ = oracle_timed([L], 0.0, nth, False, capacity=True, tokens=smp)
            est = el_r + (el_f - el_r) * L.T / len(smp)
            cpu[key] = {"value": L.T / est, "cores": nt,
                        "sample": "routing + capacity over all %d tokens %.2f s; FFN on %d tokens %.2f s, "
                                  "scaled to all tokens (extrapolated): %.1f s per layer"
                                  % (L.T, el_r, len(smp), el_f - el_r, est)}
    if rank == 0:
        print(json.dumps({"workload": "capacity-mode prefill layer: 8192 tokens (70%% visual, w~Beta(2,5)), "
                                      "hidden 2048, 128 experts, top-8, R=10, gamma=1.25, intermediate 768",
                          "metric": "prefill layer tokens/s and FFN tensor TFLOP/s",
                          "tokens_per_s": L.T * steps / (tot / 1e3), "ms_per_layer": tot / steps,
                          "ffn_ms": ffn_s * 1e3, "rows_admitted": rows[0], "active_experts": us[0],
                          "ffn_tflops": flops / ffn_s / 1e12, "peak_tflops": tf,
                          "ffn_frac": flops / ffn_s / 1e12 / tf, "steps": steps, "clocks": clocks,
                          "macs_entropy_weights_and_expert_capacity": macs, "cpu_baseline": cpu}), flush=True)
    return 0


def run_calibrate(args):
    """SERE similarity calibration: every expert's output on n = 64 synthetic
    calibration tokens, then the normalised Gram matrix (offline step)."""
    torch, moe, dev, ws, rank, local = _gpu_setup()
    from expert_routing_moe_gb300 import synthetic as syn
    from expert_routing_moe_gb300 import _abi as abi
    L = syn.decode(32)
    n = 64
    t = lambda a, dt=None: (torch.from_numpy(a).view(dt) if dt else torch.from_numpy(a)).to(dev)
    wg, wu, wd = t(L.w_gate, torch.bfloat16), t(L.w_up, torch.bfloat16), t(L.w_down, torch.bfloat16)
    x = t(syn.f32_to_bf16_bits(np.random.default_rng(1000 * syn.CONFIG_DECODE + 7).standard_normal((n, H))
                               .astype(np.float32)), torch.bfloat16)
    wsz = abi.workspace_size(abi.MOE_OP_CALIBRATE, n, H, I, N, 1, 1, False, abi.MOE_DTYPE_BF16)
    work = torch.empty(wsz, dtype=torch.uint8, device=dev)
    sim = torch.empty(N, N, dtype=torch.float32, device=dev)
    st = torch.zeros(2, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        moe.moe_similarity_calibrate(x, wg, wu, wd, sim, work, st)
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            moe.moe_similarity_calibrate(x, wg, wu, wd, sim, work, st)
    if int(st[0].item()) != 0:
        raise RuntimeError("device status %s" % st.tolist())
    steps = max(3, args.steps // 20)
    tot, _ = _timed_steps(torch, stream, [g], steps, args.warmup, ws)
    ms = tot / steps
    gram_flops = 2.0 * N * N * n * H
    ffn_flops = 2.0 * 3 * H * I * n * N
    s_h = sim.cpu().numpy()
    off = s_h[~np.eye(N, dtype=bool)]
    if rank == 0:
        print(json.dumps({"workload": "SERE similarity calibration: 128 experts (hidden 2048, intermediate 768, bf16) "
                                      "on 64 synthetic N(0,1) calibration tokens",
                          "metric": "calibration time", "ms": ms, "steps": steps,
                          "expert_weight_gbs": N * EXPERT_BYTES / (ms / 1e3) / 1e9,
                          "tflops_total": (gram_flops + ffn_flops) / (ms / 1e3) / 1e12,
                          "sim_offdiag": {"min": float(off.min()), "max": float(off.max()),
                                          "mean": float(off.mean())}}), flush=True)
    return 0


def run_stack(args):
    """48 decode layers (batch 64), each with its own ~1.2 GB of experts, router,
    similarity and protection; x_{l+1} = x_l + y_l.  One CUDA graph per step.
    Modes: plain top-8, SERE K'=2 and K'=1 at rho = 0.5, and plain top-2 (the
    fixed top-K' baseline, same weights, for the latency and union comparison
    only)."""
    torch, moe, dev, ws, rank, local = _gpu_setup()
    from expert_routing_moe_gb300 import synthetic as syn
    nl, B = args.layers, syn.STACK_BATCH
    x0f, x0b = syn.stack_tokens(B, H)
    x0_f32 = torch.from_numpy(x0f).to(dev)
    x0_bf16 = torch.from_numpy(x0b).view(torch.bfloat16).to(dev)
    layers, layers_k1, layers_top2 = [], [], []
    for l in range(nl):
        gen = torch.Generator(device=dev)
        gen.manual_seed(syn.stack_weight_seed(l))
        w = [(torch.randn(shape, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
             for shape in ((N, I, H), (N, I, H), (N, H, I))]
        w_r = torch.from_numpy(syn.stack_router(x0f, l)).to(dev)
        sim = torch.from_numpy(syn.stack_sim(l)).to(dev)
        prot = torch.from_numpy(syn.stack_protect(l)).to(dev)
        layers.append(moe.MoELayer(w_r, *w, k=K_TOP, max_tokens=B, sim=sim, protect=prot, k_primary=K_PRIMARY,
                                   rho=RHO))
        layers_k1.append(moe.MoELayer(w_r, *w, k=K_TOP, max_tokens=B, sim=sim, protect=prot, k_primary=1, rho=RHO))
        layers_top2.append(moe.MoELayer(w_r, *w, k=2, max_tokens=B))
    xres = torch.empty(B, H, dtype=torch.float32, device=dev)
    xb = torch.empty(B, H, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(stack, sere):
        xres.copy_(x0_f32)
        xb.copy_(x0_bf16)
        for lay in stack:
            lay.forward(xb, sere=sere, accumulate_into=xres)
            moe.moe_residual_to_bf16(xres, xb)

    res = {}
    for mode, stack, sere in (("top8", layers, False), ("sere_k2", layers, True), ("sere_k1", layers_k1, True),
                              ("top2", layers_top2, False)):
        step_fn = lambda: step(stack, sere)
        with torch.cuda.stream(stream):
            step_fn()
        stream.synchronize()
        us = [int(l.active[0].item()) for l in stack]
        for l in stack:
            code, detail = l.device_status()
            if code != 0:
                raise RuntimeError("device status %d detail %d" % (code, detail))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            step_fn()
            stream.synchronize()
            with torch.cuda.graph(g, stream=stream):
                step_fn()
            for _ in range(args.warmup):
                g.replay()
        torch.cuda.synchronize()
        clk = ClockSampler(local if ws > 1 else 0)
        clk.start()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        steps = max(3, args.steps // 50)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(steps):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        clocks = clk.stop()
        ms = e0.elapsed_time(e1) / steps
        byt = sum(us) * EXPERT_BYTES
        res[mode] = {"ms_per_step": ms, "tokens_per_s": B / (ms / 1e3), "active_experts_per_layer": us,
                     "active_experts_mean": float(np.mean(us)), "expert_gbs": byt / (ms / 1e3) / 1e9,
                     "steps": steps, "clocks": clocks}
        del g
    peak, peak_src = load_peaks()
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle on 4 sampled layers of the step (SERE K'=2, batch 64; one host weight
        # set, as the oracle's time does not depend on the values), scaled to all layers
        import oracle
        Lw = syn.decode(B)
        Ls = []
        for l in range(4):
            Ll = syn.decode(B, layer=l, with_weights=False)
            Ll.w_gate, Ll.w_up, Ll.w_down = Lw.w_gate, Lw.w_up, Lw.w_down
            Ll.sim, Ll.protect = syn.stack_sim(l), syn.stack_protect(l)
            Ls.append(Ll)
        cpu = {"kind": "oracle", "unit": "tokens/s"}
        for key, nth in (("all_cores", 0), ("one_core", 1)):
            nt = oracle.set_threads(nth)
            t0 = time.perf_counter()
            for Ll in Ls:
                oracle.layer(Ll, sere_on=True)
            el = time.perf_counter() - t0
            per_step = el / len(Ls) * nl
            cpu[key] = {"value": B / per_step, "cores": nt,
                        "sample": "%d sampled layers in %.1f s, scaled to %d layers (extrapolated): %.1f s per step"
                                  % (len(Ls), el, nl, per_step)}
    if rank == 0:
        print(json.dumps({"workload": "decode step over %d MoE layers, batch %d, hidden 2048, 128 experts, top-8, "
                                      "intermediate 768, %.1f GB of bf16 experts resident; SERE K'=2 and K'=1 at "
                                      "rho=0.5 with per-layer similarity and 16 protected experts, plain top-8, "
                                      "plain top-2" % (nl, B, nl * N * EXPERT_BYTES / 1e9),
                          "metric": "decode step tokens/s (one CUDA graph per step)", "peak_gbs": peak,
                          "peak_source": peak_src, "residual": "x_{l+1} = x_l + y_l in fp32 (the FFN accumulates into it), rounded to bf16 per layer by moe_residual_to_bf16",
                          "cpu_baseline": cpu, **res}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=8.0,
                    help="seconds of oracle time for each cpu_baseline leg (all cores, one core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=4, help="expert-weight copies rotated per step")
    ap.add_argument("--clock-soak", type=float, default=1.5, help="seconds of untimed load while sampling clocks")
    ap.add_argument("--workload", choices=["decode", "sweep", "prefill", "stack", "calibrate"], default="decode",
                    help="decode (the headline line) or one of the further workloads")
    ap.add_argument("--layers", type=int, default=48, help="layers of the stack workload")
    ap.add_argument("--passes", type=int, default=5, help="timed passes of --steps steps (median reported)")
    ap.add_argument("--batches", type=lambda v: [int(b) for b in v.split(",")], default=[1, 8, 32, 64, 128],
                    help="comma-separated decode batches of the sweep workload (each 1..128)")
    args = ap.parse_args()
    global N_COPIES
    N_COPIES = max(1, args.copies)
    if args.warmup < 3:
        args.warmup = 3
    if args.steps < 1 or args.passes < 1:
        ap.error("--steps and --passes must be positive")
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "sweep":
        return run_sweep(args)
    if args.workload == "prefill":
        return run_prefill(args)
    if args.workload == "stack":
        return run_stack(args)
    if args.workload == "calibrate":
        return run_calibrate(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
