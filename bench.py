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
METRIC = "MoE-layer decode tokens/s (SERE K'=2, rho=0.5; top-8 alongside)"
UNIT = "tokens/s"
EXPERT_BYTES = 3 * H * I * 2


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
def oracle_sample(budget_s: float, max_batches: int = 64):
    """Times the oracle layer (router -> rank -> SERE -> permute -> FFN) on
    whole decode batches of the workload until `budget_s` is used."""
    import oracle
    from expert_routing_moe_gb300 import synthetic as syn
    L = syn.decode(T)
    L.k_primary, L.rho = K_PRIMARY, RHO
    oracle.layer(L, sere_on=True, tokens=np.arange(1))  # load + warm the library
    toks, t0, nb = 0, time.perf_counter(), 0
    while nb < max_batches:
        Lb = syn.decode(T, with_weights=False, token_stream_offset=nb)
        Lb.w_gate, Lb.w_up, Lb.w_down = L.w_gate, L.w_up, L.w_down
        oracle.layer(Lb, sere_on=True)
        toks += T
        nb += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    el = time.perf_counter() - t0
    return toks / el, el, nb


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from expert_routing_moe_gb300 import synthetic as syn
    oracle.build()
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
              "%d token(s) of it" % (T, ntok))
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": workload_config(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import expert_routing_moe_gb300 as moe
    from expert_routing_moe_gb300 import synthetic as syn

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

    # ---- inputs: one host-generated copy of the layer + device-generated copies ----
    L = syn.decode(T)
    w_r = torch.from_numpy(L.w_r).to(dev)
    sim = torch.from_numpy(L.sim).to(dev)
    copies = [tuple(torch.from_numpy(a).view(torch.bfloat16).to(dev) for a in (L.w_gate, L.w_up, L.w_down))]
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 * syn.CONFIG_DECODE + 10 * (rank + 1))
    for c in range(1, N_COPIES):
        copies.append(tuple((torch.randn(shape, generator=gen, device=dev) * 0.02).to(torch.bfloat16)
                            for shape in ((N, I, H), (N, I, H), (N, H, I))))
    xs = []
    for bidx in range(N_BATCHES):
        Lb = syn.decode(T, with_weights=False, token_stream_offset=bidx + 97 * rank)
        xs.append(torch.from_numpy(Lb.x_bf16).view(torch.bfloat16).to(dev))
    layers = [moe.MoELayer(w_r, *copies[c], k=K_TOP, max_tokens=T, sim=sim, k_primary=K_PRIMARY, rho=RHO)
              for c in range(N_COPIES)]
    stream = torch.cuda.Stream(device=dev)

    # ---- capture each (batch, copy) step as two graphs: routing+dispatch, FFN ----
    def capture(sere):
        graphs = []
        with torch.cuda.stream(stream):
            for bidx in range(N_BATCHES):
                lay = layers[bidx % N_COPIES]
                x = xs[bidx]
                for _ in range(2):  # eager warm-up on the capture stream
                    lay.forward(x, sere=sere)
                stream.synchronize()
                g1, g2 = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
                with torch.cuda.graph(g1, stream=stream):
                    lay.route(x, sere)
                    lay.dispatch(T)
                with torch.cuda.graph(g2, stream=stream):
                    lay.ffn(x)
                graphs.append((g1, g2))
        torch.cuda.synchronize()
        return graphs

    def active_counts(sere):
        us = []
        for bidx in range(N_BATCHES):
            lay = layers[bidx % N_COPIES]
            with torch.cuda.stream(stream):
                lay.forward(xs[bidx], sere=sere)
            stream.synchronize()
            code, detail = lay.device_status()
            if code != 0:
                raise RuntimeError("device status %d (%s) detail %d" % (code, moe.status_string(code, True),
                                                                          detail))
            us.append(int(lay.active[0].item()))
        return us

    def timed(graphs, us, steps, warmup):
        ev = lambda: torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for i in range(warmup):
                g1, g2 = graphs[i % N_BATCHES]
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
                g1, g2 = graphs[i % N_BATCHES]
                g1.replay()
                f0[i].record(stream)
                g2.replay()
                f1[i].record(stream)
            e1.record(stream)
        torch.cuda.synchronize()
        if ws > 1:
            torch.distributed.barrier()
        total_ms = e0.elapsed_time(e1)
        ffn_ms = [a.elapsed_time(b) for a, b in zip(f0, f1)]
        ffn_bytes = [us[i % N_BATCHES] * EXPERT_BYTES + T * H * 2 + T * H * 4 for i in range(steps)]
        return total_ms, ffn_ms, ffn_bytes

    def max_over_ranks(v):
        if ws == 1:
            return v
        t = torch.tensor([v], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        return float(t.item())

    us_sere = active_counts(True)
    us_top8 = active_counts(False)
    g_sere = capture(True)
    g_top8 = capture(False)
    launches_per_step = 4  # router, rank+SERE, permute, FFN tensor-core kernel (plus a memset node for y)

    clk = ClockSampler(local if ws > 1 else 0)
    clk.start()
    if args.clock_soak > 0:
        # untimed replays so that the clock record covers a loaded GPU, not just a few ms
        t_end = time.perf_counter() + args.clock_soak
        with torch.cuda.stream(stream):
            i = 0
            while time.perf_counter() < t_end:
                for _ in range(50):
                    g1, g2 = g_sere[i % N_BATCHES]
                    g1.replay()
                    g2.replay()
                    i += 1
                stream.synchronize()
    total_ms, ffn_ms, ffn_bytes = timed(g_sere, us_sere, args.steps, args.warmup)
    clocks = clk.stop()
    total_ms = max_over_ranks(total_ms)
    t8_ms, t8_ffn_ms, t8_bytes = timed(g_top8, us_top8, args.steps, args.warmup)
    t8_ms = max_over_ranks(t8_ms)

    # ---- end to end through the public API: pinned host x in, host y out, every step ----
    xs_host = [x.cpu().pin_memory() for x in xs]
    y_host = torch.empty(T, H, dtype=torch.float32).pin_memory()
    x_dev = [torch.empty_like(x) for x in xs]
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            lay = layers[i % N_COPIES]
            x_dev[i % N_BATCHES].copy_(xs_host[i % N_BATCHES], non_blocking=True)
            y = lay.forward(x_dev[i % N_BATCHES], sere=True)
            y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.steps):
            b_i = i % N_BATCHES
            lay = layers[b_i % N_COPIES]
            x_dev[b_i].copy_(xs_host[b_i], non_blocking=True)
            y = lay.forward(x_dev[b_i], sere=True)
            y_host.copy_(y, non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    for lay in layers:
        code, detail = lay.device_status()
        if code != 0:
            raise RuntimeError("device status %d detail %d after the timed runs" % (code, detail))

    peak, peak_src = load_peaks()
    ffn_s = sum(ffn_ms) / 1e3
    achieved = sum(ffn_bytes) / ffn_s / 1e9
    line = {
        "metric": METRIC, "value": ws * T * args.steps / (total_ms / 1e3), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded Dirichlet-skewed router logits, N(0,0.02) bf16 experts)",
        "config": workload_config({"parallelism": "replicas" if ws > 1 else "single GPU",
                                   "cuda_graphs": "per step: routing+dispatch graph, FFN graph"}),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "kernel": "moe_ffn_grouped (y clear + tcgen05 FFN kernel)",
                     "peak_source": peak_src,
                     "bytes_per_launch_mean": float(np.mean(ffn_bytes)),
                     "ms_per_launch_mean": float(np.mean(ffn_ms))},
        "active_experts": {"sere_mean": float(np.mean(us_sere)), "top8_mean": float(np.mean(us_top8))},
        "top8": {"value": ws * T * args.steps / (t8_ms / 1e3), "ms_per_step": t8_ms / args.steps,
                 "ffn_ms_mean": float(np.mean(t8_ffn_ms)),
                 "ffn_gbs": sum(t8_bytes) / (sum(t8_ffn_ms) / 1e3) / 1e9},
        "e2e": {"value": ws * T * args.steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 4},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
    }
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        v, el, nb = oracle_sample(args.cpu_budget)
        line["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle",
                                "sample": "%d whole decode batches of %d tokens through the oracle layer "
                                          "(router, rank, SERE, permute, FFN + combine) in %.1f s"
                                          % (nb, T, el)}
    elif rank == 0:
        line["cpu_baseline"] = None
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--copies", type=int, default=4, help="expert-weight copies rotated per step")
    ap.add_argument("--clock-soak", type=float, default=1.5, help="seconds of untimed load while sampling clocks")
    args = ap.parse_args()
    global N_COPIES
    N_COPIES = max(1, args.copies)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
