#!/usr/bin/env python
"""Benchmark of the MoE expert-cache layer step on GB300.

Default workload (one line of JSON on stdout): A3B-style decode, 48 MoE layers,
d=2048, E=128 routed experts, top-8, SwiGLU f=768, bf16 weights N(0, 0.02) in a
57.98 GB pinned host pool, batch 1, AR(1) hidden states (rho = 0.9), a shared
LRU cache of 1536 slots (25% of 48x128), BP/BH = 1, K_max = 128.  One step is
one decode token through all 48 layers: routing, cache control, fills from the
host pool, expert FFNs and merge, replayed as one CUDA graph per token.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload a3b_decode|tiny_decode|v4_decode|a3b_prefill|control_stress]

Under torchrun (N > 1) every rank runs an independent replica of the workload
on its own GPU (the path has no exchange step); rank 0 prints the line with
value = units of all ranks / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import ftsynth  # noqa: E402

WORKLOADS = {
    "a3b_decode": dict(L=48, E=128, k=8, d=2048, f=768, dtype=0, S=1536, K_max=128, T=1, rho=0.9, r=(1, 1),
                       steps=512,
                       desc="A3B-style decode: 48 layers, d=2048, E=128, top-8, f=768, bf16, batch 1, "
                            "S=1536 (25% of 6144), BP/BH=1, K_max=128, AR(1) rho=0.9"),
    "tiny_decode": dict(L=1, E=16, k=2, d=256, f=128, dtype=0, S=8, K_max=16, T=1, rho=0.9, r=(1, 1), steps=32,
                        desc="tiny: 1 layer, d=256, E=16, top-2, f=128, S=8, BP/BH=1"),
}
L2_BYTES = 129 * 2 ** 20


# ----------------------------------------------------------------------------- helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def replica_reduce(elapsed_s: float, units: float, world_size: int):
    """Max of the elapsed time and sum of the units over ranks (replicas only:
    this is the only cross-rank communication)."""
    if world_size == 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return dict(hbm_gbs=float(d["hbm_gbs"]), bf16_tflops=float(d["bf16_tflops"]),
                    bf16_tflops_sustained=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="ftclk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200", "-f", self.path],
                                         stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as fh:
                for line in fh:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- decode workload

def decode_inputs(w, n_steps, seed=0):
    """AR(1) hidden [steps, L, T, d] bf16 and logits [steps, L, T, E] float32."""
    L, E, d, T = w["L"], w["E"], w["d"], w["T"]
    wr = ftsynth.router_weights(seed, L, E, d)
    hid = np.empty((n_steps, L, T, d), dtype=np.uint16)
    for l in range(L):
        for b in range(T):
            hid[:, l, b, :] = ftsynth.ar1_hidden(seed, l, b, n_steps, d, w["rho"])
    lg = np.stack([ftsynth.router_logits(hid[:, l], wr[l]) for l in range(L)], axis=1)
    return hid, np.ascontiguousarray(lg)


def run_ours_decode(args, w, world, rank, local, pool, hid, lg, t_gen):
    import torch

    import expert_cache_host_gb300 as ft
    from expert_cache_host_gb300 import build as ftbuild

    ftbuild.build()
    torch.cuda.set_device(local)
    L, E, k, d, f, T = w["L"], w["E"], w["k"], w["d"], w["f"], w["T"]
    bx = ftsynth.expert_bytes(d, f, w["dtype"])
    W, K = args.warmup, args.steps
    P = min(K, args.profile_steps)
    E2E = min(K, args.e2e_steps)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=w["dtype"],
                         num_slots=w["S"], k_max=w["K_max"], t_max=T, r_num=w["r"][0], r_den=w["r"][1])
    t0 = time.time()
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    t_init = time.time() - t0
    try:
        d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
        d_lg = torch.from_numpy(lg).cuda()
        cur_hid = torch.empty((L, T, d), dtype=torch.int16, device="cuda")
        cur_lg = torch.empty((L, T, E), dtype=torch.float32, device="cuda")
        out = torch.empty((L, T, d), dtype=torch.float32, device="cuda")
        stream = torch.cuda.Stream()
        h_hid = torch.from_numpy(hid.view(np.int16)).pin_memory()
        h_lg = torch.from_numpy(lg).pin_memory()
        h_out = torch.empty((L, T, d), dtype=torch.float32).pin_memory()

        def token(st):
            for l in range(L):
                ft.ft_cache_step(ctx, l, cur_lg[l].data_ptr(), T, st)
                ft.ft_moe_forward(ctx, l, ft.FT_DECODE_CACHED, 0, cur_hid[l].data_ptr(), T, 0, out[l].data_ptr(), st)

        with torch.cuda.stream(stream):
            st = stream.cuda_stream
            # one eager token (step 0) to set up kernel attributes, then capture
            cur_hid.copy_(d_hid[0])
            cur_lg.copy_(d_lg[0])
            token(st)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                token(torch.cuda.current_stream().cuda_stream)
            s = 1
            for _ in range(W - 1):
                cur_hid.copy_(d_hid[s]); cur_lg.copy_(d_lg[s]); graph.replay(); s += 1
            stream.synchronize()
            if world > 1:
                torch.distributed.barrier()
            c0 = ft.ft_get_counters(ctx, L)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with ClockSampler(local) as clk:
                stream.synchronize()
                ev0.record(stream)
                for _ in range(K):
                    cur_hid.copy_(d_hid[s]); cur_lg.copy_(d_lg[s]); graph.replay(); s += 1
                ev1.record(stream)
                ev1.synchronize()
            elapsed = ev0.elapsed_time(ev1) / 1e3
            if world > 1:
                torch.distributed.barrier()
            c1 = ft.ft_get_counters(ctx, L)
            clocks = clk.summary()

            # per-kernel durations: the same steps run eagerly with event timing
            ft.ft_profile_enable(ctx, True)
            ft.ft_profile_read(ctx, reset=True)
            cp0 = ft.ft_get_counters(ctx, L)
            for _ in range(P):
                cur_hid.copy_(d_hid[s]); cur_lg.copy_(d_lg[s]); token(st); s += 1
            prof = ft.ft_profile_read(ctx, reset=True)
            cp1 = ft.ft_get_counters(ctx, L)
            ft.ft_profile_enable(ctx, False)

            # end to end: pinned host inputs in, layer outputs back, per token
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            stream.synchronize()
            e0.record(stream)
            for _ in range(E2E):
                cur_hid.copy_(h_hid[s], non_blocking=True)
                cur_lg.copy_(h_lg[s], non_blocking=True)
                graph.replay()
                h_out.copy_(out, non_blocking=True)
                s += 1
            e1.record(stream)
            e1.synchronize()
            e2e_elapsed = e0.elapsed_time(e1) / 1e3
        status = ft.ft_get_status(ctx)
    finally:
        ft.ft_moe_destroy(ctx)

    dc = (c1 - c0).astype(np.float64)
    hits, misses, fills, cpu = dc[:, 0].sum(), dc[:, 1].sum(), dc[:, 2].sum(), dc[:, 3].sum()
    elapsed_max, units = replica_reduce(elapsed, K * T, world)
    value = units / elapsed_max
    peaks = measured_peaks()
    dp = (cp1 - cp0).astype(np.float64)
    groups_p = dp[:, 0].sum() + dp[:, 2].sum()
    fills_p = dp[:, 2].sum()
    tot_ms = sum(v[0] for v in prof.values())
    shares = {kname: (round(v[0] / tot_ms, 4) if tot_ms else 0.0) for kname, v in prof.items() if v[1]}
    ex_ms, ex_n = prof["experts"]
    fill_ms, fill_n = prof["fill"]
    ex_bytes = groups_p * bx  # algorithmic: each executed expert's weights read once
    ex_gbs = ex_bytes / (ex_ms / 1e3) / 1e9 if ex_ms else 0.0
    fill_gbs = fills_p * bx / (fill_ms / 1e3) / 1e9 if fill_ms else 0.0
    per_launch_bytes = ex_bytes / ex_n if ex_n else 0.0
    h2d = (lg[0].nbytes + hid[0].nbytes)
    d2h = L * T * d * 4
    line = {
        "metric": "MoE decode tok/s (A3B-style, batch 1, GPU side; CPU-routed experts arrive as a partial sum)",
        "value": round(value, 3),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(elapsed_max / K * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w["desc"], "graph": "one CUDA graph per token", "batch": T,
                   "l2": "inputs larger than L2: %.2f GB of expert weights read per token" % (L * k * bx / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "kernel": "decode experts", "achieved": round(ex_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ex_gbs / peaks["hbm_gbs"], 4),
                     "traffic": None, "peak_source": peaks["source"],
                     "bytes_per_launch": round(per_launch_bytes), "avg_launch_us": round(ex_ms / ex_n * 1e3, 2) if ex_n else None},
        "components": {
            "kernel_share": shares,
            "kernel_ms_per_token": {kname: round(v[0] / P, 4) for kname, v in prof.items() if v[1]},
            "fill_link_gbs": round(fill_gbs, 1),
            "control_us_per_layer_step": round(prof["control"][0] / max(1, prof["control"][1]) * 1e3, 3),
            "hit_rate": round(hits / max(1.0, hits + misses), 4),
            "fills_per_token": round(fills / K, 3),
            "cpu_routes_per_token": round(cpu / K, 3),
            "eager_ms_per_token_profiled": round(tot_ms / P, 4) if P else None,
            "setup_s": {"generate": round(t_gen, 1), "init_pin": round(t_init, 1)},
            "device_status": status,
        },
        "clocks": clocks,
        "e2e": {"value": round(E2E * T / e2e_elapsed, 3), "unit": "tok/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h)},
        "gpu_launches": int(K * L * (5 if w["dtype"] == 0 else 5)),
    }
    return line


# ----------------------------------------------------------------------------- oracle (CPU baseline / reference arm)

def oracle_decode_rate(w, pool, hid, lg, budget_s, min_tokens=1, max_tokens=None):
    """Time the oracle on the decode workload from a cold cache: whole tokens
    (routing, cache step and fp64 experts for every layer) until budget_s.
    Returns (tokens/s, tokens, seconds, threads used)."""
    import oracle
    L, E, k, d, f, T = w["L"], w["E"], w["k"], w["d"], w["f"], w["T"]
    bx = ftsynth.expert_bytes(d, f, w["dtype"])
    n_tok = min(hid.shape[0], max_tokens or hid.shape[0])
    cache = oracle.Cache(L * E, w["S"])
    done, t_spent = 0, 0.0
    for s in range(n_tok):
        t0 = time.time()
        for l in range(L):
            ids, wt = oracle.route(lg[s, l], k)
            ref = cache.step(l, E, ids, w["r"][0], w["r"][1], w["K_max"])
            oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, w["dtype"], d, f, ids, wt, hid[s, l],
                               slot_ids=ref.slot_ids.reshape(T, k))
        t_spent += time.time() - t0
        done += 1
        if done >= min_tokens and t_spent >= budget_s:
            break
    # the expert evaluations of one layer run in parallel over its T*k routes
    threads = min(oracle.threads(), T * k)
    return done * T / t_spent, done, t_spent, threads


def run_reference(args, w):
    """The oracle as the reference arm: same metric and unit, CPU cores."""
    budget = args.ref_budget_s
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02)
    hid, lg = decode_inputs(w, max(2, min(args.steps, 64)))
    rate, n, t, threads = oracle_decode_rate(w, pool, hid, lg, budget, min_tokens=max(1, min(args.steps, 2)),
                                              max_tokens=max(1, args.steps))
    sample = f"{n} decode tokens x {w['L']} layers from a cold cache ({t:.1f} s of oracle work)"
    return {
        "impl": "reference",
        "metric": "MoE decode tok/s (A3B-style, batch 1, GPU side; CPU-routed experts arrive as a partial sum)",
        "value": round(rate, 5), "unit": "tok/s", "n_gpus": 1, "steps": n, "warmup": 0,
        "ms_per_step": round(t / max(1, n) * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w["desc"]},
        "cpu_baseline": {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(rate, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- main

def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=448)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="a3b_decode")
    ap.add_argument("--profile-steps", type=int, default=32)
    ap.add_argument("--e2e-steps", type=int, default=128)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=0, help="override L (small profiling cases, not a bench line)")
    ap.add_argument("--slots", type=int, default=0, help="override S (small profiling cases, not a bench line)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    w = dict(WORKLOADS[args.workload])
    if args.layers or args.slots:
        w["L"] = args.layers or w["L"]
        w["S"] = args.slots or w["S"]
        w["desc"] = w["desc"] + f" [profiling case: L={w['L']}, S={w['S']}]"

    if world > 1:
        import torch
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args, w)), flush=True)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    t0 = time.time()
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02)
    hid, lg = decode_inputs(w, args.warmup + args.steps + min(args.steps, args.profile_steps)
                            + min(args.steps, args.e2e_steps))
    t_gen = time.time() - t0
    line = run_ours_decode(args, w, world, rank, local, pool, hid, lg, t_gen)
    if rank == 0 and not args.no_cpu_baseline:
        rate, n, t, threads = oracle_decode_rate(w, pool, hid, lg, args.cpu_budget_s)
        line["cpu_baseline"] = {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} decode tokens x {w['L']} layers from a cold cache, "
                                          f"{t:.1f} s of oracle work"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
