#!/usr/bin/env python
"""Benchmark of the MoE expert-cache layer step on GB300.

One JSON line on stdout.  The headline (value) is A3B-style decode: 48 MoE
layers, d=2048, E=128 routed experts, top-8, SwiGLU f=768, bf16 weights
N(0, 0.02) in a 57.98 GB pinned host pool, batch 1, AR(1) hidden states
(rho = 0.9), a shared LRU cache of 1536 slots (25% of 48x128), BP/BH = 1,
K_max = 128.  One step is one decode token through all 48 layers -- routing,
cache control, fills from the host pool, expert FFNs and merge -- replayed as
one CUDA graph per token.  The same run adds, as components, the 8192-token
prefill chunk of the same model (full-layer double buffer on and off, grouped
GEMM throughput with weights resident) and the cache-control stress workload
(48 layers x 64 tokens x top-8, 6144 slots, Zipf routes).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the decode
workload on its own GPU (the path has no exchange step); rank 0 prints the
line with value = tokens of all ranks / the slowest rank's time.
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

METRIC = "MoE decode tok/s (A3B-style, batch 1, GPU side; CPU-routed experts arrive as a partial sum)"
V4 = dict(L=43, E=256, k=6, d=4096, f=2048, dtype=1, S=2393, K_max=256, T=1, rho=0.9, r=(1, 1),
          desc="V4-Flash-style decode: 43 layers, d=4096, E=256, top-6, f=2048, MXFP4 experts (147 GB pool), "
               "S=2393 (32 GB budget), BP/BH=1, K_max=256, AR(1) rho=0.9")
A3B = dict(L=48, E=128, k=8, d=2048, f=768, dtype=0, S=1536, K_max=128, T=1, rho=0.9, r=(1, 1),
           desc="A3B-style decode: 48 layers, d=2048, E=128, top-8, f=768, bf16, batch 1, "
                "S=1536 (25% of 6144), BP/BH=1, K_max=128, AR(1) rho=0.9")
L2_BYTES = 129 * 2 ** 20

# DRAM bytes per launch from ncu captures (profiles/); None once the kernel changed.
# dram__bytes_read + dram__bytes_write / algorithmic bytes of the decode expert
# kernels over the launches captured with ncu (--set full): three A3B bf16
# launches (6 + 2 + 5 experts) and two V4 MXFP4 launches (4 + 2 experts); the
# traffic reported per launch is this ratio times the launch's algorithmic bytes
NCU_TRAFFIC_RATIO = {
    "decode_experts": 123_111_424 / 122_683_392,
    "decode_experts_mxfp4": 80_432_896 / 80_216_064,
}


# ----------------------------------------------------------------------------- helpers

def dist_env():
    return int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0"))


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
        self.gpu, self.proc, self.path = gpu_index, None, None

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
                rows = [p for p in ([x.strip() for x in line.split(",")] for line in fh) if len(p) >= 9]
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        num = lambda s: s.replace(".", "", 1).isdigit()
        sm = [float(r[1]) for r in rows if num(r[1])]
        mx = [float(r[2]) for r in rows if num(r[2])]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


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


def timed(stream, fn, reps=1):
    import torch
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    stream.synchronize()
    e0.record(stream)
    for _ in range(reps):
        fn()
    e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1) / 1e3


def link_peak_gbs(pool, nbytes):
    """Best of three host->device copies of `nbytes` of the pinned pool (copy engine)."""
    import torch
    src = torch.from_numpy(pool[:nbytes])
    dst = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream()
    best = min(timed(s, lambda: dst.copy_(src, non_blocking=True)) for _ in range(3))
    del dst
    return nbytes / best / 1e9


def experts_alone(w, pool, hid, reps=40):
    """The bf16 decode expert kernel with its merge, outside the step: the
    first k experts of layer 0 resident in a scratch arena, one token, L2
    flushed (256 MB written) before every call, CUDA events around the call
    (route grouping + experts + merge of the allocation-free entry).  Returns
    {experts: median seconds} for k and for 2 experts."""
    import torch

    import expert_cache_host_gb300 as ft
    d, f, k = w["d"], w["f"], w["k"]
    bx = ftsynth.expert_bytes(d, f, 0)
    arena = torch.from_numpy(pool[:k * bx]).cuda()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    x = torch.from_numpy(hid[0, 0, :1].view(np.int16)).cuda()
    out = torch.empty((1, d), dtype=torch.float32, device="cuda")
    st = torch.cuda.current_stream()
    res = {}
    for n in (k, 2):
        sid = torch.arange(n, dtype=torch.int32, device="cuda")
        wt = torch.full((n,), 1.0 / n, dtype=torch.float32, device="cuda")
        ts = []
        for r in range(reps + 3):
            flush.add_(1)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            ft.ft_decode_experts_noalloc(arena.data_ptr(), k, d, f, n, 1, sid.data_ptr(), wt.data_ptr(), x.data_ptr(),
                                         0, out.data_ptr(), 0, st.cuda_stream)
            e1.record(st)
            e1.synchronize()
            if r >= 3:
                ts.append(e0.elapsed_time(e1) / 1e3)
        res[n] = statistics.median(ts)
    del arena, flush
    return res


# ----------------------------------------------------------------------------- decode (headline)

def run_decode_leg(args, w, world, local, pool, hid, lg):
    import torch

    import expert_cache_host_gb300 as ft

    L, E, k, d, f, T = w["L"], w["E"], w["k"], w["d"], w["f"], w["T"]
    bx = ftsynth.expert_bytes(d, f, w["dtype"])
    W, K = args.warmup, args.steps
    P, E2E = min(K, args.profile_steps), min(K, args.e2e_steps)
    cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, dtype=w["dtype"],
                         num_slots=w["S"], k_max=w["K_max"], t_max=T, r_num=w["r"][0], r_den=w["r"][1])
    t0 = time.time()
    ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
    t_init = time.time() - t0
    try:
        if args.cpu_exec:
            ft.ft_cpu_executor(ctx, args.cpu_exec)
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
            cur_hid.copy_(d_hid[0])
            cur_lg.copy_(d_lg[0])
            token(st)  # one eager token (step 0): kernel attributes are set outside the capture
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                token(torch.cuda.current_stream().cuda_stream)
            s = 1

            def step():
                nonlocal s
                cur_hid.copy_(d_hid[s])
                cur_lg.copy_(d_lg[s])
                graph.replay()
                s += 1

            for _ in range(W - 1):
                step()
            stream.synchronize()
            if world > 1:
                torch.distributed.barrier()
            c0 = ft.ft_get_counters(ctx, L)
            with ClockSampler(local) as clk:
                elapsed = timed(stream, step, K)
            if world > 1:
                torch.distributed.barrier()
            c1 = ft.ft_get_counters(ctx, L)
            clocks = clk.summary()

            # per-kernel durations: the following steps run eagerly with event timing
            ft.ft_profile_enable(ctx, True)
            ft.ft_profile_read(ctx, reset=True)
            cp0 = ft.ft_get_counters(ctx, L)
            for _ in range(P):
                cur_hid.copy_(d_hid[s])
                cur_lg.copy_(d_lg[s])
                token(st)
                s += 1
            prof = ft.ft_profile_read(ctx, reset=True)
            cp1 = ft.ft_get_counters(ctx, L)
            ft.ft_profile_enable(ctx, False)

            # end to end: pinned host inputs in, every layer's output back, per token
            def e2e_step():
                nonlocal s
                cur_hid.copy_(h_hid[s], non_blocking=True)
                cur_lg.copy_(h_lg[s], non_blocking=True)
                graph.replay()
                h_out.copy_(out, non_blocking=True)
                s += 1

            e2e_elapsed = timed(stream, e2e_step, E2E)
        status = ft.ft_get_status(ctx)
    finally:
        ft.ft_moe_destroy(ctx)

    dc = (c1 - c0).astype(np.float64)
    hits, misses, fills, cpu = (dc[:, i].sum() for i in range(4))
    elapsed_max, units = replica_reduce(elapsed, K * T, world)
    dp = (cp1 - cp0).astype(np.float64)
    groups_p, fills_p = dp[:, 0].sum() + dp[:, 2].sum(), dp[:, 2].sum()
    tot_ms = sum(v[0] for v in prof.values())
    ex_ms, ex_n = prof["experts"]
    fill_ms, fill_n = prof["fill"]
    return dict(
        value=units / elapsed_max, elapsed=elapsed_max, K=K, W=W, T=T, clocks=clocks, status=status,
        t_init=t_init, hits=hits, misses=misses, fills=fills, cpu=cpu, P=P,
        shares={n: round(v[0] / tot_ms, 4) for n, v in prof.items() if v[1]},
        ms_per_token={n: round(v[0] / P, 4) for n, v in prof.items() if v[1]},
        launches={n: v[1] for n, v in prof.items() if v[1]},
        ex_bytes=groups_p * bx, ex_ms=ex_ms, ex_n=ex_n, fill_bytes=fills_p * bx, fill_ms=fill_ms, fill_n=fill_n,
        control_us=prof["control"][0] / max(1, prof["control"][1]) * 1e3,
        route_us=prof["route"][0] / max(1, prof["route"][1]) * 1e3,
        eager_ms=tot_ms / P if P else None,
        e2e=E2E * T / e2e_elapsed, h2d=int(lg[0].nbytes + hid[0].nbytes), d2h=int(L * T * d * 4),
    )


# ----------------------------------------------------------------------------- prefill chunk

def run_prefill_leg(args, w, pool):
    import torch

    import expert_cache_host_gb300 as ft

    L = args.prefill_layers or w["L"]
    E, k, d, f, T = w["E"], w["k"], w["d"], w["f"], args.prefill_tokens
    bx = ftsynth.expert_bytes(d, f, 0)
    wr = ftsynth.router_weights(0, L, E, d)
    hid = np.stack([ftsynth.prefill_hidden(0, l, T, d) for l in range(L)])
    lg = np.stack([ftsynth.router_logits(hid[l], wr[l]) for l in range(L)])
    d_hid = torch.from_numpy(hid.view(np.int16)).cuda()
    d_lg = torch.from_numpy(lg).cuda()
    del hid, lg
    out = torch.empty((T, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()
    res = {}
    for buffers in (2, 1):
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=1, k_max=1, t_max=1,
                             prefill_buffers=buffers, prefill_t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            with torch.cuda.stream(stream):
                st = stream.cuda_stream

                def chunk():
                    for l in range(L):
                        ft.ft_moe_forward(ctx, l, ft.FT_PREFILL_LAYER, d_lg[l].data_ptr(), d_hid[l].data_ptr(), T, 0,
                                          out.data_ptr(), st)

                chunk()  # warm-up chunk (each chunk re-uploads the whole pool: layer 0 is not resident)
                times = [timed(stream, chunk) for _ in range(2)]
                res[buffers] = min(times)
                if buffers == 2:
                    # upload rate and grouped-GEMM throughput, weights resident (layer 0 twice in a row)
                    ft.ft_profile_enable(ctx, True)
                    ft.ft_profile_read(ctx, reset=True)
                    chunk()
                    prof_chunk = ft.ft_profile_read(ctx, reset=True)
                    for _ in range(3):
                        ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lg[0].data_ptr(), d_hid[0].data_ptr(), T, 0,
                                          out.data_ptr(), st)
                    ft.ft_moe_forward(ctx, 0, ft.FT_PREFILL_LAYER, d_lg[0].data_ptr(), d_hid[0].data_ptr(), T, 0,
                                      out.data_ptr(), st)
                    prof_res = ft.ft_profile_read(ctx, reset=True)
                    ft.ft_profile_enable(ctx, False)
            status = ft.ft_get_status(ctx)
        finally:
            ft.ft_moe_destroy(ctx)
    pool_bytes = L * E * bx
    up_ms, up_n = prof_chunk["upload"]
    gemm_ms, gemm_n = prof_res["gemm"]
    flops_layer = T * k * 3 * d * f * 2  # 3 matrices of d*f MACs per (token, expert), 2 flops per MAC
    gemm_tflops = flops_layer / (gemm_ms / gemm_n / 1e3) / 1e12 if gemm_n else 0.0
    upload_gbs = up_n * E * bx / (up_ms / 1e3) / 1e9 if up_n else 0.0
    return dict(L=L, T=T, chunk_s=res[2], chunk_s_single_buffer=res[1], pool_bytes=pool_bytes,
                link_gbs=pool_bytes / res[2] / 1e9, upload_gbs=upload_gbs, gemm_tflops=gemm_tflops,
                gemm_ms_per_layer=gemm_ms / max(1, gemm_n), status=status,
                overlap_loss_without_double_buffer=1.0 - res[2] / res[1])


# ----------------------------------------------------------------------------- control stress

def run_control_leg(args):
    import torch

    import expert_cache_host_gb300 as ft

    L, E, k, T, steps = 48, 128, 8, 64, args.control_steps
    d, f = 256, 128  # the control kernel never reads expert bytes: smallest legal expert shape
    pool = np.zeros(L * E * ftsynth.expert_bytes(d, f, 0), dtype=np.uint8)
    stream = torch.cuda.Stream()
    cases = [(6144, km, s) for s in (0.6, 1.2) for km in (8, 64, 128, 512)] + \
            [(S, 128, s) for S in (1536, 512) for s in (0.6, 1.2)]
    routes = {}
    for s in (0.6, 1.2):
        r = np.stack([ftsynth.zipf_routes(0, l, E, T, k, s, 0, steps) for l in range(L)], axis=1)
        routes[s] = torch.from_numpy(r).cuda()  # [steps, L, T, k]
    out = []
    for S, km, s in cases:
        cfg = ft.make_config(num_layers=L, num_experts=E, top_k=k, hidden=d, inter=f, num_slots=S, k_max=km, t_max=T)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            cur = torch.empty((L, T, k), dtype=torch.int32, device="cuda")
            with torch.cuda.stream(stream):
                cur.copy_(routes[s][0])
                for l in range(L):
                    ft.ft_cache_control(ctx, l, cur[l].data_ptr(), T, stream.cuda_stream)
                stream.synchronize()
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    for l in range(L):
                        ft.ft_cache_control(ctx, l, cur[l].data_ptr(), T, torch.cuda.current_stream().cuda_stream)
                i = 1

                def step():
                    nonlocal i
                    cur.copy_(routes[s][i])
                    g.replay()
                    i += 1

                warm = min(100, steps // 4)
                for _ in range(warm):
                    step()
                c0 = ft.ft_get_counters(ctx, L)
                el = timed(stream, step, steps - 1 - warm)
                c1 = ft.ft_get_counters(ctx, L)
            dc = (c1 - c0).astype(np.float64)
            n_ls = (steps - 1 - warm) * L
            out.append(dict(S=S, K_max=km, zipf_s=s, us_per_layer_step=round(el / n_ls * 1e6, 3),
                            miss_rate=round(dc[:, 1].sum() / max(1.0, dc[:, 0].sum() + dc[:, 1].sum()), 4),
                            fills_per_layer_step=round(dc[:, 2].sum() / n_ls, 3), status=ft.ft_get_status(ctx)))
        finally:
            ft.ft_moe_destroy(ctx)
    return out


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
    layer_steps, t_spent = 0, 0.0
    for s in range(n_tok):
        for l in range(L):
            t0 = time.time()
            ids, wt = oracle.route(lg[s, l], k)
            ref = cache.step(l, E, ids, w["r"][0], w["r"][1], w["K_max"])
            oracle.moe_forward(pool[l * E * bx:(l + 1) * E * bx], bx, w["dtype"], d, f, ids, wt, hid[s, l],
                               slot_ids=ref.slot_ids.reshape(T, k))
            t_spent += time.time() - t0
            layer_steps += 1
            if layer_steps >= min_tokens * L and t_spent >= budget_s:
                break
        else:
            continue
        break
    # the expert evaluations of one layer run in parallel over its T*k routes
    threads = min(oracle.threads(), T * k)
    tokens = layer_steps / L
    return tokens * T / t_spent, tokens, t_spent, threads


def run_reference(args, w):
    """The oracle as the reference arm: same metric and unit, host cores."""
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02)
    hid, lg = decode_inputs(w, max(2, min(args.steps, 64)))
    rate, n, t, threads = oracle_decode_rate(w, pool, hid, lg, args.ref_budget_s, min_tokens=max(1, min(args.steps, 2)),
                                              max_tokens=max(1, args.steps))
    sample = f"{n:.2f} decode tokens x {w['L']} layers from a cold cache ({t:.1f} s of oracle work)"
    return {
        "impl": "reference", "metric": METRIC, "value": round(rate, 5), "unit": "tok/s", "n_gpus": 1, "steps": n,
        "warmup": 0, "ms_per_step": round(t / max(1, n) * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": {"workload": w["desc"]},
        "cpu_baseline": {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(rate, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------- sweeps (report mode)

def run_sweep(args, w, world, local):
    """One JSON line per point.  capacity: the decode step at S = 5, 10, 25 and
    50 % of the pool's experts (the synthetic counterpart of the article's
    miss rate versus cache capacity, Figure 4b); prompt: the prefill chunk at
    4096, 8192 and 16384 tokens with and without the double buffer (Figure 4a)."""
    hp, pool, _ = make_host_pool(args, w)
    try:
        if args.sweep == "capacity":
            e_tot = w["L"] * w["E"]
            hid, lg = decode_inputs(w, args.warmup + args.steps + min(args.steps, args.profile_steps)
                                    + min(args.steps, args.e2e_steps))
            for pct in (5, 10, 25, 50):
                ws = dict(w, S=max(w["k"] * w["T"], e_tot * pct // 100))
                dec = run_decode_leg(args, ws, world, local, pool, hid, lg)
                routes = dec["hits"] + dec["misses"]
                print(json.dumps({
                    "sweep": "capacity", "workload": w["desc"].split(":")[0], "slots": ws["S"],
                    "capacity_pct": pct, "tok_s": round(dec["value"], 3),
                    "expert_miss_rate": round(dec["misses"] / max(1.0, routes), 4),
                    "fills_per_token": round(dec["fills"] / (dec["K"] * dec["T"]), 3),
                    "timed_tokens": dec["K"], "warmup_tokens": dec["W"], "device_status": dec["status"]}), flush=True)
        else:
            w = dict(w, dtype=0)
            for tokens in (4096, 8192, 16384):
                args.prefill_tokens = tokens
                pre = run_prefill_leg(args, w, pool)
                print(json.dumps({
                    "sweep": "prompt", "tokens": tokens, "chunk_s": round(pre["chunk_s"], 4),
                    "chunk_s_single_buffer": round(pre["chunk_s_single_buffer"], 4),
                    "tok_s": round(tokens / pre["chunk_s"], 1), "link_gbs": round(pre["link_gbs"], 1),
                    "gemm_tflops": round(pre["gemm_tflops"], 1), "device_status": pre["status"]}), flush=True)
    finally:
        if hp:
            del pool
            hp.free()


# ----------------------------------------------------------------------------- main

def make_host_pool(args, w):
    """The expert pool, written in the canonical layout.  "pinned": into
    ft_host_alloc memory (mapped in the GPU page tables before the write);
    "registered": into pageable memory that ft_moe_init pins after the write.
    Returns (HostPool or None, uint8 array, seconds to allocate and write)."""
    import expert_cache_host_gb300 as ft
    t0 = time.time()
    n = w["L"] * w["E"] * ftsynth.expert_bytes(w["d"], w["f"], w["dtype"])
    hp = ft.HostPool(n) if args.pool == "pinned" else None
    pool = ftsynth.make_pool(0, w["L"], w["E"], w["d"], w["f"], w["dtype"], 0.02, out=hp.array if hp else None)
    return hp, pool, time.time() - t0


def metric_name(args, w):
    m = METRIC.replace("batch 1", f"batch {w['T']}") if w["dtype"] == 0 else \
        METRIC.replace("A3B-style, batch 1", f"V4-Flash-style MXFP4, batch {w['T']}")
    if args.cpu_exec:
        m = m.replace("GPU side; CPU-routed experts arrive as a partial sum", "GPU + CPU expert executor")
    return m


def build_line(args, w, world, dec, link_gbs, pre, ctl, peaks):
    ex_gbs = dec["ex_bytes"] / (dec["ex_ms"] / 1e3) / 1e9 if dec["ex_ms"] else 0.0
    fill_gbs = dec["fill_bytes"] / (dec["fill_ms"] / 1e3) / 1e9 if dec["fill_ms"] else 0.0
    bx = ftsynth.expert_bytes(w["d"], w["f"], w["dtype"])
    line = {
        "metric": metric_name(args, w),
        "value": round(dec["value"], 3), "unit": "tok/s", "n_gpus": world, "steps": dec["K"],
        "warmup": dec["W"], "ms_per_step": round(dec["elapsed"] / dec["K"] * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if w["dtype"] == 0 else "e2m1*e8m0 x bf16 -> f16/f32",
        "data": "synthetic",
        "config": {"workload": w["desc"], "graph": "one CUDA graph per token", "batch": dec["T"],
                   "l2": "inputs larger than L2: %.2f GB of expert weights per token" % (w["L"] * w["k"] * bx / 1e9),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        # the dominant kernel by time is the fill: host-link bound
        "roofline": {"bound": "host_link", "kernel": "decode fill (host pool -> slots)", "achieved": round(fill_gbs, 1),
                     "peak": round(link_gbs, 1), "unit": "GB/s", "frac": round(fill_gbs / link_gbs, 4) if link_gbs else None,
                     "traffic": None, "peak_source": "measured in this run: 1.21 GB pinned H2D cudaMemcpyAsync, best of 3",
                     "share": dec["shares"].get("fill")},
        "roofline_experts": {"bound": "hbm", "kernel": "decode experts", "achieved": round(ex_gbs, 1),
                             "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(ex_gbs / peaks["hbm_gbs"], 4),
                             "traffic": round(NCU_TRAFFIC_RATIO["decode_experts" if w["dtype"] == 0 else "decode_experts_mxfp4"]
                                              * dec["ex_bytes"] / max(1, dec["ex_n"])),
                             "traffic_source": "ncu ratio x algorithmic bytes per launch", "peak_source": peaks["source"],
                             "bytes_per_launch": round(dec["ex_bytes"] / max(1, dec["ex_n"])),
                             "avg_launch_us": round(dec["ex_ms"] / max(1, dec["ex_n"]) * 1e3, 2),
                             "share": dec["shares"].get("experts")},
        "components": {
            "kernel_share": dec["shares"],
            "kernel_ms_per_token": {n: round(v / dec["T"], 4) for n, v in dec["ms_per_token"].items()},
            "route_control_us_per_layer_step": round(dec["control_us"], 3),
            "hit_rate": round(dec["hits"] / max(1.0, dec["hits"] + dec["misses"]), 4),
            "fills_per_token": round(dec["fills"] / (dec["K"] * dec["T"]), 3),
            "cpu_routes_per_token": round(dec["cpu"] / (dec["K"] * dec["T"]), 3),
            "fills_per_step": round(dec["fills"] / dec["K"], 3), "tokens_per_step": dec["T"],
            "eager_ms_per_token_profiled": round(dec["eager_ms"] / dec["T"], 4) if dec["eager_ms"] else None,
            "init_pin_s": round(dec["t_init"], 2), "device_status": dec["status"],
        },
        "clocks": dec["clocks"],
        "e2e": {"value": round(dec["e2e"], 3), "unit": "tok/s", "h2d_bytes_per_step": dec["h2d"],
                "d2h_bytes_per_step": dec["d2h"]},
        # per layer: route + control (one kernel), fill, resident experts, installed experts, merge
        "gpu_launches": int(dec["K"] * w["L"] * 5),
    }
    if pre:
        line["prefill"] = {
            "workload": f"{pre['T']}-token chunk, A3B-style, {pre['L']} layers, full-layer double buffer",
            "chunk_s": round(pre["chunk_s"], 4), "chunk_s_single_buffer": round(pre["chunk_s_single_buffer"], 4),
            "loss_without_double_buffer": round(pre["overlap_loss_without_double_buffer"], 4),
            "tok_s": round(pre["T"] / pre["chunk_s"], 1), "pool_gb": round(pre["pool_bytes"] / 1e9, 2),
            "link_gbs_effective": round(pre["link_gbs"], 1), "upload_gbs": round(pre["upload_gbs"], 1),
            "link_frac": round(pre["link_gbs"] / link_gbs, 4) if link_gbs else None,
            "device_status": pre["status"],
            "roofline_gemm": {"bound": "tensor", "kernel": "grouped SwiGLU GEMMs (tcgen05), weights resident",
                              "achieved": round(pre["gemm_tflops"], 1), "peak": peaks["bf16_tflops"],
                              "unit": "TFLOP/s", "frac": round(pre["gemm_tflops"] / peaks["bf16_tflops"], 4),
                              "ms_per_layer": round(pre["gemm_ms_per_layer"], 3), "traffic": None,
                              "peak_source": peaks["source"] + " (burst bf16)"},
        }
    if ctl:
        line["control_stress"] = {
            "workload": "control kernel alone, 48 layers x 64 tokens x top-8, E=128, Zipf routes, graph replay",
            "steps": args.control_steps, "cases": ctl,
        }
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=448)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--profile-steps", type=int, default=32)
    ap.add_argument("--e2e-steps", type=int, default=128)
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-budget-s", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-control", action="store_true")
    ap.add_argument("--prefill-tokens", type=int, default=8192)
    ap.add_argument("--prefill-layers", type=int, default=0)
    ap.add_argument("--control-steps", type=int, default=10000)
    ap.add_argument("--prefill-only", action="store_true", help="profiling case: the prefill leg alone")
    ap.add_argument("--workload", choices=("a3b", "v4"), default="a3b",
                    help="a3b: bf16 A3B-style decode (default line); v4: MXFP4 V4-Flash-style decode")
    ap.add_argument("--batch", type=int, default=0, help="decode tokens per step (default 1)")
    ap.add_argument("--layers", type=int, default=0, help="override L (small profiling cases, not a bench line)")
    ap.add_argument("--slots", type=int, default=0, help="override S (small profiling cases, not a bench line)")
    ap.add_argument("--sweep", choices=("capacity", "prompt"), default=None,
                    help="report mode (not the bench line): decode miss rate and tok/s over cache capacities of "
                         "5/10/25/50%% of the pool, or prefill chunk time over prompt lengths 4k/8k/16k with and "
                         "without the double buffer")
    ap.add_argument("--ratio", default=None, help="r = BP/BH as NUM/DEN for the decode workload (default 1/1: every "
                    "miss filled)")
    ap.add_argument("--cpu-exec", type=int, default=0, help="variant: the context's CPU expert executor with this many "
                    "host threads computes the misses that are not filled (not the bench line)")
    ap.add_argument("--pool", choices=("pinned", "registered"), default="pinned",
                    help="pinned: pool written into ft_host_alloc memory; registered: pageable pool pinned by "
                         "ft_moe_init after the write")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_env()
    w = dict(A3B if args.workload == "a3b" else V4)
    if args.batch:
        w["T"] = args.batch
        w["desc"] = w["desc"].replace("batch 1, ", "") + f", batch {args.batch}"
    if args.workload == "v4":
        # keep the per-layer shapes; drop layers only if the host cannot hold the pinned pool
        avail = 0
        with open("/proc/meminfo") as fh:
            for line in fh:
                if line.startswith("MemAvailable:"):
                    avail = int(line.split()[1]) * 1024
        per_layer = w["E"] * ftsynth.expert_bytes(w["d"], w["f"], 1)
        fit = int(max(0, avail - (24 << 30)) // per_layer)
        if fit < w["L"]:
            w["L"] = max(1, fit)
            w["desc"] += f" [host RAM holds {w['L']} of the 43 layers]"
        args.no_prefill = args.no_control = True
    if args.ratio:
        num, den = (int(x) for x in args.ratio.split("/"))
        w["r"] = (num, den)
        w["desc"] = w["desc"].replace("BP/BH=1", f"BP/BH={num}/{den}")
    if args.cpu_exec:
        w["desc"] += f", CPU executor with {args.cpu_exec} host threads for the unfilled misses"
    if args.layers or args.slots:
        w["L"], w["S"] = args.layers or w["L"], args.slots or w["S"]
        w["desc"] += f" [profiling case: L={w['L']}, S={w['S']}]"

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

    import torch

    from expert_cache_host_gb300 import build as ftbuild
    ftbuild.build()
    torch.cuda.set_device(local)
    if args.prefill_only:
        # profiling case: the prefill leg alone on the first --prefill-layers layers (not a bench line)
        w["L"] = args.prefill_layers or w["L"]
        w["dtype"] = 0
        hp, pool, _ = make_host_pool(args, w)
        print(json.dumps({"profiling_case": "prefill", **run_prefill_leg(args, w, pool)}), flush=True)
        if hp:
            del pool
            hp.free()
        return
    if args.sweep:
        run_sweep(args, w, world, local)
        return
    hp, pool, t_pool = make_host_pool(args, w)
    hid, lg = decode_inputs(w, args.warmup + args.steps + min(args.steps, args.profile_steps)
                            + min(args.steps, args.e2e_steps))
    dec = run_decode_leg(args, w, world, local, pool, hid, lg)
    pre = ctl = alone = None
    link = 0.0
    if rank == 0:
        import expert_cache_host_gb300 as ft
        # the pool is registered (pinned, mapped) for the measurement below by a throwaway context
        cfg = ft.make_config(num_layers=w["L"], num_experts=w["E"], top_k=w["k"], hidden=w["d"], inter=w["f"],
                             dtype=w["dtype"], num_slots=1, k_max=1, t_max=1)
        ctx = ft.ft_moe_init(cfg, pool.ctypes.data, pool.nbytes)
        try:
            link = link_peak_gbs(pool, w["E"] * ftsynth.expert_bytes(w["d"], w["f"], w["dtype"]))
        finally:
            ft.ft_moe_destroy(ctx)
        if w["dtype"] == 0:
            alone = experts_alone(w, pool, hid)
        if not args.no_prefill and not args.layers:
            pre = run_prefill_leg(args, w, pool)
        if not args.no_control and not args.layers:
            ctl = run_control_leg(args)
    peaks = measured_peaks()
    if rank == 0:
        line = build_line(args, w, world, dec, link, pre, ctl, peaks)
        if alone:
            bx = ftsynth.expert_bytes(w["d"], w["f"], 0)
            t8 = alone[w["k"]]
            line["roofline_experts_alone"] = {
                "bound": "hbm", "kernel": f"decode experts + merge outside the step ({w['k']} resident experts, "
                                          "batch 1, L2 flushed; allocation-free entry: route grouping, experts, merge)",
                "achieved": round(w["k"] * bx / t8 / 1e9, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(w["k"] * bx / t8 / 1e9 / peaks["hbm_gbs"], 4), "us": round(t8 * 1e6, 2),
                "us_2_experts": round(alone[2] * 1e6, 2), "peak_source": peaks["source"]}
        if not args.no_cpu_baseline:
            rate, n, t, threads = oracle_decode_rate(w, pool, hid, lg, args.cpu_budget_s,
                                                     min_tokens=1.0 if w["T"] == 1 else 1.0 / w["L"])
            line["cpu_baseline"] = {"value": round(rate, 5), "unit": "tok/s", "cores": threads, "kind": "oracle",
                                    "sample": f"{n:.2f} decode tokens x {w['L']} layers from a cold cache, "
                                              f"{t:.1f} s of oracle work"}
        line["config"]["pool"] = (f"{args.pool}: {pool.nbytes / 1e9:.2f} GB, allocated and written in {t_pool:.1f} s")
        print(json.dumps(line), flush=True)
    if hp:
        del pool
        hp.free()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
